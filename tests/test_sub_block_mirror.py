"""The tensor-core kernel's chunk algebra, unit by unit, in both of its forms, checked
on the CPU against the oracle (no GPU).

`tests/chunked_mirror.chunked_forward_units` restates in float64 what the kernel
computes: the plan's units (each from a zero state; the rows of a unit's first
chunk before its cut belong to the previous unit), and per chunk either the
whole-chunk factorisation (Qt = q exp(-Suf), Ktb = beta k exp(Suf), Suf summed to
the chunk's end) or, for strongly decaying chunks, the sub-block form (Suf summed
to the end of each 16-row sub-block, A' kept on the diagonal blocks, and the
state read out and updated once per sub-block with that sub-block's masks). In
float64 both forms are exact, so each must reproduce the oracle's token
recurrence to rounding error on every layout, cut set and decay strength. A
slip in a sub-block mask (which rows read the incoming state, which rows feed
the state, whether the state carries through) fails here.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.chunked_mirror import chunked_forward_units


def _inputs(rng, N, H, D, strong_channels=0, strong_g=-3.0):
    q = rng.standard_normal((N, H, D)) / np.sqrt(D)
    k = rng.standard_normal((N, H, D)) / np.sqrt(D)
    v = rng.standard_normal((N, H, D))
    g = -np.exp(rng.normal(-2.0, 0.5, (N, H, D)))
    if strong_channels:
        ch = rng.choice(D, size=strong_channels, replace=False)
        g[:, :, ch] = strong_g * (0.5 + rng.random((N, H, strong_channels)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((N, H))))
    return q, k, v, g, beta


def _layouts():
    rng = np.random.default_rng(17)
    out = []
    for (B, T, max_len, pad) in [(1, 64 * 4 + 9, 200, 0.0), (2, 150, 40, 0.15), (1, 256, 7, 0.1),
                                 (3, 100, 90, 0.2), (1, 320, 1, 0.0)]:
        out.append(synth.random_segment_ids(rng, B, T, max_len=max_len, pad_prob=pad))
    seg = np.ones((2, 200), np.int32)           # boundaries on sub-block and chunk edges
    seg[0, 16:] = 2
    seg[0, 63:] = 3
    seg[0, 64 + 31:] = 4
    seg[1, 47:60] = 0
    seg[1, 60:] = 5
    out.append(seg)
    return out


@pytest.mark.parametrize("mode", ["never", "always", "auto"])
@pytest.mark.parametrize("strong", [0, 3])
def test_units_and_forms_match_the_oracle(mode, strong):
    rng = np.random.default_rng(100 + strong)
    for li, seg in enumerate(_layouts()):
        B, T = seg.shape
        N, H, D = B * T, 2, 16
        q, k, v, g, beta = _inputs(rng, N, H, D, strong_channels=strong)
        ref = oracle.kda_fwd(*(torch.from_numpy(x) for x in (q, k, v, g, beta)),
                             torch.from_numpy(seg), B, T, scale=0.7).numpy()
        cut_sets = [None]
        # a random subset of the candidate chunks as cuts (longer units, more carried state)
        n_chunks = (N + 63) // 64
        cand = [c for c in range(n_chunks)
                if (seg.reshape(-1)[c * 64:(c + 1) * 64] == 0).any()
                or any(p % T == 0 or seg.reshape(-1)[p] != seg.reshape(-1)[p - 1]
                       for p in range(c * 64, min((c + 1) * 64, N)) if seg.reshape(-1)[p] != 0)]
        if len(cand) > 2:
            cut_sets.append(sorted(rng.choice(cand, size=max(1, len(cand) // 2), replace=False)))
        for cuts in cut_sets:
            o, n_sub = chunked_forward_units(q, k, v, g, beta, seg, B, T, scale=0.7, cuts=cuts,
                                             mode=mode)
            o = o.numpy()
            rms = np.sqrt((ref ** 2).mean())
            assert np.abs(o - ref).max() <= 1e-10 * max(rms, 1e-300), \
                f"layout {li} cuts {cuts}: {np.abs(o - ref).max():.3e}"
            if mode == "auto":
                assert (n_sub > 0) == (strong > 0)


def test_planted_sub_block_mask_mistakes_are_caught():
    """Two plausible slips in the sub-block form, planted in a copy of the mirror's step:
    the state carried through a sub-block that holds a start, and the A' mask spanning
    all earlier rows instead of the row's own sub-block. Each moves the result off the
    oracle."""
    import tests.chunked_mirror as cm
    src = open(cm.__file__).read()
    rng = np.random.default_rng(3)
    seg = _layouts()[5]
    B, T = seg.shape
    q, k, v, g, beta = _inputs(rng, B * T, 1, 16, strong_channels=2)
    ref = oracle.kda_fwd(*(torch.from_numpy(x) for x in (q, k, v, g, beta)),
                         torch.from_numpy(seg), B, T).numpy()
    mutations = [
        ("if in_b and not cutb.any():", "if in_b:"),
        ("lo = np.maximum(lo, rows // 16 * 16)", "lo = lo"),
    ]
    for old, new in mutations:
        assert old in src
        ns = {}
        exec(compile(src.replace(old, new), "mutant", "exec"), ns)
        o, _ = ns["chunked_forward_units"](q, k, v, g, beta, seg, B, T, mode="always")
        assert np.abs(o.numpy() - ref).max() > 1e-6, f"mutation not caught: {new}"
