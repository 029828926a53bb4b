"""The chunk algebra of the tensor-core backward (tests/chunked_bwd_mirror.py), on the CPU.

It must reproduce the oracle's reverse-mode gradients to float64 rounding on layouts that
reach every case of the algebra: boundaries inside chunks and on their edges, chains over
many chunks, padding inside and at the end, ragged T, arbitrary ids and no ids. Cutting the
scans' long chains into pieces (end states, combine, seeded export) must not change the
result beyond rounding. A planted mistake in the algebra (the carry past the chunk dropped,
the carried state's decay P left out) fails it.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import tests.chunked_bwd_mirror as mirror


def _inputs(B, T, H, D, seed, seg=None, decay=1.0, **kw):
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    if seg is None:
        seg = torch.from_numpy(synth.random_segment_ids(rng, B, T, **kw))
    N = B * T
    q = torch.nn.functional.normalize(torch.randn(N, H, D, generator=gen, dtype=torch.float64), dim=-1)
    k = torch.nn.functional.normalize(torch.randn(N, H, D, generator=gen, dtype=torch.float64), dim=-1)
    v = torch.randn(N, H, D, generator=gen, dtype=torch.float64)
    g = -decay * torch.exp(torch.randn(N, H, D, generator=gen, dtype=torch.float64) * 0.5 - 2.0)
    beta = torch.sigmoid(torch.randn(N, H, generator=gen, dtype=torch.float64))
    do = torch.randn(N, H, D, generator=gen, dtype=torch.float64)
    return q, k, v, g, beta, do, seg


def _close(got, ref, label):
    for name, a, b in zip(("dq", "dk", "dv", "dg", "dbeta"), got, ref):
        b = b.numpy() if isinstance(b, torch.Tensor) else b
        rms = np.sqrt((b ** 2).mean()) + 1e-300
        err = np.abs(a - b).max() / rms
        assert err < 1e-11, f"{label} {name}: {err:.2e} RMS"


LAYOUTS = [
    dict(B=1, T=64 * 5 + 17, max_len=70),
    dict(B=3, T=100, max_len=9, pad_prob=0.25),
    dict(B=2, T=120, max_len=3, ids="arbitrary"),
    dict(B=1, T=64 * 6, max_len=400, pad_prob=0.05),
    dict(B=1, T=130, max_len=1),
]


@pytest.mark.parametrize("lay", range(len(LAYOUTS)))
def test_chunk_algebra_equals_the_oracle(lay):
    c = dict(LAYOUTS[lay])
    B, T = c.pop("B"), c.pop("T")
    q, k, v, g, beta, do, seg = _inputs(B, T, 2, 8, seed=400 + lay, **c)
    got = mirror.chunked_backward(q, k, v, g, beta, do, seg, B, T, scale=0.7)
    ref = oracle.kda_bwd(q, k, v, g, beta, do, seg, B, T, scale=0.7)
    _close(got, ref, f"layout {lay}")


def test_every_boundary_offset_and_no_ids():
    """A boundary at each offset of a chunk between two carried chunks; and one segment per
    row (segment_ids None) across chunks."""
    B, T = 8, 64 * 3
    seg = torch.ones(B, T, dtype=torch.int32)
    for b in range(B):
        seg[b, 64 + 8 * b + 3:] = 2
    q, k, v, g, beta, do, _ = _inputs(B, T, 1, 8, seed=5, seg=seg)
    _close(mirror.chunked_backward(q, k, v, g, beta, do, seg, B, T, scale=0.9),
           oracle.kda_bwd(q, k, v, g, beta, do, seg, B, T, scale=0.9), "offsets")
    x = [t[:192] for t in (q, k, v, g, beta, do)]
    _close(mirror.chunked_backward(*x, None, 2, 96), oracle.kda_bwd(*x, None, 2, 96), "no ids")


def test_scans_in_pieces_change_nothing():
    """Chains cut into pieces of 3 chunks (when longer than 4): S_in and D_end are written for
    the same chunks and agree to rounding with the uncut scans; so do the gradients."""
    B, T = 2, 64 * 11 + 5
    q, k, v, g, beta, do, seg = _inputs(B, T, 1, 8, seed=9, max_len=64 * 9, pad_prob=0.02)
    N = B * T
    n, start, valid, fc = mirror.chunk_layout(seg, N, T)
    assert max(cb - ca for ca, cb in mirror._chains(n, fc)) >= 7     # three pieces or more
    pad = n * 64 - N
    ext = [np.concatenate([mirror._np(x), np.zeros((pad,) + x.shape[1:])]) for x in (q, k, v, g, do)]
    be = np.concatenate([mirror._np(beta), np.zeros((pad, 1))])
    s0, d0 = mirror.scans(ext[0], ext[1], ext[2], ext[3], be, ext[4], n, start, valid, fc, 0, 0.6)
    s1, d1 = mirror.scans(ext[0], ext[1], ext[2], ext[3], be, ext[4], n, start, valid, fc, 0, 0.6,
                          piece=3, split_min=4)
    assert (np.isnan(s0) == np.isnan(s1)).all() and (np.isnan(d0) == np.isnan(d1)).all()
    assert np.nanmax(np.abs(s0 - s1)) < 1e-12 and np.nanmax(np.abs(d0 - d1)) < 1e-12
    got = mirror.chunked_backward(q, k, v, g, beta, do, seg, B, T, scale=0.6, piece=3, split_min=4)
    _close(got, oracle.kda_bwd(q, k, v, g, beta, do, seg, B, T, scale=0.6), "pieces")


def test_planted_mistakes_fail():
    """The carry past the chunk and the carried state's decay P are each needed: the mirror
    with either one taken out misses the oracle by far more than rounding."""
    B, T = 1, 64 * 4
    # weak decay, so that a state carried over a whole chunk still matters
    q, k, v, g, beta, do, seg = _inputs(B, T, 1, 8, seed=13, max_len=200, decay=0.02)
    ref = oracle.kda_bwd(q, k, v, g, beta, do, seg, B, T)
    src = open(mirror.__file__).read()
    for bad, planted in (("carry += P * (S0 * DE).sum(1)", "carry += 0.0 * (S0 * DE).sum(1)"),
                         ("(P[:, None] * S0).T", "S0.T")):
        assert src.count(bad) == 1
        ns = {}
        exec(compile(src.replace(bad, planted), mirror.__file__, "exec"), ns)
        got = ns["chunked_backward"](q, k, v, g, beta, do, seg, B, T)
        errs = [np.abs(a - b.numpy()).max() / np.sqrt((b.numpy() ** 2).mean())
                for a, b in zip(got, ref)]
        assert max(errs) > 1e-3, f"planted mistake not caught: {planted}"
