"""The per-segment state split of the bf16 path, checked on the CPU (no GPU).

The tensor-core kernel carries one state per unit through whole chunks. To hand
each segment its own initial state and return its final state, the bf16 path:
- seeds the carried state, at the chunk where a segment starts and carries on,
  with that segment's initial state decayed to the chunk's end;
- keeps the state carried into the chunk where a segment ends;
- then, per chunk, rewrites the rows of each segment in the chunk where it
  starts, and forms final states from the kept states and the chunk's own
  tokens.
`tests/chunked_mirror.chunked_forward_state` restates those steps in float64,
with the kernels' decisions: which chunks seed, which export, and which
segments the state pass takes. Here that restatement must reproduce the
oracle's token recurrence to rounding error on layouts that exercise every
case:
- segments starting and ending inside one chunk, at chunk edges, and across
  many chunks;
- padding inside and at the end of chunks;
- ragged T and several rows;
- slots for only some of the segments.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.chunked_mirror import chunked_forward_state


def _inputs(rng, N, H, D):
    q = rng.standard_normal((N, H, D)) / np.sqrt(D)
    k = rng.standard_normal((N, H, D)) / np.sqrt(D)
    v = rng.standard_normal((N, H, D))
    g = -np.exp(rng.normal(-2.0, 0.5, (N, H, D)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((N, H))))
    return q, k, v, g, beta


def _layouts():
    rng = np.random.default_rng(5)
    out = []
    # long documents crossing chunk edges, one ending exactly on an edge
    out.append(("long", 1, 320, np.array([[1] * 150 + [2] * 42 + [3] * 128], dtype=np.int32)))
    # documents aligned to chunk edges, then a padded tail
    out.append(("aligned", 1, 256, np.array([[1] * 64 + [2] * 128 + [0] * 64], dtype=np.int32)))
    # many short documents per chunk, padding inside chunks, ragged T, two rows
    seg = np.zeros((2, 150), dtype=np.int32)
    for b in range(2):
        t, sid = 0, 1
        while t < 150:
            n = int(rng.integers(1, 20))
            if rng.random() < 0.15:
                t += n                              # padding run
                continue
            seg[b, t:t + n] = sid
            sid += 1
            t += n
    out.append(("short", 2, 150, seg))
    # length-1 documents on both sides of every chunk edge, and a document ending on row 63
    s = [1] * 63 + [2] + [3] + [4] * 62 + [5] + [6] * 65
    out.append(("edges", 1, len(s), np.array([s], dtype=np.int32)))
    return out


@pytest.mark.parametrize("name,B,T,seg", _layouts(), ids=lambda x: x if isinstance(x, str) else "")
@pytest.mark.parametrize("mode", ["init+final", "init", "final", "half-slots"])
def test_split_reproduces_oracle(name, B, T, seg, mode):
    rng = np.random.default_rng(len(name) * 7 + len(mode))
    H, D = 2, 4
    q, k, v, g, beta = _inputs(rng, B * T, H, D)
    starts = (seg != 0) & ((np.arange(T)[None, :] == 0) |
                           (seg != np.concatenate([np.zeros((B, 1), seg.dtype), seg[:, :-1]], 1)))
    n = int(starts.sum())
    n_state = max(1, n // 2) if mode == "half-slots" else n
    init = rng.standard_normal((n_state, H, D, D)) * 0.5 if mode != "final" else None
    want = mode != "init"
    ref_o, ref_f = oracle.kda_fwd_state(q, k, v, g, beta, seg, B, T, initial_state=init,
                                        n_state=n_state, want_final=want, scale=0.7)
    o, f = chunked_forward_state(q, k, v, g, beta, seg, B, T, init=init, n_state=n_state,
                                 want_final=want, scale=0.7)
    assert torch.allclose(o, ref_o.to(torch.float64), rtol=1e-10, atol=1e-12), name
    if want:
        assert torch.allclose(f, ref_f.to(torch.float64), rtol=1e-10, atol=1e-12), name
