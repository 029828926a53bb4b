"""Pins for the oracle's per-segment state (no GPU).

[RFC-0026] passes `initial_state` and `output_final_state` to the chunked KDA
call: each packed sequence (segment) may start from a given state instead of
zero, and the state after its last token can be returned. The oracle takes
both per segment, indexed by the segment's rank in flattened token order (the
order of cu_seqlens). These tests pin that against:
- the plain path (zero initial state, no state written);
- brute-force closed forms of the final state and of the outputs under an
  initial state, summed term by term;
- the chaining identity: a document cut in two, with the first part's final
  state handed to the second part, gives the uncut document's outputs and
  final state.
"""
import numpy as np
import torch

import oracle


def _inputs(rng, N, H, Dk, Dv):
    q = rng.standard_normal((N, H, Dk)) / np.sqrt(Dk)
    k = rng.standard_normal((N, H, Dk)) / np.sqrt(Dk)
    v = rng.standard_normal((N, H, Dv))
    g = -np.exp(rng.normal(-2.0, 0.5, (N, H, Dk)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((N, H))))
    return q, k, v, g, beta


def _segments(seg):
    """(row, first, one-past-last) of every segment in flattened order."""
    out = []
    B, T = seg.shape
    for b in range(B):
        t = 0
        while t < T:
            s = seg[b, t]
            if s == 0:
                t += 1
                continue
            e = t + 1
            while e < T and seg[b, e] == s:
                e += 1
            out.append((b, t, e))
            t = e
    return out


def test_zero_initial_state_equals_plain_path():
    rng = np.random.default_rng(1)
    B, T, H, D = 2, 23, 2, 4
    q, k, v, g, beta = _inputs(rng, B * T, H, D, D)
    seg = np.array([[1] * 9 + [2] * 7 + [0] * 2 + [3] * 5, [5] * 11 + [6] * 12], dtype=np.int32)
    o_plain = oracle.kda_fwd(q, k, v, g, beta, seg)
    n = len(_segments(seg))
    o0, fin = oracle.kda_fwd_state(q, k, v, g, beta, seg, initial_state=np.zeros((n, H, D, D)),
                                   n_state=n, want_final=True)
    assert torch.equal(o0, o_plain)
    o1, none = oracle.kda_fwd_state(q, k, v, g, beta, seg)
    assert torch.equal(o1, o_plain) and none is None
    assert fin.shape == (n, H, D, D) and torch.isfinite(fin).all()


def test_closed_forms_bruteforce():
    """S_final = (prod of e over the segment) * S0 + sum_j (prod of e after j) * beta_j k_j v_j^T
    and o_t = scale * q_t^T [(prod of e up to t) * S0 + sum_{j<=t} (prod of e over j<u<=t) * beta_j k_j v_j^T],
    with the products taken elementwise per key channel, summed term by term."""
    rng = np.random.default_rng(2)
    B, T, H, Dk, Dv = 1, 13, 2, 3, 2
    q, k, v, g, beta = _inputs(rng, B * T, H, Dk, Dv)
    seg = np.array([[4] * 5 + [0] + [7] * 7], dtype=np.int32)
    segs = _segments(seg)
    S0 = rng.standard_normal((len(segs), H, Dk, Dv))
    scale = 0.7
    o, fin = oracle.kda_fwd_state(q, k, v, g, beta, seg, scale=scale, initial_state=S0,
                                  n_state=len(segs), want_final=True)
    o, fin = o.numpy(), fin.numpy()
    e = np.exp(g)
    for r, (b, t0, t1) in enumerate(segs):
        for h in range(H):
            for t in range(t0, t1):
                St = np.prod(e[t0:t + 1, h], axis=0)[:, None] * S0[r, h]
                for j in range(t0, t + 1):
                    dec = np.prod(e[j + 1:t + 1, h], axis=0) if j < t else np.ones(Dk)
                    St = St + dec[:, None] * beta[j, h] * np.outer(k[j, h], v[j, h])
                np.testing.assert_allclose(o[t, h], scale * St.T @ q[t, h], rtol=1e-12, atol=1e-12)
            SF = np.prod(e[t0:t1, h], axis=0)[:, None] * S0[r, h]
            for j in range(t0, t1):
                SF = SF + np.prod(e[j + 1:t1, h], axis=0)[:, None] * beta[j, h] * np.outer(k[j, h], v[j, h])
            np.testing.assert_allclose(fin[r, h], SF, rtol=1e-12, atol=1e-12)
    assert np.all(o[5] == 0.0)                        # padding


def test_chaining_identity():
    """Cutting a document at m and handing part A's final state to part B is the uncut run."""
    rng = np.random.default_rng(3)
    T, H, D, m = 40, 2, 5, 17
    q, k, v, g, beta = _inputs(rng, T, H, D, D)
    S0 = rng.standard_normal((1, H, D, D))
    whole = np.ones((1, T), dtype=np.int32)
    o_w, f_w = oracle.kda_fwd_state(q, k, v, g, beta, whole, initial_state=S0, n_state=1,
                                    want_final=True)
    cut = np.array([[1] * m + [2] * (T - m)], dtype=np.int32)
    # part A alone gives the state at the cut; part B (rank 1) starts from it
    _, f_a = oracle.kda_fwd_state(q, k, v, g, beta, cut, initial_state=np.concatenate([S0, S0]),
                                  n_state=2, want_final=True)
    init = np.stack([S0[0], f_a[0].numpy()])
    o_c, f_c = oracle.kda_fwd_state(q, k, v, g, beta, cut, initial_state=init, n_state=2,
                                    want_final=True)
    np.testing.assert_allclose(o_c.numpy(), o_w.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(f_c[1].numpy(), f_w[0].numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(f_c[0].numpy(), f_a[0].numpy(), rtol=0, atol=0)


def test_state_slots_beyond_n_state_and_ranks():
    """Segments at rank >= n_state start from zero; ranks follow flattened order
    (rows first), padding is no segment, and segment_ids=None makes each row one."""
    rng = np.random.default_rng(4)
    B, T, H, D = 2, 9, 1, 3
    q, k, v, g, beta = _inputs(rng, B * T, H, D, D)
    seg = np.array([[2, 2, 0, 3, 3, 3, 2, 2, 2], [2, 2, 2, 2, 1, 1, 1, 1, 1]], dtype=np.int32)
    segs = _segments(seg)
    assert [s[1:] for s in segs] == [(0, 2), (3, 6), (6, 9), (0, 4), (4, 9)]
    S0 = rng.standard_normal((2, H, D, D))
    o, fin = oracle.kda_fwd_state(q, k, v, g, beta, seg, initial_state=S0, n_state=2,
                                  want_final=True)
    o_plain = oracle.kda_fwd(q, k, v, g, beta, seg)
    # ranks 0 and 1 (row 0, tokens 0-1 and 3-5) differ from the zero-state run, the rest agree
    diff = (o - o_plain).abs().amax(dim=(1, 2)).numpy()
    assert np.all(diff[[0, 1, 3, 4, 5]] > 0) and np.all(diff[[2, 6, 7, 8]] == 0)
    assert np.all(diff[9:] == 0)
    # each row one segment: rank = row
    S1 = rng.standard_normal((B, H, D, D))
    o_n, f_n = oracle.kda_fwd_state(q, k, v, g, beta, None, B=B, T=T, initial_state=S1,
                                    n_state=B, want_final=True)
    ones = np.ones((B, T), dtype=np.int32)
    o_1, f_1 = oracle.kda_fwd_state(q, k, v, g, beta, ones, initial_state=S1, n_state=B,
                                    want_final=True)
    assert torch.equal(o_n, o_1) and torch.equal(f_n, f_1)
