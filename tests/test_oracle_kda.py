"""Pins for the oracle's token-by-token KDA recurrence (no GPU).

The recurrence is RFC-0026 "Ling3 KDA Varlen 支持", 背景 "KDA 状态泄漏问题"
(S'_t = S_{t-1} exp(g_t), S_t = S'_t + beta_t k_t v_t^T), read out as
o_t = scale * S_t^T q_t, with the reset rule of §3.1.1 (zero S where the id
changes and at t = 0 of each row; id 0 is padding).

Pins, each chosen so that a plausible slip in the oracle fails one of them:
  * the unrolled closed form o_t = scale * sum_{j<=t, same segment}
    beta_j v_j sum_c q_tc k_jc exp(G_tc - G_jc) (G = inclusive prefix sum of g),
    computed by brute force;  [catches a wrong decay index/sign or order]
  * g = 0 reduces to causal linear attention, a textbook matrix formula;
  * length-1 documents: o_t = scale * beta_t (q_t . k_t) v_t;
  * Dk = Dv = 1 with constant decay is a first-order IIR filter
    (scipy.signal.lfilter);  [catches decay applied after the update]
  * gate injection (RFC-0026 备选方案 "Gate 注入法"): one continuous segment
    with g = -inf at every document start gives the packed result;
  * isolation (测试方案 test_packed_equivalence_with_per_doc): packed output
    equals each document run alone;
  * segment_ids=None equals all-ones ids (test_segment_ids_none_fallback);
  * row independence (test_row_independence_under_vmap), scale linearity,
    padding output exactly zero;
  * a hand-worked 3-token example.
"""
import math

import numpy as np
import pytest
import scipy.signal
import torch

import oracle
import synth

f64 = torch.float64


def _rand_inputs(N, H, Dk, Dv, gen, g_scale=0.3):
    q = torch.randn(N, H, Dk, generator=gen, dtype=f64)
    k = torch.randn(N, H, Dk, generator=gen, dtype=f64)
    v = torch.randn(N, H, Dv, generator=gen, dtype=f64)
    g = -g_scale * torch.rand(N, H, Dk, generator=gen, dtype=f64)
    beta = torch.rand(N, H, generator=gen, dtype=f64)
    return q, k, v, g, beta


def _segments(seg_row):
    """Maximal runs of equal non-zero ids in one row: list of (start, end)."""
    out, t, T = [], 0, len(seg_row)
    while t < T:
        if seg_row[t] == 0:
            t += 1
            continue
        e = t + 1
        while e < T and seg_row[e] == seg_row[t]:
            e += 1
        out.append((t, e))
        t = e
    return out


def _closed_form(q, k, v, g, beta, seg, B, T, scale):
    N, H, Dk = q.shape
    Dv = v.shape[-1]
    o = torch.zeros(N, H, Dv, dtype=f64)
    for b in range(B):
        for (s, e) in _segments(seg[b].tolist()):
            for h in range(H):
                for t in range(s, e):
                    pt = b * T + t
                    acc = torch.zeros(Dv, dtype=f64)
                    for j in range(s, t + 1):
                        pj = b * T + j
                        # G_t - G_j = sum of g over tokens j+1 .. t
                        dG = g[b * T + j + 1: pt + 1, h].sum(0) if t > j else torch.zeros(Dk, dtype=f64)
                        w = (q[pt, h] * k[pj, h] * torch.exp(dG)).sum()
                        acc += beta[pj, h] * w * v[pj, h]
                    o[pt, h] = scale * acc
    return o


def test_closed_form_bruteforce():
    gen = torch.Generator().manual_seed(1)
    B, T, H, Dk, Dv = 2, 23, 2, 5, 3
    seg = torch.from_numpy(synth.random_segment_ids(np.random.default_rng(1), B, T,
                                                    max_len=9, pad_prob=0.15))
    q, k, v, g, beta = _rand_inputs(B * T, H, Dk, Dv, gen)
    o = oracle.kda_fwd(q, k, v, g, beta, seg, B, T, scale=0.7, n_threads=3)
    ref = _closed_form(q, k, v, g, beta, seg, B, T, 0.7)
    assert torch.allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_hand_worked_three_tokens():
    # H = 1, Dk = 2, Dv = 1, one segment of 3 tokens.
    q = torch.tensor([[[1.0, 0.0]], [[0.0, 1.0]], [[1.0, 1.0]]], dtype=f64)
    k = torch.tensor([[[1.0, 0.0]], [[0.0, 2.0]], [[1.0, 0.0]]], dtype=f64)
    v = torch.tensor([[[3.0]], [[5.0]], [[7.0]]], dtype=f64)
    g = torch.log(torch.tensor([[[0.5, 1.0]], [[0.5, 0.25]], [[1.0, 0.5]]], dtype=f64))
    beta = torch.tensor([[1.0], [0.5], [2.0]], dtype=f64)
    # S1 = diag(.5,1)*0 + 1*[1,0]^T*3           = [[3],[0]]     o1 = q1.S1 = 3
    # S2 = diag(.5,.25)*S1 + .5*[0,2]^T*5        = [[1.5],[5]]   o2 = 5
    # S3 = diag(1,.5)*S2 + 2*[1,0]^T*7           = [[15.5],[2.5]] o3 = 18
    o = oracle.kda_fwd(q, k, v, g, beta, torch.ones(1, 3, dtype=torch.int32))
    assert o[:, 0, 0].tolist() == pytest.approx([3.0, 5.0, 18.0], abs=1e-14)


def test_zero_decay_is_causal_linear_attention():
    gen = torch.Generator().manual_seed(2)
    B, T, H, Dk, Dv = 1, 40, 3, 8, 6
    seg_np = synth.random_segment_ids(np.random.default_rng(2), B, T, max_len=15)
    seg = torch.from_numpy(seg_np)
    q, k, v, _, beta = _rand_inputs(B * T, H, Dk, Dv, gen)
    g = torch.zeros(B * T, H, Dk, dtype=f64)
    o = oracle.kda_fwd(q, k, v, g, beta, seg, B, T)
    ids = seg.reshape(-1)
    same = (ids[:, None] == ids[None, :]) & (ids[:, None] != 0)
    mask = torch.tril(torch.ones(T, T, dtype=torch.bool)) & same
    for h in range(H):
        A = (q[:, h] @ k[:, h].T) * mask
        ref = A @ (beta[:, h, None] * v[:, h])
        assert torch.allclose(o[:, h], ref, rtol=1e-12, atol=1e-12)


def test_length_one_documents():
    gen = torch.Generator().manual_seed(3)
    T, H, Dk, Dv = 12, 2, 4, 5
    seg = torch.arange(1, T + 1, dtype=torch.int32)[None]
    q, k, v, g, beta = _rand_inputs(T, H, Dk, Dv, gen)
    o = oracle.kda_fwd(q, k, v, g, beta, seg, 1, T, scale=1.3)
    ref = 1.3 * beta[..., None] * (q * k).sum(-1, keepdim=True) * v
    assert torch.allclose(o, ref, rtol=1e-13, atol=1e-13)


def test_scalar_channel_is_first_order_filter():
    gen = torch.Generator().manual_seed(4)
    T = 300
    a = 0.93
    q = torch.randn(T, 1, 1, generator=gen, dtype=f64)
    k = torch.randn(T, 1, 1, generator=gen, dtype=f64)
    v = torch.randn(T, 1, 1, generator=gen, dtype=f64)
    beta = torch.rand(T, 1, generator=gen, dtype=f64)
    g = torch.full((T, 1, 1), math.log(a), dtype=f64)
    o = oracle.kda_fwd(q, k, v, g, beta, None, 1, T)
    u = (beta[:, 0] * k[:, 0, 0] * v[:, 0, 0]).numpy()
    s = scipy.signal.lfilter([1.0], [1.0, -a], u)    # s_t = a s_{t-1} + u_t
    assert np.allclose(o[:, 0, 0].numpy(), q[:, 0, 0].numpy() * s, rtol=1e-11, atol=1e-12)


def test_gate_injection_equivalence():
    gen = torch.Generator().manual_seed(5)
    B, T, H, Dk, Dv = 1, 70, 2, 6, 4
    seg_np = synth.random_segment_ids(np.random.default_rng(5), B, T, max_len=20)
    seg = torch.from_numpy(seg_np)
    q, k, v, g, beta = _rand_inputs(B * T, H, Dk, Dv, gen)
    o_packed = oracle.kda_fwd(q, k, v, g, beta, seg, B, T)
    g_inj = g.clone()
    for t in range(1, T):
        if seg_np[0, t] != seg_np[0, t - 1]:
            g_inj[t] = -math.inf                      # exp(-inf) = 0 clears S at the start
    o_inj = oracle.kda_fwd(q, k, v, g_inj, beta, None, B, T)
    assert torch.allclose(o_packed, o_inj, rtol=1e-13, atol=1e-13)


def test_isolation_packed_equals_per_document():
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_kda_inputs(wl)
    o = oracle.kda_fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.segment_ids, wl.B, wl.T)
    t = 0
    for L in inp.doc_lengths[0]:
        sl = slice(t, t + L)
        alone = oracle.kda_fwd(inp.q[sl], inp.k[sl], inp.v[sl], inp.g[sl], inp.beta[sl],
                               None, 1, L)
        assert torch.equal(o[sl], alone)      # bit-exact: same arithmetic, same order
        t += L


def test_none_equals_all_ones_and_rows_independent():
    gen = torch.Generator().manual_seed(6)
    B, T, H, Dk, Dv = 3, 17, 2, 4, 4
    q, k, v, g, beta = _rand_inputs(B * T, H, Dk, Dv, gen)
    o_none = oracle.kda_fwd(q, k, v, g, beta, None, B, T)
    o_ones = oracle.kda_fwd(q, k, v, g, beta, torch.ones(B, T, dtype=torch.int32), B, T)
    assert torch.equal(o_none, o_ones)
    # changing row 2's ids leaves rows 0 and 1 bitwise unchanged
    seg = torch.ones(B, T, dtype=torch.int32)
    seg2 = seg.clone()
    seg2[2, 5:] = 2
    a = oracle.kda_fwd(q, k, v, g, beta, seg, B, T)
    b = oracle.kda_fwd(q, k, v, g, beta, seg2, B, T)
    assert torch.equal(a[: 2 * T], b[: 2 * T])
    assert not torch.equal(a[2 * T:], b[2 * T:])


def test_scale_linearity_and_padding_zero():
    gen = torch.Generator().manual_seed(7)
    B, T, H, Dk, Dv = 2, 30, 2, 4, 3
    seg = torch.from_numpy(synth.random_segment_ids(np.random.default_rng(7), B, T,
                                                    max_len=8, pad_prob=0.3))
    q, k, v, g, beta = _rand_inputs(B * T, H, Dk, Dv, gen)
    o1 = oracle.kda_fwd(q, k, v, g, beta, seg, B, T, scale=1.0)
    o2 = oracle.kda_fwd(q, k, v, g, beta, seg, B, T, scale=0.25)
    assert torch.allclose(o2, 0.25 * o1, rtol=1e-14, atol=0)
    pad = seg.reshape(-1) == 0
    assert pad.any()
    assert torch.count_nonzero(o1[pad]).item() == 0
    # padding inputs are ignored entirely, even non-finite ones
    q2 = q.clone()
    q2[pad] = float("nan")
    v2 = v.clone()
    v2[pad] = float("inf")
    o3 = oracle.kda_fwd(q2, k, v2, g, beta, seg, B, T)
    assert torch.equal(o1, o3)


def test_threads_do_not_change_result():
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_kda_inputs(wl)
    a = oracle.kda_fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.segment_ids, 1, wl.T, n_threads=1)
    b = oracle.kda_fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.segment_ids, 1, wl.T, n_threads=5)
    assert torch.equal(a, b)
