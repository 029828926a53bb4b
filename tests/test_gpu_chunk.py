"""GPU parity and invariants for kda_chunk_fwd_varlen.

Bar (per head, over real tokens): max|o - o_ref| <= 2e-2 RMS(o_ref) for bf16
inputs, <= 1e-4 RMS(o_ref) for fp32 inputs; padding outputs exactly 0.
Small workloads are compared in full; the large ones at their full size, in
the launch configuration the bench times: ling3 and short on every head, the
long workloads on sampled heads that the oracle computes in seconds. Bit-exact invariants: documents do not leak into each
other, rows are independent, segment_ids=None equals all-ones ids, reruns are
deterministic. Within the bound: a packed call equals its documents run alone.
"""
import numpy as np
import pytest
import torch

import kda_segids_cu_gb300 as kda
import oracle
import synth
from tests.parity import check_kda_output

pytestmark = pytest.mark.gpu


def _gpu_fwd(inp, B, T, scale=1.0, seg="inputs", out_dtype=None):
    s = inp.segment_ids if seg == "inputs" else seg
    o = kda.kda_chunk_fwd_varlen(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.g.cuda(),
                                 inp.beta.cuda(), None if s is None else s.cuda(), scale=scale,
                                 B=B, T=T, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return o


def _oracle(inp, B, T, heads=None, scale=1.0, seg="inputs"):
    s = inp.segment_ids if seg == "inputs" else seg
    if heads is None:
        return oracle.kda_fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, s, B, T, scale=scale)
    hs = torch.tensor(heads)
    pick = lambda t: t.index_select(1, hs.to(t.device)).cpu()
    return oracle.kda_fwd(pick(inp.q), pick(inp.k), pick(inp.v), pick(inp.g), pick(inp.beta),
                          None if s is None else s.cpu(), B, T, scale=scale)


@pytest.mark.parametrize("name", ["tiny", "b2"])
def test_small_workloads_full(name):
    wl = synth.WORKLOADS[name]
    inp = synth.make_kda_inputs(wl)
    ref = _oracle(inp, wl.B, wl.T)
    # fp32 output: the strict per-head bound; input-dtype output: plus its rounding
    o32 = _gpu_fwd(inp, wl.B, wl.T, out_dtype=torch.float32)
    check_kda_output(o32, ref, inp.segment_ids, wl.dtype, label=name + "/f32 out")
    o = _gpu_fwd(inp, wl.B, wl.T)
    assert o.dtype == wl.dtype
    check_kda_output(o, ref, inp.segment_ids, wl.dtype, label=name)


@pytest.mark.parametrize("name,heads", [("ling3", None), ("short", None),
                                        ("long", [0, 31]), ("long_none", [5])])
def test_large_workloads(name, heads):
    """ling3 and short on every head; long and long_none on sampled heads."""
    wl = synth.WORKLOADS[name]
    inp = synth.make_kda_inputs(wl, device="cuda")
    ref = _oracle(inp, wl.B, wl.T, heads=heads)
    o = _gpu_fwd(inp, wl.B, wl.T)
    check_kda_output(o, ref, inp.segment_ids, wl.dtype, heads=heads, label=name)
    o32 = _gpu_fwd(inp, wl.B, wl.T, out_dtype=torch.float32)
    check_kda_output(o32, ref, inp.segment_ids, wl.dtype, heads=heads, label=name + "/f32 out")
    # the bf16 output is the fp32 output rounded once to nearest even
    assert torch.equal(o, o32.to(wl.dtype))


def test_long_none_equals_single_segment():
    # segment_ids=None on the long workload equals one all-ones segment, bitwise
    wl = synth.WORKLOADS["long_none"]
    inp = synth.make_kda_inputs(wl, device="cuda", heads=4)
    a = _gpu_fwd(inp, wl.B, wl.T)
    b = _gpu_fwd(inp, wl.B, wl.T, seg=torch.ones(wl.B, wl.T, dtype=torch.int32))
    assert torch.equal(a, b)


def _small_random(B, T, H, D, dtype, seed, max_len=80, pad_prob=0.0, ids="increasing"):
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    seg = torch.from_numpy(synth.random_segment_ids(rng, B, T, max_len=max_len,
                                                    pad_prob=pad_prob, ids=ids))
    N = B * T
    q = torch.nn.functional.normalize(torch.randn(N, H, D, generator=gen), dim=-1).to(dtype)
    k = torch.nn.functional.normalize(torch.randn(N, H, D, generator=gen), dim=-1).to(dtype)
    v = torch.randn(N, H, D, generator=gen).to(dtype)
    g = (-torch.exp(torch.randn(N, H, D, generator=gen) * 0.5 - 2.0)).to(dtype)
    beta = torch.sigmoid(torch.randn(N, H, generator=gen)).to(dtype)
    return synth.KdaInputs(q, k, v, g, beta, seg, [])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D", [64, 128])
def test_boundary_sweep(dtype, D):
    """Ragged T, several chunks, boundaries at every in-chunk offset, length-1
    documents, interior and leading padding, arbitrary (non-monotone) ids."""
    cases = [
        dict(B=1, T=64 * 5 + 17, max_len=70),
        dict(B=3, T=100, max_len=9, pad_prob=0.25),
        dict(B=2, T=200, max_len=3, ids="arbitrary"),
        dict(B=1, T=333, max_len=200, pad_prob=0.1),
        dict(B=1, T=130, max_len=1),
    ]
    for i, c in enumerate(cases):
        B, T = c.pop("B"), c.pop("T")
        inp = _small_random(B, T, 2, D, dtype, seed=100 * D + i, **c)
        o = _gpu_fwd(inp, B, T, scale=0.5)
        ref = _oracle(inp, B, T, scale=0.5)
        check_kda_output(o, ref, inp.segment_ids, dtype, label=f"case{i}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_every_boundary_offset(dtype):
    # one document boundary at each offset 1..64 of the second chunk (64-wide heads: the
    # token recurrence)
    for off in range(1, 65):
        T = 192
        seg = torch.ones(1, T, dtype=torch.int32)
        seg[0, 64 + off:] = 2
        inp = _small_random(1, T, 1, 64, dtype, seed=off)
        inp.segment_ids = seg
        check_kda_output(_gpu_fwd(inp, 1, T), _oracle(inp, 1, T), seg, dtype, label=f"off{off}")


@pytest.mark.parametrize("out_dtype", [None, torch.float32])
def test_every_boundary_offset_tensor_core(out_dtype):
    """bf16 with 128-wide heads (the tcgen05 kernel): a boundary at each offset 0..63 of a
    chunk in two rows whose second row starts inside a chunk (T = 200: flat 200 is offset 8
    of chunk 3), plus a boundary on the first and on the last row of another chunk and a
    padding run, so that row masks, the A' mask, first cuts and carried states all see
    every in-chunk position."""
    B, T, H = 2, 200, 2
    for off in range(64):
        seg = torch.ones(B, T, dtype=torch.int32)
        seg[0, 64 + off:] = 2                  # row 0: chunk 1, offset off
        seg[0, 128:] = 3                       # row 0: first row of chunk 2
        seg[0, 191:] = 4                       # row 0: last row of chunk 2
        seg[1, 56 + off:] = 5                  # row 1 (flat 200..399): chunk 4, offset off
        seg[1, 120 + (off % 7):126 + (off % 7)] = 0     # padding inside chunk 5
        inp = _small_random(B, T, H, 128, torch.bfloat16, seed=500 + off)
        inp.segment_ids = seg
        o = _gpu_fwd(inp, B, T, scale=0.75, out_dtype=out_dtype)
        check_kda_output(o, _oracle(inp, B, T, scale=0.75), seg, torch.bfloat16,
                         label=f"tc off{off}")


def test_isolation_bitwise():
    """Changing one document's values leaves every other document's output bitwise
    unchanged (no state leaks across a boundary)."""
    wl = synth.WORKLOADS["b2"]
    inp = synth.make_kda_inputs(wl)
    o1 = _gpu_fwd(inp, wl.B, wl.T).cpu()
    seg = inp.segment_ids.reshape(-1)
    victim = (seg == 3)
    victim[wl.T:] = False                     # document 3 of row 0
    inp2 = synth.KdaInputs(inp.q.clone(), inp.k.clone(), inp.v.clone(), inp.g.clone(),
                           inp.beta.clone(), inp.segment_ids, [])
    inp2.v[victim] = -inp2.v[victim] * 3
    inp2.q[victim] = inp2.k[victim]
    o2 = _gpu_fwd(inp2, wl.B, wl.T).cpu()
    assert torch.equal(o1[~victim], o2[~victim])
    assert not torch.equal(o1[victim], o2[victim])


def test_packed_equals_per_document():
    """Each document run alone (its own call: B=1, T its length, no ids) gives the packed
    call's output for its tokens within the bf16 bound. Packing changes only where the
    document's tokens fall on the 64-token chunk grid."""
    wl = synth.WORKLOADS["b2"]
    inp = synth.make_kda_inputs(wl)
    packed = _gpu_fwd(inp, wl.B, wl.T, out_dtype=torch.float32).cpu()
    seg = inp.segment_ids.reshape(-1)
    N = wl.B * wl.T
    alone = torch.zeros_like(packed)
    n_docs, p = 0, 0
    while p < N:
        if seg[p] == 0:
            p += 1
            continue
        e = p + 1
        while e < N and e % wl.T != 0 and seg[e] == seg[p]:
            e += 1
        one = synth.KdaInputs(inp.q[p:e], inp.k[p:e], inp.v[p:e], inp.g[p:e], inp.beta[p:e],
                              None, [])
        alone[p:e] = _gpu_fwd(one, 1, e - p, seg=None, out_dtype=torch.float32).cpu()
        n_docs += 1
        p = e
    assert n_docs >= 8
    assert (packed[seg == 0] == 0).all()
    check_kda_output(packed, alone.double(), inp.segment_ids, wl.dtype, label="packed vs alone")


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.bfloat16, 64),
                                     (torch.float32, 64)])
def test_planned_calls_match_plain_call(dtype, D):
    """A plan made on another stream, then planned forwards on it (the second reuses the
    plan: the kernel rewinds its work counter), give the plain call's output bit for bit."""
    B, T, H = 2, 700, 3
    inp = _small_random(B, T, H, D, dtype, seed=31, max_len=150, pad_prob=0.05)
    q, k, v, g, beta = (t.cuda().contiguous() for t in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    seg = inp.segment_ids.cuda().contiguous()
    plain = kda.kda_chunk_fwd_varlen(q, k, v, g, beta, seg, B=B, T=T)
    ws = torch.empty(max(kda.chunk_fwd_workspace_bytes(B, T, H, D, D, dtype), 256),
                     dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        kda.kda_chunk_plan_varlen(seg, B, T, H, D, D, dtype, ws)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        o = kda.kda_chunk_fwd_varlen(q, k, v, g, beta, seg, B=B, T=T, workspace=ws,
                                     planned=True)
        torch.cuda.synchronize()
        assert torch.equal(o, plain)
    # segment_ids=None: the plan of whole rows
    plain = kda.kda_chunk_fwd_varlen(q, k, v, g, beta, None, B=B, T=T)
    kda.kda_chunk_plan_varlen(None, B, T, H, D, D, dtype, ws)
    o = kda.kda_chunk_fwd_varlen(q, k, v, g, beta, None, B=B, T=T, workspace=ws, planned=True)
    torch.cuda.synchronize()
    assert torch.equal(o, plain)


def test_row_independence_and_determinism():
    B, T = 3, 300
    inp = _small_random(B, T, 2, 128, torch.bfloat16, seed=9, max_len=90)
    a = _gpu_fwd(inp, B, T).cpu()
    seg2 = inp.segment_ids.clone()
    seg2[2] = torch.from_numpy(synth.random_segment_ids(np.random.default_rng(1), 1, T, 20))[0]
    b = _gpu_fwd(inp, B, T, seg=seg2).cpu()
    assert torch.equal(a[: 2 * T], b[: 2 * T])
    c = _gpu_fwd(inp, B, T).cpu()
    assert torch.equal(a, c)


def test_none_equals_all_ones():
    B, T = 2, 257
    for dtype in (torch.bfloat16, torch.float32):
        inp = _small_random(B, T, 2, 64, dtype, seed=3)
        a = _gpu_fwd(inp, B, T, seg=None)
        b = _gpu_fwd(inp, B, T, seg=torch.ones(B, T, dtype=torch.int32))
        assert torch.equal(a, b)
        check_kda_output(a, _oracle(inp, B, T, seg=None), None, dtype, label="none")


def test_all_padding_and_tiny_shapes():
    for (B, T) in [(1, 1), (1, 63), (2, 65), (5, 3)]:
        inp = _small_random(B, T, 3, 64, torch.bfloat16, seed=B * 100 + T, max_len=5)
        check_kda_output(_gpu_fwd(inp, B, T), _oracle(inp, B, T), inp.segment_ids,
                         torch.bfloat16, label=f"{B}x{T}")
    inp = _small_random(2, 70, 2, 64, torch.bfloat16, seed=1)
    zeros = torch.zeros(2, 70, dtype=torch.int32)
    o = _gpu_fwd(inp, 2, 70, seg=zeros)
    assert torch.count_nonzero(o).item() == 0
