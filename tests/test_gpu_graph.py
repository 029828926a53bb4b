"""Every libkda call can be captured in a CUDA graph (no host round trip, no
allocation, launches only on the caller's stream): a whole step -- cu_seqlens, a
masked conv, the chunked forward (planner and chunk kernel, chained by
programmatic dependent launch) and the per-segment state call -- is captured
once and replayed on new inputs, and every replay equals the eager calls bit for
bit (the kernels are deterministic)."""
import pytest
import torch

import kda_segids_cu_gb300 as kda
from tests.test_gpu_chunk import _small_random

pytestmark = pytest.mark.gpu


def _fill(dst, src):
    dst.copy_(src.to(dst.device))


def test_step_captured_in_a_graph_matches_eager():
    B, T, H, D, K = 2, 300, 4, 128, 4
    F = H * D
    dev = torch.device("cuda")
    first = _small_random(B, T, H, D, torch.bfloat16, seed=11, max_len=90, pad_prob=0.1)
    # static buffers the graph reads and writes
    seg = first.segment_ids.to(dev).contiguous()
    q, k, v, g, beta = (t.to(dev).contiguous() for t in (first.q, first.k, first.v, first.g,
                                                          first.beta))
    x = torch.randn(B, T, F, device=dev).bfloat16()
    w = (torch.randn(K, F, device=dev) * 0.5).bfloat16()
    max_segs = 64
    n_state = 8
    init = torch.randn(n_state, H, D, D, device=dev) * 0.1

    def step():
        cu, n = kda.kda_segids_to_cu_seqlens(seg, max_segs)
        y = kda.kda_short_conv_varlen(x, w, seg)
        o = kda.kda_chunk_fwd_varlen(q, k, v, g, beta, seg, B=B, T=T)
        o2, fin = kda.kda_chunk_fwd_varlen_state(q, k, v, g, beta, seg, B=B, T=T,
                                                 initial_state=init, output_final_state=True)
        return cu, n, y, o, o2, fin

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        step()                                   # first calls set kernel attributes
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        outs = step()
    torch.cuda.synchronize()

    for trial in range(3):
        new = _small_random(B, T, H, D, torch.bfloat16, seed=20 + trial, max_len=70,
                            pad_prob=0.1)
        for dst, src in ((seg, new.segment_ids), (q, new.q), (k, new.k), (v, new.v),
                         (g, new.g), (beta, new.beta)):
            _fill(dst, src)
        x.copy_(torch.randn(B, T, F, device=dev).bfloat16())
        graph.replay()
        torch.cuda.synchronize()
        eager = step()
        torch.cuda.synchronize()
        for name, a, b in zip(("cu_seqlens", "n_segs", "conv", "o", "o (state)", "final state"),
                              outs, eager):
            assert torch.equal(a, b), f"trial {trial}: graph replay differs from eager: {name}"


def test_two_stream_step_with_a_plan_matches_plain_calls():
    """The bench's step shape: the scan and the chunk plan on a side stream of the graph,
    beside the conv; the planned forward after the join. Replays on new inputs equal the
    plain eager calls bit for bit."""
    B, T, H, D, K = 2, 640, 4, 128, 4
    F = H * D
    dev = torch.device("cuda")
    first = _small_random(B, T, H, D, torch.bfloat16, seed=41, max_len=200, pad_prob=0.05)
    seg = first.segment_ids.to(dev).contiguous()
    g, beta = first.g.to(dev).contiguous(), first.beta.to(dev).contiguous()
    xs = [torch.randn(B, T, F, device=dev).bfloat16() for _ in range(3)]
    w = (torch.randn(K, F, device=dev) * 0.5).bfloat16()
    ys = [torch.empty_like(x) for x in xs]
    cu = torch.empty(65, dtype=torch.int32, device=dev)
    nseg = torch.empty(1, dtype=torch.int32, device=dev)
    o = torch.empty(B * T, H, D, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(kda.chunk_fwd_workspace_bytes(B, T, H, D, D, torch.bfloat16), 256),
                     dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream()

    def step():
        cur = torch.cuda.current_stream()
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            kda.kda_segids_to_cu_seqlens(seg, 64, out=cu, n_segs_out=nseg)
            kda.kda_chunk_plan_varlen(seg, B, T, H, D, D, torch.bfloat16, ws)
        for x, y in zip(xs, ys):
            kda.kda_short_conv_varlen(x, w, seg, out=y)
        cur.wait_stream(side)
        qkv = [y.view(B * T, H, D) for y in ys]
        kda.kda_chunk_fwd_varlen(qkv[0], qkv[1], qkv[2], g, beta, seg, B=B, T=T, out=o,
                                 workspace=ws, planned=True)

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    torch.cuda.synchronize()
    for trial in range(3):
        new = _small_random(B, T, H, D, torch.bfloat16, seed=50 + trial, max_len=120,
                            pad_prob=0.05)
        _fill(seg, new.segment_ids)
        _fill(g, new.g)
        _fill(beta, new.beta)
        for x in xs:
            x.copy_(torch.randn(B, T, F, device=dev).bfloat16())
        graph.replay()
        torch.cuda.synchronize()
        cu_e, n_e = kda.kda_segids_to_cu_seqlens(seg, 64)
        ys_e = [kda.kda_short_conv_varlen(x, w, seg) for x in xs]
        o_e = kda.kda_chunk_fwd_varlen(*[y.view(B * T, H, D) for y in ys_e], g, beta, seg, B=B,
                                       T=T)
        torch.cuda.synchronize()
        assert torch.equal(cu, cu_e) and torch.equal(nseg, n_e.reshape(nseg.shape))
        for y, y_e in zip(ys, ys_e):
            assert torch.equal(y, y_e)
        assert torch.equal(o, o_e), f"trial {trial}: planned replay differs from the plain call"


def test_backward_captured_in_a_graph_matches_eager():
    B, T, H, D = 2, 200, 2, 128
    dev = torch.device("cuda")
    first = _small_random(B, T, H, D, torch.bfloat16, seed=31, max_len=80, pad_prob=0.1)
    seg = first.segment_ids.to(dev).contiguous()
    q, k, v, g, beta = (t.to(dev).contiguous() for t in (first.q, first.k, first.v, first.g,
                                                          first.beta))
    d_o = torch.randn(q.shape, device=dev).bfloat16()
    ws = torch.empty(int(kda.load_library().kda_chunk_bwd_varlen_workspace_size(
        B, T, H, D, D, kda.KDA_BF16)), dtype=torch.uint8, device=dev)

    def step():
        return kda.kda_chunk_bwd_varlen(q, k, v, g, beta, d_o, seg, B=B, T=T, workspace=ws)

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        step()                                   # first call sets kernel attributes
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        outs = step()
    torch.cuda.synchronize()
    for trial in range(2):
        new = _small_random(B, T, H, D, torch.bfloat16, seed=40 + trial, max_len=60, pad_prob=0.1)
        for dst, src in ((seg, new.segment_ids), (q, new.q), (k, new.k), (v, new.v),
                         (g, new.g), (beta, new.beta)):
            _fill(dst, src)
        d_o.copy_(torch.randn(q.shape, device=dev).bfloat16())
        graph.replay()
        torch.cuda.synchronize()
        eager = step()
        torch.cuda.synchronize()
        for name, a, b in zip(("dq", "dk", "dv", "dg", "dbeta"), outs, eager):
            assert torch.equal(a, b), f"trial {trial}: graph replay differs from eager: {name}"
