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
