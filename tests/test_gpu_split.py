"""GPU parity when long segments are split into pieces.

The state is serial along a segment, so a document much longer than one CTA's
share of the work (chunks x heads / SMs) would keep one SM busy while the
others idle. With room in the workspace, the plan cuts such a unit into
leading pieces of at most 64 chunks and a last piece of one share. A
state-only pass computes each leading piece's end state from a zero start and
hands each piece's start state to the next along the segment (a decoupled
look-back through flags in the workspace); the forward then runs every piece
from its start state.

The cases force splits at small sizes (few heads make a CTA's share a few
chunks), and each reads the plan's count of split pieces from the workspace to
be sure the path ran. Outputs are held to the oracle at the bf16 bound, and to
an unsplit call (the minimum workspace) at the same bound; planned calls on one
plan and replays of a captured forward equal the plain call bit for bit (the
look-back flags carry a per-call epoch).
"""
import numpy as np
import pytest
import torch

import kda_segids_cu_gb300 as kda
import oracle
import synth
from tests.parity import check_kda_output
from tests.test_gpu_decay import _strong_inputs

pytestmark = pytest.mark.gpu


def _workspace(B, T, H, minimum=False):
    n = kda.chunk_fwd_workspace_bytes(B, T, H, 128, 128, torch.bfloat16, minimum=minimum)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")


def _n_split(ws):
    """Split pieces with a successor in the last plan written to ws (plan counter 7)."""
    return int(ws[:64].view(torch.int32)[7].item())


def _layouts():
    rng = np.random.default_rng(41)
    one = np.ones((1, 64 * 300), np.int32)                       # one long document
    mixed = np.zeros((2, 64 * 150 + 17), np.int32)               # long and short documents
    mixed[0, :9000] = 1
    mixed[0, 9000:9100] = 0
    mixed[0, 9100:] = 2
    mixed[1] = synth.random_segment_ids(rng, 1, mixed.shape[1], max_len=40, pad_prob=0.1)[0]
    mixed[1, 500:8000] = 7
    padded = np.ones((1, 64 * 200 + 33), np.int32)               # a start inside a chunk, padding
    padded[0, :101] = 3
    padded[0, 101:12000] = 4
    padded[0, 12000:12050] = 0
    padded[0, 12050:] = 5
    return [torch.from_numpy(s) for s in (one, mixed, padded)]


@pytest.mark.parametrize("out_dtype", [None, torch.float32])
def test_split_matches_oracle_and_unsplit(out_dtype):
    for i, seg in enumerate(_layouts()):
        B, T = seg.shape
        H = 2
        args = [t.cuda() for t in _strong_inputs(seg, H, 128, torch.bfloat16, seed=70 + i,
                                                 n_strong=0)]
        ws = _workspace(B, T, H)
        o = kda.kda_chunk_fwd_varlen(*args, seg.cuda(), workspace=ws, out_dtype=out_dtype)
        assert _n_split(ws) > 0, f"layout {i}: nothing was split"
        ws_min = _workspace(B, T, H, minimum=True)
        o_min = kda.kda_chunk_fwd_varlen(*args, seg.cuda(), workspace=ws_min,
                                         out_dtype=out_dtype)
        assert _n_split(ws_min) == 0
        ref = oracle.kda_fwd(*(t.cpu() for t in args), seg, B, T)
        check_kda_output(o, ref, seg, torch.bfloat16, label=f"split layout {i}")
        check_kda_output(o, o_min.double().cpu(), seg, torch.bfloat16,
                         label=f"split vs unsplit layout {i}")


def test_split_planned_calls_and_graph_replay():
    seg = _layouts()[1]
    B, T = seg.shape
    H = 3
    usual = [t.cuda() for t in _strong_inputs(seg, H, 128, torch.bfloat16, seed=3, n_strong=0)]
    other = [t.cuda() for t in _strong_inputs(seg, H, 128, torch.bfloat16, seed=4, n_strong=0)]
    segd = seg.cuda()
    ws = _workspace(B, T, H)
    kda.kda_chunk_plan_varlen(segd, B, T, H, 128, 128, torch.bfloat16, ws)
    assert _n_split(ws) > 0
    for inp in (usual, other, usual, usual):
        plain = kda.kda_chunk_fwd_varlen(*inp, segd)
        o = kda.kda_chunk_fwd_varlen(*inp, segd, workspace=ws, planned=True)
        torch.cuda.synchronize()
        assert torch.equal(o, plain)
    bufs = [t.clone() for t in usual]
    out = torch.empty_like(bufs[2])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        kda.kda_chunk_fwd_varlen(*bufs, segd, workspace=ws, planned=True, out=out, status=status)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        kda.kda_chunk_fwd_varlen(*bufs, segd, workspace=ws, planned=True, out=out, status=status)
    for inp in (other, usual, other):
        for dst, src in zip(bufs, inp):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, kda.kda_chunk_fwd_varlen(*inp, segd))
    assert int(status.item()) == 0


def test_split_with_strong_decay():
    """Split pieces whose chunks leave the whole-chunk form's range: the safe kernel reruns
    those pieces from their start states."""
    seg = _layouts()[0]
    B, T = seg.shape
    args = [t.cuda() for t in _strong_inputs(seg, 2, 128, torch.bfloat16, seed=12, n_strong=6)]
    ws = _workspace(B, T, 2)
    o = kda.kda_chunk_fwd_varlen(*args, seg.cuda(), workspace=ws, out_dtype=torch.float32)
    assert _n_split(ws) > 0
    check_kda_output(o, oracle.kda_fwd(*(t.cpu() for t in args), seg, B, T), seg,
                     torch.bfloat16, label="split strong")


def test_long_workloads_are_split():
    """The long workload's plan splits its two longest documents; long_none its one."""
    for name in ("long", "long_none"):
        wl = synth.WORKLOADS[name]
        inp = synth.make_kda_inputs(wl, device="cuda", heads=2)
        ws = _workspace(wl.B, wl.T, wl.H)
        seg = inp.segment_ids
        kda.kda_chunk_plan_varlen(seg, wl.B, wl.T, wl.H, 128, 128, torch.bfloat16, ws)
        assert _n_split(ws) > 0, name
