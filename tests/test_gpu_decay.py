"""GPU parity under strong decay (log-decays far below the synthetic workloads').

The tensor-core kernel factorises exp(G_i - G_j) as exp(-Suf_i) exp(Suf_j). With a
reference point at the chunk's end, that leaves fp32's range once a key channel
decays by more than about e^-80 over a chunk (a per-token average below -1.25).
The fast chunk kernel has only that form; it lists the units holding such a chunk,
and the safe chunk kernel, launched after it, reruns those units with the choice of
the sub-block form per chunk: the reference at the end of each 16-row sub-block,
which holds while every 16-row sub-block stays above e^-80 (an average above -5 per
token). RFC-0026 §3.3's gate kwargs (lower_bound, safe_gate) are there for gates
this strong.

- Decay of about -3 per token (range -1.5 .. -4.5) on some channels, mixed with the
  usual decay on the others, on layouts with boundaries at every sub-block position,
  padding and several rows: o within the bf16 bound of the oracle for either output
  dtype, with the status word clean. Chunks of both forms follow one another inside
  a unit, so the state carries from one form to the other.
- The same for the per-segment state call (initial states in, final states out).
- The 64-wide and fp32 paths (the token recurrence) under the same decay.
- Decay below the sub-block form's range sets KDA_DEV_DECAY_RANGE; the wrappers
  raise KdaDeviceError by default.
"""
import numpy as np
import pytest
import torch

import kda_segids_cu_gb300 as kda
import oracle
import synth
from tests.parity import check_kda_output
from tests.test_gpu_state import _check_states, _n_segments

pytestmark = pytest.mark.gpu


def _strong_inputs(seg, H, D, dtype, seed, n_strong=8, mean=-3.0, chunk_mask=None):
    """q, k L2-normalised, v ~ N(0,1), beta = sigmoid(N(0,1)); g = -exp(N(-2, 0.5)) except on
    n_strong channels per head, where g = mean * U(0.5, 1.5) (only in the chunks that
    chunk_mask marks, if given)."""
    B, T = seg.shape
    N = B * T
    gen = torch.Generator().manual_seed(seed)
    q = torch.nn.functional.normalize(torch.randn(N, H, D, generator=gen), dim=-1)
    k = torch.nn.functional.normalize(torch.randn(N, H, D, generator=gen), dim=-1)
    v = torch.randn(N, H, D, generator=gen)
    g = -torch.exp(torch.randn(N, H, D, generator=gen) * 0.5 - 2.0)
    beta = torch.sigmoid(torch.randn(N, H, generator=gen))
    for h in range(H):
        ch = torch.randperm(D, generator=gen)[:n_strong]
        strong = mean * (0.5 + torch.rand(N, n_strong, generator=gen))
        if chunk_mask is not None:
            rows = torch.from_numpy(np.repeat(chunk_mask, 64)[:N])
            strong = torch.where(rows[:, None], strong, g[:, h][:, ch])
        g[:, h, ch] = strong
    return [t.to(dtype) for t in (q, k, v, g, beta)]


def _layouts():
    rng = np.random.default_rng(23)
    out = [synth.random_segment_ids(rng, 2, 700, max_len=300, pad_prob=0.05),
           synth.random_segment_ids(rng, 1, 1000, max_len=20, pad_prob=0.1),
           np.ones((1, 64 * 9 + 5), np.int32)]
    seg = np.ones((2, 300), np.int32)            # boundaries on and next to sub-block edges
    for i, p in enumerate([15, 16, 17, 31, 32, 47, 63, 64, 65, 100, 127, 128]):
        seg[0, p:] = i + 2
    seg[1, 40:56] = 0
    seg[1, 56:] = 30
    seg[1, 200:] = 31
    out.append(seg)
    return [torch.from_numpy(s) for s in out]


@pytest.mark.parametrize("out_dtype", [None, torch.float32])
def test_strong_decay_tensor_core(out_dtype):
    for i, seg in enumerate(_layouts()):
        B, T = seg.shape
        q, k, v, g, beta = _strong_inputs(seg, 3, 128, torch.bfloat16, seed=40 + i)
        ref = oracle.kda_fwd(q, k, v, g, beta, seg, B, T, scale=0.9)
        o = kda.kda_chunk_fwd_varlen(*(t.cuda() for t in (q, k, v, g, beta)), seg.cuda(),
                                     scale=0.9, out_dtype=out_dtype)   # raises on a status bit
        check_kda_output(o, ref, seg, torch.bfloat16, label=f"strong layout {i}")


def test_strong_decay_in_some_chunks():
    """One long segment whose strong decay comes and goes chunk by chunk: consecutive
    chunks of one unit alternate between the two forms."""
    rng = np.random.default_rng(5)
    T = 64 * 40
    seg = torch.ones(1, T, dtype=torch.int32)
    mask = rng.random(40) < 0.5
    q, k, v, g, beta = _strong_inputs(seg, 2, 128, torch.bfloat16, seed=77, chunk_mask=mask)
    ref = oracle.kda_fwd(q, k, v, g, beta, seg, 1, T)
    o = kda.kda_chunk_fwd_varlen(*(t.cuda() for t in (q, k, v, g, beta)), seg.cuda(),
                                 out_dtype=torch.float32)
    check_kda_output(o, ref, seg, torch.bfloat16, label="alternating forms")
    o_none = kda.kda_chunk_fwd_varlen(*(t.cuda() for t in (q, k, v, g, beta)), None, B=1, T=T,
                                      out_dtype=torch.float32)
    assert torch.equal(o, o_none)


def test_strong_decay_ling3_shape():
    """The ling3 workload's shape and documents with 16 strongly decaying channels per head,
    all heads against the oracle."""
    wl = synth.WORKLOADS["ling3"]
    seg_np, _ = synth.make_segment_ids(wl, synth.default_seed(wl.name))
    seg = torch.from_numpy(seg_np)
    q, k, v, g, beta = _strong_inputs(seg, wl.H, wl.d_qk, torch.bfloat16, seed=91, n_strong=16)
    ref = oracle.kda_fwd(q, k, v, g, beta, seg, wl.B, wl.T)
    o = kda.kda_chunk_fwd_varlen(*(t.cuda() for t in (q, k, v, g, beta)), seg.cuda())
    check_kda_output(o, ref, seg, torch.bfloat16, label="ling3 strong")


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.bfloat16, 64),
                                     (torch.float32, 64)])
def test_strong_decay_state_call(dtype, D):
    for i, seg in enumerate(_layouts()[:2] + _layouts()[3:]):
        B, T = seg.shape
        H = 2
        q, k, v, g, beta = _strong_inputs(seg, H, D, dtype, seed=60 + i)
        n = _n_segments(seg, B)
        init = torch.randn(n, H, D, D, generator=torch.Generator().manual_seed(i)) * 0.3
        ref, ref_fin = oracle.kda_fwd_state(q, k, v, g, beta, seg, B, T, initial_state=init,
                                            n_state=n, want_final=True)
        o, fin = kda.kda_chunk_fwd_varlen_state(*(t.cuda() for t in (q, k, v, g, beta)),
                                                seg.cuda(), initial_state=init.cuda(),
                                                output_final_state=True,
                                                out_dtype=torch.float32)
        bound = dtype if (dtype == torch.bfloat16 and D == 128) else torch.float32
        check_kda_output(o, ref, seg, bound, label=f"state strong {i} D={D}")
        _check_states(fin, ref_fin, f"state strong {i} D={D}")


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 64), (torch.float32, 64)])
def test_strong_decay_token_recurrence(dtype, D):
    for i, seg in enumerate(_layouts()):
        B, T = seg.shape
        q, k, v, g, beta = _strong_inputs(seg, 2, D, dtype, seed=80 + i, n_strong=4, mean=-6.0)
        ref = oracle.kda_fwd(q, k, v, g, beta, seg, B, T)
        o = kda.kda_chunk_fwd_varlen(*(t.cuda() for t in (q, k, v, g, beta)), seg.cuda())
        check_kda_output(o, ref, seg, dtype, label=f"recurrence strong {i}")


def test_decay_beyond_the_range_is_reported():
    """A channel decaying by about -8 per token leaves even a 16-row sub-block's range: the
    kernel sets KDA_DEV_DECAY_RANGE and the default wrapper raises; with check=False the
    word is the caller's to read."""
    seg = torch.ones(1, 256, dtype=torch.int32)
    q, k, v, g, beta = _strong_inputs(seg, 1, 128, torch.bfloat16, seed=3, n_strong=1, mean=-8.0)
    args = [t.cuda() for t in (q, k, v, g, beta)]
    with pytest.raises(kda.KdaDeviceError) as e:
        kda.kda_chunk_fwd_varlen(*args, seg.cuda())
    assert e.value.bits & kda.KDA_DEV_DECAY_RANGE
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_chunk_fwd_varlen(*args, seg.cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & kda.KDA_DEV_DECAY_RANGE
    # the usual decay leaves the word clean
    q, k, v, g, beta = _strong_inputs(seg, 1, 128, torch.bfloat16, seed=3, n_strong=0)
    status.zero_()
    kda.kda_chunk_fwd_varlen(*(t.cuda() for t in (q, k, v, g, beta)), seg.cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_strong_decay_planned_calls_and_graph_replay():
    """The fast chunk kernel leaves units with a chunk out of its range to the safe kernel,
    through a list in the workspace that the safe kernel empties again. Planned calls that
    reuse one plan, alternating strong and usual decay, and replays of a captured forward
    each equal the plain call bit for bit."""
    B, T, H, D = 2, 640, 3, 128
    rng = np.random.default_rng(9)
    seg = torch.from_numpy(synth.random_segment_ids(rng, B, T, max_len=400, pad_prob=0.05))
    strong = [t.cuda() for t in _strong_inputs(seg, H, D, torch.bfloat16, seed=5)]
    usual = [t.cuda() for t in _strong_inputs(seg, H, D, torch.bfloat16, seed=6, n_strong=0)]
    segd = seg.cuda()
    ws = torch.empty(max(kda.chunk_fwd_workspace_bytes(B, T, H, D, D, torch.bfloat16), 256),
                     dtype=torch.uint8, device="cuda")
    kda.kda_chunk_plan_varlen(segd, B, T, H, D, D, torch.bfloat16, ws)
    for inp in (strong, usual, strong, strong, usual):
        plain = kda.kda_chunk_fwd_varlen(*inp, segd)
        o = kda.kda_chunk_fwd_varlen(*inp, segd, workspace=ws, planned=True)
        torch.cuda.synchronize()
        assert torch.equal(o, plain)
    ref = oracle.kda_fwd(*(t.cpu() for t in strong), seg, B, T)
    check_kda_output(kda.kda_chunk_fwd_varlen(*strong, segd), ref, seg, torch.bfloat16,
                     label="planned strong")
    # a captured planned forward, replayed on strong then usual inputs
    bufs = [t.clone() for t in strong]
    out = torch.empty_like(bufs[2])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        kda.kda_chunk_fwd_varlen(*bufs, segd, workspace=ws, planned=True, out=out, status=status)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        kda.kda_chunk_fwd_varlen(*bufs, segd, workspace=ws, planned=True, out=out, status=status)
    for inp in (strong, usual, strong):
        for dst, src in zip(bufs, inp):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, kda.kda_chunk_fwd_varlen(*inp, segd))
    assert int(status.item()) == 0
