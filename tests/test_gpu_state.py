"""GPU parity for kda_chunk_fwd_varlen_state (per-segment initial and final state).

Segment r (flattened token order) starts from initial_state[r] and returns its
state after its last token in final[r]. Outputs are held to the bounds of
kda_chunk_fwd_varlen (this entry runs the fp32 token recurrence for every dtype,
so the fp32 bound 1e-4 RMS applies to fp32 outputs of either input dtype); final
states to max|S - S_ref| <= 1e-4 RMS(S_ref) per (segment, head).
"""
import numpy as np
import pytest
import torch

import kda_segids_cu_gb300 as kda
import oracle
import synth
from tests.parity import check_kda_output
from tests.test_gpu_chunk import _small_random

pytestmark = pytest.mark.gpu


def _n_segments(seg, B):
    if seg is None:
        return B
    s = seg.cpu().numpy()
    prev = np.concatenate([np.zeros((s.shape[0], 1), s.dtype), s[:, :-1]], axis=1)
    start = (s != 0) & ((s != prev) | (np.arange(s.shape[1])[None, :] == 0))
    return int(start.sum())


def _check_states(fin, ref, label):
    fin = fin.double().cpu()
    for r in range(ref.shape[0]):
        for h in range(ref.shape[1]):
            rms = ref[r, h].pow(2).mean().sqrt().item()
            err = (fin[r, h] - ref[r, h]).abs().max().item()
            assert err <= 1e-4 * rms + 1e-30, f"{label}: state [{r},{h}] err {err:.3e} rms {rms:.3e}"


def _run(inp, B, T, init, n_state, out_dtype=None, seg="inputs"):
    s = inp.segment_ids if seg == "inputs" else seg
    o, fin = kda.kda_chunk_fwd_varlen_state(
        inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.g.cuda(), inp.beta.cuda(),
        None if s is None else s.cuda(), B=B, T=T,
        initial_state=None if init is None else init.cuda(), output_final_state=True,
        n_state=n_state, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return o, fin


@pytest.mark.parametrize("name", ["tiny", "b2"])
def test_states_match_oracle(name):
    wl = synth.WORKLOADS[name]
    inp = synth.make_kda_inputs(wl)
    n = _n_segments(inp.segment_ids, wl.B)
    H, D = wl.H, wl.d_qk
    init = torch.randn(n, H, D, D, generator=torch.Generator().manual_seed(7)) * 0.5
    ref, ref_fin = oracle.kda_fwd_state(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.segment_ids,
                                        wl.B, wl.T, initial_state=init, n_state=n,
                                        want_final=True)
    o32, fin = _run(inp, wl.B, wl.T, init, n, out_dtype=torch.float32)
    check_kda_output(o32, ref, inp.segment_ids, torch.float32, label=name + "/f32 out")
    _check_states(fin, ref_fin, name)
    o, fin2 = _run(inp, wl.B, wl.T, init, n)
    check_kda_output(o, ref, inp.segment_ids, wl.dtype, label=name)
    assert torch.equal(fin, fin2)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D", [64, 128])
def test_partial_slots_and_zero_state(dtype, D):
    """Segments past n_state start from zero and are not written; a zero initial
    state gives the plain entry point's result (fp32: the same kernel, bit for bit)."""
    B, T, H = 2, 150, 2
    inp = _small_random(B, T, H, D, dtype, seed=D, max_len=40, pad_prob=0.1)
    seg = inp.segment_ids
    n = _n_segments(seg, B)
    k = max(1, n // 2)
    init = torch.randn(k, H, D, D, generator=torch.Generator().manual_seed(1)) * 0.3
    ref, ref_fin = oracle.kda_fwd_state(inp.q, inp.k, inp.v, inp.g, inp.beta, seg, B, T,
                                        initial_state=init, n_state=k, want_final=True)
    o32, fin = _run(inp, B, T, init, k, out_dtype=torch.float32)
    check_kda_output(o32, ref, seg, torch.float32, label=f"partial D={D}")
    _check_states(fin, ref_fin, f"partial D={D}")
    zero = torch.zeros(n, H, D, D)
    oz, _ = _run(inp, B, T, zero, n, out_dtype=torch.float32)
    plain = kda.kda_chunk_fwd_varlen(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.g.cuda(),
                                     inp.beta.cuda(), seg.cuda(), B=B, T=T,
                                     out_dtype=torch.float32)
    if dtype == torch.float32:
        assert torch.equal(oz, plain)
    else:
        check_kda_output(oz, oracle.kda_fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, seg, B, T),
                         seg, torch.float32, label=f"zero state D={D}")
        check_kda_output(plain, oracle.kda_fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, seg, B, T),
                         seg, dtype, label=f"plain D={D}")


def test_chaining_on_gpu():
    """A document cut in two with part A's final state handed to part B is the uncut run."""
    T, H, D, m = 300, 2, 128, 131
    whole = torch.ones(1, T, dtype=torch.int32)
    cut = torch.tensor([[1] * m + [2] * (T - m)], dtype=torch.int32)
    inp = _small_random(1, T, H, D, torch.float32, seed=3)
    inp.segment_ids = whole
    init = torch.randn(1, H, D, D, generator=torch.Generator().manual_seed(2)) * 0.3
    o_w, f_w = _run(inp, 1, T, init, 1, seg=whole)
    _, f_a = _run(inp, 1, T, torch.cat([init, init]), 2, seg=cut)
    o_c, f_c = _run(inp, 1, T, torch.cat([init, f_a[:1].cpu()]), 2, seg=cut)
    rms = o_w.double().pow(2).mean().sqrt().item()
    assert (o_c.double() - o_w.double()).abs().max().item() <= 1e-5 * rms
    srms = f_w.double().pow(2).mean().sqrt().item()
    assert (f_c[1].double() - f_w[0].double()).abs().max().item() <= 1e-5 * srms


def test_segment_ids_none_ranks_rows():
    B, T, H, D = 3, 70, 1, 64
    ones = torch.ones(B, T, dtype=torch.int32)
    inp = _small_random(B, T, H, D, torch.float32, seed=5)
    inp.segment_ids = ones
    init = torch.randn(B, H, D, D, generator=torch.Generator().manual_seed(4))
    o1, f1 = _run(inp, B, T, init, B, seg=ones)
    on, fn = _run(inp, B, T, init, B, seg=None)
    assert torch.equal(o1, on) and torch.equal(f1, fn)
