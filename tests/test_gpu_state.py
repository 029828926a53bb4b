"""GPU parity for kda_chunk_fwd_varlen_state (per-segment initial and final state).

Segment r (flattened token order) starts from initial_state[r] and returns its
state after its last token in final[r]. Outputs are held to the bounds of
kda_chunk_fwd_varlen for the input dtype. bf16 inputs with 128-wide heads run the
tensor-core chunked form plus the state pass, so they get the bf16 bound for
either output dtype. The other cases run the fp32 token recurrence, so their fp32
outputs get the fp32 bound of 1e-4 RMS. Final states are held to
max|S - S_ref| <= 1e-4 RMS(S_ref) per (segment, head).
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


def _first_chunk_rows(seg):
    """Mask of the flattened tokens that lie in their segment's first 64-token chunk."""
    s = seg.reshape(-1).numpy()
    B, T = seg.shape
    out = np.zeros(s.shape[0], bool)
    p = 0
    while p < s.shape[0]:
        if s[p] == 0:
            p += 1
            continue
        e = p + 1
        while e < s.shape[0] and s[e] == s[p] and e % T != 0:
            e += 1
        out[p:min(e, (p // 64 + 1) * 64)] = True
        p = e
    return torch.from_numpy(out).cuda()


def _check_states(fin, ref, label):
    fin = fin.double().cpu()
    for r in range(ref.shape[0]):
        for h in range(ref.shape[1]):
            rms = ref[r, h].pow(2).mean().sqrt().item()
            err = (fin[r, h] - ref[r, h]).abs().max().item()
            assert err <= 1e-4 * rms + 1e-30, f"{label}: state [{r},{h}] err {err:.3e} rms {rms:.3e}"


def _o_bound(dtype, D):
    """Input dtype whose bound an fp32 output of the state call meets."""
    return dtype if (dtype == torch.bfloat16 and D == 128) else torch.float32


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
    check_kda_output(o32, ref, inp.segment_ids, _o_bound(wl.dtype, D), label=name + "/f32 out")
    _check_states(fin, ref_fin, name)
    o, fin2 = _run(inp, wl.B, wl.T, init, n)
    check_kda_output(o, ref, inp.segment_ids, wl.dtype, label=name)
    assert torch.equal(fin, fin2)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D", [64, 128])
def test_partial_slots_and_zero_state(dtype, D):
    """Segments past n_state start from zero and are not written. A zero initial state
    gives the plain entry point's result bit for bit: the same kernels, and on the
    tensor-core path a seed of zeros adds nothing. The exception is the rows of each
    segment in the chunk where it starts, which the state pass rewrites in fp32."""
    B, T, H = 2, 150, 2
    inp = _small_random(B, T, H, D, dtype, seed=D, max_len=40, pad_prob=0.1)
    seg = inp.segment_ids
    n = _n_segments(seg, B)
    k = max(1, n // 2)
    init = torch.randn(k, H, D, D, generator=torch.Generator().manual_seed(1)) * 0.3
    ref, ref_fin = oracle.kda_fwd_state(inp.q, inp.k, inp.v, inp.g, inp.beta, seg, B, T,
                                        initial_state=init, n_state=k, want_final=True)
    o32, fin = _run(inp, B, T, init, k, out_dtype=torch.float32)
    check_kda_output(o32, ref, seg, _o_bound(dtype, D), label=f"partial D={D}")
    _check_states(fin, ref_fin, f"partial D={D}")
    zero = torch.zeros(n, H, D, D)
    oz, _ = _run(inp, B, T, zero, n, out_dtype=torch.float32)
    plain = kda.kda_chunk_fwd_varlen(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.g.cuda(),
                                     inp.beta.cuda(), seg.cuda(), B=B, T=T,
                                     out_dtype=torch.float32)
    if dtype == torch.bfloat16 and D == 128:
        keep = ~_first_chunk_rows(seg)
        assert torch.equal(oz[keep], plain[keep])
        check_kda_output(oz, oracle.kda_fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, seg, B, T),
                         seg, dtype, label=f"zero state D={D}")
    else:
        assert torch.equal(oz, plain)
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


def _layout_inputs(kind, seed):
    """bf16, 128-wide heads: layouts that exercise every case of the state split."""
    if kind == "long":          # documents across many chunks, one ending on a chunk edge
        B, T = 1, 1100
        ids = [1] * 600 + [2] * 104 + [3] * 396
    elif kind == "edges":       # length-1 documents on both sides of chunk edges
        ids = [1] * 63 + [2] + [3] + [4] * 62 + [5] + [6] * 129 + [7] * 64
        B, T = 1, len(ids)
    elif kind == "aligned":     # documents on chunk edges, then padding
        B, T = 2, 256
        ids = [1] * 64 + [2] * 128 + [0] * 64 + [3] * 192 + [4] * 64
    else:
        ids = None
    if ids is not None:
        inp = _small_random(B, T, 3, 128, torch.bfloat16, seed=seed)
        inp.segment_ids = torch.tensor(ids, dtype=torch.int32).reshape(B, T)
        return inp, B, T
    B, T = 2, 300               # many short documents per chunk, padding, ragged T
    return _small_random(B, T, 3, 128, torch.bfloat16, seed=seed, max_len=20, pad_prob=0.1), B, T


@pytest.mark.parametrize("kind", ["long", "edges", "aligned", "short"])
@pytest.mark.parametrize("mode", ["init+final", "init", "final", "half-slots"])
def test_tensor_core_state_layouts(kind, mode):
    inp, B, T = _layout_inputs(kind, seed=len(kind) + 3 * len(mode))
    n = _n_segments(inp.segment_ids, B)
    H, D = 3, 128
    n_state = max(1, n // 2) if mode == "half-slots" else n
    gen = torch.Generator().manual_seed(n_state)
    init = torch.randn(n_state, H, D, D, generator=gen) * 0.5 if mode != "final" else None
    want = mode != "init"
    ref, ref_fin = oracle.kda_fwd_state(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.segment_ids,
                                        B, T, initial_state=init, n_state=n_state,
                                        want_final=want)
    o, fin = kda.kda_chunk_fwd_varlen_state(
        inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.g.cuda(), inp.beta.cuda(),
        inp.segment_ids.cuda(), B=B, T=T, initial_state=None if init is None else init.cuda(),
        output_final_state=want, n_state=n_state)
    torch.cuda.synchronize()
    check_kda_output(o, ref, inp.segment_ids, torch.bfloat16, label=f"{kind}/{mode}")
    if want:
        _check_states(fin, ref_fin, f"{kind}/{mode}")


def test_tensor_core_chaining():
    """bf16, 128-wide heads: a document cut in two (mid-chunk), with part A's final state
    handed to part B, gives the uncut document's outputs and final state."""
    T, H, D, m = 700, 2, 128, 333
    inp = _small_random(1, T, H, D, torch.bfloat16, seed=9)
    whole = torch.ones(1, T, dtype=torch.int32)
    cut = torch.tensor([[1] * m + [2] * (T - m)], dtype=torch.int32)
    init = torch.randn(1, H, D, D, generator=torch.Generator().manual_seed(2)) * 0.3
    ref, ref_fin = oracle.kda_fwd_state(inp.q, inp.k, inp.v, inp.g, inp.beta, whole, 1, T,
                                        initial_state=init, n_state=1, want_final=True)
    _, f_a = _run(inp, 1, T, torch.cat([init, init]), 2, seg=cut)
    o_c, f_c = _run(inp, 1, T, torch.cat([init, f_a[:1].cpu()]), 2, seg=cut)
    check_kda_output(o_c, ref, whole, torch.bfloat16, label="chained")
    _check_states(f_c[1:], ref_fin, "chained")


@pytest.mark.parametrize("name,heads", [("ling3", [0, 9]), ("short", [3]), ("long", [0, 31])])
def test_large_workloads_state_sampled_heads(name, heads):
    """Full-size workloads in bench.py's configuration (every segment with an initial and
    a final state), held to the oracle on sampled heads: outputs on every token of those
    heads, final states of every segment."""
    wl = synth.WORKLOADS[name]
    inp = synth.make_kda_inputs(wl, device="cuda")
    seg = inp.segment_ids
    n = _n_segments(seg.cpu() if seg is not None else None, wl.B)
    H, D = wl.H, wl.d_qk
    gen = torch.Generator(device="cuda").manual_seed(17)
    init = torch.randn(n, H, D, D, device="cuda", generator=gen) * 0.1
    o, fin = kda.kda_chunk_fwd_varlen_state(inp.q, inp.k, inp.v, inp.g, inp.beta, seg, B=wl.B,
                                            T=wl.T, initial_state=init, output_final_state=True)
    torch.cuda.synchronize()
    hs = torch.tensor(heads, device="cuda")
    pick = lambda t: t.index_select(1, hs).cpu()     # noqa: E731
    ref, ref_fin = oracle.kda_fwd_state(pick(inp.q), pick(inp.k), pick(inp.v), pick(inp.g),
                                        pick(inp.beta), None if seg is None else seg.cpu(),
                                        wl.B, wl.T, initial_state=pick(init), n_state=n,
                                        want_final=True)
    check_kda_output(o, ref, None if seg is None else seg.cpu(), wl.dtype, heads=heads,
                     label=name)
    _check_states(pick(fin), ref_fin, name)


def test_tensor_core_state_segment_ids_none():
    """bf16, 128-wide heads, segment_ids=None: row b is segment b. Equal bit for bit to
    all-ones ids, and held to the oracle."""
    B, T, H, D = 3, 200, 2, 128
    inp = _small_random(B, T, H, D, torch.bfloat16, seed=21)
    ones = torch.ones(B, T, dtype=torch.int32)
    inp.segment_ids = ones
    init = torch.randn(B, H, D, D, generator=torch.Generator().manual_seed(8)) * 0.3
    o1, f1 = _run(inp, B, T, init, B, seg=ones)
    on, fn = _run(inp, B, T, init, B, seg=None)
    assert torch.equal(o1, on) and torch.equal(f1, fn)
    ref, ref_fin = oracle.kda_fwd_state(inp.q, inp.k, inp.v, inp.g, inp.beta, None, B, T,
                                        initial_state=init, n_state=B, want_final=True)
    check_kda_output(on, ref, None, torch.bfloat16, label="None")
    _check_states(fn, ref_fin, "None")
