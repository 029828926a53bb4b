"""GPU parity for the tensor-core backward (kda_chunk_bwd_varlen, method="auto", bf16
inputs with d_qk = d_v = 128).

Its operands are bf16 (the decayed ones as hi + lo pairs) with fp32 accumulation, like
the forward kernel's, so every gradient is held to the bf16 bound of the forward's output,
max|x - x_ref| <= 2e-2 RMS(x_ref) per head over real tokens (plus half a bf16 ulp when the
gradient is stored in bf16); padding tokens get exact zeros. The oracle is the fp64
derivative of the token recurrence (oracle.kda_bwd).
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

NAMES = ("dq", "dk", "dv", "dg", "dbeta")


def _d_o(shape, seed, dtype=torch.bfloat16):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=gen).to(dtype)


def _check(grads, refs, seg, heads=None, label=""):
    worst = {}
    for name, got, ref in zip(NAMES, grads, refs):
        if name == "dbeta":
            got, ref = got.unsqueeze(-1), ref.unsqueeze(-1)
        r = check_kda_output(got, ref, seg, torch.bfloat16, heads=heads, label=f"{label} {name}")
        worst[name] = r["worst_ratio"]
    return worst


def _gpu(inp, B, T, d_o, scale=1.0, grad_dtype=None, method="auto", seg="inputs", status=None):
    s = inp.segment_ids if seg == "inputs" else seg
    out = kda.kda_chunk_bwd_varlen(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.g.cuda(),
                                   inp.beta.cuda(), d_o.cuda(), None if s is None else s.cuda(),
                                   scale=scale, B=B, T=T, grad_dtype=grad_dtype, method=method,
                                   status=status, check=None if status is None else False)
    torch.cuda.synchronize()
    return out


def _ref(inp, B, T, d_o, scale=1.0):
    return oracle.kda_bwd(inp.q, inp.k, inp.v, inp.g, inp.beta, d_o, inp.segment_ids, B, T,
                          scale=scale)


def test_boundary_sweep():
    """Ragged T, several chunks, long and length-1 documents, interior and leading padding,
    arbitrary ids; fp32 and bf16 gradients."""
    cases = [
        dict(B=1, T=64 * 5 + 17, max_len=70),
        dict(B=3, T=100, max_len=9, pad_prob=0.25),
        dict(B=2, T=200, max_len=3, ids="arbitrary"),
        dict(B=1, T=333, max_len=200, pad_prob=0.1),
        dict(B=1, T=130, max_len=1),
        dict(B=2, T=64 * 9, max_len=400),
    ]
    for i, c in enumerate(cases):
        B, T = c.pop("B"), c.pop("T")
        inp = _small_random(B, T, 2, 128, torch.bfloat16, seed=700 + i, **c)
        d_o = _d_o(inp.v.shape, 50 + i)
        ref = _ref(inp, B, T, d_o, scale=0.5)
        _check(_gpu(inp, B, T, d_o, scale=0.5, grad_dtype=torch.float32), ref, inp.segment_ids,
               label=f"case{i}/f32")
        _check(_gpu(inp, B, T, d_o, scale=0.5), ref, inp.segment_ids, label=f"case{i}")


def test_every_boundary_offset():
    """One boundary at each in-chunk offset 0..63, in a chunk between two carried chunks, so
    that the carried-in state, the state carried out and the cut all meet in one chunk."""
    T = 64 * 3
    B = 64
    seg = torch.ones(B, T, dtype=torch.int32)
    for b in range(B):
        seg[b, 64 + b:] = 2
    inp = _small_random(B, T, 2, 128, torch.bfloat16, seed=11)
    inp = synth.KdaInputs(inp.q, inp.k, inp.v, inp.g, inp.beta, seg, [])
    d_o = _d_o(inp.v.shape, 12)
    _check(_gpu(inp, B, T, d_o, scale=0.7), _ref(inp, B, T, d_o, scale=0.7), seg,
           label="offsets")


def test_long_segment_and_none():
    """One segment over 40 chunks (the scans' chains); segment_ids None equals all-ones."""
    B, T = 1, 64 * 40
    inp = _small_random(B, T, 2, 128, torch.bfloat16, seed=21, max_len=T)
    inp = synth.KdaInputs(inp.q, inp.k, inp.v, inp.g, inp.beta,
                          torch.ones(B, T, dtype=torch.int32), [])
    d_o = _d_o(inp.v.shape, 22)
    a = _gpu(inp, B, T, d_o)
    _check(a, _ref(inp, B, T, d_o), inp.segment_ids, label="long")
    b = _gpu(inp, B, T, d_o, seg=None)
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_long_chains_in_pieces():
    """Chains longer than 32 chunks run in 16-chunk pieces (end states from zero, a combine
    pass, then the export from the true piece starts): a 70-chunk document, a ragged tail, and
    a row whose documents end inside chunks, with padding between them."""
    B, T = 2, 64 * 70 + 13
    seg = torch.ones(B, T, dtype=torch.int32)
    seg[1, 2000:2050] = 0
    seg[1, 2050:4100] = 2
    seg[1, 4100:] = 3
    inp = _small_random(B, T, 2, 128, torch.bfloat16, seed=61, max_len=T)
    inp = synth.KdaInputs(inp.q, inp.k, inp.v, inp.g, inp.beta, seg, [])
    d_o = _d_o(inp.v.shape, 62)
    _check(_gpu(inp, B, T, d_o, scale=0.6, grad_dtype=torch.float32),
           _ref(inp, B, T, d_o, scale=0.6), seg, label="pieces")


def test_deterministic_and_agrees_with_walks():
    inp = _small_random(2, 300, 3, 128, torch.bfloat16, seed=31, max_len=120, pad_prob=0.05)
    d_o = _d_o(inp.v.shape, 32)
    a = _gpu(inp, 2, 300, d_o, grad_dtype=torch.float32)
    b = _gpu(inp, 2, 300, d_o, grad_dtype=torch.float32)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    w = _gpu(inp, 2, 300, d_o, grad_dtype=torch.float32, method="walk")
    # both paths hold their bounds against the oracle; the walks are the stricter one
    ref = _ref(inp, 2, 300, d_o)
    _check(a, ref, inp.segment_ids, label="tc")
    for name, got, r in zip(NAMES, w, ref):
        if name == "dbeta":
            got, r = got.unsqueeze(-1), r.unsqueeze(-1)
        check_kda_output(got, r, inp.segment_ids, torch.float32, label=f"walk {name}")


@pytest.mark.parametrize("name", ["ling3", "short"])
def test_full_size_sampled_heads(name):
    """The full-size workloads on the GPU; the oracle checks sampled heads."""
    wl = synth.WORKLOADS[name]
    inp = synth.make_kda_inputs(wl, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(5)
    d_o = torch.randn(inp.v.shape, device="cuda", generator=gen).to(wl.dtype)
    grads = kda.kda_chunk_bwd_varlen(inp.q, inp.k, inp.v, inp.g, inp.beta, d_o, inp.segment_ids,
                                     B=wl.B, T=wl.T, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    heads = [0, 7]
    hs = torch.tensor(heads, device="cuda")
    pick = lambda t: t.index_select(1, hs).cpu()     # noqa: E731
    ref = oracle.kda_bwd(pick(inp.q), pick(inp.k), pick(inp.v), pick(inp.g), pick(inp.beta),
                         pick(d_o), inp.segment_ids.cpu(), wl.B, wl.T)
    _check(grads, ref, inp.segment_ids.cpu(), heads=heads, label=name)


def test_strong_decay_takes_the_fp32_redo():
    """Chunks whose log-decay falls below -80 on some channel are outside the factorised
    form's range: the gradient kernel lists them and an fp32 token walk over each such chunk
    (from the stored S_in and D_end) rewrites their gradients. A segment boundary falls inside
    the strong chunks, and one head stays in range."""
    B, T = 2, 64 * 4
    inp = _small_random(B, T, 2, 128, torch.bfloat16, seed=41, max_len=T)
    seg = torch.ones(B, T, dtype=torch.int32)
    seg[0, 100:] = 2
    seg[1, 150:200] = 0                               # padding inside a strong chunk
    seg[1, 200:] = 3
    g = inp.g.clone().view(B, T, 2, 128)
    g[0, 64:192, 0, 5] = -3.0                         # 64 x -3 = -192 per chunk, head 0
    g[1, 128:256, 0, 77] = -2.0
    inp = synth.KdaInputs(inp.q, inp.k, inp.v, g.view(B * T, 2, 128), inp.beta, seg, [])
    d_o = _d_o(inp.v.shape, 42)
    ref = _ref(inp, B, T, d_o, scale=0.8)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _gpu(inp, B, T, d_o, scale=0.8, grad_dtype=torch.float32, status=status)
    assert int(status.item()) == 0
    _check(got, ref, seg, label="redo")
    w = _gpu(inp, B, T, d_o, scale=0.8, grad_dtype=torch.float32, method="walk")
    for name, gw, r in zip(NAMES, w, ref):
        if name == "dbeta":
            gw, r = gw.unsqueeze(-1), r.unsqueeze(-1)
        check_kda_output(gw, r, seg, torch.float32, label=f"walk {name}")
