"""GPU parity for kda_chunk_bwd_varlen's fp32 walks (method="walk").

The walks run in fp32 arithmetic from the stored inputs, so every gradient is
held to the fp32 bound max|x - x_ref| <= 1e-4 RMS(x_ref) per head, over real
tokens, for either input dtype; gradients stored in bf16 get half a bf16 ulp more
for their rounding. Padding tokens get exact zeros. The tensor-core path (the
default for bf16 with 128-wide heads) is tested in test_gpu_bwd_tc.py.
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


def _d_o(inp, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(inp.v.shape, generator=gen).to(inp.v.dtype)


def _check(grads, refs, seg, heads=None, label=""):
    for name, got, ref in zip(NAMES, grads, refs):
        if name == "dbeta":
            got, ref = got.unsqueeze(-1), ref.unsqueeze(-1)
        check_kda_output(got, ref, seg, torch.float32, heads=heads, label=f"{label} {name}")


def _run(inp, B, T, d_o, scale=1.0, grad_dtype=None, seg="inputs", dev=None, method="walk"):
    s = inp.segment_ids if seg == "inputs" else seg
    to = (lambda t: t.cuda()) if dev is None else (lambda t: t)
    out = kda.kda_chunk_bwd_varlen(to(inp.q), to(inp.k), to(inp.v), to(inp.g), to(inp.beta),
                                   to(d_o), None if s is None else to(s), scale=scale, B=B, T=T,
                                   grad_dtype=grad_dtype, method=method)
    torch.cuda.synchronize()
    return out


def _oracle(inp, B, T, d_o, scale=1.0, heads=None):
    s = inp.segment_ids
    if heads is None:
        return oracle.kda_bwd(inp.q, inp.k, inp.v, inp.g, inp.beta, d_o, s, B, T, scale=scale)
    hs = torch.tensor(heads)
    pick = lambda t: t.index_select(1, hs.to(t.device)).cpu()     # noqa: E731
    return oracle.kda_bwd(pick(inp.q), pick(inp.k), pick(inp.v), pick(inp.g), pick(inp.beta),
                          pick(d_o), None if s is None else s.cpu(), B, T, scale=scale)


@pytest.mark.parametrize("name", ["tiny", "b2"])
def test_small_workloads(name):
    wl = synth.WORKLOADS[name]
    inp = synth.make_kda_inputs(wl)
    d_o = _d_o(inp, 1)
    ref = _oracle(inp, wl.B, wl.T, d_o, scale=0.9)
    _check(_run(inp, wl.B, wl.T, d_o, scale=0.9, grad_dtype=torch.float32), ref,
           inp.segment_ids, label=name + "/f32")
    g_in = _run(inp, wl.B, wl.T, d_o, scale=0.9)
    assert all(t.dtype == wl.dtype for t in g_in)
    _check(g_in, ref, inp.segment_ids, label=name)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D", [64, 128])
def test_boundary_sweep(dtype, D):
    """Ragged T, several windows, length-1 documents, padding, arbitrary ids, None."""
    cases = [
        dict(B=1, T=64 * 3 + 17, max_len=70),
        dict(B=3, T=100, max_len=9, pad_prob=0.25),
        dict(B=2, T=120, max_len=3, ids="arbitrary"),
        dict(B=1, T=130, max_len=1),
    ]
    for i, c in enumerate(cases):
        B, T = c.pop("B"), c.pop("T")
        inp = _small_random(B, T, 2, D, dtype, seed=300 + 10 * D + i, **c)
        d_o = _d_o(inp, i)
        _check(_run(inp, B, T, d_o, scale=0.5, grad_dtype=torch.float32),
               _oracle(inp, B, T, d_o, scale=0.5), inp.segment_ids, label=f"case{i}")
    inp = _small_random(2, 90, 2, D, dtype, seed=7)
    d_o = _d_o(inp, 9)
    a = _run(inp, 2, 90, d_o, seg=None)
    b = _run(inp, 2, 90, d_o, seg=torch.ones(2, 90, dtype=torch.int32))
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_ling3_sampled_heads():
    wl = synth.WORKLOADS["ling3"]
    inp = synth.make_kda_inputs(wl, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(5)
    d_o = torch.randn(inp.v.shape, device="cuda", generator=gen).to(wl.dtype)
    heads = [0, 11]
    grads = _run(inp, wl.B, wl.T, d_o, grad_dtype=torch.float32, dev="cuda")
    _check(grads, _oracle(inp, wl.B, wl.T, d_o, heads=heads), inp.segment_ids.cpu(),
           heads=heads, label="ling3")


def test_autograd_function():
    """kda_varlen's backward is kda_chunk_bwd_varlen, bit for bit, and its forward is
    kda_chunk_fwd_varlen."""
    B, T, H, D = 2, 150, 2, 128
    inp = _small_random(B, T, H, D, torch.bfloat16, seed=4, max_len=60, pad_prob=0.1)
    seg = inp.segment_ids.cuda()
    leaves = [t.cuda().requires_grad_(True) for t in (inp.q, inp.k, inp.v, inp.g, inp.beta)]
    o = kda.kda_varlen(*leaves, seg, scale=0.8)
    d_o = _d_o(inp, 3).cuda()
    o.backward(d_o)
    direct = kda.kda_chunk_bwd_varlen(*[t.detach() for t in leaves], d_o, seg, scale=0.8)
    for leaf, ref in zip(leaves, direct):
        assert torch.equal(leaf.grad, ref)
    plain = kda.kda_chunk_fwd_varlen(*[t.detach() for t in leaves], seg, scale=0.8)
    assert torch.equal(o.detach(), plain)
