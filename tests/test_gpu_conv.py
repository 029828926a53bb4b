"""GPU parity: kda_short_conv_varlen against the oracle's fp64 sum rounded once.

Bound (derived in tests/parity.py): |y - ref| <= ulp(ref) + K 2^-23 sum|w x|.
"""
import numpy as np
import pytest
import torch

import kda_segids_cu_gb300 as kda
import oracle
import synth
from tests.parity import check_conv_output

pytestmark = pytest.mark.gpu


def _run(x, w, seg, K, label, row_subset=None):
    y = kda.kda_short_conv_varlen(x.cuda(), w.cuda(), None if seg is None else seg.cuda())
    torch.cuda.synchronize()
    xs, ys, ss = x, y.cpu(), seg
    if row_subset is not None:
        xs, ys = x[row_subset], ys[row_subset]
        ss = None if seg is None else seg[row_subset]
    ref = oracle.short_conv(xs, w, ss, out_dtype=torch.float64)
    absr = oracle.short_conv(xs.abs(), w.abs(), ss, out_dtype=torch.float64)
    exact = check_conv_output(ys, ref, absr, x.dtype, K, label)
    return exact


@pytest.mark.parametrize("name", ["tiny", "b2"])
def test_workloads_full(name):
    wl = synth.WORKLOADS[name]
    ci = synth.make_conv_inputs(wl)
    exact = _run(ci.x, ci.w, ci.segment_ids, wl.k_conv, name)
    if wl.dtype == torch.bfloat16:
        # bf16 products are exact in fp32: nearly every output is the correctly rounded sum
        assert exact > 0.99


@pytest.mark.parametrize("name", ["ling3", "short", "long"])
def test_workloads_large_feature_sample(name):
    # full token range, a slice of 64 features (the kernel treats features independently)
    wl = synth.WORKLOADS[name]
    ci = synth.make_conv_inputs(wl, device="cuda")
    F = ci.x.shape[-1]
    y = kda.kda_short_conv_varlen(ci.x, ci.w, ci.segment_ids)
    torch.cuda.synchronize()
    for f0 in (0, F - 64):
        xs = ci.x[..., f0:f0 + 64].cpu()
        ws = ci.w[:, f0:f0 + 64].cpu()
        seg = ci.segment_ids.cpu()
        ref = oracle.short_conv(xs, ws, seg, out_dtype=torch.float64)
        absr = oracle.short_conv(xs.abs(), ws.abs(), seg, out_dtype=torch.float64)
        exact = check_conv_output(y[..., f0:f0 + 64].cpu(), ref, absr, xs.dtype, wl.k_conv,
                                  f"{name}[{f0}]")
        assert exact > 0.99


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("K", [1, 2, 3, 4, 5, 8])
def test_widths_and_segments(dtype, K):
    rng = np.random.default_rng(K)
    g = torch.Generator().manual_seed(K)
    B, T, F = 3, 101, 64
    seg = torch.from_numpy(synth.random_segment_ids(rng, B, T, max_len=7, pad_prob=0.2))
    x = torch.randn(B, T, F, generator=g).to(dtype)
    w = (torch.randn(K, F, generator=g) * 0.5).to(dtype)
    _run(x, w, seg, K, f"K={K}")
    _run(x, w, None, K, f"K={K} no ids")


def test_edges():
    g = torch.Generator().manual_seed(0)
    for (B, T, F) in [(1, 1, 8), (2, 17, 8), (1, 15, 16), (1, 16, 24), (4, 33, 2048)]:
        x = torch.randn(B, T, F, generator=g).bfloat16()
        w = torch.randn(4, F, generator=g).bfloat16()
        seg = torch.ones(B, T, dtype=torch.int32)
        _run(x, w, seg, 4, f"{B}x{T}x{F}")
    # length-1 documents: y = w[0] * x, bit-exact (one product, one rounding)
    x = torch.randn(1, 64, 16, generator=g).bfloat16()
    w = torch.randn(4, 16, generator=g).bfloat16()
    seg = torch.arange(1, 65, dtype=torch.int32)[None]
    y = kda.kda_short_conv_varlen(x.cuda(), w.cuda(), seg.cuda()).cpu()
    assert torch.equal(y, (x.double() * w[0].double()).bfloat16())
