"""Pins for the oracle's segment-masked causal short convolution (no GPU).

Definition: RFC-0025 "支持 Attention Varlen 功能并对齐 Loss", 方案 §3
"ShortConvolution segment 边界 mask". Pins: without segment ids it equals
torch's depthwise conv1d (a library routine) with the taps time-reversed and
K-1 zeros of left padding; a packed row equals the concatenation of each
document convolved alone; a length-1 document gives w[0]*x; an impulse
returns the weights, cut where its document ends; padding destinations only see
padding sources.
"""
import numpy as np
import pytest
import torch

import oracle
import synth


def _torch_conv_ref(x, w):
    # x [B, T, F] float64, w [K, F]: y[t] = sum_j w[j] x[t-j]
    B, T, F = x.shape
    K = w.shape[0]
    weight = torch.flip(w, dims=[0]).t().reshape(F, 1, K)  # conv1d is a correlation
    xp = torch.nn.functional.pad(x.permute(0, 2, 1), (K - 1, 0))
    return torch.nn.functional.conv1d(xp, weight, groups=F).permute(0, 2, 1)


@pytest.mark.parametrize("K", [1, 2, 4, 7])
def test_no_segments_equals_library_conv1d(K):
    g = torch.Generator().manual_seed(K)
    x = torch.randn(2, 37, 9, generator=g, dtype=torch.float64)
    w = torch.randn(K, 9, generator=g, dtype=torch.float64)
    y = oracle.short_conv(x, w, None, out_dtype=torch.float64)
    ref = _torch_conv_ref(x, w)
    assert torch.allclose(y, ref, rtol=1e-13, atol=1e-13)
    # a single segment covering each row gives the same result
    seg = torch.ones(2, 37, dtype=torch.int32)
    assert torch.equal(oracle.short_conv(x, w, seg, out_dtype=torch.float64), y)


def test_packed_equals_concatenated_documents():
    rng = np.random.default_rng(11)
    g = torch.Generator().manual_seed(11)
    for trial in range(20):
        T = int(rng.integers(5, 90))
        seg = synth.random_segment_ids(rng, 1, T, max_len=9)
        x = torch.randn(1, T, 6, generator=g, dtype=torch.float64)
        w = torch.randn(4, 6, generator=g, dtype=torch.float64)
        y = oracle.short_conv(x, w, torch.from_numpy(seg), out_dtype=torch.float64)
        t = 0
        while t < T:
            e = t + 1
            while e < T and seg[0, e] == seg[0, t]:
                e += 1
            alone = _torch_conv_ref(x[:, t:e], w)
            assert torch.allclose(y[:, t:e], alone, rtol=1e-13, atol=1e-13)
            t = e


def test_length_one_document_and_impulse():
    seg = torch.tensor([[1, 1, 1, 2, 3, 3, 3, 3, 3]], dtype=torch.int32)
    w = torch.tensor([[0.5], [0.25], [-2.0], [3.0]], dtype=torch.float64)
    x = torch.zeros(1, 9, 1, dtype=torch.float64)
    x[0, 3, 0] = 1.7                      # the length-1 document
    y = oracle.short_conv(x, w, seg, out_dtype=torch.float64)
    assert y[0, 3, 0].item() == 0.5 * 1.7
    assert torch.count_nonzero(y).item() == 1
    x = torch.zeros(1, 9, 1, dtype=torch.float64)
    x[0, 5, 0] = 1.0                      # impulse inside document 3 (starts at 4)
    y = oracle.short_conv(x, w, seg, out_dtype=torch.float64)
    assert y[0, :, 0].tolist() == [0, 0, 0, 0, 0, 0.5, 0.25, -2.0, 3.0]
    x = torch.zeros(1, 9, 1, dtype=torch.float64)
    x[0, 7, 0] = 1.0                      # near the row end: the response is cut there
    y = oracle.short_conv(x, w, seg, out_dtype=torch.float64)
    assert y[0, :, 0].tolist() == [0, 0, 0, 0, 0, 0, 0, 0.5, 0.25]
    # the same impulse one step after a boundary reaches no earlier token
    x = torch.zeros(1, 9, 1, dtype=torch.float64)
    x[0, 2, 0] = 1.0                      # last token of document 1
    y = oracle.short_conv(x, w, seg, out_dtype=torch.float64)
    assert y[0, :, 0].tolist() == [0, 0, 0.5, 0, 0, 0, 0, 0, 0]


def test_padding_destinations_see_only_padding():
    seg = torch.tensor([[1, 1, 0, 0, 2]], dtype=torch.int32)
    w = torch.ones(3, 1, dtype=torch.float64)
    x = torch.tensor([[[1.0], [2.0], [4.0], [8.0], [16.0]]], dtype=torch.float64)
    y = oracle.short_conv(x, w, seg, out_dtype=torch.float64)
    assert y[0, :, 0].tolist() == [1.0, 3.0, 4.0, 12.0, 16.0]


def test_rows_are_independent_and_rounding_is_single():
    seg = torch.tensor([[1, 1, 1], [1, 1, 1]], dtype=torch.int32)
    x = torch.tensor([[[1.0], [1.0], [1.0]], [[2.0], [2.0], [2.0]]], dtype=torch.float64)
    w = torch.tensor([[1.0], [1.0]], dtype=torch.float64)
    y = oracle.short_conv(x, w, seg, out_dtype=torch.float64)
    assert y[1, 0, 0].item() == 2.0       # row 1 does not see row 0's last token
    # bf16 output: the exact sum rounded once to nearest-even
    xb = torch.tensor([[[1.0], [2.0 ** -8]]], dtype=torch.bfloat16)
    wb = torch.tensor([[1.0], [1.0]], dtype=torch.bfloat16)
    yb = oracle.short_conv(xb, wb, torch.ones(1, 2, dtype=torch.int32))
    assert yb.dtype == torch.bfloat16
    assert yb[0, 1, 0].item() == 1.0      # 1 + 2^-8 ties to even (1.0) in bf16
