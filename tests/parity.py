"""Comparison helpers for GPU-vs-oracle parity tests."""
from __future__ import annotations

import math

import torch

# Per-head bound max|o - o_ref| <= tol * RMS(o_ref), over real (non-padding) tokens.
TOL_BF16 = 2e-2
TOL_F32 = 1e-4


def tolerance(dtype: torch.dtype) -> float:
    return TOL_BF16 if dtype == torch.bfloat16 else TOL_F32


def check_kda_output(o_gpu: torch.Tensor, o_ref: torch.Tensor, seg: torch.Tensor | None,
                     dtype: torch.dtype, heads: list[int] | None = None, label: str = "") -> dict:
    """o_gpu [N, H, Dv], o_ref [N, H_sel, Dv] float64 for `heads`; `dtype` is the
    input dtype, which sets the tolerance.

    Real tokens, per head: |o - ref| <= tol * RMS(ref) elementwise, plus -- only
    when o is stored in bf16 -- half a bf16 ulp of o for its final rounding
    (rounding the exact result itself to bf16 already moves outliers of ~10x
    RMS by more than 2e-2 RMS). Padding tokens: exactly 0.
    Returns the worst ratio max|diff| / (tol * RMS) (storage rounding included).
    """
    stored_bf16 = o_gpu.dtype == torch.bfloat16
    o = o_gpu.detach().to("cpu", torch.float64)
    if heads is not None:
        o = o[:, heads]
    assert o.shape == o_ref.shape, (o.shape, o_ref.shape)
    assert torch.isfinite(o).all(), f"{label}: non-finite output"
    if seg is not None:
        real = (seg.reshape(-1).to("cpu") != 0)
    else:
        real = torch.ones(o.shape[0], dtype=torch.bool)
    tol = tolerance(dtype)
    worst = 0.0
    for h in range(o.shape[1]):
        ref = o_ref[real, h]
        got = o[real, h]
        if ref.numel() == 0:
            continue
        rms = ref.pow(2).mean().sqrt().item()
        diff = (got - ref).abs()
        allow = torch.full_like(diff, tol * rms)
        if stored_bf16:
            allow = allow + 0.5 * ulp(got, torch.bfloat16)
        excess = (diff - allow).max().item()
        err = diff.max().item()
        ratio = err / (tol * rms) if rms > 0 else (0.0 if err == 0 else math.inf)
        worst = max(worst, ratio)
        assert excess <= 0, (f"{label} head {h}: max|diff| {err:.3e} exceeds {tol} * RMS "
                             f"{rms:.3e}{' + half a bf16 ulp' if stored_bf16 else ''}")
    pad = ~real
    if pad.any():
        assert torch.count_nonzero(o[pad]).item() == 0, f"{label}: padding outputs not zero"
    return {"worst_ratio": worst}


def ulp(x: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    """Spacing of `dtype` numbers at |x| (float64 result)."""
    mant = 8 if dtype == torch.bfloat16 else 24
    a = x.abs().clamp_min(torch.finfo(dtype).tiny)
    e = torch.floor(torch.log2(a))
    return torch.pow(2.0, e - (mant - 1))


def check_conv_output(y_gpu: torch.Tensor, y_ref64: torch.Tensor, abs_terms: torch.Tensor,
                      dtype: torch.dtype, K: int, label: str = "") -> float:
    """Conv bound: |y - ref| <= ulp_dtype(ref) + K * 2^-23 * sum_j |w_j x_j|.

    The GPU sums K exact-or-fp32 products in fp32 (error <= K 2^-24 sum|w x|)
    and rounds once to dtype (<= 1/2 ulp, and at most 1 ulp with the fp32 error).
    Returns the fraction of elements that match the oracle's single rounding exactly.
    """
    y = y_gpu.detach().to("cpu", torch.float64)
    bound = ulp(y_ref64, dtype) + K * 2.0 ** -23 * abs_terms
    diff = (y - y_ref64).abs()
    bad = diff > bound
    assert not bad.any(), f"{label}: {int(bad.sum())} elements outside the bound, worst " \
                          f"{(diff - bound).max().item():.3e}"
    exact = (y == y_ref64.to(dtype).to(torch.float64)).double().mean().item()
    return exact
