"""Seeded synthetic inputs for the packed (varlen) Kimi Delta Attention forward.

This module is shared by the CUDA-path tests, the oracle tests and the bench.
It draws document lengths, segment ids and tensor values with the shapes and
distributions of the workloads; it holds none of the method's arithmetic.

Workloads (shapes follow RFC-0026 "Ling3 KDA Varlen 支持", 背景 "当前 packing 状态":
8193-token samples, EOD-separated documents; the batch is flattened to
[1, B*T] as in RFC-0025 "支持 Attention Varlen 功能并对齐 Loss", 方案 §2):

  tiny   B=1 T=256    H=2  D=64  fp32  docs 100/37/119             max_segs 4
  b2     B=2 T=2048   H=8  D=128 bf16  geometric(mean 300) docs,   max_segs 64
                                       last 64 tokens of row 1 are padding (id 0)
  ling3  B=4 T=8192   H=16 D=128 bf16  lognormal(median 800, sigma 1) docs
                                       clipped to [1, 8192]        max_segs 128
  short  B=1 T=65536  H=16 D=128 bf16  uniform{1..64} docs         max_segs 4096
  long   B=1 T=131072 H=32 D=128 bf16  docs 65536/32768/24576/8192 max_segs 8

Values: q, k ~ N(0,1)/sqrt(64) then L2-normalised per (token, head); v ~ N(0,1);
g = -exp(N(-2, 0.5)) per (token, head, key channel); beta = sigmoid(N(0,1)) per
(token, head); conv input x ~ N(0,1) of shape [B, T, H*D_qk]; conv weights
N(0, 0.5) of shape [K_conv, H*D_qk]. Values are drawn in fp32 and rounded to
nearest-even into the workload dtype.

Segment ids restart at 1 in every row and increase by one per document; the
last document of a row is truncated at T.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    d_qk: int
    d_v: int
    dtype: torch.dtype
    max_segs: int
    doc_kind: str                    # "fixed" | "geometric" | "lognormal" | "uniform"
    doc_param: tuple = ()
    tail_pad_last_row: int = 0       # trailing padding tokens in the last row
    k_conv: int = 4
    segmented: bool = True           # False: segment_ids is None (one segment per row)

    @property
    def N(self) -> int:
        return self.B * self.T

    @property
    def F(self) -> int:
        return self.H * self.d_qk


WORKLOADS = {
    "tiny": Workload("tiny", 1, 256, 2, 64, 64, torch.float32, 4, "fixed", (100, 37, 119)),
    "b2": Workload("b2", 2, 2048, 8, 128, 128, torch.bfloat16, 64, "geometric", (300.0,),
                   tail_pad_last_row=64),
    "ling3": Workload("ling3", 4, 8192, 16, 128, 128, torch.bfloat16, 128, "lognormal",
                      (800.0, 1.0, 1, 8192)),
    "short": Workload("short", 1, 65536, 16, 128, 128, torch.bfloat16, 4096, "uniform", (1, 64)),
    "long": Workload("long", 1, 131072, 32, 128, 128, torch.bfloat16, 8, "fixed",
                     (65536, 32768, 24576, 8192)),
    "long_none": Workload("long_none", 1, 131072, 32, 128, 128, torch.bfloat16, 8, "fixed",
                          (131072,), segmented=False),
}

# Index of each workload in the fixed seed scheme: seed = 1000 + index.
WORKLOAD_INDEX = {"tiny": 1, "b2": 2, "ling3": 3, "short": 4, "long": 5, "long_none": 5}


def default_seed(name: str) -> int:
    return 1000 + WORKLOAD_INDEX[name]


def _row_doc_lengths(wl: Workload, rng: np.random.Generator, budget: int) -> list[int]:
    """Document lengths for one row, drawn until `budget` tokens are filled (last truncated)."""
    out: list[int] = []
    total = 0
    if wl.doc_kind == "fixed":
        for L in wl.doc_param:
            if total >= budget:
                break
            L = min(int(L), budget - total)
            out.append(L)
            total += L
        if total < budget:
            out.append(budget - total)
        return out
    while total < budget:
        if wl.doc_kind == "geometric":
            L = int(rng.geometric(1.0 / wl.doc_param[0]))
        elif wl.doc_kind == "lognormal":
            median, sigma, lo, hi = wl.doc_param
            L = int(round(math.exp(math.log(median) + sigma * rng.standard_normal())))
            L = max(lo, min(hi, L))
        elif wl.doc_kind == "uniform":
            lo, hi = wl.doc_param
            L = int(rng.integers(lo, hi + 1))
        else:
            raise ValueError(wl.doc_kind)
        L = min(L, budget - total)
        out.append(L)
        total += L
    return out


def make_segment_ids(wl: Workload, seed: int) -> tuple[np.ndarray, list[list[int]]]:
    """int32 [B, T] segment ids and the per-row real document lengths.

    Ids are 1, 2, 3, ... per row; padding is 0.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    seg = np.zeros((wl.B, wl.T), dtype=np.int32)
    lengths: list[list[int]] = []
    for b in range(wl.B):
        budget = wl.T - (wl.tail_pad_last_row if b == wl.B - 1 else 0)
        row = _row_doc_lengths(wl, rng, budget)
        if wl.doc_kind == "uniform" and b == 0 and 1 not in row and len(row) > 1:
            # the short-document workload must hold at least one length-1 document
            row[0] -= 1
            row.insert(0, 1)
            row = [L for L in row if L > 0]
        t = 0
        for i, L in enumerate(row):
            seg[b, t:t + L] = i + 1
            t += L
        lengths.append(row)
    return seg, lengths


def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 64 + stream)
    return g


def _l2norm_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


@dataclass
class KdaInputs:
    q: torch.Tensor          # [B*T, H, d_qk]
    k: torch.Tensor          # [B*T, H, d_qk]
    v: torch.Tensor          # [B*T, H, d_v]
    g: torch.Tensor          # [B*T, H, d_qk] log-decay (<= 0)
    beta: torch.Tensor       # [B*T, H]
    segment_ids: torch.Tensor | None   # [B, T] int32, or None
    doc_lengths: list = field(default_factory=list)


def make_kda_inputs(wl: Workload, seed: int | None = None, device="cpu",
                    heads: int | None = None) -> KdaInputs:
    """Inputs of the chunk forward in the flattened [B*T, H, D] layout.

    `heads` (optional) draws only that many heads; the values of head h do not
    depend on `heads` only in the sense that the recipe is the same.
    """
    seed = default_seed(wl.name) if seed is None else seed
    seg_np, lengths = make_segment_ids(wl, seed)
    H = wl.H if heads is None else heads
    N = wl.N
    gen = _gen(device, seed, 1)
    f32 = torch.float32

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=device, dtype=f32)

    q = _l2norm_rows(randn(N, H, wl.d_qk) / 8.0).to(wl.dtype)
    k = _l2norm_rows(randn(N, H, wl.d_qk) / 8.0).to(wl.dtype)
    v = randn(N, H, wl.d_v).to(wl.dtype)
    g = (-torch.exp(randn(N, H, wl.d_qk) * 0.5 - 2.0)).to(wl.dtype)
    beta = torch.sigmoid(randn(N, H)).to(wl.dtype)
    seg = torch.from_numpy(seg_np).to(device) if wl.segmented else None
    return KdaInputs(q, k, v, g, beta, seg, lengths)


@dataclass
class ConvInputs:
    x: torch.Tensor          # [B, T, F]
    w: torch.Tensor          # [K_conv, F]
    segment_ids: torch.Tensor | None


def make_conv_inputs(wl: Workload, seed: int | None = None, device="cpu",
                     features: int | None = None) -> ConvInputs:
    seed = default_seed(wl.name) if seed is None else seed
    seg_np, _ = make_segment_ids(wl, seed)
    F = wl.F if features is None else features
    gen = _gen(device, seed, 2)
    x = torch.randn(wl.B, wl.T, F, generator=gen, device=device,
                    dtype=torch.float32).to(wl.dtype)
    w = (torch.randn(wl.k_conv, F, generator=gen, device=device,
                     dtype=torch.float32) * 0.5).to(wl.dtype)
    seg = torch.from_numpy(seg_np).to(device) if wl.segmented else None
    return ConvInputs(x, w, seg)


def random_segment_ids(rng: np.random.Generator, B: int, T: int, max_len: int = 80,
                       pad_prob: float = 0.0, ids: str = "increasing") -> np.ndarray:
    """Small random segment-id arrays for sweeps: random document lengths in
    [1, max_len], optional padding runs, ids increasing from 1 per row (or
    arbitrary non-zero ids when ids == "arbitrary")."""
    seg = np.zeros((B, T), dtype=np.int32)
    for b in range(B):
        t = 0
        nxt = 1
        while t < T:
            L = int(rng.integers(1, max_len + 1))
            L = min(L, T - t)
            if pad_prob > 0 and rng.random() < pad_prob:
                seg[b, t:t + L] = 0
            else:
                if ids == "arbitrary":
                    seg[b, t:t + L] = int(rng.integers(1, 4))
                else:
                    seg[b, t:t + L] = nxt
                    nxt += 1
            t += L
    return seg
