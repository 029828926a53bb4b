"""A CPU restatement of the chunked KDA forward used by the tensor-core kernel.

Not the oracle: this is the chunk algebra (64-token chunks, per-token decay
factors, segment masks, carried state) written out in numpy float64, with
optional rounding to bf16 at the points where the kernel stores bf16 tensor-core
operands. The tests use it to check that the algebra reproduces the oracle's
token recurrence to rounding error (fp64) and to bound what bf16 operand
rounding alone costs, separately from the CUDA code.
"""
from __future__ import annotations

import numpy as np
import torch

C = 64


def _bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16) \
        .to(torch.float64).numpy()


def chunked_forward(q, k, v, g, beta, seg, B, T, scale=1.0, round_bf16=False,
                    ref_mode="last"):
    """q, k, g: [N, H, Dk]; v: [N, H, Dv]; beta: [N, H]; seg: [B, T] or None.

    Every row of the flattened sequence is walked chunk by chunk on the global
    64-token grid; state carries across chunk edges, masks handle starts inside
    a chunk. round_bf16 rounds Qt, Kt, Qd, beta*V, A and S_in to bf16.
    """
    f = (lambda t: t.detach().to(torch.float64).numpy()) if isinstance(q, torch.Tensor) else np.asarray
    q, k, v, g, beta = (f(t) for t in (q, k, v, g, beta))
    N, H, Dk = q.shape
    Dv = v.shape[-1]
    if seg is None:
        ids = np.ones(N, dtype=np.int64)
    else:
        ids = (seg.numpy() if isinstance(seg, torch.Tensor) else np.asarray(seg)).reshape(-1)
    p = np.arange(N)
    valid_all = ids != 0
    prev = np.concatenate([[0], ids[:-1]])
    start_all = valid_all & ((p % T == 0) | (ids != prev))
    rnd = _bf16 if round_bf16 else (lambda x: x)
    o = np.zeros((N, H, Dv))
    n_chunks = (N + C - 1) // C
    for h in range(H):
        S = np.zeros((Dk, Dv))
        for c in range(n_chunks):
            lo_p, hi_p = c * C, min((c + 1) * C, N)
            n = hi_p - lo_p
            valid = np.zeros(C, bool)
            start = np.zeros(C, bool)
            valid[:n] = valid_all[lo_p:hi_p]
            start[:n] = start_all[lo_p:hi_p]
            cut = np.nonzero(start | ~valid)[0]
            first_cut = cut[0] if len(cut) else C
            starts = np.nonzero(start)[0]
            last_start = starts[-1] if len(starts) else 0
            tail_live = valid[C - 1]
            gg = np.zeros((C, Dk))
            gg[:n] = np.where(valid[:n, None], g[lo_p:hi_p, h], 0.0)
            e = np.exp(gg)
            P = np.cumprod(e, axis=0)                      # P_i = prod_{u<=i} e_u
            R = np.ones((C, Dk))
            R[:-1] = np.cumprod(e[::-1], axis=0)[::-1][1:]  # R_j = prod_{u>j} e_u
            qq = np.zeros((C, Dk)); kk = np.zeros((C, Dk)); vv = np.zeros((C, Dv)); bb = np.zeros(C)
            qq[:n], kk[:n], vv[:n], bb[:n] = q[lo_p:hi_p, h], k[lo_p:hi_p, h], v[lo_p:hi_p, h], beta[lo_p:hi_p, h]
            rows = np.arange(C)
            Qd = np.where((valid & (rows < first_cut))[:, None], qq * P, 0.0)
            Qt = np.where(valid[:, None], qq * P / P[-1], 0.0)
            Kt = np.where(valid[:, None], kk * R, 0.0)
            Kh = np.where((valid & (rows >= last_start) & tail_live)[:, None], Kt, 0.0)
            bV = np.where(valid[:, None], bb[:, None] * vv, 0.0)
            A = rnd(Qt) @ rnd(Kt).T
            lo = np.zeros(C, int)
            for i in range(C):
                s = np.nonzero(start[: i + 1])[0]
                lo[i] = s[-1] if len(s) else 0
            jj = np.arange(C)[None, :]
            mask = valid[:, None] & (jj >= lo[:, None]) & (jj <= rows[:, None])
            A = np.where(mask, A, 0.0)
            read_state = first_cut > 0 and c > 0
            carry = first_cut == C and c > 0
            O = rnd(A) @ rnd(bV)
            if read_state:
                O = O + rnd(Qd) @ rnd(S)
            S_new = rnd(Kh).T @ rnd(bV)
            if carry:
                S_new = S_new + P[-1][:, None] * S
            S = S_new
            o[lo_p:hi_p, h] = scale * O[:n]
    return torch.from_numpy(o)
