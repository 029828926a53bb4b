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


def chunked_forward_state(q, k, v, g, beta, seg, B, T, init=None, n_state=0, want_final=False,
                          scale=1.0):
    """The per-segment state split of the bf16 path, in float64: the chunk walk above
    with the state seeded at the chunk where a segment starts (its initial state decayed
    to the chunk's end) and the state carried into the chunk where a segment ends kept
    aside; then the per-chunk pass that writes the rows of each segment in its first
    chunk whole and forms the final states. Segment r (flattened order) has slot r if
    r < n_state. Returns (o [N, H, Dv], final [n_state, H, Dk, Dv] or None)."""
    f = (lambda t: t.detach().to(torch.float64).numpy()) if isinstance(q, torch.Tensor) else np.asarray
    q, k, v, g, beta = (f(t) for t in (q, k, v, g, beta))
    S0 = None if init is None else f(init)
    N, H, Dk = q.shape
    Dv = v.shape[-1]
    ids = np.ones(N, dtype=np.int64) if seg is None else \
        (seg.numpy() if isinstance(seg, torch.Tensor) else np.asarray(seg)).reshape(-1)
    p = np.arange(N)
    valid_all = ids != 0
    prev = np.concatenate([[0], ids[:-1]])
    start_all = valid_all & ((p % T == 0) | (ids != prev))
    n_chunks = (N + C - 1) // C

    def chunk_masks(c):
        lo_p, hi_p = c * C, min((c + 1) * C, N)
        valid = np.zeros(C, bool)
        start = np.zeros(C, bool)
        valid[: hi_p - lo_p] = valid_all[lo_p:hi_p]
        start[: hi_p - lo_p] = start_all[lo_p:hi_p]
        return valid, start

    first_cut = np.zeros(n_chunks, int)
    rank_base = np.zeros(n_chunks, int)
    run = 0
    for c in range(n_chunks):
        valid, start = chunk_masks(c)
        cut = np.nonzero(start | ~valid)[0]
        first_cut[c] = cut[0] if len(cut) else C
        rank_base[c] = run
        run += int(start.sum())
    fin = np.zeros((n_state, H, Dk, Dv)) if want_final else None
    o = np.zeros((N, H, Dv))

    def rows_of(c, h, arr):
        lo_p, hi_p = c * C, min((c + 1) * C, N)
        out = np.zeros((C,) + arr.shape[2:])
        out[: hi_p - lo_p] = arr[lo_p:hi_p, h]
        return out

    for h in range(H):
        # ---- chunk walk (the tensor-core kernel): zero start, seeds, exports ----
        S = np.zeros((Dk, Dv))
        for c in range(n_chunks):
            lo_p, hi_p = c * C, min((c + 1) * C, N)
            n = hi_p - lo_p
            valid, start = chunk_masks(c)
            fc = first_cut[c]
            starts = np.nonzero(start)[0]
            last_start = starts[-1] if len(starts) else 0
            tail_live = valid[C - 1]
            next_cut = c + 1 >= n_chunks or first_cut[c + 1] == 0
            read_state = fc > 0 and c > 0
            carry = fc == C and c > 0
            gg = np.where(valid[:, None], rows_of(c, h, g), 0.0)
            G = np.cumsum(gg, axis=0)                      # G_i, inclusive
            qq, kk, vv, bb = rows_of(c, h, q), rows_of(c, h, k), rows_of(c, h, v), rows_of(c, h, beta)
            rows = np.arange(C)
            lo = np.array([(np.nonzero(start[: i + 1])[0][-1] if start[: i + 1].any() else 0)
                           for i in range(C)])
            if want_final and read_state and (fc < C or next_cut) and rank_base[c] - 1 < n_state:
                fin[rank_base[c] - 1, h] = S                # exported S_in
            O = np.zeros((C, Dv))
            for i in range(C):
                if not valid[i]:
                    continue
                for j in range(lo[i], i + 1):
                    O[i] += (qq[i] * np.exp(G[i] - G[j])) @ kk[j] * bb[j] * vv[j]
                if read_state and i < fc:
                    O[i] += (qq[i] * np.exp(G[i])) @ S
            Snew = np.zeros((Dk, Dv))
            if tail_live:
                for j in range(last_start, C):
                    Snew += np.outer(kk[j] * bb[j] * np.exp(G[-1] - G[j]), vv[j])
            if carry:
                Snew += np.exp(G[-1])[:, None] * S
            rl = rank_base[c] + len(starts) - 1
            if S0 is not None and tail_live and len(starts) and rl < n_state:
                base = G[last_start - 1] if last_start > 0 else np.zeros(Dk)
                Snew += np.exp(G[-1] - base)[:, None] * S0[rl, h]
            S = Snew
            o[lo_p:hi_p, h] = scale * O[:n]
        # ---- the state pass: per chunk, local work ----
        for c in range(n_chunks):
            lo_p, hi_p = c * C, min((c + 1) * C, N)
            valid, start = chunk_masks(c)
            fc = first_cut[c]
            next_cut = c + 1 >= n_chunks or first_cut[c + 1] == 0
            rb = rank_base[c]
            cut = start | ~valid
            gg = np.where(valid[:, None], rows_of(c, h, g), 0.0)
            G = np.cumsum(gg, axis=0)
            Gm = lambda i: G[i] if i >= 0 else np.zeros(Dk)   # noqa: E731
            qq, kk, vv, bb = rows_of(c, h, q), rows_of(c, h, k), rows_of(c, h, v), rows_of(c, h, beta)

            def final(a, e, base):
                Sx = np.zeros((Dk, Dv)) if base is None else np.exp(G[e] - Gm(a - 1))[:, None] * base
                for j in range(a, e + 1):
                    Sx = Sx + np.outer(bb[j] * kk[j] * np.exp(G[e] - G[j]), vv[j])
                return Sx

            if want_final and fc > 0 and (fc < C or next_cut) and rb - 1 < n_state:
                fin[rb - 1, h] = final(0, min(fc, C) - 1, fin[rb - 1, h])
            for idx, r in enumerate(np.nonzero(start)[0]):
                rank = rb + idx
                if rank >= n_state:
                    break
                after = np.nonzero(cut[r + 1:])[0]
                end = r + 1 + after[0] if len(after) else C
                ends_here = len(after) > 0 or next_cut
                if S0 is not None:
                    for t in range(r, end):
                        acc = (qq[t] * np.exp(G[t] - Gm(r - 1))) @ S0[rank, h]
                        for j in range(r, t + 1):
                            acc = acc + (qq[t] * np.exp(G[t] - G[j])) @ kk[j] * bb[j] * vv[j]
                        o[lo_p + t, h] = scale * acc
                if want_final and ends_here:
                    fin[rank, h] = final(r, end - 1, None if S0 is None else S0[rank, h])
    return torch.from_numpy(o), (None if fin is None else torch.from_numpy(fin))


def chunk_units(first_cut, cuts=None):
    """Units of the tensor-core kernel's plan: a unit runs from a cut chunk (from its first
    start-or-padding row) to the next cut chunk (up to that chunk's first cut row).
    `cuts` (chunk indices, sorted) defaults to every chunk holding a start or padding; the
    first of those is always included. Returns [(c0, c1, row_lo, row_hi)]."""
    n_chunks = len(first_cut)
    cand = [c for c in range(n_chunks) if first_cut[c] < C]
    cuts = cand if cuts is None else sorted(set(cuts) | {cand[0]})
    units = []
    for i, c0 in enumerate(cuts):
        if i + 1 < len(cuts):
            cn = cuts[i + 1]
            sn = first_cut[cn]
            c1, row_hi = (cn, sn) if sn > 0 else (cn - 1, C)
        else:
            c1, row_hi = n_chunks - 1, C
        units.append((c0, c1, int(first_cut[c0]), row_hi))
    return units


def chunked_forward_units(q, k, v, g, beta, seg, B, T, scale=1.0, cuts=None, mode="auto",
                          group_floor=-10.0):
    """The tensor-core kernel's algebra in float64, unit by unit, with its masks and its two
    forms. Per chunk: Suf_i sums g over the real rows after i up to the chunk's end (the
    whole-chunk form) or up to the end of row i's 16-row sub-block (the sub-block form,
    taken when `mode` is "always", or for "auto" when some channel's sum over an 8-row group
    falls below `group_floor`); Qt = q exp(-Suf), Ktb = beta k exp(Suf); A' = the masked
    Qt Ktb^T (only the diagonal 16x16 blocks in the sub-block form); O = A' V plus the
    read-out of the incoming state, and the state update, once per chunk or once per
    sub-block with the sub-block's masks (in_b, Kh' rows from the last start, Qt rows before
    the first cut). Each unit starts from a zero state; rows outside [row_lo, row_hi) of its
    first and last chunks belong to the neighbouring units. Returns (o [N, H, Dv] float64,
    the number of chunk-heads that took the sub-block form)."""
    f = (lambda t: t.detach().to(torch.float64).numpy()) if isinstance(q, torch.Tensor) else np.asarray
    q, k, v, g, beta = (f(t) for t in (q, k, v, g, beta))
    N, H, Dk = q.shape
    Dv = v.shape[-1]
    ids = np.ones(N, dtype=np.int64) if seg is None else \
        (seg.numpy() if isinstance(seg, torch.Tensor) else np.asarray(seg)).reshape(-1)
    p = np.arange(N)
    valid_all = ids != 0
    prev = np.concatenate([[0], ids[:-1]])
    start_all = valid_all & ((p % T == 0) | (ids != prev))
    n_chunks = (N + C - 1) // C
    masks = []
    first_cut = np.zeros(n_chunks, int)
    for c in range(n_chunks):
        lo_p, hi_p = c * C, min((c + 1) * C, N)
        valid = np.zeros(C, bool)
        start = np.zeros(C, bool)
        valid[: hi_p - lo_p] = valid_all[lo_p:hi_p]
        start[: hi_p - lo_p] = start_all[lo_p:hi_p]
        masks.append((valid, start))
        cut = np.nonzero(start | ~valid)[0]
        first_cut[c] = cut[0] if len(cut) else C
    rows = np.arange(C)
    o = np.zeros((N, H, Dv))
    n_sub = 0

    def rows_of(c, h, arr):
        lo_p, hi_p = c * C, min((c + 1) * C, N)
        out = np.zeros((C,) + arr.shape[2:])
        out[: hi_p - lo_p] = arr[lo_p:hi_p, h]
        return out

    for (c0, c1, row_lo, row_hi) in chunk_units(first_cut, cuts):
        for h in range(H):
            S = np.zeros((Dk, Dv))
            for c in range(c0, c1 + 1):
                valid, start = masks[c]
                unit_first = c == c0
                lo_row = row_lo if unit_first else 0
                hi_row = row_hi if c == c1 else C
                fc = first_cut[c]
                starts = np.nonzero(start)[0]
                last_start = starts[-1] if len(starts) else 0
                tail_live = valid[C - 1]
                read_state = (not unit_first) and fc > 0
                carry = (not unit_first) and fc == C
                gg = np.where(valid[:, None], rows_of(c, h, g), 0.0)
                groups = gg.reshape(8, 8, Dk).sum(axis=1)
                sub = mode == "always" or (mode == "auto" and bool((groups < group_floor).any()))
                n_sub += int(sub)
                span = 16 if sub else C
                Suf = np.zeros((C, Dk))
                for i in range(C):
                    end = (i // span + 1) * span
                    Suf[i] = gg[i + 1:end].sum(axis=0)
                qq, kk, vv, bb = rows_of(c, h, q), rows_of(c, h, k), rows_of(c, h, v), rows_of(c, h, beta)
                Qt = np.where(valid[:, None], qq * np.exp(-Suf), 0.0)
                Ktb = np.where(valid[:, None], kk * bb[:, None] * np.exp(Suf), 0.0)
                lo = np.array([(np.nonzero(start[: i + 1])[0][-1] if start[: i + 1].any() else 0)
                               for i in range(C)])
                if sub:
                    lo = np.maximum(lo, rows // 16 * 16)
                jj = rows[None, :]
                keep = valid[:, None] & (jj >= lo[:, None]) & (jj <= rows[:, None])
                O = np.where(keep, Qt @ Ktb.T, 0.0) @ vv
                if not sub:
                    kh_lo = last_start if tail_live else C
                    q_hi = fc if (read_state and fc < C) else C
                    P = np.exp(gg.sum(axis=0))
                    if read_state:
                        O += np.where((rows < q_hi)[:, None], Qt, 0.0) @ (P[:, None] * S)
                    Snew = np.where((rows >= kh_lo)[:, None], Ktb, 0.0).T @ vv
                    if carry:
                        Snew += P[:, None] * S
                    S = Snew
                else:
                    for b in range(4):
                        rb = slice(16 * b, 16 * b + 16)
                        stb, vab = start[rb], valid[rb]
                        cutb = stb | ~vab
                        in_b = (not unit_first) or 16 * b > lo_row
                        kh_lo = (16 * b + (np.nonzero(stb)[0][-1] if stb.any() else 0)) if vab[-1] else C
                        q_hi = 16 * b + np.nonzero(cutb)[0][0] if (in_b and cutb.any()) else C
                        P = np.exp(gg[rb].sum(axis=0))
                        Sdec = P[:, None] * S if in_b else np.zeros((Dk, Dv))
                        O[rb] += np.where((rows[rb] < q_hi)[:, None], Qt[rb], 0.0) @ Sdec
                        Snew = np.where((rows[rb] >= kh_lo)[:, None], Ktb[rb], 0.0).T @ vv[rb]
                        if in_b and not cutb.any():
                            Snew += P[:, None] * S
                        S = Snew
                lo_p = c * C
                for i in range(lo_row, min(hi_row, N - lo_p)):
                    o[lo_p + i, h] = scale * O[i]
    return torch.from_numpy(o), n_sub
