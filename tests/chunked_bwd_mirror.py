"""A CPU restatement of the chunked KDA backward used by the tensor-core kernels.

Not the oracle: this is the chunk algebra of the backward (chains of chunks, the two state
scans with their optional cut into pieces, the per-chunk gradient formulas with their
segment masks, and dg's part past the chunk) written out in numpy float64. The tests hold it
to the oracle's step-by-step reverse-mode gradients, so that the algebra the kernels follow
is checked on the CPU, apart from the CUDA code.

Per chunk c and head (G the chunk-local cumulative log-decay over real rows, Suf_t the sum of
g over the chunk's real rows after t, P = exp of the chunk's whole real g):
    S_in  = the state the carried segment brings into the chunk (forward scan)
    D_end = dL/dS at the chunk's last row for the segment that goes on (reverse scan)
    Qt = q exp(-Suf), Ktb = beta k exp(Suf), M = same-segment causal mask (real rows)
    W  = M (dO V^T),  A' = scale M (Qt Ktb^T)
    dq_t = scale exp(-Suf_t) [ (W Ktb)_t + [t carried] P (S_in do_t) ]
    dk_s = beta_s exp(Suf_s) [ scale (W^T Qt)_s + [s in the last segment] D_end v_s ]
    dv_s = (A'^T dO)_s + [s in the last segment] D_end^T Ktb_s
    dbeta_s = k_s . (dk_s / beta_s)
    dg_t = sum over u >= t in t's segment within the chunk of (q_u dq_u - k_u dk_u)
           + [t in the last segment] rowdot(S_out, D_end);  0 at a segment's first row
"""
from __future__ import annotations

import numpy as np
import torch

C = 64


def _np(t):
    return t.detach().to(torch.float64).numpy() if isinstance(t, torch.Tensor) else np.asarray(t)


def chunk_layout(seg, N: int, T: int):
    """Per chunk (64-token grid of the flattened rows): start and real masks [n, 64] and the
    first start-or-padding row (64 if none)."""
    n = (N + C - 1) // C
    ids = np.ones(N, np.int64) if seg is None else _np(seg).reshape(-1).astype(np.int64)
    start = np.zeros(n * C, bool)
    valid = np.zeros(n * C, bool)
    for p in range(N):
        valid[p] = ids[p] != 0
        start[p] = valid[p] and (p % T == 0 or ids[p] != ids[p - 1])
    start, valid = start.reshape(n, C), valid.reshape(n, C)
    fc = [int(np.argmax(start[c] | ~valid[c])) if (start[c] | ~valid[c]).any() else C
          for c in range(n)]
    return n, start, valid, fc


def _chains(n, fc):
    heads = [c for c in range(n) if c == 0 or fc[c] < C]
    return list(zip(heads, heads[1:] + [n]))


def _pieces(items, piece, split_min):
    """The run of chunks `items` (in scan order) as pieces: one piece when it is short, else
    pieces of `piece` chunks."""
    if piece is None or len(items) <= split_min:
        return [items]
    return [items[i:i + piece] for i in range(0, len(items), piece)]


def scans(q, k, v, g, beta, do, n, start, valid, fc, h, scale, piece=None, split_min=None):
    """S_in and D_end for every chunk (NaN where the kernels write nothing), for head h.

    With `piece`, chains longer than `split_min` chunks run as pieces: each piece but the last
    from a zero state (its end state E_j and decay product Pi_j), then the true piece starts
    T_{j+1} = Pi_j T_j + E_j, then every piece from its true start."""
    D = q.shape[-1]
    split_min = piece if split_min is None else split_min
    S_in = np.full((n, D, D), np.nan)
    D_end = np.full((n, D, D), np.nan)

    def chunk_p(c):
        return np.exp(np.where(valid[c][:, None], g[c * C:(c + 1) * C, h], 0.0).sum(0))

    def fwd_step(S, c, first, lo):
        if not first:
            S = chunk_p(c)[:, None] * S
        for t in range(lo, C):
            p = c * C + t
            suf = g[p + 1:(c + 1) * C, h].sum(0)
            S = S + np.outer(beta[p, h] * k[p, h] * np.exp(suf), v[p, h])
        return S

    def rev_step(Dm, c, first, hi):
        if not first:
            Dm = chunk_p(c)[:, None] * Dm
        G = np.zeros(D)
        for t in range(hi):
            p = c * C + t
            G = G + g[p, h]
            Dm = Dm + np.outer(scale * q[p, h] * np.exp(G), do[p, h])
        return Dm

    def run(pieces, step, rows_of, export, post):
        # the end-state pass and the combine
        T = [None]
        if len(pieces) > 1:
            E, PI = [], []
            for pcs in pieces[:-1]:
                X = np.zeros((D, D))
                pi = np.ones(D)
                for i, c in enumerate(pcs):
                    X = step(X, c, i == 0, rows_of(c))
                    pi = pi * chunk_p(c)
                E.append(X)
                PI.append(pi)
            T.append(E[0])
            for j in range(1, len(pieces) - 1):
                T.append(PI[j][:, None] * T[j] + E[j])
        # the export pass
        for j, pcs in enumerate(pieces):
            X = np.zeros((D, D))
            for i, c in enumerate(pcs):
                if i == 0 and j > 0:
                    X = T[j]
                    export(c, X)
                    X = step(X, c, False, rows_of(c))
                else:
                    if i > 0:
                        export(c, X)
                    X = step(X, c, i == 0, rows_of(c))
            if j == len(pieces) - 1:
                post(X)

    for ca, cb in _chains(n, fc):
        def lo_of(c, ca=ca):
            if c != ca:
                return 0
            st = np.nonzero(start[c])[0]
            return (int(st[-1]) if len(st) else 0) if valid[c, C - 1] else C

        def post_f(X, cb=cb):
            if cb < n and fc[cb] > 0:
                S_in[cb] = X

        run(_pieces(list(range(ca, cb)), piece, split_min), fwd_step, lo_of,
            lambda c, X: S_in.__setitem__(c, X), post_f)
        head = cb < n and fc[cb] > 0
        c_from = cb if head else cb - 1
        items = list(range(c_from, ca, -1))
        if not items:
            continue

        def hi_of(c, cb=cb):
            return fc[c] if c == cb else C

        run(_pieces(items, piece, split_min), rev_step, hi_of,
            lambda c, X: D_end.__setitem__(c, X), lambda X, ca=ca: D_end.__setitem__(ca, X))
    return S_in, D_end


def chunked_backward(q, k, v, g, beta, do, seg, B, T, scale=1.0, piece=None, split_min=None):
    """(dq, dk, dv, dg, dbeta) shaped like the inputs, from the chunk algebra (float64)."""
    q, k, v, g, beta, do = (_np(t) for t in (q, k, v, g, beta, do))
    N, H, D = q.shape
    n, start, valid, fc = chunk_layout(seg, N, T)
    pad = n * C - N
    if pad:
        q, k, v, g, do = (np.concatenate([x, np.zeros((pad,) + x.shape[1:])]) for x in (q, k, v, g, do))
        beta = np.concatenate([beta, np.zeros((pad, H))])
    dq, dk, dv, dg = (np.zeros_like(q) for _ in range(4))
    db = np.zeros_like(beta)
    for h in range(H):
        S_in, D_end = scans(q, k, v, g, beta, do, n, start, valid, fc, h, scale, piece, split_min)
        for c in range(n):
            rows = slice(c * C, (c + 1) * C)
            st, va = start[c], valid[c]
            cin = fc[c] > 0
            cout = c + 1 < n and fc[c + 1] > 0
            starts = np.nonzero(st)[0]
            lo_last = int(starts[-1]) if len(starts) else 0
            gg = np.where(va[:, None], g[rows, h], 0.0)
            suf = np.array([gg[t + 1:].sum(0) for t in range(C)])
            Qt = np.where(va[:, None], q[rows, h] * np.exp(-suf), 0.0)
            Ktb = np.where(va[:, None], k[rows, h] * beta[rows, h][:, None] * np.exp(suf), 0.0)
            P = np.exp(gg.sum(0))
            M = np.zeros((C, C))
            for t in range(C):
                if va[t]:
                    s0 = max([r for r in range(t + 1) if st[r]], default=0)
                    M[t, s0:t + 1] = 1.0
            A = scale * M * (Qt @ Ktb.T)
            W = M * (do[rows, h] @ v[rows, h].T)
            S0 = S_in[c] if cin else np.zeros((D, D))
            DE = D_end[c] if cout else np.zeros((D, D))
            Qs = do[rows, h] @ (P[:, None] * S0).T     # [t][key]
            T2 = v[rows, h] @ DE.T                      # [s][key]
            Vs = Ktb @ DE                               # [s][v]
            dQ, dK, dV = W @ Ktb, W.T @ Qt, A.T @ do[rows, h]
            carry = np.zeros(D)
            if cout:
                if fc[c] == C:
                    carry += P * (S0 * DE).sum(1)
                for s in range(lo_last, C):
                    carry += Ktb[s] * T2[s]
            run = carry
            for t in range(C - 1, -1, -1):
                p = c * C + t
                if not va[t]:
                    run = np.zeros(D)
                    continue
                last = cout and t >= lo_last
                qsum = dQ[t] + (Qs[t] if t < fc[c] else 0.0)
                ksum = scale * dK[t] + (T2[t] if last else 0.0)
                dq[p, h] = scale * np.exp(-suf[t]) * qsum
                dkr = np.exp(suf[t]) * ksum
                dk[p, h] = beta[p, h] * dkr
                dv[p, h] = dV[t] + (Vs[t] if last else 0.0)
                db[p, h] = (k[p, h] * dkr).sum()
                run = run + scale * Qt[t] * qsum - Ktb[t] * ksum
                dg[p, h] = 0.0 if st[t] else run
                if st[t]:
                    run = np.zeros(D)
    return tuple(x[:N] for x in (dq, dk, dv, dg)) + (db[:N],)
