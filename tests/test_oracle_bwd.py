"""Pins for the oracle's gradients (no GPU).

The pages give the forward recurrence only; `oracle.kda_bwd` differentiates it
step by step in reverse. Two checks that do not go through that code:
- central finite differences of the oracle's own forward (a brute-force
  derivative) on a tiny packed batch with padding, a length-1 document and two
  rows;
- automatic differentiation (torch, float64) of the brute-force closed form
  o_t = scale sum_{j<=t, same segment} beta_j v_j sum_c q_t[c] k_j[c] exp(G_t[c] - G_j[c]),
  with G the cumulative sum of g, on a larger batch.
"""
import numpy as np
import torch

import oracle


def _inputs(rng, N, H, Dk, Dv):
    q = rng.standard_normal((N, H, Dk)) / np.sqrt(Dk)
    k = rng.standard_normal((N, H, Dk)) / np.sqrt(Dk)
    v = rng.standard_normal((N, H, Dv))
    g = -np.exp(rng.normal(-2.0, 0.5, (N, H, Dk)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((N, H))))
    d_o = rng.standard_normal((N, H, Dv))
    return q, k, v, g, beta, d_o


def test_finite_differences():
    rng = np.random.default_rng(3)
    B, T, H, Dk, Dv = 2, 7, 2, 3, 2
    seg = np.array([[4, 4, 4, 0, 9, 9, 9], [1, 2, 2, 2, 2, 0, 0]], dtype=np.int32)
    q, k, v, g, beta, d_o = _inputs(rng, B * T, H, Dk, Dv)
    scale = 0.7
    grads = oracle.kda_bwd(q, k, v, g, beta, d_o, seg, B, T, scale=scale)

    def loss(qq, kk, vv, gg, bb):
        o = oracle.kda_fwd(qq, kk, vv, gg, bb, seg, B, T, scale=scale, n_threads=1)
        return float((o.numpy() * d_o).sum())

    args = [q, k, v, g, beta]
    eps = 1e-6
    for which, (x, gr) in enumerate(zip(args, grads)):
        gr = gr.numpy()
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            ap, am = list(args), list(args)
            ap[which], am[which] = xp, xm
            fd = (loss(*ap) - loss(*am)) / (2 * eps)
            assert abs(fd - gr[idx]) <= 1e-7 + 1e-6 * abs(fd), (which, idx, fd, gr[idx])
    # padding tokens have zero gradients
    pad = (seg.reshape(-1) == 0)
    for gr in grads:
        assert torch.all(gr[torch.from_numpy(pad)] == 0)


def _closed_form(q, k, v, g, beta, seg, B, T, scale):
    """o by the O(T^2) closed form, differentiable in torch (float64)."""
    N, H, Dk = q.shape
    out = []
    for b in range(B):
        sl = slice(b * T, (b + 1) * T)
        s = seg[b]
        t_idx = torch.arange(T)
        same = (s[:, None] == s[None, :]) & (s[:, None] != 0)
        # same segment = same id and no break (different id or padding) in between
        run = torch.cumsum(torch.cat([torch.ones(1, dtype=torch.long),
                                      (s[1:] != s[:-1]).long()]), 0)
        same = same & (run[:, None] == run[None, :]) & (t_idx[None, :] <= t_idx[:, None])
        G = torch.cumsum(g[sl], 0)                             # [T, H, Dk]
        E = G[:, None] - G[None, :]                            # [t, j, H, Dk]
        E = torch.where(same[:, :, None, None], E, torch.zeros_like(E))
        A = torch.einsum("thc,jhc,tjhc->tjh", q[sl], k[sl], torch.exp(E))
        A = A * same[:, :, None]
        out.append(scale * torch.einsum("tjh,jh,jhd->thd", A, beta[sl], v[sl]))
    return torch.cat(out, 0)


def test_autograd_of_closed_form():
    rng = np.random.default_rng(11)
    B, T, H, Dk, Dv = 2, 40, 2, 4, 3
    seg = np.zeros((B, T), dtype=np.int32)
    seg[0, :13], seg[0, 13:14], seg[0, 14:30], seg[0, 33:] = 5, 6, 5, 2   # 30-32 padding
    seg[1, 0:1], seg[1, 1:25], seg[1, 25:] = 3, 1, 7
    q, k, v, g, beta, d_o = _inputs(rng, B * T, H, Dk, Dv)
    scale = 1.3
    ts = [torch.tensor(a, requires_grad=True) for a in (q, k, v, g, beta)]
    o = _closed_form(*ts, torch.from_numpy(seg), B, T, scale)
    (o * torch.from_numpy(d_o)).sum().backward()
    got = oracle.kda_bwd(q, k, v, g, beta, d_o, seg, B, T, scale=scale)
    for name, t, gr in zip(("dq", "dk", "dv", "dg", "dbeta"), ts, got):
        ref = t.grad
        err = (gr - ref).abs().max().item()
        assert err <= 1e-10 * max(1.0, ref.abs().max().item()), (name, err)


def test_segment_ids_none_and_isolation():
    """seg=None equals all-ones; a packed batch's gradients equal each document's own."""
    rng = np.random.default_rng(5)
    T, H, D = 30, 1, 3
    q, k, v, g, beta, d_o = _inputs(rng, T, H, D, D)
    a = oracle.kda_bwd(q, k, v, g, beta, d_o, None, 1, T)
    b = oracle.kda_bwd(q, k, v, g, beta, d_o, np.ones((1, T), np.int32), 1, T)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    seg = np.array([[1] * 12 + [2] * 18], dtype=np.int32)
    packed = oracle.kda_bwd(q, k, v, g, beta, d_o, seg, 1, T)
    first = oracle.kda_bwd(q[:12], k[:12], v[:12], g[:12], beta[:12], d_o[:12], None, 1, 12)
    second = oracle.kda_bwd(q[12:], k[12:], v[12:], g[12:], beta[12:], d_o[12:], None, 1, 18)
    for x, y1, y2 in zip(packed, first, second):
        assert torch.equal(x, torch.cat([y1, y2], 0))
