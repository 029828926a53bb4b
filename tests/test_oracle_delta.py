"""Pins of the oracle's delta rule (oracle.kda_fwd_delta), on the CPU.

RFC-0026 names the method Kimi Delta Attention but states only the additive update; the
delta rule is the reading of that name (the gated delta rule with a decay per key channel):
    S'_t = S_{t-1} exp(g_t) (key rows),  S_t = S'_t + beta_t k_t (v_t - S'_t^T k_t)^T,
    o_t = scale S_t^T q_t,
reset at segment starts like the additive rule. The pins do not retype the oracle's loops:
- the rule's defining property: with beta = 1 and a unit key, the new state reads back
  exactly v_t along k_t, whatever the decay before it (so q = k gives o_t = scale v_t);
- the projector form (I - beta k k^T) S' + beta k v^T, evaluated as matrix products;
- at a segment's first token the state before it is zero, so the delta rule equals the
  additive rule there;
- beta = 0 writes nothing; the output is linear in v for fixed q, k, g, beta;
- segments are independent and padding outputs are zero.
A slip in the oracle (a dropped or mis-signed correction, the decay applied after the write,
beta inside the correction, a transposed state) fails at least one of them.
"""
import numpy as np
import torch

import oracle
import synth


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _inputs(rng, N, H, Dk, Dv, beta_one=False):
    q = rng.standard_normal((N, H, Dk))
    k = _unit(rng.standard_normal((N, H, Dk)))
    v = rng.standard_normal((N, H, Dv))
    g = -np.exp(rng.standard_normal((N, H, Dk)) * 0.5 - 1.0)
    beta = np.ones((N, H)) if beta_one else 1.0 / (1.0 + np.exp(-rng.standard_normal((N, H))))
    return [torch.from_numpy(a) for a in (q, k, v, g, beta)]


def test_unit_keys_read_back_their_values():
    rng = np.random.default_rng(1)
    seg = torch.from_numpy(synth.random_segment_ids(rng, 2, 90, max_len=40, pad_prob=0.1))
    N, H, D = 180, 3, 16
    _, k, v, g, beta = _inputs(rng, N, H, D, D, beta_one=True)
    o = oracle.kda_fwd_delta(k, k, v, g, beta, seg, 2, 90, scale=0.7)
    real = (seg.reshape(-1) != 0)
    assert torch.allclose(o[real], 0.7 * v[real], rtol=0, atol=1e-12)
    assert torch.all(o[~real] == 0)


def _projector_form(q, k, v, g, beta, seg_row, scale):
    """One row: the state as matrices, S_t = (I - b k k^T) diag(exp g) S_{t-1} + b k v^T."""
    T, H, Dk = q.shape
    Dv = v.shape[-1]
    out = np.zeros((T, H, Dv))
    for h in range(H):
        S = np.zeros((Dk, Dv))
        for t in range(T):
            if seg_row[t] == 0:
                S = np.zeros((Dk, Dv))
                continue
            if t == 0 or seg_row[t - 1] != seg_row[t]:
                S = np.zeros((Dk, Dv))
            kt = k[t, h][:, None]
            P = np.eye(Dk) - beta[t, h] * (kt @ kt.T)
            S = P @ (np.diag(np.exp(g[t, h])) @ S) + beta[t, h] * (kt @ v[t, h][None, :])
            out[t, h] = scale * (S.T @ q[t, h])
    return out


def test_projector_form():
    rng = np.random.default_rng(2)
    seg = np.array([[1, 1, 1, 2, 2, 0, 3, 3, 3, 3, 3, 1, 1]], np.int32)   # an id comes back
    T = seg.shape[1]
    q, k, v, g, beta = (t.numpy() for t in _inputs(rng, T, 2, 5, 4))
    k = k * rng.uniform(0.5, 1.5, size=(T, 2, 1))                        # keys of any length
    ref = _projector_form(q, k, v, g, beta, seg[0], 0.9)
    o = oracle.kda_fwd_delta(*(torch.from_numpy(a) for a in (q, k, v, g, beta)),
                             torch.from_numpy(seg), 1, T, scale=0.9)
    assert np.allclose(o.numpy(), ref, rtol=1e-12, atol=1e-13)


def test_first_token_of_a_segment_is_the_additive_rule():
    rng = np.random.default_rng(3)
    seg_np = synth.random_segment_ids(rng, 2, 120, max_len=30, pad_prob=0.05)
    seg = torch.from_numpy(seg_np)
    q, k, v, g, beta = _inputs(rng, 240, 2, 8, 8)
    d = oracle.kda_fwd_delta(q, k, v, g, beta, seg, 2, 120)
    a = oracle.kda_fwd(q, k, v, g, beta, seg, 2, 120)
    flat = seg_np.reshape(-1)
    first = [p for p in range(240) if flat[p] != 0 and (p % 120 == 0 or flat[p - 1] != flat[p])]
    assert len(first) > 5
    assert torch.allclose(d[first], a[first], rtol=0, atol=1e-14)
    # later tokens differ: the correction is there
    later = [p for p in range(240) if flat[p] != 0 and p not in first]
    assert (d[later] - a[later]).abs().max() > 1e-3


def test_zero_beta_writes_nothing_and_linearity_in_v():
    rng = np.random.default_rng(4)
    seg = torch.ones(1, 50, dtype=torch.int32)
    q, k, v, g, beta = _inputs(rng, 50, 2, 6, 5)
    assert torch.all(oracle.kda_fwd_delta(q, k, v, g, torch.zeros_like(beta), seg, 1, 50) == 0)
    v2 = torch.from_numpy(rng.standard_normal(v.shape))
    o1 = oracle.kda_fwd_delta(q, k, v, g, beta, seg, 1, 50)
    o2 = oracle.kda_fwd_delta(q, k, v2, g, beta, seg, 1, 50)
    o12 = oracle.kda_fwd_delta(q, k, v + 2.5 * v2, g, beta, seg, 1, 50)
    assert torch.allclose(o12, o1 + 2.5 * o2, rtol=1e-12, atol=1e-12)


def test_segments_are_independent():
    rng = np.random.default_rng(5)
    q, k, v, g, beta = _inputs(rng, 60, 2, 8, 8)
    seg = torch.tensor([[1] * 25 + [0] * 5 + [2] * 30], dtype=torch.int32)
    whole = oracle.kda_fwd_delta(q, k, v, g, beta, seg, 1, 60)
    a = oracle.kda_fwd_delta(*(t[:25] for t in (q, k, v, g, beta)), None, 1, 25)
    b = oracle.kda_fwd_delta(*(t[30:] for t in (q, k, v, g, beta)), None, 1, 30)
    assert torch.equal(whole[:25], a) and torch.equal(whole[30:], b)
    assert torch.all(whole[25:30] == 0)
