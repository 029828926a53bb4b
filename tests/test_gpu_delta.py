"""GPU parity of kda_delta_fwd_varlen, the delta-rule form of the recurrence.

RFC-0026 names the method Kimi Delta Attention but states only the additive update; the
delta rule S_t = S'_t + beta_t k_t (v_t - S'_t^T k_t)^T is the reading of that name, and
oracle.kda_fwd_delta is its fp64 reference (pinned in tests/test_oracle_delta.py). The kernel
runs the token recurrence in fp32 arithmetic, so outputs are held to the fp32 bound of the
oracle's output RMS for either input dtype (bf16 inputs are exact in both), plus half a bf16
ulp when stored in bf16. The cases cover segments with padding, several ragged rows, both
head widths, both dtypes, no ids, and the rule's defining property on the device: with
beta = 1 and unit keys, q = k reads back scale * v.
"""
import numpy as np
import pytest
import torch

import kda_segids_cu_gb300 as kda
import oracle
import synth
from tests.parity import check_kda_output

pytestmark = pytest.mark.gpu


def _inputs(N, H, D, dtype, seed, beta_one=False):
    gen = torch.Generator().manual_seed(seed)
    q = torch.nn.functional.normalize(torch.randn(N, H, D, generator=gen), dim=-1)
    k = torch.nn.functional.normalize(torch.randn(N, H, D, generator=gen), dim=-1)
    v = torch.randn(N, H, D, generator=gen)
    g = -torch.exp(torch.randn(N, H, D, generator=gen) * 0.5 - 2.0)
    beta = torch.ones(N, H) if beta_one else torch.sigmoid(torch.randn(N, H, generator=gen))
    return [t.to(dtype) for t in (q, k, v, g, beta)]


@pytest.mark.parametrize("dtype,D", [(torch.float32, 64), (torch.float32, 128),
                                     (torch.bfloat16, 64), (torch.bfloat16, 128)])
def test_delta_matches_oracle(dtype, D):
    rng = np.random.default_rng(7)
    layouts = [synth.random_segment_ids(rng, 2, 300, max_len=120, pad_prob=0.1),
               synth.random_segment_ids(rng, 3, 97, max_len=40, pad_prob=0.05),
               np.ones((1, 400), np.int32)]
    for i, seg_np in enumerate(layouts):
        seg = torch.from_numpy(seg_np)
        B, T = seg.shape
        H = 2
        args = _inputs(B * T, H, D, dtype, seed=10 * i + D)
        ref = oracle.kda_fwd_delta(*args, seg, B, T, scale=0.8)
        for out_dtype in (None, torch.float32):
            o = kda.kda_delta_fwd_varlen(*(t.cuda() for t in args), seg.cuda(), scale=0.8,
                                         out_dtype=out_dtype)
            check_kda_output(o, ref, seg, torch.float32, label=f"delta {dtype} D={D} layout {i}")


def test_delta_without_ids():
    B, T, H, D = 2, 150, 2, 64
    args = _inputs(B * T, H, D, torch.float32, seed=3)
    o = kda.kda_delta_fwd_varlen(*(t.cuda() for t in args), None, B=B, T=T)
    ref = oracle.kda_fwd_delta(*args, None, B, T)
    check_kda_output(o, ref, None, torch.float32, label="delta no ids")


def test_unit_keys_read_back_their_values_on_the_device():
    """beta = 1, unit keys and q = k: o_t = scale v_t whatever the decay and history."""
    rng = np.random.default_rng(9)
    seg = torch.from_numpy(synth.random_segment_ids(rng, 2, 256, max_len=200, pad_prob=0.05))
    B, T = seg.shape
    _, k, v, g, beta = _inputs(B * T, 3, 128, torch.float32, seed=4, beta_one=True)
    o = kda.kda_delta_fwd_varlen(k.cuda(), k.cuda(), v.cuda(), g.cuda(), beta.cuda(), seg.cuda(),
                                 scale=0.5).cpu()
    real = seg.reshape(-1) != 0
    err = (o[real] - 0.5 * v[real]).abs().max().item()
    assert err < 1e-4 * 0.5 * v[real].abs().max().item() * 10, err
    assert torch.all(o[~real] == 0)
