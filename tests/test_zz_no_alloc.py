"""kda_chunk_fwd_varlen_noalloc: the forward for callers that cannot allocate.

Some callers hold no device allocator (a C host program handed buffers by
another runtime, or a serving loop whose pool owns all free device memory and
forbids cudaMalloc/cudaFree on its hot path), so they cannot pass the scratch
workspace that kda_chunk_fwd_varlen takes. This entry point uses a scratch
array built into the library instead.

The GPU test calls it through the C ABI several times in a row, on different
inputs and on both paths (the tensor-core path for bf16 with 128-wide heads,
the token recurrence for fp32 and for 64-wide heads). The no-allocation call
runs the same kernels on the same plan as the allocating entry point, so the
two outputs must be equal bit for bit: a stale word in the shared array that
perturbed an output would show here. Each output is also held to the oracle
within the parity tolerance. The file is collected last and passes alone or
after the rest. The size and argument-order checks run on the host only.
"""
import ctypes

import numpy as np
import pytest
import torch

import kda_segids_cu_gb300 as kda
import oracle
import synth
from tests.parity import check_kda_output

SCRATCH_BYTES = 4 << 20          # KDA_NOALLOC_SCRATCH_BYTES in include/kda.h
MAX_TOKENS = 524_256             # the largest B*T whose workspace fits the array


def _noalloc_fn():
    lib = kda.load_library()
    f = lib.kda_chunk_fwd_varlen_noalloc
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    f.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, i32, ctypes.c_float, ctypes.c_int,
                  ctypes.c_int, vp, vp, vp]
    f.restype = ctypes.c_int
    return f


def _inputs(B, T, H, D, dtype, seed, max_len):
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    seg = torch.from_numpy(synth.random_segment_ids(rng, B, T, max_len=max_len, pad_prob=0.1))
    N = B * T
    q = torch.nn.functional.normalize(torch.randn(N, H, D, generator=gen), dim=-1).to(dtype)
    k = torch.nn.functional.normalize(torch.randn(N, H, D, generator=gen), dim=-1).to(dtype)
    v = torch.randn(N, H, D, generator=gen).to(dtype)
    g = (-torch.exp(torch.randn(N, H, D, generator=gen) * 0.5 - 2.0)).to(dtype)
    beta = torch.sigmoid(torch.randn(N, H, generator=gen)).to(dtype)
    return q, k, v, g, beta, seg


def _call_noalloc(f, q, k, v, g, beta, seg, B, T, scale, status=None):
    H, D = q.shape[-2], q.shape[-1]
    o = torch.full_like(v, float("nan"))
    dt = kda.KDA_BF16 if q.dtype == torch.bfloat16 else kda.KDA_F32
    st = f(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(), seg.data_ptr(),
           B, T, H, D, D, ctypes.c_float(scale), dt, dt, o.data_ptr(),
           None if status is None else status.data_ptr(),
           torch.cuda.current_stream().cuda_stream)
    assert st == 0, f"kda_chunk_fwd_varlen_noalloc returned {st}"
    return o


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.bfloat16, 64),
                                     (torch.float32, 64)])
def test_noalloc_matches_allocating_entry_point(dtype, D):
    f = _noalloc_fn()
    cases = [(2, 700, 4, 9, 120, 1.0), (1, 1500, 2, 10, 30, 0.5), (3, 257, 3, 11, 64, 1.0)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for (B, T, H, seed, max_len, scale) in cases:           # calls in a row on the one array
        cpu = _inputs(B, T, H, D, dtype, seed, max_len)
        q, k, v, g, beta, seg = (t.cuda() for t in cpu)
        o_na = _call_noalloc(f, q, k, v, g, beta, seg, B, T, scale, status)
        o_ref = kda.kda_chunk_fwd_varlen(q, k, v, g, beta, seg, scale=scale, check=False)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(o_na, o_ref), f"B={B} T={T}: outputs differ from the allocating call"
        ref = oracle.kda_fwd(*cpu[:5], cpu[5], B, T, scale=scale)
        check_kda_output(o_na, ref, cpu[5], dtype, label=f"noalloc B={B} T={T}")


def test_noalloc_size_limit_on_the_host():
    """The array's size bounds the problem: the least workspace of MAX_TOKENS tokens fits it
    and one token more does not, for either dtype and head width (no launch). A problem
    that fits uses whatever room is left for splitting long segments."""
    lib = kda.load_library()
    for dt, D in ((kda.KDA_BF16, 128), (kda.KDA_BF16, 64), (kda.KDA_F32, 64)):
        for H in (1, 16, 64):
            assert lib.kda_chunk_fwd_varlen_workspace_min(1, MAX_TOKENS, H, D, D, dt) <= \
                SCRATCH_BYTES
            assert lib.kda_chunk_fwd_varlen_workspace_min(1, MAX_TOKENS + 1, H, D, D, dt) > \
                SCRATCH_BYTES
            assert lib.kda_chunk_fwd_varlen_workspace_min(4, MAX_TOKENS // 4, H, D, D, dt) <= \
                SCRATCH_BYTES


def test_noalloc_refuses_on_the_host():
    """Refusals happen before any launch: a problem one token past the limit returns
    KDA_ERR_WORKSPACE, and a null or misaligned tensor returns KDA_ERR_INVALID_ARG first,
    whatever the size (the pointers are never dereferenced)."""
    f = _noalloc_fn()
    p = ctypes.c_void_p(4096)
    odd = ctypes.c_void_p(4098)
    args = lambda T, q=p: (q, p, p, p, p, None, 1, T, 1, 128, 128, ctypes.c_float(1.0),
                           kda.KDA_BF16, kda.KDA_BF16, p, None, None)
    assert f(*args(MAX_TOKENS + 1)) == -4           # KDA_ERR_WORKSPACE
    assert f(*args(600_000)) == -4
    assert f(*args(600_000, q=None)) == -1          # KDA_ERR_INVALID_ARG before the size
    assert f(*args(600_000, q=odd)) == -1
    assert f(*args(MAX_TOKENS, q=None)) == -1
