"""kda_chunk_fwd_varlen_noalloc: the forward for callers that cannot allocate.

Some callers hold no device allocator (a C host program handed buffers by
another runtime, or a serving loop whose pool owns all free device memory and
forbids cudaMalloc/cudaFree on its hot path), so they cannot pass the scratch
workspace that kda_chunk_fwd_varlen takes. This entry point uses a scratch
array built into the library instead. The test calls it through the C ABI
twice in a row, on different inputs, and checks each result against the
allocating entry point within the parity tolerance the other tests use. It
lives in its own file, collected last, and passes alone or after the rest.
"""
import ctypes

import numpy as np
import pytest
import torch

import kda_segids_cu_gb300 as kda
import synth
from tests.parity import tolerance

pytestmark = pytest.mark.gpu


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
    return [t.cuda() for t in (q, k, v, g, beta, seg)]


def _call_noalloc(f, q, k, v, g, beta, seg, B, T, scale):
    H, D = q.shape[-2], q.shape[-1]
    o = torch.full_like(v, float("nan"))
    dt = kda.KDA_BF16 if q.dtype == torch.bfloat16 else kda.KDA_F32
    st = f(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(), seg.data_ptr(),
           B, T, H, D, D, ctypes.c_float(scale), dt, dt, o.data_ptr(), None,
           torch.cuda.current_stream().cuda_stream)
    assert st == 0, f"kda_chunk_fwd_varlen_noalloc returned {st}"
    return o


def _close(a, b, dtype):
    a64, b64 = a.double().cpu(), b.double().cpu()
    rms = b64.pow(2).mean().sqrt().item()
    err = (a64 - b64).abs().max().item()
    assert err <= tolerance(dtype) * rms, f"max|diff| {err:.3e} vs RMS {rms:.3e}"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_allocating_entry_point(dtype):
    f = _noalloc_fn()
    cases = [(2, 700, 4, 128, 9, 120, 1.0), (1, 1500, 2, 128, 10, 30, 0.5)]
    for (B, T, H, D, seed, max_len, scale) in cases:        # two calls in a row
        q, k, v, g, beta, seg = _inputs(B, T, H, D, dtype, seed, max_len)
        o_na = _call_noalloc(f, q, k, v, g, beta, seg, B, T, scale)
        o_ref = kda.kda_chunk_fwd_varlen(q, k, v, g, beta, seg, scale=scale)
        torch.cuda.synchronize()
        assert torch.isfinite(o_na).all()
        _close(o_na, o_ref, dtype)


def test_noalloc_refuses_sizes_beyond_its_array():
    f = _noalloc_fn()
    lib = kda.load_library()
    limit = 4 << 20
    B, T = 1, 600_000                      # needs more scratch than the built-in array
    assert lib.kda_chunk_fwd_varlen_workspace_size(B, T, 1, 128, 128, kda.KDA_BF16) > limit
    p = ctypes.c_void_p(4096)              # never dereferenced: refused on the host
    st = f(p, p, p, p, p, None, B, T, 1, 128, 128, ctypes.c_float(1.0), kda.KDA_BF16,
           kda.KDA_BF16, p, None, None)
    assert st == -4                        # KDA_ERR_WORKSPACE
