"""The C ABI library loads, exports every function include/kda.h declares,
and rejects invalid arguments on the host before touching the GPU (no GPU)."""
import ctypes

import pytest

import kda_segids_cu_gb300 as kda


@pytest.fixture(scope="module")
def lib():
    return kda.load_library()


def test_exports_every_declared_function(lib):
    names = kda.header_functions()
    assert {"kda_segids_to_cu_seqlens", "kda_short_conv_varlen", "kda_chunk_fwd_varlen",
            "kda_chunk_fwd_varlen_workspace_size", "kda_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"libkda.so does not export {n}"


def test_status_strings(lib):
    for code, name in [(0, b"KDA_OK"), (-1, b"KDA_ERR_INVALID_ARG"), (-2, b"KDA_ERR_UNSUPPORTED"),
                       (-3, b"KDA_ERR_CUDA"), (-4, b"KDA_ERR_WORKSPACE")]:
        assert lib.kda_status_string(code) == name


def test_workspace_size_host_logic(lib):
    f = lib.kda_chunk_fwd_varlen_workspace_size
    assert f(4, 8192, 16, 128, 128, kda.KDA_BF16) > 0
    assert f(1, 256, 2, 64, 64, kda.KDA_F32) > 0
    assert f(0, 8, 1, 64, 64, kda.KDA_F32) == 0          # invalid sizes
    assert f(1, 8, 0, 64, 64, kda.KDA_F32) == 0
    assert f(1 << 20, 1 << 12, 1, 64, 64, kda.KDA_F32) == 0   # B*T >= 2^31
    assert f(1, 8, 1, 64, 64, 7) == 0                     # unknown dtype
    # the minimum is the plan (or the token recurrence's list); the full size adds one 64 KB
    # state per head per 64 chunks for splitting long segments (bf16, 128-wide heads only)
    m = lib.kda_chunk_fwd_varlen_workspace_min
    for (B, T, H) in ((4, 8192, 16), (1, 131072, 32), (2, 100, 3)):
        n_chunks = (B * T + 63) // 64
        full, least = f(B, T, H, 128, 128, kda.KDA_BF16), m(B, T, H, 128, 128, kda.KDA_BF16)
        assert full >= least and full >= -(-n_chunks // 64) * H * 128 * 128 * 4
        assert m(B, T, H, 64, 64, kda.KDA_BF16) == f(B, T, H, 64, 64, kda.KDA_BF16)
        assert m(B, T, H, 64, 64, kda.KDA_F32) == f(B, T, H, 64, 64, kda.KDA_F32) == 8 * B * T + 256
    assert m(0, 8, 1, 64, 64, kda.KDA_F32) == 0


FAKE = ctypes.c_void_p(4096)    # aligned, never dereferenced: validation fails first
ODD = ctypes.c_void_p(4098)


def test_segids_rejects_invalid_arguments(lib):
    f = lib.kda_segids_to_cu_seqlens
    assert f(None, 1, 4, 4, FAKE, None, None) == -1
    assert f(FAKE, 1, 4, 4, None, None, None) == -1
    assert f(FAKE, 0, 4, 4, FAKE, None, None) == -1
    assert f(FAKE, 1, 0, 4, FAKE, None, None) == -1
    assert f(FAKE, 1, 4, 0, FAKE, None, None) == -1
    assert f(ODD, 1, 4, 4, FAKE, None, None) == -1
    assert f(FAKE, 1 << 20, 1 << 12, 4, FAKE, None, None) == -1


def test_conv_rejects_invalid_arguments(lib):
    f = lib.kda_short_conv_varlen
    assert f(None, FAKE, None, FAKE, 1, 4, 8, 4, 1, None) == -1
    assert f(FAKE, FAKE, None, FAKE, 1, 4, 8, 0, 1, None) == -2     # k_conv out of range
    assert f(FAKE, FAKE, None, FAKE, 1, 4, 8, 9, 1, None) == -2
    assert f(FAKE, FAKE, None, FAKE, 1, 4, 7, 4, 1, None) == -2     # F*2 not a multiple of 16
    assert f(ODD, FAKE, None, FAKE, 1, 4, 8, 4, 1, None) == -1      # misaligned
    assert f(FAKE, FAKE, None, FAKE, 1, 4, 8, 4, 3, None) == -1     # dtype


@pytest.mark.parametrize("fname", ["kda_chunk_fwd_varlen", "kda_chunk_fwd_varlen_planned",
                                   "kda_delta_fwd_varlen"])
def test_chunk_rejects_invalid_arguments(lib, fname):
    f = getattr(lib, fname)
    ws = lib.kda_chunk_fwd_varlen_workspace_min(1, 64, 2, 64, 64, kda.KDA_BF16)
    args = [FAKE] * 5 + [None, 1, 64, 2, 64, 64, ctypes.c_float(1.0), kda.KDA_BF16, kda.KDA_BF16,
                         FAKE, FAKE, ws, None, None]

    def call(**over):
        a = list(args)
        idx = {"q": 0, "seg": 5, "B": 6, "H": 8, "dk": 9, "dv": 10, "dtype": 12, "out_dtype": 13,
               "o": 14, "ws": 15, "ws_bytes": 16, "status": 17}
        for k, v in over.items():
            a[idx[k]] = v
        return f(*a)

    assert call(q=None) == -1
    assert call(o=None) == -1
    assert call(q=ODD) == -1
    assert call(B=0) == -1
    assert call(dtype=5) == -1
    assert call(out_dtype=5) == -1
    assert call(dtype=kda.KDA_F32, out_dtype=kda.KDA_BF16) == -2   # no narrowing output
    assert call(dk=96, dv=96) == -2
    assert call(dk=64, dv=128) == -2
    assert call(ws=None) == -4
    assert call(ws_bytes=ws - 1) == -4
    assert call(ws=ctypes.c_void_p(4096 + 16)) == -4          # workspace must be 256-aligned
    assert call(status=ODD) == -1


def test_chunk_conv_rejects_invalid_arguments(lib):
    """kda_chunk_fwd_varlen_conv: the forward's checks, then its own (no launch is reached)."""
    f = lib.kda_chunk_fwd_varlen_conv
    ws = lib.kda_chunk_fwd_varlen_workspace_min(1, 64, 2, 128, 128, kda.KDA_BF16)
    args = [FAKE] * 6 + [4, FAKE, FAKE, None, 1, 64, 2, 128, 128, ctypes.c_float(1.0),
                         kda.KDA_BF16, kda.KDA_BF16, FAKE, FAKE, ws, 0, None, None]

    def call(**over):
        a = list(args)
        idx = {"xq": 0, "wq": 3, "wv": 5, "K": 6, "g": 7, "seg": 9, "B": 10, "H": 12, "dk": 13,
               "dv": 14, "dtype": 16, "out_dtype": 17, "o": 18, "ws": 19, "ws_bytes": 20,
               "status": 22}
        for k, v in over.items():
            a[idx[k]] = v
        return f(*a)

    assert call(xq=None) == -1
    assert call(wq=None) == -1
    assert call(wv=ODD) == -1
    assert call(g=ODD) == -1
    assert call(o=None) == -1
    assert call(B=0) == -1
    assert call(dtype=5) == -1
    assert call(ws=None) == -4
    assert call(ws_bytes=ws - 1) == -4
    # the fused path: bf16, 128-wide heads, up to 4 taps (other forms run the convs apart)
    assert call(K=0) == -2
    assert call(K=5) == -2
    assert call(dtype=kda.KDA_F32, out_dtype=kda.KDA_F32,
                ws_bytes=lib.kda_chunk_fwd_varlen_workspace_min(1, 64, 2, 128, 128,
                                                                kda.KDA_F32)) == -2
    ws64 = lib.kda_chunk_fwd_varlen_workspace_min(1, 64, 2, 64, 64, kda.KDA_BF16)
    assert call(dk=64, dv=64, ws_bytes=ws64) == -2
    assert call(dk=96, dv=96) == -2


def test_selftest_wait_timeout_rejects_invalid_arguments(lib):
    """The bounded-wait self-test checks its arguments before any launch."""
    f = lib.kda_selftest_wait_timeout
    assert f(50_000_000, None, None) == -1                     # no status word
    assert f(50_000_000, ODD, None) == -1                      # misaligned
    assert f(999_999, FAKE, None) == -1                        # below 1 ms
    assert f(10_000_000_001, FAKE, None) == -1                 # above 10 s


def test_chunk_plan_rejects_invalid_arguments(lib):
    f = lib.kda_chunk_plan_varlen
    ws = lib.kda_chunk_fwd_varlen_workspace_min(1, 64, 2, 128, 128, kda.KDA_BF16)
    args = [FAKE, 1, 64, 2, 128, 128, kda.KDA_BF16, FAKE, ws, None]

    def call(**over):
        a = list(args)
        idx = {"seg": 0, "B": 1, "T": 2, "H": 3, "dk": 4, "dv": 5, "dtype": 6, "ws": 7,
               "ws_bytes": 8}
        for k, v in over.items():
            a[idx[k]] = v
        return f(*a)

    assert call(seg=ODD) == -1
    assert call(B=0) == -1
    assert call(T=0) == -1
    assert call(H=0) == -1
    assert call(dtype=5) == -1
    assert call(dk=96, dv=96) == -2
    assert call(dk=64, dv=128) == -2
    assert call(ws=None) == -4
    assert call(ws_bytes=ws - 1) == -4
    assert call(ws=ctypes.c_void_p(4096 + 16)) == -4


def test_chunk_state_rejects_invalid_arguments(lib):
    f = lib.kda_chunk_fwd_varlen_state
    ws = lib.kda_chunk_fwd_varlen_workspace_min(1, 64, 2, 64, 64, kda.KDA_BF16)
    args = [FAKE] * 5 + [None, 1, 64, 2, 64, 64, ctypes.c_float(1.0), kda.KDA_BF16, kda.KDA_BF16,
                         FAKE, FAKE, FAKE, 3, FAKE, ws, None, None]

    def call(**over):
        a = list(args)
        idx = {"q": 0, "B": 6, "dk": 9, "dv": 10, "o": 14, "init": 15, "fin": 16, "n_state": 17,
               "ws": 18, "ws_bytes": 19}
        for k, v in over.items():
            a[idx[k]] = v
        return f(*a)

    assert call(q=None) == -1
    assert call(o=None) == -1
    assert call(B=0) == -1
    assert call(n_state=-1) == -1
    assert call(init=ODD) == -1
    assert call(fin=ODD) == -1
    assert call(dk=96, dv=96) == -2
    assert call(ws=None) == -4
    assert call(ws_bytes=ws - 1) == -4


def test_chunk_bwd_rejects_invalid_arguments(lib):
    f = lib.kda_chunk_bwd_varlen
    ws = lib.kda_chunk_bwd_varlen_workspace_size(1, 64, 2, 64, 64, kda.KDA_BF16)
    assert ws > 0
    assert lib.kda_chunk_bwd_varlen_workspace_size(1, 64, 2, 96, 96, kda.KDA_BF16) == 0
    args = [FAKE] * 5 + [None, 1, 64, 2, 64, 64, ctypes.c_float(1.0), kda.KDA_BF16, FAKE,
                         kda.KDA_BF16] + [FAKE] * 5 + [FAKE, ws, None]

    def call(**over):
        a = list(args)
        idx = {"q": 0, "B": 6, "dk": 9, "dv": 10, "d_o": 13, "gdt": 14, "dq": 15, "dbeta": 19,
               "ws": 20, "ws_bytes": 21}
        for k, v in over.items():
            a[idx[k]] = v
        return f(*a)

    assert call(q=None) == -1
    assert call(d_o=None) == -1
    assert call(dbeta=None) == -1
    assert call(dq=ODD) == -1
    assert call(B=0) == -1
    assert call(dk=96, dv=96) == -2
    assert call(gdt=kda.KDA_BF16 + 7) == -1
    assert call(ws=None) == -4
    assert call(ws_bytes=ws - 1) == -4


def test_chunk_bwd_ex_rejects_invalid_arguments(lib):
    """kda_chunk_bwd_varlen_ex: kda_chunk_bwd_varlen's checks, plus the method and the status
    word's alignment; the workspace size covers either method."""
    f = lib.kda_chunk_bwd_varlen_ex
    ws = lib.kda_chunk_bwd_varlen_workspace_size(1, 64, 2, 128, 128, kda.KDA_BF16)
    # the tensor-core path keeps two fp32-sized states per chunk and head (2 x 64 KB)
    assert ws >= 2 * 2 * 65536
    assert lib.kda_chunk_bwd_varlen_workspace_size(1, 64, 2, 128, 128, kda.KDA_F32) < ws
    args = [FAKE] * 5 + [None, 1, 64, 2, 128, 128, ctypes.c_float(1.0), kda.KDA_BF16, FAKE,
                         kda.KDA_BF16] + [FAKE] * 5 + [FAKE, ws, kda.KDA_BWD_AUTO, None, None]

    def call(**over):
        a = list(args)
        idx = {"q": 0, "B": 6, "dk": 9, "dv": 10, "d_o": 13, "dq": 15, "ws": 20,
               "ws_bytes": 21, "method": 22, "status": 23}
        for k, v in over.items():
            a[idx[k]] = v
        return f(*a)

    assert call(q=None) == -1
    assert call(dq=ODD) == -1
    assert call(method=2) == -1
    assert call(method=-1) == -1
    assert call(status=ODD) == -1
    assert call(dk=96, dv=96) == -2
    assert call(ws_bytes=ws - 1) == -4
    assert call(method=kda.KDA_BWD_WALK, ws=None) == -4
