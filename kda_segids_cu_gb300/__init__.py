"""libkda: packed (varlen) Kimi Delta Attention forward for NVIDIA GB300.

A thin ctypes binding over the C ABI in include/kda.h. Every step of the
computation runs in libkda's CUDA kernels; this module only checks tensor
properties, allocates outputs and workspace with torch, and passes device
pointers plus the current CUDA stream. There is no CPU fallback: if
libkda.so is missing or a call fails, an exception is raised.

Calls (same names as the C ABI; segids_to_cu_seqlens, short_conv_varlen and
chunk_fwd_varlen are the same functions under shorter names):
  kda_segids_to_cu_seqlens(segment_ids, max_segs) -> (cu_seqlens, n_segs)
  kda_short_conv_varlen(x, weight, segment_ids=None) -> y
  kda_chunk_fwd_varlen(q, k, v, g, beta, segment_ids=None, scale=1.0) -> o
  kda_chunk_plan_varlen / kda_chunk_fwd_varlen(..., planned=True), the same in two calls
  kda_chunk_fwd_varlen_state(...) -> (o, final states): per-segment initial/final state
  kda_chunk_bwd_varlen(...) -> (dq, dk, dv, dg, dbeta), and kda_varlen (autograd)
The forward wrappers read the kernels' device status word after the call and
raise KdaDeviceError when a bit is set, unless told not to (check=False) or
given a status tensor of the caller's.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "kda.h")

KDA_OK = 0
KDA_F32 = 0
KDA_BF16 = 1
KDA_DEV_DECAY_RANGE = 0x1
KDA_DEV_TIMEOUT = 0x2

_lib = None


class KdaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        name = load_library().kda_status_string(status).decode()
        super().__init__(f"{fn} failed: {name} ({status})")


class KdaDeviceError(RuntimeError):
    """A condition the kernels reported through the device status word (KDA_DEV_* bits)."""

    def __init__(self, fn: str, bits: int):
        self.bits = bits
        names = [n for b, n in ((KDA_DEV_DECAY_RANGE, "KDA_DEV_DECAY_RANGE"),
                                (KDA_DEV_TIMEOUT, "KDA_DEV_TIMEOUT")) if bits & b]
        super().__init__(f"{fn}: device status {bits:#x} ({', '.join(names) or 'unknown'}); "
                         "the outputs of this call are unreliable")


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libkda.so (built by __graft_entry__.build() or kda_segids_cu_gb300.build)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libkda.so not found at {p}: build it with "
                           "`python -m kda_segids_cu_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(p)
    vp, i64, i32, u32p = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_segids_to_cu_seqlens.argtypes = [vp, i64, i64, i32, vp, vp, vp]
    lib.kda_segids_to_cu_seqlens.restype = ctypes.c_int
    lib.kda_short_conv_varlen.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, ctypes.c_int, vp]
    lib.kda_short_conv_varlen.restype = ctypes.c_int
    lib.kda_chunk_fwd_varlen_workspace_size.argtypes = [i64, i64, i32, i32, i32, ctypes.c_int]
    lib.kda_chunk_fwd_varlen_workspace_size.restype = ctypes.c_size_t
    lib.kda_chunk_fwd_varlen_workspace_min.argtypes = [i64, i64, i32, i32, i32, ctypes.c_int]
    lib.kda_chunk_fwd_varlen_workspace_min.restype = ctypes.c_size_t
    lib.kda_chunk_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, i32,
                                         ctypes.c_float, ctypes.c_int, ctypes.c_int, vp, vp,
                                         ctypes.c_size_t, u32p, vp]
    lib.kda_chunk_fwd_varlen.restype = ctypes.c_int
    lib.kda_chunk_plan_varlen.argtypes = [vp, i64, i64, i32, i32, i32, ctypes.c_int, vp,
                                          ctypes.c_size_t, vp]
    lib.kda_chunk_plan_varlen.restype = ctypes.c_int
    lib.kda_chunk_fwd_varlen_planned.argtypes = lib.kda_chunk_fwd_varlen.argtypes
    lib.kda_chunk_fwd_varlen_planned.restype = ctypes.c_int
    lib.kda_chunk_fwd_varlen_conv.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, i64, i64,
                                              i32, i32, i32, ctypes.c_float, ctypes.c_int,
                                              ctypes.c_int, vp, vp, ctypes.c_size_t, ctypes.c_int,
                                              u32p, vp]
    lib.kda_chunk_fwd_varlen_conv.restype = ctypes.c_int
    lib.kda_delta_fwd_varlen.argtypes = lib.kda_chunk_fwd_varlen.argtypes
    lib.kda_delta_fwd_varlen.restype = ctypes.c_int
    lib.kda_selftest_wait_timeout.argtypes = [ctypes.c_uint64, u32p, vp]
    lib.kda_selftest_wait_timeout.restype = ctypes.c_int
    lib.kda_chunk_fwd_varlen_state.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, i32,
                                               ctypes.c_float, ctypes.c_int, ctypes.c_int, vp,
                                               vp, vp, i64, vp, ctypes.c_size_t, u32p, vp]
    lib.kda_chunk_fwd_varlen_state.restype = ctypes.c_int
    lib.kda_chunk_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, i32,
                                         ctypes.c_float, ctypes.c_int, vp, ctypes.c_int, vp, vp,
                                         vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.kda_chunk_bwd_varlen.restype = ctypes.c_int
    lib.kda_chunk_bwd_varlen_ex.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, i32,
                                            ctypes.c_float, ctypes.c_int, vp, ctypes.c_int, vp,
                                            vp, vp, vp, vp, vp, ctypes.c_size_t, i32, u32p, vp]
    lib.kda_chunk_bwd_varlen_ex.restype = ctypes.c_int
    lib.kda_chunk_bwd_varlen_workspace_size.argtypes = [i64, i64, i32, i32, i32, ctypes.c_int]
    lib.kda_chunk_bwd_varlen_workspace_size.restype = ctypes.c_size_t
    if path is None:
        _lib = lib
    return lib


def header_functions(header: str = HEADER) -> list[str]:
    """Names of the functions that include/kda.h declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return KDA_BF16
    if t == torch.float32:
        return KDA_F32
    raise TypeError(f"unsupported dtype {t}: libkda takes bfloat16 or float32")


def _stream_ptr(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(fn: str, status: int) -> None:
    if status != KDA_OK:
        raise KdaError(fn, status)


def _status_word(status: torch.Tensor | None, check: bool | None, device, stream):
    """The device status word of a forward call and whether the wrapper reads it.

    check=None (the default) reads it when the wrapper owns the word (status is None) and
    the stream is not being captured; check=True always reads it (not under capture);
    check=False never does. Reading means waiting for the stream."""
    s = torch.cuda.current_stream(device) if stream is None else stream
    capturing = torch.cuda.is_current_stream_capturing()
    if check is None:
        check = status is None and not capturing
    elif check and capturing:
        raise ValueError("check=True cannot wait under stream capture: pass a status tensor "
                         "and read it after the graph runs")
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=device)
    elif check:
        status.zero_()
    return status, check, s


def _raise_on_status(fn: str, status: torch.Tensor, stream) -> None:
    stream.synchronize()
    bits = int(status.item()) & 0xffffffff
    if bits:
        raise KdaDeviceError(fn, bits)


def kda_segids_to_cu_seqlens(segment_ids: torch.Tensor, max_segs: int, stream=None,
                             out: torch.Tensor | None = None,
                             n_segs_out: torch.Tensor | None = None):
    """[B, T] int32 ids -> (cu_seqlens int32 [max_segs+1], n_segs int32 [1]) on the device."""
    seg = _dev(segment_ids, "segment_ids")
    if seg.dtype != torch.int32 or seg.dim() != 2:
        raise ValueError("segment_ids must be int32 [B, T]")
    B, T = seg.shape
    cu = out if out is not None else torch.empty(max_segs + 1, dtype=torch.int32, device=seg.device)
    n = n_segs_out if n_segs_out is not None else torch.empty(1, dtype=torch.int32, device=seg.device)
    _check("kda_segids_to_cu_seqlens",
           load_library().kda_segids_to_cu_seqlens(_ptr(seg), B, T, int(max_segs), _ptr(cu),
                                                   _ptr(n), _stream_ptr(stream)))
    return cu, n


def kda_short_conv_varlen(x: torch.Tensor, weight: torch.Tensor,
                          segment_ids: torch.Tensor | None = None, stream=None,
                          out: torch.Tensor | None = None) -> torch.Tensor:
    """Segment-masked causal depthwise conv: x [B, T, F], weight [K, F] -> y [B, T, F]."""
    x = _dev(x, "x")
    weight = _dev(weight, "weight")
    if x.dim() != 3 or weight.dim() != 2 or weight.shape[1] != x.shape[2]:
        raise ValueError("expected x [B, T, F] and weight [K, F]")
    if weight.dtype != x.dtype:
        raise ValueError("x and weight must share a dtype")
    B, T, F = x.shape
    seg = None
    if segment_ids is not None:
        seg = _dev(segment_ids, "segment_ids")
        if seg.dtype != torch.int32 or tuple(seg.shape) != (B, T):
            raise ValueError("segment_ids must be int32 [B, T]")
    y = out if out is not None else torch.empty_like(x)
    _check("kda_short_conv_varlen",
           load_library().kda_short_conv_varlen(_ptr(x), _ptr(weight), _ptr(seg), _ptr(y), B, T,
                                                F, weight.shape[0], _dtype_code(x.dtype),
                                                _stream_ptr(stream)))
    return y


def chunk_fwd_workspace_bytes(B: int, T: int, H: int, d_qk: int, d_v: int, dtype,
                              minimum: bool = False) -> int:
    """Workspace bytes of the forward: the full size (room to split long segments) or, with
    minimum=True, the least the entry points accept."""
    lib = load_library()
    fn = lib.kda_chunk_fwd_varlen_workspace_min if minimum else lib.kda_chunk_fwd_varlen_workspace_size
    return int(fn(B, T, H, d_qk, d_v, _dtype_code(dtype)))


def _chunk_args(q, k, v, g, beta, segment_ids, B, T, out, workspace, out_dtype,
                workspace_size=None, want_out=True):
    """Checks and marshals the arguments the chunk entry points share; allocates o (if
    want_out) and the workspace (workspace_size(B, T, H, Dk, Dv, dtype code) bytes, by
    default the forward's) when they are not given."""
    q, k, v, g, beta = (_dev(t, n) for t, n in ((q, "q"), (k, "k"), (v, "v"), (g, "g"),
                                                 (beta, "beta")))
    H, Dk = q.shape[-2], q.shape[-1]
    Dv = v.shape[-1]
    N = q.numel() // (H * Dk)
    if segment_ids is not None:
        seg = _dev(segment_ids, "segment_ids")
        if seg.dtype != torch.int32 or seg.dim() != 2:
            raise ValueError("segment_ids must be int32 [B, T]")
        B, T = seg.shape
    else:
        seg = None
        if B is None or T is None:
            if q.dim() == 4:
                B, T = q.shape[0], q.shape[1]
            else:
                B, T = 1, N
    if B * T != N:
        raise ValueError(f"token count mismatch: B*T = {B * T}, tensors hold {N}")
    for t, n, d in ((k, "k", Dk), (g, "g", Dk), (v, "v", Dv)):
        if t.numel() != N * H * d or t.shape[-1] != d or t.dtype != q.dtype:
            raise ValueError(f"{n} has an unexpected shape or dtype")
    if beta.numel() != N * H or beta.dtype != q.dtype:
        raise ValueError("beta must hold B*T*H values of q's dtype")
    dt = _dtype_code(q.dtype)
    out_dtype = q.dtype if out_dtype is None else out_dtype
    if out is not None:
        out_dtype = out.dtype
        if out.numel() != v.numel() or not out.is_contiguous():
            raise ValueError("out must be a contiguous tensor with v's element count")
    odt = _dtype_code(out_dtype)
    o = None
    if want_out:
        o = out if out is not None else torch.empty(v.shape, dtype=out_dtype, device=v.device)
    if workspace is None:
        if workspace_size is None:
            need = chunk_fwd_workspace_bytes(B, T, H, Dk, Dv, q.dtype)
        else:
            need = int(workspace_size(B, T, H, Dk, Dv, dt))
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    return q, k, v, g, beta, seg, B, T, H, Dk, Dv, dt, odt, o, workspace


def kda_chunk_fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                         beta: torch.Tensor, segment_ids: torch.Tensor | None = None,
                         scale: float = 1.0, B: int | None = None, T: int | None = None,
                         stream=None, out: torch.Tensor | None = None,
                         workspace: torch.Tensor | None = None,
                         status: torch.Tensor | None = None,
                         out_dtype: torch.dtype | None = None,
                         planned: bool = False, check: bool | None = None) -> torch.Tensor:
    """Packed KDA forward. q, k, g: [B, T, H, Dk], [1, B*T, H, Dk] or [B*T, H, Dk];
    v like q with Dv; beta [..., H]; segment_ids int32 [B, T] or None.
    Returns o shaped like v, of `out_dtype` (default: the input dtype; float32
    is also accepted). planned=True skips the planning: `workspace` must hold the
    plan of these segment ids and sizes from kda_chunk_plan_varlen.

    Device-side conditions (KDA_DEV_* bits) go to `status`, an int32 device tensor
    ORed into and never cleared by the kernels. By default (status None, check None)
    the wrapper allocates the word, waits for the stream after the launch and raises
    KdaDeviceError if a bit is set. Pass check=False to skip that wait (the word is
    then the caller's to read), or pass your own `status` to read it yourself; under
    stream capture the wrapper never waits."""
    if planned and workspace is None:
        raise ValueError("planned=True needs the workspace that holds the plan")
    q, k, v, g, beta, seg, B, T, H, Dk, Dv, dt, odt, o, workspace = _chunk_args(
        q, k, v, g, beta, segment_ids, B, T, out, workspace, out_dtype)
    status, check, st = _status_word(status, check, q.device, stream)
    lib = load_library()
    fn, name = ((lib.kda_chunk_fwd_varlen_planned, "kda_chunk_fwd_varlen_planned") if planned
                else (lib.kda_chunk_fwd_varlen, "kda_chunk_fwd_varlen"))
    _check(name, fn(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(seg), B, T, H, Dk, Dv,
                    float(scale), dt, odt, _ptr(o), _ptr(workspace), workspace.numel(),
                    _ptr(status), _stream_ptr(st)))
    if check:
        _raise_on_status(name, status, st)
    return o


def kda_chunk_fwd_varlen_conv(x_q: torch.Tensor, x_k: torch.Tensor, x_v: torch.Tensor,
                              w_q: torch.Tensor, w_k: torch.Tensor, w_v: torch.Tensor,
                              g: torch.Tensor, beta: torch.Tensor,
                              segment_ids: torch.Tensor | None = None, scale: float = 1.0,
                              B: int | None = None, T: int | None = None, stream=None,
                              out: torch.Tensor | None = None,
                              workspace: torch.Tensor | None = None,
                              status: torch.Tensor | None = None,
                              out_dtype: torch.dtype | None = None, planned: bool = False,
                              check: bool | None = None) -> torch.Tensor:
    """kda_chunk_fwd_varlen on q, k, v = the segment-masked short convs of x_q, x_k, x_v
    (weights w_q, w_k, w_v [K, H*D], as kda_short_conv_varlen), with the convs done inside
    the chunk kernel. The result equals the three conv calls followed by
    kda_chunk_fwd_varlen bit for bit. x_*: [B, T, H*D] or shaped like g. bf16, 128-wide
    heads and K <= 4; other arguments as in kda_chunk_fwd_varlen."""
    if planned and workspace is None:
        raise ValueError("planned=True needs the workspace that holds the plan")
    g = _dev(g, "g")
    xs = []
    for x, n in ((x_q, "x_q"), (x_k, "x_k"), (x_v, "x_v")):
        x = _dev(x, n)
        if x.numel() != g.numel():
            raise ValueError(f"{n} must hold as many values as g")
        xs.append(x.view(g.shape))
    ws_ = []
    for w, n in ((w_q, "w_q"), (w_k, "w_k"), (w_v, "w_v")):
        w = _dev(w, n)
        if w.dim() != 2 or w.shape[1] != g.shape[-2] * g.shape[-1] or w.dtype != g.dtype:
            raise ValueError(f"{n} must be [K, H*D] of g's dtype")
        ws_.append(w)
    if not (ws_[0].shape == ws_[1].shape == ws_[2].shape):
        raise ValueError("the three conv weights must have one shape")
    q, k, v, g, beta, seg, B, T, H, Dk, Dv, dt, odt, o, workspace = _chunk_args(
        xs[0], xs[1], xs[2], g, beta, segment_ids, B, T, out, workspace, out_dtype)
    status, check, st = _status_word(status, check, q.device, stream)
    name = "kda_chunk_fwd_varlen_conv"
    _check(name, load_library().kda_chunk_fwd_varlen_conv(
        _ptr(q), _ptr(k), _ptr(v), _ptr(ws_[0]), _ptr(ws_[1]), _ptr(ws_[2]), ws_[0].shape[0],
        _ptr(g), _ptr(beta), _ptr(seg), B, T, H, Dk, Dv, float(scale), dt, odt, _ptr(o),
        _ptr(workspace), workspace.numel(), int(planned), _ptr(status), _stream_ptr(st)))
    if check:
        _raise_on_status(name, status, st)
    return o


def kda_delta_fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                         beta: torch.Tensor, segment_ids: torch.Tensor | None = None,
                         scale: float = 1.0, B: int | None = None, T: int | None = None,
                         stream=None, out: torch.Tensor | None = None,
                         workspace: torch.Tensor | None = None,
                         status: torch.Tensor | None = None,
                         out_dtype: torch.dtype | None = None,
                         check: bool | None = None) -> torch.Tensor:
    """The delta-rule form of the recurrence, S_t = S'_t + beta_t k_t (v_t - S'_t^T k_t)^T
    (the reading of the method's name; the pages state only the additive update), as a
    token recurrence in fp32 arithmetic. Arguments as kda_chunk_fwd_varlen."""
    q, k, v, g, beta, seg, B, T, H, Dk, Dv, dt, odt, o, workspace = _chunk_args(
        q, k, v, g, beta, segment_ids, B, T, out, workspace, out_dtype)
    status, check, st = _status_word(status, check, q.device, stream)
    name = "kda_delta_fwd_varlen"
    _check(name, load_library().kda_delta_fwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(seg), B, T, H, Dk, Dv,
        float(scale), dt, odt, _ptr(o), _ptr(workspace), workspace.numel(), _ptr(status),
        _stream_ptr(st)))
    if check:
        _raise_on_status(name, status, st)
    return o


def kda_selftest_wait_timeout(timeout_s: float = 0.05, status: torch.Tensor | None = None,
                              stream=None) -> torch.Tensor:
    """Runs the library's bounded in-kernel wait on a barrier that nothing arrives on, for
    about timeout_s seconds of GPU time; the kernel then sets KDA_DEV_TIMEOUT in `status`
    (an int32 device word, allocated if None) and returns. Returns the word, unread."""
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
    status = _dev(status, "status")
    _check("kda_selftest_wait_timeout",
           load_library().kda_selftest_wait_timeout(int(timeout_s * 1e9), _ptr(status),
                                                    _stream_ptr(stream)))
    return status


def kda_chunk_plan_varlen(segment_ids: torch.Tensor | None, B: int, T: int, H: int, d_qk: int,
                          d_v: int, dtype: torch.dtype, workspace: torch.Tensor,
                          stream=None) -> torch.Tensor:
    """Writes the plan of a forward over these segment ids and sizes into `workspace`
    (the forward's workspace), for kda_chunk_fwd_varlen(..., planned=True). Reads only
    segment_ids; returns the workspace."""
    seg = None
    if segment_ids is not None:
        seg = _dev(segment_ids, "segment_ids")
        if seg.dtype != torch.int32 or tuple(seg.shape) != (B, T):
            raise ValueError("segment_ids must be int32 [B, T]")
    ws = _dev(workspace, "workspace")
    _check("kda_chunk_plan_varlen",
           load_library().kda_chunk_plan_varlen(_ptr(seg), B, T, H, d_qk, d_v,
                                                _dtype_code(dtype), _ptr(ws), ws.numel(),
                                                _stream_ptr(stream)))
    return ws


def kda_chunk_fwd_varlen_state(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                               g: torch.Tensor, beta: torch.Tensor,
                               segment_ids: torch.Tensor | None = None, scale: float = 1.0,
                               B: int | None = None, T: int | None = None,
                               initial_state: torch.Tensor | None = None,
                               output_final_state: bool = False, n_state: int | None = None,
                               stream=None, out: torch.Tensor | None = None,
                               workspace: torch.Tensor | None = None,
                               status: torch.Tensor | None = None,
                               out_dtype: torch.dtype | None = None,
                               check: bool | None = None):
    """kda_chunk_fwd_varlen with per-segment state: segment r (flattened token order,
    as in cu_seqlens) starts from initial_state[r] ([n_state, H, Dk, Dv] float32) and,
    with output_final_state, its state after its last token is returned in
    final[r]. n_state defaults to initial_state's first dimension (else 0).
    Returns (o, final or None). `status` and `check` as in kda_chunk_fwd_varlen."""
    q, k, v, g, beta, seg, B, T, H, Dk, Dv, dt, odt, o, workspace = _chunk_args(
        q, k, v, g, beta, segment_ids, B, T, out, workspace, out_dtype)
    status, check, st = _status_word(status, check, q.device, stream)
    if n_state is None:
        n_state = initial_state.shape[0] if initial_state is not None else 0
    init = None
    if initial_state is not None:
        init = _dev(initial_state, "initial_state")
        if init.dtype != torch.float32 or init.numel() != n_state * H * Dk * Dv:
            raise ValueError("initial_state must be float32 [n_state, H, Dk, Dv]")
    fin = None
    if output_final_state:
        fin = torch.zeros((n_state, H, Dk, Dv), dtype=torch.float32, device=q.device)
    _check("kda_chunk_fwd_varlen_state",
           load_library().kda_chunk_fwd_varlen_state(
               _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(seg), B, T, H, Dk, Dv,
               float(scale), dt, odt, _ptr(o), _ptr(init), _ptr(fin), int(n_state),
               _ptr(workspace), workspace.numel(), _ptr(status), _stream_ptr(st)))
    if check:
        _raise_on_status("kda_chunk_fwd_varlen_state", status, st)
    return o, fin


KDA_BWD_AUTO = 0
KDA_BWD_WALK = 1
_BWD_METHODS = {"auto": KDA_BWD_AUTO, "walk": KDA_BWD_WALK}


def kda_chunk_bwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                         beta: torch.Tensor, d_o: torch.Tensor,
                         segment_ids: torch.Tensor | None = None, scale: float = 1.0,
                         B: int | None = None, T: int | None = None, stream=None,
                         workspace: torch.Tensor | None = None,
                         grad_dtype: torch.dtype | None = None, method: str = "auto",
                         status: torch.Tensor | None = None, check: bool | None = None):
    """Gradients of kda_chunk_fwd_varlen for the upstream gradient d_o (shaped like v, of
    the input dtype). Returns (dq, dk, dv, dg, dbeta) shaped like q, k, v, g, beta, of
    `grad_dtype` (default: the input dtype; float32 is also accepted).

    method="auto" runs bf16 inputs with 128-wide heads on the tensor-core path (the bf16
    bound) and everything else on the fp32 walks; method="walk" forces the walks (the fp32
    bound). The device status word is handled as in kda_chunk_fwd_varlen."""
    if method not in _BWD_METHODS:
        raise ValueError(f"method must be one of {sorted(_BWD_METHODS)}")
    q, k, v, g, beta, seg, B, T, H, Dk, Dv, dt, _, _, workspace = _chunk_args(
        q, k, v, g, beta, segment_ids, B, T, None, workspace, None,
        workspace_size=load_library().kda_chunk_bwd_varlen_workspace_size, want_out=False)
    d_o = _dev(d_o, "d_o")
    if d_o.numel() != v.numel() or d_o.dtype != q.dtype:
        raise ValueError("d_o must be shaped like v, of the input dtype")
    grad_dtype = q.dtype if grad_dtype is None else grad_dtype
    gdt = _dtype_code(grad_dtype)
    dq, dk, dv, dg, db = (torch.empty(t.shape, dtype=grad_dtype, device=q.device)
                          for t in (q, k, v, g, beta))
    status, check, st = _status_word(status, check, q.device, stream)
    _check("kda_chunk_bwd_varlen",
           load_library().kda_chunk_bwd_varlen_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                                  _ptr(seg), B, T, H, Dk, Dv, float(scale), dt,
                                                  _ptr(d_o), gdt, _ptr(dq), _ptr(dk), _ptr(dv),
                                                  _ptr(dg), _ptr(db), _ptr(workspace),
                                                  workspace.numel(), _BWD_METHODS[method],
                                                  _ptr(status), _stream_ptr(st)))
    if check:
        _raise_on_status("kda_chunk_bwd_varlen", status, st)
    return dq, dk, dv, dg, db


class _KdaVarlen(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, g, beta, segment_ids, scale, B, T):
        ctx.save_for_backward(q, k, v, g, beta, segment_ids)
        ctx.scale, ctx.B, ctx.T = scale, B, T
        return kda_chunk_fwd_varlen(q, k, v, g, beta, segment_ids, scale=scale, B=B, T=T)

    @staticmethod
    def backward(ctx, d_o):
        q, k, v, g, beta, seg = ctx.saved_tensors
        grads = kda_chunk_bwd_varlen(q, k, v, g, beta, d_o.contiguous(), seg, scale=ctx.scale,
                                     B=ctx.B, T=ctx.T)
        return (*grads, None, None, None, None)


def kda_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
               beta: torch.Tensor, segment_ids: torch.Tensor | None = None, scale: float = 1.0,
               B: int | None = None, T: int | None = None) -> torch.Tensor:
    """kda_chunk_fwd_varlen as a differentiable op: its backward runs kda_chunk_bwd_varlen."""
    return _KdaVarlen.apply(q, k, v, g, beta, segment_ids, scale, B, T)


# The shorter names the boundary's description uses, for the same calls.
segids_to_cu_seqlens = kda_segids_to_cu_seqlens
short_conv_varlen = kda_short_conv_varlen
chunk_fwd_varlen = kda_chunk_fwd_varlen

__all__ = ["segids_to_cu_seqlens", "short_conv_varlen", "chunk_fwd_varlen",
           "kda_segids_to_cu_seqlens", "kda_short_conv_varlen", "kda_chunk_fwd_varlen",
           "kda_chunk_plan_varlen", "kda_chunk_fwd_varlen_state", "kda_chunk_bwd_varlen", "kda_varlen",
           "chunk_fwd_workspace_bytes", "load_library", "header_functions", "KdaError",
           "KdaDeviceError", "KDA_DEV_DECAY_RANGE", "KDA_DEV_TIMEOUT", "KDA_BWD_AUTO", "KDA_BWD_WALK"]
