"""fp64 CPU oracle for the packed (varlen) Kimi Delta Attention forward.

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import this package. It shares no code with the
CUDA library (``kda_segids_cu_gb300``) and never imports it.

The arithmetic lives in ``kda_oracle.c`` (plain C, fp64), built with gcc into
``libkda_oracle.so`` beside it; this module only marshals arrays:

  cu_seqlens(seg, max_segs)            RFC-0025 方案 §1 (with two amendments,
                                       both switchable to the page's reading)
  short_conv(x, w, seg, out_dtype)     RFC-0025 方案 §3
  kda_fwd(q, k, v, g, beta, seg, ...)  RFC-0026 背景 "KDA 状态泄漏问题" and
                                       §3.1.1 reset semantics
  kda_fwd_state(...)                   the same with per-segment initial and
                                       final states (RFC-0026's kwargs)
  kda_bwd(q, k, v, g, beta, do, seg)   gradients of kda_fwd, by reverse-mode
                                       differentiation of the recurrence
  kda_fwd_delta(...)                   the delta-rule update, the reading of the
                                       method's name (the pages state only the
                                       additive update)

Parity pins live in tests/test_oracle_*.py. Parity status of each function:
cu_seqlens, short_conv, kda_fwd and kda_fwd_state are pinned (worked examples
from the page, library routines, closed forms, brute force and invariants);
kda_bwd is pinned by finite differences of kda_fwd and by automatic
differentiation of the brute-force closed form; kda_fwd_delta by the delta
rule's defining property (with beta = 1 and unit keys the state reads back v_t
along k_t exactly), its projector form and its first-token reduction.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile kda_oracle.c with gcc (portable flags only) and return the .so path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, dp, ip = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p
            lib.oracle_cu_seqlens.argtypes = [ip, i64, i64, i32, ctypes.c_int, ctypes.c_int,
                                              ip, ctypes.POINTER(ctypes.c_int64)]
            lib.oracle_cu_seqlens.restype = ctypes.c_int
            lib.oracle_short_conv.argtypes = [dp, dp, ip, i64, i64, i64, i32, dp]
            lib.oracle_short_conv.restype = ctypes.c_int
            lib.oracle_kda_fwd.argtypes = [dp, dp, dp, dp, dp, ip, i64, i64, i64, i64, i64,
                                           ctypes.c_double, dp, ctypes.c_int]
            lib.oracle_kda_fwd.restype = ctypes.c_int
            lib.oracle_kda_fwd_delta.argtypes = lib.oracle_kda_fwd.argtypes
            lib.oracle_kda_fwd_delta.restype = ctypes.c_int
            lib.oracle_kda_fwd_state.argtypes = [dp, dp, dp, dp, dp, ip, i64, i64, i64, i64, i64,
                                                 ctypes.c_double, dp, dp, i64, dp, ctypes.c_int]
            lib.oracle_kda_fwd_state.restype = ctypes.c_int
            lib.oracle_kda_bwd.argtypes = [dp, dp, dp, dp, dp, ip, i64, i64, i64, i64, i64,
                                           ctypes.c_double, dp, dp, dp, dp, dp, dp, ctypes.c_int]
            lib.oracle_kda_bwd.restype = ctypes.c_int
            _lib = lib
    return _lib


def _np(x, dtype) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().to("cpu")
        if x.dtype == torch.bfloat16:
            x = x.to(torch.float32)   # exact widening
        x = x.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=dtype))


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def cu_seqlens(seg, max_segs: int, force_row_starts: bool = True,
               end_rule: str = "last_real") -> tuple[np.ndarray, int]:
    """RFC-0025 方案 §1 conversion of [B, T] int32 ids to int32 [max_segs+1].

    force_row_starts=True forces a segment start at t = 0 of every row
    (RFC-0026 §3.1.1); end_rule "last_real" ends the last real segment one
    past the last non-padding position, "count" uses the page's count of
    non-padding positions. Returns (cu_seqlens, n_segs).
    """
    s = _np(seg, np.int32)
    if s.ndim == 1:
        s = s[None, :]
    B, T = s.shape
    cu = np.zeros(max_segs + 1, dtype=np.int32)
    n = ctypes.c_int64(0)
    rc = _load().oracle_cu_seqlens(_ptr(s), B, T, int(max_segs), int(force_row_starts),
                                   1 if end_rule == "last_real" else 0, _ptr(cu),
                                   ctypes.byref(n))
    if rc != 0:
        raise ValueError("oracle_cu_seqlens: bad arguments")
    return cu, int(n.value)


def short_conv(x, w, seg=None, out_dtype=None) -> torch.Tensor:
    """RFC-0025 方案 §3 masked causal depthwise conv; x [B, T, F], w [K, F].

    The fp64 sum is rounded once (nearest-even) to `out_dtype` (default: x's
    dtype; torch.float64 keeps it unrounded).
    """
    if out_dtype is None:
        out_dtype = x.dtype if isinstance(x, torch.Tensor) else torch.float64
    xa = _np(x, np.float64)
    wa = _np(w, np.float64)
    B, T, F = xa.shape
    K = wa.shape[0]
    sa = None if seg is None else _np(seg, np.int32).reshape(B, T)
    y = np.zeros_like(xa)
    rc = _load().oracle_short_conv(_ptr(xa), _ptr(wa), _ptr(sa), B, T, F, K, _ptr(y))
    if rc != 0:
        raise ValueError("oracle_short_conv: bad arguments")
    return torch.from_numpy(y).to(out_dtype)


def kda_fwd(q, k, v, g, beta, seg=None, B: int | None = None, T: int | None = None,
            scale: float = 1.0, n_threads: int | None = None,
            out_dtype=torch.float64) -> torch.Tensor:
    """Token-by-token fp64 KDA recurrence (RFC-0026 背景, §3.1.1).

    q, k, g: [B*T, H, Dk] (or [B, T, H, Dk]); v: [B*T, H, Dv]; beta: [B*T, H];
    seg: [B, T] int32 or None (each row one segment). Returns o [B*T, H, Dv]
    (float64 unless out_dtype says otherwise).
    """
    o, _ = kda_fwd_state(q, k, v, g, beta, seg, B=B, T=T, scale=scale, n_threads=n_threads,
                         out_dtype=out_dtype)
    return o


def kda_fwd_delta(q, k, v, g, beta, seg=None, B: int | None = None, T: int | None = None,
                  scale: float = 1.0, n_threads: int | None = None,
                  out_dtype=torch.float64) -> torch.Tensor:
    """The delta-rule recurrence in fp64: S'_t = S_{t-1} exp(g_t) (key rows), S_t = S'_t +
    beta_t k_t (v_t - S'_t^T k_t)^T, o_t = scale S_t^T q_t, with kda_fwd's segments and
    layouts. RFC-0026 names the method Kimi Delta Attention but states only the additive
    update; this is the reading of that name (the gated delta rule, decay per key channel)."""
    qa, ka, va, ga = (_np(t, np.float64) for t in (q, k, v, g))
    ba = _np(beta, np.float64)
    if seg is not None:
        sa = _np(seg, np.int32)
        if sa.ndim == 1:
            sa = sa[None, :]
        if B is None:
            B, T = sa.shape
        sa = sa.reshape(B, T)
    else:
        sa = None
        if B is None:
            B, T = 1, qa.reshape(-1, *qa.shape[-2:]).shape[0]
    Dk, Dv = qa.shape[-1], va.shape[-1]
    H = qa.shape[-2]
    N = B * T
    qa, ka, ga = (a.reshape(N, H, Dk) for a in (qa, ka, ga))
    va = va.reshape(N, H, Dv)
    ba = ba.reshape(N, H)
    o = np.zeros((N, H, Dv), dtype=np.float64)
    nt = default_threads() if n_threads is None else n_threads
    rc = _load().oracle_kda_fwd_delta(_ptr(qa), _ptr(ka), _ptr(va), _ptr(ga), _ptr(ba),
                                      _ptr(sa), B, T, H, Dk, Dv, float(scale), _ptr(o), int(nt))
    if rc != 0:
        raise ValueError("oracle_kda_fwd_delta: bad arguments")
    return torch.from_numpy(o).to(out_dtype)


def kda_fwd_state(q, k, v, g, beta, seg=None, B: int | None = None, T: int | None = None,
                  scale: float = 1.0, initial_state=None, n_state: int = 0,
                  want_final: bool = False, n_threads: int | None = None,
                  out_dtype=torch.float64):
    """The recurrence with per-segment state in and out (RFC-0026, the initial_state /
    output_final_state kwargs of the chunk_kda call).

    Segment r (counted in flattened token order, as in cu_seqlens) starts from
    initial_state[r] ([n_state, H, Dk, Dv]) instead of zero when r < n_state; with
    want_final, final[r] is its state after its last token (zero for r >= the
    segment count). Returns (o, final or None), both float64 unless out_dtype says
    otherwise.
    """
    qa, ka, va, ga = (_np(t, np.float64) for t in (q, k, v, g))
    ba = _np(beta, np.float64)
    if seg is not None:
        sa = _np(seg, np.int32)
        if sa.ndim == 1:
            sa = sa[None, :]
        if B is None:
            B, T = sa.shape
        sa = sa.reshape(B, T)
    else:
        sa = None
        if B is None:
            B, T = 1, qa.reshape(-1, *qa.shape[-2:]).shape[0]
    Dk, Dv = qa.shape[-1], va.shape[-1]
    H = qa.shape[-2]
    N = B * T
    qa, ka, ga = (a.reshape(N, H, Dk) for a in (qa, ka, ga))
    va = va.reshape(N, H, Dv)
    ba = ba.reshape(N, H)
    o = np.zeros((N, H, Dv), dtype=np.float64)
    ia = None
    if initial_state is not None:
        ia = _np(initial_state, np.float64).reshape(n_state, H, Dk, Dv)
    fa = np.zeros((n_state, H, Dk, Dv), dtype=np.float64) if want_final else None
    nt = default_threads() if n_threads is None else n_threads
    rc = _load().oracle_kda_fwd_state(_ptr(qa), _ptr(ka), _ptr(va), _ptr(ga), _ptr(ba),
                                      _ptr(sa), B, T, H, Dk, Dv, float(scale), _ptr(ia),
                                      _ptr(fa), int(n_state), _ptr(o), int(nt))
    if rc != 0:
        raise ValueError("oracle_kda_fwd_state: bad arguments")
    fin = torch.from_numpy(fa).to(out_dtype) if fa is not None else None
    return torch.from_numpy(o).to(out_dtype), fin


def kda_bwd(q, k, v, g, beta, d_o, seg=None, B: int | None = None, T: int | None = None,
            scale: float = 1.0, n_threads: int | None = None, out_dtype=torch.float64):
    """Gradients of kda_fwd with respect to q, k, v, g and beta for the upstream
    gradient d_o ([B*T, H, Dv]). Returns (dq, dk, dv, dg, dbeta), float64 unless
    out_dtype says otherwise; all zero on padding tokens."""
    qa, ka, va, ga, da = (_np(t, np.float64) for t in (q, k, v, g, d_o))
    ba = _np(beta, np.float64)
    if seg is not None:
        sa = _np(seg, np.int32)
        if sa.ndim == 1:
            sa = sa[None, :]
        if B is None:
            B, T = sa.shape
        sa = sa.reshape(B, T)
    else:
        sa = None
        if B is None:
            B, T = 1, qa.reshape(-1, *qa.shape[-2:]).shape[0]
    Dk, Dv = qa.shape[-1], va.shape[-1]
    H = qa.shape[-2]
    N = B * T
    qa, ka, ga = (a.reshape(N, H, Dk) for a in (qa, ka, ga))
    va, da = va.reshape(N, H, Dv), da.reshape(N, H, Dv)
    ba = ba.reshape(N, H)
    dq, dk, dg = (np.zeros((N, H, Dk)) for _ in range(3))
    dv = np.zeros((N, H, Dv))
    db = np.zeros((N, H))
    nt = default_threads() if n_threads is None else n_threads
    rc = _load().oracle_kda_bwd(_ptr(qa), _ptr(ka), _ptr(va), _ptr(ga), _ptr(ba), _ptr(sa), B, T,
                                H, Dk, Dv, float(scale), _ptr(da), _ptr(dq), _ptr(dk), _ptr(dv),
                                _ptr(dg), _ptr(db), int(nt))
    if rc != 0:
        raise ValueError("oracle_kda_bwd: bad arguments or out of memory")
    return tuple(torch.from_numpy(a).to(out_dtype) for a in (dq, dk, dv, dg, db))
