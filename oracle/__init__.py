"""Float64 CPU oracle for exact attention forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never imports, loads or
calls anything here, and this package imports nothing from the product.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, OpenMP
over rows); this module builds it with gcc on first use and wraps it with
ctypes.  Every function takes float32 arrays that hold exactly the values the
GPU sees (bf16 values are widened to float32 without rounding) and returns
float64 arrays.

Parity status per function (what pins it, in ``tests/test_oracle.py``):

* ``attn_fwd``             pinned: closed forms (one key, uniform scores,
                           two keys), shift and permutation invariance, a hand
                           worked example in ``tests/golden``, a float64
                           library cross-check.
* ``attn_fwd_rows``        pinned against ``attn_fwd`` row by row plus the
                           same closed forms.
* ``probs_row``            pinned: rows sum to one, masked keys are zero,
                           ``probs_row @ V`` reproduces the output.
* ``online_replay``        pinned: equals the one-shot result for tile sizes
                           1, 2, N/2, N and the hand two-tile example.
* ``row_softmax``          pinned: closed forms and a library cross-check.
* ``attn_bwd``             pinned: central finite differences of the oracle
                           forward, a float64 library autograd cross-check,
                           and dV = P^T dO row sums.
* ``add_rmsnorm``          pinned: constant rows, a hand-worked row, scale
                           invariance, and a library cross-check.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None

_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``oracle/_build/liboracle.so`` with gcc.

    ``-ffp-contract=off`` keeps the double arithmetic free of fused
    multiply-adds so the oracle rounds the same way on x86 and Arm hosts.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_attn_fwd.argtypes = [_f32p, _f32p, _f32p, _f64p, _f64p,
                                        _i64, _i64, _i64, _i64,
                                        ctypes.c_double, ctypes.c_int, ctypes.c_int]
        lib.oracle_attn_fwd_rows.argtypes = [_f32p, _f32p, _f32p,
                                             _i64, _i64, _i64, _i64,
                                             ctypes.c_double, ctypes.c_int,
                                             _i64p, _i64p, _i64, _f64p, _f64p,
                                             ctypes.c_int]
        lib.oracle_probs_row.argtypes = [_f32p, _f32p, _i64, _i64, _i64,
                                         ctypes.c_double, ctypes.c_int, _f64p]
        lib.oracle_online_replay.argtypes = [_f32p, _f32p, _f32p, _i64, _i64,
                                             ctypes.c_double, ctypes.c_int, _i64,
                                             _f64p, _f64p]
        lib.oracle_row_softmax.argtypes = [_f32p, _i64, _i64, _f64p, _f64p,
                                           ctypes.c_int]
        lib.oracle_add_rmsnorm.argtypes = [_f32p, ctypes.c_void_p, _f32p, _i64, _i64,
                                           ctypes.c_double, _f64p, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_attn_bwd.argtypes = [_f32p, _f32p, _f32p, _f32p, _f32p, _f32p,
                                        _i64, _i64, _i64, _i64, ctypes.c_double, ctypes.c_int,
                                        _f64p, _f64p, _f64p, ctypes.c_int]
        lib.oracle_max_threads.argtypes = []
        for name in ("oracle_attn_fwd", "oracle_attn_fwd_rows", "oracle_probs_row",
                     "oracle_online_replay", "oracle_row_softmax",
                     "oracle_add_rmsnorm", "oracle_attn_bwd", "oracle_max_threads"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _as_f32(x) -> np.ndarray:
    """Widen to a contiguous float32 numpy array (exact for bf16 and fp32)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float32).contiguous().numpy()
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    a = np.ascontiguousarray(x)
    if a.dtype != np.float32:
        if a.dtype == np.float64:
            raise TypeError("oracle inputs must be representable in float32; "
                            "pass float32 (or bf16 widened to float32)")
        a = a.astype(np.float32)
    return a


def max_threads() -> int:
    """Threads the oracle's OpenMP regions use by default."""
    return int(_load().oracle_max_threads())


def attn_fwd(q, k, v, scale: float, causal: bool = False, nthreads: int = 0):
    """O [B,H,N,d] and LSE [B,H,N] by the plain formula, in float64."""
    q, k, v = _as_f32(q), _as_f32(k), _as_f32(v)
    if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share a [B, H, N, d] shape")
    B, H, N, d = q.shape
    o = np.empty((B, H, N, d), np.float64)
    lse = np.empty((B, H, N), np.float64)
    rc = _load().oracle_attn_fwd(q, k, v, o, lse, B, H, N, d, float(scale),
                                 int(bool(causal)), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attn_fwd failed")
    return o, lse


def attn_fwd_rows(q, k, v, scale: float, causal: bool, bh, rows, nthreads: int = 0):
    """Output rows ``rows[t]`` of slices ``bh[t]`` (bh = b*H + h): ([n,d], [n])."""
    q, k, v = _as_f32(q), _as_f32(k), _as_f32(v)
    if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share a [B, H, N, d] shape")
    B, H, N, d = q.shape
    bh = np.ascontiguousarray(bh, dtype=np.int64).ravel()
    rows = np.ascontiguousarray(rows, dtype=np.int64).ravel()
    if bh.shape != rows.shape:
        raise ValueError("bh and rows must have the same length")
    n = bh.shape[0]
    o = np.empty((n, d), np.float64)
    lse = np.empty((n,), np.float64)
    rc = _load().oracle_attn_fwd_rows(q, k, v, B, H, N, d, float(scale),
                                      int(bool(causal)), bh, rows, n, o, lse,
                                      int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attn_fwd_rows failed (bad index?)")
    return o, lse


def probs_row(q2, k2, i: int, scale: float, causal: bool = False):
    """P[i, :] of one (batch, head) slice; q2, k2 are [N, d]."""
    q2, k2 = _as_f32(q2), _as_f32(k2)
    N, d = q2.shape
    p = np.empty((N,), np.float64)
    rc = _load().oracle_probs_row(q2, k2, N, d, int(i), float(scale),
                                  int(bool(causal)), p)
    if rc != 0:
        raise RuntimeError("oracle_probs_row failed")
    return p


def online_replay(q2, k2, v2, scale: float, causal: bool, tile: int):
    """Tile-by-tile online-softmax replay over one slice: ([N,d], [N])."""
    q2, k2, v2 = _as_f32(q2), _as_f32(k2), _as_f32(v2)
    N, d = q2.shape
    o = np.empty((N, d), np.float64)
    lse = np.empty((N,), np.float64)
    rc = _load().oracle_online_replay(q2, k2, v2, N, d, float(scale),
                                      int(bool(causal)), int(tile), o, lse)
    if rc != 0:
        raise RuntimeError("oracle_online_replay failed")
    return o, lse


def row_softmax(x, nthreads: int = 0):
    """Row softmax of a [rows, width] matrix: (y [rows,width], lse [rows])."""
    x = _as_f32(x)
    if x.ndim != 2:
        raise ValueError("row_softmax expects a matrix")
    rows, width = x.shape
    y = np.empty((rows, width), np.float64)
    lse = np.empty((rows,), np.float64)
    rc = _load().oracle_row_softmax(x, rows, width, y, lse, int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_row_softmax failed")
    return y, lse


def add_rmsnorm(x, residual, weight, eps: float, nthreads: int = 0):
    """Residual add + RMSNorm: (out [rows, width], h = x + residual) in float64."""
    x = _as_f32(x)
    if x.ndim != 2:
        raise ValueError("add_rmsnorm expects a matrix")
    rows, width = x.shape
    w = _as_f32(weight).reshape(-1)
    if w.shape[0] != width:
        raise ValueError("weight must have one entry per column")
    r = None if residual is None else _as_f32(residual)
    if r is not None and r.shape != x.shape:
        raise ValueError("residual must match x")
    out = np.empty((rows, width), np.float64)
    h = np.empty((rows, width), np.float64)
    rc = _load().oracle_add_rmsnorm(x, None if r is None else r.ctypes.data, w, rows, width,
                                    float(eps), out, h.ctypes.data, int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_add_rmsnorm failed")
    return out, h


def attn_bwd(q, k, v, o, dout, lse, scale: float, causal: bool = False, nthreads: int = 0):
    """Gradients (dQ, dK, dV) in float64, given the forward's O and LSE."""
    arrs = [_as_f32(t) for t in (q, k, v, o, dout)]
    lse = _as_f32(lse)
    shape = arrs[0].shape
    if len(shape) != 4 or any(a.shape != shape for a in arrs):
        raise ValueError("q, k, v, o, dout must share a [B, H, N, d] shape")
    B, H, N, d = shape
    if lse.shape != (B, H, N):
        raise ValueError("lse must be [B, H, N]")
    dq = np.empty(shape, np.float64)
    dk = np.empty(shape, np.float64)
    dv = np.empty(shape, np.float64)
    rc = _load().oracle_attn_bwd(*arrs, lse, B, H, N, d, float(scale), int(bool(causal)),
                                 dq, dk, dv, int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attn_bwd failed")
    return dq, dk, dv
