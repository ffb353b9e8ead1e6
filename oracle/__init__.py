"""ORACLE -- plain fp64 CPU attention forward.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  It shares no code with the CUDA library
(``exact_attention_forward_fa2_gb300``) and never imports it; the product path
never calls it.

``fa2_oracle.c`` holds the arithmetic (see its header for the definition and the
passages it follows); this file only compiles it with gcc and marshals numpy
arrays through ctypes.  Pins that tie the oracle to the pages and to mathematics
live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa2_oracle.c")
_LIB = os.path.join(_HERE, "libfa2_oracle.so")
_lock = threading.Lock()
_lib = None

_DTYPE_CODE = {np.dtype(np.uint16): 0, np.dtype(np.float32): 1, np.dtype(np.float64): 2}


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle (gcc -O2, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load the oracle library (building it if needed)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    vp, i32, dbl, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_int64
    lib.oracle_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, dbl, i32, i32]
    lib.oracle_attn_fwd.restype = i32
    lib.oracle_attn_fwd_rows.argtypes = [vp, vp, vp, vp, i64, vp, vp, i32, i32, i32, i32, i32,
                                         dbl, i32, i32]
    lib.oracle_attn_fwd_rows.restype = i32
    lib.oracle_attn_fwd_tiled.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, dbl, i32,
                                          i32, i32, i32]
    lib.oracle_attn_fwd_tiled.restype = i32
    lib.oracle_attn_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, dbl, i32,
                                        i32]
    lib.oracle_attn_fwd_gqa.restype = i32
    lib.oracle_attn_fwd_gqa_rows.argtypes = [vp, vp, vp, vp, i64, vp, vp, i32, i32, i32, i32, i32,
                                             i32, dbl, i32, i32]
    lib.oracle_attn_fwd_gqa_rows.restype = i32
    lib.oracle_attn_fwd_mod.argtypes = [vp, vp, vp, vp, i64, vp, vp, i32, i32, i32, i32, i32, i32,
                                        dbl, i32, i32, i32, dbl, vp, i64, i32]
    lib.oracle_attn_fwd_mod.restype = i32
    lib.oracle_attn_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                        dbl, i32, i32]
    lib.oracle_attn_bwd_gqa.restype = i32
    lib.oracle_omp_threads.argtypes = []
    lib.oracle_omp_threads.restype = i32
    return lib


def _prep(q, k, v, gqa=False):
    q, k, v = (np.ascontiguousarray(t) for t in (q, k, v))
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in _DTYPE_CODE:
        raise TypeError("q, k, v must share one dtype: uint16 (bf16 bits), float32 or float64")
    if q.ndim != 4 or k.ndim != 4 or v.shape != k.shape or q.shape[0] != k.shape[0] \
            or q.shape[3] != k.shape[3]:
        raise ValueError("expected q [B,H,M,D] and k, v [B,Hkv,N,D]")
    if (not gqa and q.shape[1] != k.shape[1]) or q.shape[1] % k.shape[1] != 0:
        raise ValueError("k, v head count must equal (or, for grouped-query attention, divide) H")
    B, H, M, D = q.shape
    N = k.shape[2]
    return q, k, v, B, H, M, N, D, _DTYPE_CODE[q.dtype]


def omp_threads(lib=None) -> int:
    """Threads the oracle's OpenMP regions run with in this process."""
    lib = lib or load()
    return int(lib.oracle_omp_threads())


def attn_fwd(q, k, v, scale: float, causal: bool, lib=None):
    """Every row: returns (O [B,H,M,D] fp64, L [B,H,M] fp64)."""
    lib = lib or load()
    q, k, v, B, H, M, N, D, code = _prep(q, k, v)
    o = np.empty((B, H, M, D), np.float64)
    lse = np.empty((B, H, M), np.float64)
    rc = lib.oracle_attn_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, o.ctypes.data,
                             lse.ctypes.data, B, H, M, N, D, float(scale), int(causal), code)
    if rc:
        raise RuntimeError(f"oracle_attn_fwd failed: {rc}")
    return o, lse


def attn_fwd_rows(q, k, v, scale: float, causal: bool, rows, lib=None):
    """Selected rows (flat index (b*H+h)*M+i): returns (O [n,D], L [n]) fp64."""
    lib = lib or load()
    q, k, v, B, H, M, N, D, code = _prep(q, k, v)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.empty((rows.size, D), np.float64)
    lse = np.empty((rows.size,), np.float64)
    rc = lib.oracle_attn_fwd_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, rows.ctypes.data,
                                  rows.size, o.ctypes.data, lse.ctypes.data, B, H, M, N, D,
                                  float(scale), int(causal), code)
    if rc:
        raise RuntimeError(f"oracle_attn_fwd_rows failed: {rc}")
    return o, lse


def attn_fwd_tiled(q, k, v, scale: float, causal: bool, block_m: int, block_n: int, lib=None):
    """The fp64 tiled online-softmax recurrence: returns (O, L) like attn_fwd."""
    lib = lib or load()
    q, k, v, B, H, M, N, D, code = _prep(q, k, v)
    o = np.empty((B, H, M, D), np.float64)
    lse = np.empty((B, H, M), np.float64)
    rc = lib.oracle_attn_fwd_tiled(q.ctypes.data, k.ctypes.data, v.ctypes.data, o.ctypes.data,
                                   lse.ctypes.data, B, H, M, N, D, float(scale), int(causal),
                                   code, int(block_m), int(block_n))
    if rc:
        raise RuntimeError(f"oracle_attn_fwd_tiled failed: {rc}")
    return o, lse


def attn_fwd_gqa(q, k, v, scale: float, causal: bool, lib=None):
    """Grouped-query attention: q [B,H,M,D], k and v [B,Hkv,N,D] with Hkv | H;
    returns (O [B,H,M,D], L [B,H,M]) fp64."""
    lib = lib or load()
    q, k, v, B, H, M, N, D, code = _prep(q, k, v, gqa=True)
    Hkv = k.shape[1]
    o = np.empty((B, H, M, D), np.float64)
    lse = np.empty((B, H, M), np.float64)
    rc = lib.oracle_attn_fwd_gqa(q.ctypes.data, k.ctypes.data, v.ctypes.data, o.ctypes.data,
                                 lse.ctypes.data, B, H, Hkv, M, N, D, float(scale), int(causal), code)
    if rc:
        raise RuntimeError(f"oracle_attn_fwd_gqa failed: {rc}")
    return o, lse


def attn_fwd_gqa_rows(q, k, v, scale: float, causal: bool, rows, lib=None):
    """Selected rows of grouped-query attention: returns (O [n,D], L [n]) fp64."""
    lib = lib or load()
    q, k, v, B, H, M, N, D, code = _prep(q, k, v, gqa=True)
    Hkv = k.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.empty((rows.size, D), np.float64)
    lse = np.empty((rows.size,), np.float64)
    rc = lib.oracle_attn_fwd_gqa_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                      rows.ctypes.data, rows.size, o.ctypes.data, lse.ctypes.data,
                                      B, H, Hkv, M, N, D, float(scale), int(causal), code)
    if rc:
        raise RuntimeError(f"oracle_attn_fwd_gqa_rows failed: {rc}")
    return o, lse


def attn_fwd_mod(q, k, v, scale: float, causal: bool, window=(-1, -1), softcap: float = 0.0,
                 alibi_slopes=None, rows=None, lib=None):
    """Attention with score modifiers (sliding window, softcap, ALiBi; see
    ``fa2_oracle.c`` for the reading).  q [B,H,M,D], k and v [B,Hkv,N,D];
    ``window`` = (left, right), negative = unbounded; ``alibi_slopes`` None,
    [H] (shared by every batch entry) or [B,H].  With ``rows`` None returns
    (O [B,H,M,D], L [B,H,M]), else (O [n,D], L [n]) for the listed flat rows."""
    lib = lib or load()
    q, k, v, B, H, M, N, D, code = _prep(q, k, v, gqa=True)
    Hkv = k.shape[1]
    slopes_ptr, sb = None, 0
    if alibi_slopes is not None:
        sl = np.ascontiguousarray(alibi_slopes, dtype=np.float64)
        if sl.shape == (H,):
            sb = 0
        elif sl.shape == (B, H):
            sb = H
        else:
            raise ValueError("alibi_slopes must be [H] or [B, H]")
        slopes_ptr = sl.ctypes.data
    if rows is None:
        rows_arr, n, rows_ptr = None, B * H * M, None
        o = np.empty((B, H, M, D), np.float64)
        lse = np.empty((B, H, M), np.float64)
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n, rows_ptr = rows_arr.size, rows_arr.ctypes.data
        o = np.empty((n, D), np.float64)
        lse = np.empty((n,), np.float64)
    wl, wr = (int(x) for x in window)
    rc = lib.oracle_attn_fwd_mod(q.ctypes.data, k.ctypes.data, v.ctypes.data, rows_ptr, n,
                                 o.ctypes.data, lse.ctypes.data, B, H, Hkv, M, N, D, float(scale),
                                 int(causal), wl, wr, float(softcap), slopes_ptr, sb, code)
    if rc:
        raise RuntimeError(f"oracle_attn_fwd_mod failed: {rc}")
    return o, lse


def attn_bwd(q, k, v, dout, scale: float, causal: bool, lib=None):
    """Gradients of the forward for upstream gradient ``dout`` (same shape and
    dtype as q): returns (dQ [B,H,M,D], dK [B,Hkv,N,D], dV [B,Hkv,N,D]) fp64.
    k and v may hold fewer heads than q (grouped-query attention)."""
    lib = lib or load()
    q, k, v, B, H, M, N, D, code = _prep(q, k, v, gqa=True)
    dout = np.ascontiguousarray(dout)
    if dout.shape != q.shape or dout.dtype != q.dtype:
        raise ValueError("dout must have the shape and dtype of q")
    Hkv = k.shape[1]
    dq = np.empty((B, H, M, D), np.float64)
    dk = np.empty((B, Hkv, N, D), np.float64)
    dv = np.empty((B, Hkv, N, D), np.float64)
    rc = lib.oracle_attn_bwd_gqa(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data,
                                 dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, B, H, Hkv, M, N, D,
                                 float(scale), int(causal), code)
    if rc:
        raise RuntimeError(f"oracle_attn_bwd_gqa failed: {rc}")
    return dq, dk, dv
