"""Seeded synthetic inputs shared by the fp64 oracle and the GPU path.

This module draws the Q, K, V tensors of an attention workload and rounds them
to the storage dtype. It holds none of the attention arithmetic, and neither the
oracle nor the CUDA library is imported here.

The generator is counter based (SplitMix64 over a Weyl sequence, Box-Muller
normals; see gen.c), so element ``i`` of a stream is a pure function of
``(seed, stream, i)``: the same on x86 and Arm, and any slice can be drawn on
its own. Q, K and V of a workload use streams 1, 2 and 3 of the workload's seed.

Workload shapes follow the pages' problem statement: Q [B,H,M,D], K/V [B,H,N,D]
(FlashAttention 2 in Triton tutorial, Step 2 and Step 6; drew-chen
flash-attention README, "Implementations").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libseeded_inputs.so")
_lock = threading.Lock()
_lib = None

BF16, FP32, FP64 = "bf16", "fp32", "fp64"


def build(force: bool = False) -> str:
    """Compile gen.c into an in-tree shared library (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            for name, ptr_t in (("seeded_normal_f64", ctypes.c_void_p),
                                ("seeded_normal_f32", ctypes.c_void_p),
                                ("seeded_normal_bf16", ctypes.c_void_p)):
                fn = getattr(lib, name)
                fn.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                               ctypes.c_int64, ctypes.c_double, ptr_t]
                fn.restype = None
            lib.seeded_f64_to_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
            lib.seeded_f64_to_bf16.restype = None
            _lib = lib
    return _lib


def normal(seed: int, stream: int, shape, sigma: float = 1.0, dtype: str = FP64,
           offset: int = 0) -> np.ndarray:
    """iid N(0, sigma^2) samples of ``shape``, rounded to ``dtype``.

    bf16 is returned as its raw 16-bit patterns (``np.uint16``); fp32 and fp64
    as ``np.float32`` / ``np.float64``.
    """
    lib = _load()
    n = int(np.prod(shape)) if len(shape) else 1
    if dtype == FP64:
        out = np.empty(shape, np.float64)
        lib.seeded_normal_f64(seed, stream, offset, n, sigma, out.ctypes.data)
    elif dtype == FP32:
        out = np.empty(shape, np.float32)
        lib.seeded_normal_f32(seed, stream, offset, n, sigma, out.ctypes.data)
    elif dtype == BF16:
        out = np.empty(shape, np.uint16)
        lib.seeded_normal_bf16(seed, stream, offset, n, sigma, out.ctypes.data)
    else:
        raise ValueError(f"unknown dtype {dtype!r}")
    return out


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (via fp32, both round-to-nearest-even)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    lib.seeded_f64_to_bf16(x.ctypes.data, x.size, out.ctypes.data)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class Workload:
    """One attention forward problem: sizes, dtype, mask, value recipe, seed."""
    name: str
    B: int
    H: int
    M: int
    N: int
    D: int
    dtype: str
    causal: bool
    seed: int
    sigma_qk: float = 1.0
    sigma_v: float = 1.0
    H_kv: int = 0  # key/value heads (grouped-query attention); 0 means H
    split_kv: bool = False  # measured through the split-KV entry
    window: tuple = (-1, -1)  # (left, right) sliding window; negative = unbounded
    softcap: float = 0.0  # 0 = no softcap
    alibi: bool = False  # ALiBi with alibi_slopes(H)

    @property
    def Hkv(self) -> int:
        return self.H_kv or self.H

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))

    @property
    def modified(self) -> bool:
        """A score modifier (window, softcap or ALiBi) is in use."""
        return self.window != (-1, -1) or self.softcap > 0 or self.alibi

    def visible_keys(self, i) -> np.ndarray:
        """Keys visible to query rows i (array), under the mask and window."""
        i = np.asarray(i, np.int64)
        lo = np.maximum(0, i - self.window[0]) if self.window[0] >= 0 else np.zeros_like(i)
        hi = np.full_like(i, self.N - 1)
        if self.window[1] >= 0:
            hi = np.minimum(hi, i + self.window[1])
        if self.causal:
            hi = np.minimum(hi, i)
        return np.maximum(0, hi - lo + 1)

    @property
    def flops(self) -> float:
        """4*B*H*M*N*D, halved for causal (the pages' attention FLOP count); with
        a window, 4*D per visible (query, key) pair."""
        if self.window != (-1, -1):
            return 4.0 * self.B * self.H * self.D * float(np.sum(self.visible_keys(np.arange(self.M))))
        f = 4.0 * self.B * self.H * self.M * self.N * self.D
        return f / 2 if self.causal else f

    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: read Q, K, V once; write O and fp32 L once."""
        e = 2 if self.dtype == BF16 else 4
        q_o = self.B * self.H * (2 * self.M * self.D * e + 4 * self.M)
        return q_o + self.B * self.Hkv * 2 * self.N * self.D * e


# The five workloads the method is checked and measured on. Values are iid normal;
# the cross-attention case draws Q and K with sigma 3 so softmax rows are sharp.
WORKLOADS = {
    "fp32_1x1x128x128x64": Workload("fp32_1x1x128x128x64", 1, 1, 128, 128, 64, FP32, False, 1),
    "tf32_4x12x2048x2048x64": Workload("tf32_4x12x2048x2048x64", 4, 12, 2048, 2048, 64, FP32, False, 2),
    "bf16_4x16x4096x4096x64_causal": Workload("bf16_4x16x4096x4096x64_causal", 4, 16, 4096, 4096, 64, BF16, True, 3),
    "bf16_2x16x8192x8192x128": Workload("bf16_2x16x8192x8192x128", 2, 16, 8192, 8192, 128, BF16, False, 4),
    "bf16_2x16x8192x8192x128_causal": Workload("bf16_2x16x8192x8192x128_causal", 2, 16, 8192, 8192, 128, BF16, True, 4),
    "bf16_8x32x1000x3000x128_sharp": Workload("bf16_8x32x1000x3000x128_sharp", 8, 32, 1000, 3000, 128, BF16, False, 5,
                                              sigma_qk=3.0, sigma_v=1.0),
    # grouped-query attention: 32 query heads share 8 key/value heads
    "bf16_2x32x8192x8192x128_gqa8_causal": Workload("bf16_2x32x8192x8192x128_gqa8_causal", 2, 32, 8192, 8192, 128,
                                                    BF16, True, 6, H_kv=8),
    # short queries against a long key range (a prefill chunk against a long
    # cache): 32 query-tile units cannot fill the GPU, so the key range is split
    "bf16_1x32x128x32768x128_gqa8_splitkv": Workload("bf16_1x32x128x32768x128_gqa8_splitkv", 1, 32, 128, 32768, 128,
                                                     BF16, False, 7, H_kv=8, split_kv=True),
    # decode: one query row per sequence against an 8192-key cache, grouped-query
    # heads; bound by reading K and V once from HBM
    "bf16_16x32x1x8192x128_gqa8_decode": Workload("bf16_16x32x1x8192x128_gqa8_decode", 16, 32, 1, 8192, 128, BF16,
                                                  False, 11, H_kv=8, split_kv=True),
    # score modifiers at the headline size: a 2048-key causal sliding window, a
    # softcap of 50, ALiBi with the geometric slopes below
    "bf16_2x16x8192x8192x128_causal_window2048": Workload("bf16_2x16x8192x8192x128_causal_window2048", 2, 16, 8192,
                                                          8192, 128, BF16, True, 8, window=(2048, -1)),
    "bf16_2x16x8192x8192x128_causal_softcap50": Workload("bf16_2x16x8192x8192x128_causal_softcap50", 2, 16, 8192,
                                                         8192, 128, BF16, True, 9, softcap=50.0),
    "bf16_2x16x8192x8192x128_causal_alibi": Workload("bf16_2x16x8192x8192x128_causal_alibi", 2, 16, 8192, 8192,
                                                     128, BF16, True, 10, alibi=True),
}


def alibi_slopes(H: int) -> np.ndarray:
    """ALiBi slopes, one per head: the geometric sequence 2^(-8 (h + 1) / H),
    fp32 (an input of the method, like Q, K and V)."""
    return (2.0 ** (-8.0 * np.arange(1, H + 1) / H)).astype(np.float32)


def make_qkv(w: Workload):
    """Draw (q, k, v) host arrays for workload ``w`` in its storage dtype."""
    q = normal(w.seed, 1, (w.B, w.H, w.M, w.D), w.sigma_qk, w.dtype)
    k = normal(w.seed, 2, (w.B, w.Hkv, w.N, w.D), w.sigma_qk, w.dtype)
    v = normal(w.seed, 3, (w.B, w.Hkv, w.N, w.D), w.sigma_v, w.dtype)
    return q, k, v
