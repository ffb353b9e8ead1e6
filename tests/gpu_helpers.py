"""Helpers for the GPU parity tests: host arrays to device tensors and back,
row sampling for full-size workloads, and the comparison against the oracle."""
from __future__ import annotations

import numpy as np

import seeded_inputs as si

# Tolerances: max |dO| and max |dL|, absolute, over every compared element.
TOL = {si.BF16: 1e-2, si.FP32: 5e-3}


def to_device(a: np.ndarray, dev):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


def to_host_f64(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        return si.bf16_bits_to_f32(bits).astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def sample_rows(B, H, M, N, causal, n_random=4096, seed=0, full_heads=((0, 0), (-1, -1))):
    """Flat row indices (b*H+h)*M+i to check at full size: every row of the
    first and last head, and in every head the first and last rows, rows at
    and next to the 128-row tile edges that carry the causal diagonal, the
    ragged-tail rows, plus seeded random rows."""
    rows = set()
    for b, h in full_heads:
        bh = (b % B) * H + (h % H)
        rows.update(range(bh * M, (bh + 1) * M))
    edges = {0, 1, M - 1, M - 2}
    for e in range(0, M, 128):
        edges.update({e, e + 1, e + 127, e + 128, e - 1})
    edges.update({M - 1 - (M % 128), (M // 128) * 128})
    edges = [i for i in edges if 0 <= i < M]
    for bh in range(B * H):
        rows.update(bh * M + i for i in edges)
    rng = np.random.default_rng(seed)
    rows.update(rng.integers(0, B * H * M, size=n_random).tolist())
    return np.array(sorted(rows), np.int64)


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp at |x| (8 significant bits): the largest error of
    rounding the exact value x to bf16."""
    _, ex = np.frexp(np.abs(x))
    return np.where(x == 0, 0.0, np.ldexp(1.0, ex - 9))


def compare(o_gpu, l_gpu, o_ref, l_ref, dtype):
    """Returns (max|dO|, max|dL|, max excess of |dO| over its bound).

    The bound on |dO| is TOL[dtype] on top of the unavoidable rounding of the
    exact O to the output type: for bf16 outputs that is half a bf16 ulp of
    O_ref (0.0156 for |O| in [4, 8), already above 1e-2 by itself), for fp32
    outputs it is negligible.  L is fp32 in both cases and gets TOL[dtype]."""
    assert np.all(np.isfinite(o_gpu)), "non-finite O"
    assert np.all(np.isfinite(l_gpu)), "non-finite L"
    d_o = np.abs(o_gpu - o_ref)
    bound = TOL[dtype] + (half_ulp_bf16(o_ref) if dtype == si.BF16 else 0.0)
    return float(np.max(d_o)), float(np.max(np.abs(l_gpu - l_ref))), float(np.max(d_o - bound))
