"""Helpers for the GPU parity tests: host arrays to device tensors and back, and
the comparison against the oracle (the per-element bound and its statistics)."""
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


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp at |x| (8 significant bits): the largest error of
    rounding the exact value x to bf16."""
    _, ex = np.frexp(np.abs(x))
    return np.where(x == 0, 0.0, np.ldexp(1.0, ex - 9))


# |O_ref| from which a bf16 output gets half a bf16 ulp on top of TOL: below 2 a
# half ulp is at most 2^-8, so the flat bound is attainable there; at |O| in [4, 8)
# the correctly rounded exact answer alone is up to 2^-6 = 0.0156 away.
ULP_ALLOWANCE_FROM = 2.0


def o_bound(o_ref: np.ndarray, dtype) -> np.ndarray:
    """Per-element bound on |dO|: TOL[dtype] (1e-2 for bf16, 5e-3 for fp32, the
    forward tolerances of the parity target), and for bf16 outputs with
    |O_ref| >= 2 that plus half a bf16 ulp of O_ref, the unavoidable error of
    storing the exact O in bf16."""
    if dtype != si.BF16:
        return np.full(np.shape(o_ref), TOL[dtype])
    return TOL[dtype] + np.where(np.abs(o_ref) >= ULP_ALLOWANCE_FROM, half_ulp_bf16(o_ref), 0.0)


def compare_stats(o_gpu, l_gpu, o_ref, l_ref, dtype) -> dict:
    """Error statistics of one comparison: max|dO| over all elements, over those
    with |O_ref| < 2 (flat bound) and over those with |O_ref| >= 2 (bound plus
    half a bf16 ulp), max|dL|, max|O_ref|, and the largest excess of |dO| over
    its per-element bound (<= 0 passes)."""
    assert np.all(np.isfinite(o_gpu)), "non-finite O"
    assert np.all(np.isfinite(l_gpu)), "non-finite L"
    d_o = np.abs(o_gpu - o_ref)
    big = np.abs(o_ref) >= ULP_ALLOWANCE_FROM
    small_do = d_o[~big]
    big_do = d_o[big]
    return {
        "rows": int(np.size(l_ref)),
        "max_do": float(np.max(d_o)) if d_o.size else 0.0,
        "max_do_small": float(np.max(small_do)) if small_do.size else 0.0,
        "max_do_large": float(np.max(big_do)) if big_do.size else 0.0,
        "n_large": int(np.count_nonzero(big)),
        "max_dl": float(np.max(np.abs(l_gpu - l_ref))) if np.size(l_ref) else 0.0,
        "max_abs_oref": float(np.max(np.abs(o_ref))) if np.size(o_ref) else 0.0,
        "excess": float(np.max(d_o - o_bound(o_ref, dtype))) if d_o.size else 0.0,
        "tol": TOL[dtype],
    }


def compare(o_gpu, l_gpu, o_ref, l_ref, dtype):
    """Returns (max|dO|, max|dL|, max excess of |dO| over its bound).

    The bound on |dO| is TOL[dtype] on every element, except that bf16 outputs
    with |O_ref| >= 2 get half a bf16 ulp of O_ref on top (see o_bound).  L is
    fp32 in both cases and gets TOL[dtype]."""
    st = compare_stats(o_gpu, l_gpu, o_ref, l_ref, dtype)
    return st["max_do"], st["max_dl"], st["excess"]


def record_parity(name: str, stats: dict, **extra) -> None:
    """Append one comparison's statistics as a JSON line to the file named by
    the FA2_PARITY_RECORD environment variable (nothing when it is unset)."""
    import json
    import os
    path = os.environ.get("FA2_PARITY_RECORD")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"case": name, **stats, **extra}) + "\n")
