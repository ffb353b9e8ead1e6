"""Pins for the fp64 oracle: each check ties it to something other than itself.

- hand-derived worked examples (tests/golden/worked_examples.json);
- brute force with library routines: the whole score matrix materialised by a
  numpy matmul, L from scipy's logsumexp, P = exp(S - L) (the backward-pass
  identity of "FlashAttention-2 from PyTorch to Triton", introduction);
- PyTorch's CPU scaled_dot_product_attention in fp64 as a third opinion;
- closed forms and invariants: K = 0 gives the mean of the visible V rows and
  L = ln(#visible); one key gives O = V_0; O rows are convex combinations of V
  rows; causal row 0 equals V row 0; key/value permutation invariance; affine
  equivariance in V; the tiled online recurrence equals the two-pass softmax.

test_planted_mistakes_are_caught then plants plausible mistakes in a copy of the
oracle's C source (a dropped term, a wrong sign or index, a transposed operand,
an off-by-one causal bound) and checks that every mutant fails at least one pin.
"""
import json
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import scipy.special

import oracle
import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def widen(x):
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return si.bf16_bits_to_f32(x).astype(np.float64)
    return x.astype(np.float64)


def brute_force(q, k, v, scale, causal):
    """Materialise S, mask, L = logsumexp, P = exp(S - L), O = P V (fp64)."""
    q, k, v = widen(q), widen(k), widen(v)
    M, N = q.shape[2], k.shape[2]
    s = scale * np.matmul(q, np.swapaxes(k, -1, -2))
    if causal:
        hidden = np.arange(N)[None, :] > np.arange(M)[:, None]
        s = np.where(hidden, -np.inf, s)
    lse = scipy.special.logsumexp(s, axis=-1)
    p = np.exp(s - lse[..., None])
    return np.matmul(p, v), lse


def rand_inputs(seed, B, H, M, N, D, dtype, sigma=1.0):
    q = si.normal(seed, 1, (B, H, M, D), sigma, dtype)
    k = si.normal(seed, 2, (B, H, N, D), sigma, dtype)
    v = si.normal(seed, 3, (B, H, N, D), 1.0, dtype)
    return q, k, v


def max_err(a, b):
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b))))


# ---------------------------------------------------------------- pin suite
def golden_errors(lib):
    errs = []
    with open(GOLDEN) as f:
        data = json.load(f)
    tol = data["tolerance"]
    for c in data["cases"]:
        q, k, v = (np.array(c[n], np.float64) for n in ("q", "k", "v"))
        o, lse = oracle.attn_fwd(q, k, v, c["scale"], c["causal"], lib=lib)
        e = max(max_err(o, c["o"]), max_err(lse, c["lse"]))
        if not e <= tol:
            errs.append(f"golden {c['name']}: {e}")
    return errs


BRUTE_SHAPES = [  # (B, H, M, N, D)
    (1, 1, 1, 1, 1), (1, 1, 1, 7, 2), (1, 1, 7, 1, 2), (2, 1, 3, 3, 64), (1, 2, 16, 16, 2),
    (1, 1, 37, 53, 64), (1, 1, 53, 37, 2), (2, 2, 7, 16, 1),
]


def brute_errors(lib, dtypes=(si.FP64, si.FP32, si.BF16), shapes=BRUTE_SHAPES):
    errs = []
    for si_dtype in dtypes:
        for n, (B, H, M, N, D) in enumerate(shapes):
            for causal in (False, True):
                q, k, v = rand_inputs(100 + n, B, H, M, N, D, si_dtype)
                scale = 1.0 / math.sqrt(D)
                o, lse = oracle.attn_fwd(q, k, v, scale, causal, lib=lib)
                ob, lb = brute_force(q, k, v, scale, causal)
                e = max(max_err(o, ob), max_err(lse, lb))
                if not e <= 1e-12:
                    errs.append(f"brute {si_dtype} {(B, H, M, N, D)} causal={causal}: {e}")
    return errs


def large_score_errors(lib):
    """Scores of magnitude ~1e3: exp without the max subtraction overflows."""
    errs = []
    q, k, v = rand_inputs(7, 1, 1, 9, 11, 4, si.FP64, sigma=30.0)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, 1.0, causal, lib=lib)
        ob, lb = brute_force(q, k, v, 1.0, causal)
        e = max(max_err(o, ob), max_err(lse, lb) / max(1.0, float(np.max(np.abs(lb)))))
        if not e <= 1e-12:
            errs.append(f"large scores causal={causal}: {e}")
    return errs


def invariant_errors(lib):
    errs = []
    B, H, M, N, D = 2, 2, 19, 23, 8
    q, k, v = rand_inputs(11, B, H, M, N, D, si.FP64)
    scale = 0.37
    for causal in (False, True):
        nvis = np.minimum(np.arange(M) + 1, N) if causal else np.full(M, N)
        # K == 0: uniform weights over the visible keys
        o, lse = oracle.attn_fwd(q, np.zeros_like(k), v, scale, causal, lib=lib)
        cs = np.cumsum(v, axis=2)
        mean = np.stack([cs[:, :, n - 1, :] / n for n in nvis], axis=2)
        if max_err(o, mean) > 1e-12 or max_err(lse, np.broadcast_to(np.log(nvis), lse.shape)) > 1e-12:
            errs.append(f"K=0 causal={causal}")
        # convex hull of the visible V rows
        o, lse = oracle.attn_fwd(q, k, v, scale, causal, lib=lib)
        for i in range(M):
            vis = v[:, :, : nvis[i], :]
            lo, hi = vis.min(axis=2), vis.max(axis=2)
            if np.any(o[:, :, i, :] < lo - 1e-12) or np.any(o[:, :, i, :] > hi + 1e-12):
                errs.append(f"hull row {i} causal={causal}")
                break
        # affine equivariance in V
        a, c = -1.75, 0.5
        o2, lse2 = oracle.attn_fwd(q, k, a * v + c, scale, causal, lib=lib)
        if max_err(o2, a * o + c) > 1e-12 or max_err(lse2, lse) > 0:
            errs.append(f"affine causal={causal}")
        # causal row 0 is V row 0 and its L is its own score
        if causal:
            if max_err(o[:, :, 0, :], v[:, :, 0, :]) > 1e-12:
                errs.append("causal row 0 != V row 0")
            s00 = scale * np.sum(q[:, :, 0, :] * k[:, :, 0, :], axis=-1)
            if max_err(lse[:, :, 0], s00) > 1e-12:
                errs.append("causal row 0 L != s_00")
    # key/value permutation (non-causal only)
    perm = np.random.default_rng(3).permutation(N)
    o, lse = oracle.attn_fwd(q, k, v, scale, False, lib=lib)
    o2, lse2 = oracle.attn_fwd(q, k[:, :, perm], v[:, :, perm], scale, False, lib=lib)
    if max_err(o, o2) > 1e-12 or max_err(lse, lse2) > 1e-12:
        errs.append("permutation")
    # a single key: O = V_0, L = scale q.k_0
    o, lse = oracle.attn_fwd(q, k[:, :, :1], v[:, :, :1], scale, False, lib=lib)
    if max_err(o, np.broadcast_to(v[:, :, :1], o.shape)) > 1e-12:
        errs.append("N=1 O")
    if max_err(lse, scale * np.einsum("bhmd,bhd->bhm", q, k[:, :, 0])) > 1e-12:
        errs.append("N=1 L")
    return errs


def rows_errors(lib):
    errs = []
    B, H, M, N, D = 2, 3, 21, 17, 16
    q, k, v = rand_inputs(5, B, H, M, N, D, si.BF16)
    rows = np.array([0, 5, 20, 21, 62, B * H * M - 1], np.int64)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, 0.25, causal, lib=lib)
        orow, lrow = oracle.attn_fwd_rows(q, k, v, 0.25, causal, rows, lib=lib)
        if max_err(orow, o.reshape(-1, D)[rows]) > 0 or max_err(lrow, lse.reshape(-1)[rows]) > 0:
            errs.append(f"rows causal={causal}")
    return errs


TILINGS = [(1, 1), (16, 16), (7, 5), (128, 128), (64, 37), (3, 64)]


def tiled_errors(lib):
    errs = []
    for n, (B, H, M, N, D) in enumerate([(1, 2, 70, 70, 8), (2, 1, 33, 100, 4), (1, 1, 100, 33, 16)]):
        for dtype in (si.FP64, si.BF16):
            q, k, v = rand_inputs(40 + n, B, H, M, N, D, dtype, sigma=2.0)
            for causal in (False, True):
                ob, lb = brute_force(q, k, v, 0.3, causal)
                for bm, bn in TILINGS:
                    o, lse = oracle.attn_fwd_tiled(q, k, v, 0.3, causal, bm, bn, lib=lib)
                    e = max(max_err(o, ob), max_err(lse, lb))
                    if not e <= 1e-12:
                        errs.append(f"tiled {bm}x{bn} {(B, H, M, N, D)} causal={causal}: {e}")
    return errs


def gqa_errors(lib):
    """Grouped-query attention equals multi-head attention on K/V heads repeated
    H/Hkv times (numpy brute force), for MQA, GQA and MHA groupings."""
    errs = []
    for n, (B, H, Hkv, M, N, D) in enumerate([(2, 4, 1, 9, 13, 8), (3, 6, 2, 17, 5, 4),
                                              (1, 8, 4, 12, 20, 16), (2, 3, 3, 7, 7, 2)]):
        for dtype in (si.FP64, si.BF16):
            q = si.normal(70 + n, 1, (B, H, M, D), 1.0, dtype)
            k = si.normal(70 + n, 2, (B, Hkv, N, D), 1.0, dtype)
            v = si.normal(70 + n, 3, (B, Hkv, N, D), 1.0, dtype)
            rk, rv = (np.repeat(t, H // Hkv, axis=1) for t in (k, v))
            for causal in (False, True):
                o, lse = oracle.attn_fwd_gqa(q, k, v, 0.4, causal, lib=lib)
                ob, lb = brute_force(q, rk, rv, 0.4, causal)
                e = max(max_err(o, ob), max_err(lse, lb))
                rows = np.array([0, M - 1, B * H * M - 1, (B * H * M) // 2], np.int64)
                orow, lrow = oracle.attn_fwd_gqa_rows(q, k, v, 0.4, causal, rows, lib=lib)
                e = max(e, max_err(orow, ob.reshape(-1, D)[rows]), max_err(lrow, lb.reshape(-1)[rows]))
                if not e <= 1e-12:
                    errs.append(f"gqa {(B, H, Hkv, M, N, D)} {dtype} causal={causal}: {e}")
    return errs


def brute_force_mod(q, k, v, scale, causal, window=(-1, -1), softcap=0.0, slopes=None):
    """Materialise S with the score modifiers, mask, logsumexp (fp64); rows
    without a visible key get O = 0 and L = -inf.  k, v may hold fewer heads
    (grouped-query attention): they are repeated to H heads."""
    q, k, v = widen(q), widen(k), widen(v)
    B, H, M, _ = q.shape
    N = k.shape[2]
    k, v = (np.repeat(t, H // t.shape[1], axis=1) for t in (k, v))
    s = scale * np.matmul(q, np.swapaxes(k, -1, -2))
    if softcap > 0:
        s = softcap * np.tanh(s / softcap)
    i, j = np.arange(M)[:, None], np.arange(N)[None, :]
    if slopes is not None:
        a = np.broadcast_to(np.asarray(slopes, np.float64).reshape(-1, H), (B, H))
        s = s - a[:, :, None, None] * np.abs(i - j)[None, None]
    vis = np.ones((M, N), bool)
    if causal:
        vis &= j <= i
    if window[0] >= 0:
        vis &= j >= i - window[0]
    if window[1] >= 0:
        vis &= j <= i + window[1]
    s = np.where(vis, s, -np.inf)
    with np.errstate(invalid="ignore", divide="ignore"):
        lse = scipy.special.logsumexp(s, axis=-1)
        p = np.where(vis, np.exp(s - lse[..., None]), 0.0)
    return np.matmul(p, v), lse


def same(a, b, tol):
    """Elementwise |a - b| <= tol, with equal infinities counted as equal."""
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    inf = np.isinf(a) | np.isinf(b)
    return bool(np.all(a[inf] == b[inf]) and np.all(np.abs(a[~inf] - b[~inf]) <= tol))


MOD_CASES = [  # (B, H, Hkv, M, N, D, causal, window, softcap, slopes shape)
    (1, 2, 2, 17, 23, 8, False, (-1, -1), 0.0, None),
    (2, 2, 1, 19, 19, 4, True, (-1, -1), 0.0, None),
    (1, 3, 3, 21, 13, 8, False, (4, 2), 0.0, None),
    (2, 2, 2, 30, 9, 2, False, (3, -1), 0.0, None),   # rows past N + 3 see no key
    (1, 2, 1, 16, 27, 8, True, (5, -1), 0.0, None),
    (1, 2, 2, 11, 40, 4, False, (-1, 6), 0.0, None),
    (2, 1, 1, 12, 12, 16, False, (-1, -1), 2.5, None),
    (1, 4, 2, 13, 17, 8, True, (-1, -1), 0.0, "h"),
    (2, 3, 3, 15, 20, 4, False, (-1, -1), 0.0, "bh"),
    (2, 2, 2, 25, 18, 8, True, (6, 0), 1.5, "bh"),
    (1, 2, 2, 9, 30, 8, False, (2, 3), 4.0, "h"),
]


def mod_brute_errors(lib):
    """Score modifiers against the numpy brute force, every row and the row
    entry, bf16 and fp64 inputs."""
    errs = []
    for n, (B, H, Hkv, M, N, D, causal, window, cap, sl) in enumerate(MOD_CASES):
        for dtype in (si.FP64, si.BF16):
            q = si.normal(80 + n, 1, (B, H, M, D), 2.0, dtype)
            k = si.normal(80 + n, 2, (B, Hkv, N, D), 2.0, dtype)
            v = si.normal(80 + n, 3, (B, Hkv, N, D), 1.0, dtype)
            slopes = None
            if sl == "h":
                slopes = 0.5 ** np.arange(1, H + 1)
            elif sl == "bh":
                slopes = 0.3 * np.arange(1, B * H + 1).reshape(B, H) / (B * H)
            o, lse = oracle.attn_fwd_mod(q, k, v, 0.35, causal, window, cap, slopes, lib=lib)
            ob, lb = brute_force_mod(q, k, v, 0.35, causal, window, cap, slopes)
            rows = np.array([0, M - 1, B * H * M - 1, (B * H * M) // 3], np.int64)
            orow, lrow = oracle.attn_fwd_mod(q, k, v, 0.35, causal, window, cap, slopes, rows=rows,
                                             lib=lib)
            if not (same(o, ob, 1e-12) and same(lse, lb, 1e-12) and same(orow, o.reshape(-1, D)[rows], 0)
                    and same(lrow, lse.reshape(-1)[rows], 0)):
                errs.append(f"mod brute case {n} {dtype}")
    return errs


def mod_reduction_errors(lib):
    """Modifiers that reduce to plain attention: defaults, a window as wide as
    the problem, zero slopes, a huge softcap; window (unbounded, 0) == causal."""
    errs = []
    B, H, M, N, D = 2, 2, 14, 19, 8
    q, k, v = rand_inputs(91, B, H, M, N, D, si.FP64)
    for causal in (False, True):
        ob, lb = brute_force(q, k, v, 0.4, causal)
        for kw in (dict(), dict(window=(M, N)), dict(alibi_slopes=np.zeros(H)),
                   dict(softcap=1e7)):
            o, lse = oracle.attn_fwd_mod(q, k, v, 0.4, causal, lib=lib, **kw)
            if not (same(o, ob, 1e-10) and same(lse, lb, 1e-10)):
                errs.append(f"reduction {sorted(kw)} causal={causal}")
    ob, lb = brute_force(q, k, v, 0.4, True)
    o, lse = oracle.attn_fwd_mod(q, k, v, 0.4, False, window=(-1, 0), lib=lib)
    if not (same(o, ob, 1e-12) and same(lse, lb, 1e-12)):
        errs.append("window (-1, 0) != causal")
    return errs


def mod_closed_form_errors(lib):
    errs = []
    # K = 0 under a window: the mean of the V rows in [i - wl, i + wr] (clipped
    # to the keys, and to j <= i when causal), L = ln(count); no key: O = 0, L = -inf
    B, H, M, N, D = 1, 2, 14, 6, 3
    _, _, v = rand_inputs(92, B, H, M, N, D, si.FP64)
    for wl, wr in ((0, 0), (2, 1), (3, -1), (-1, 2), (5, 0), (1, 4)):
        for causal in (False, True):
            o, lse = oracle.attn_fwd_mod(np.ones((B, H, M, D)), np.zeros((B, H, N, D)), v, 1.0, causal,
                                         window=(wl, wr), lib=lib)
            for i in range(M):
                lo = max(0, i - wl) if wl >= 0 else 0
                hi = min(N - 1, i + wr) if wr >= 0 else N - 1
                if causal:
                    hi = min(hi, i)
                cnt = hi - lo + 1
                want_o = v[:, :, lo:hi + 1].mean(axis=2) if cnt > 0 else np.zeros((B, H, D))
                want_l = math.log(cnt) if cnt > 0 else -math.inf
                if not (same(o[:, :, i], want_o, 1e-14) and same(lse[:, :, i], np.full((B, H), want_l), 1e-14)):
                    errs.append(f"K=0 window ({wl},{wr}) causal={causal} row {i}")
                    break
    # ALiBi with K = 0 and V = identity: O[i, j] = r^|i-j| / Z_i with r = exp(-a)
    # and Z_i the two geometric sums to the left and right of i
    B, H, M, N = 2, 3, 7, 9
    slopes = np.array([[0.25, 0.5, 1.0], [0.125, 2.0, 0.75]])
    for causal in (False, True):
        o, lse = oracle.attn_fwd_mod(np.ones((B, H, M, N)), np.zeros((B, H, N, N)),
                                     np.broadcast_to(np.eye(N), (B, H, N, N)), 0.5, causal,
                                     alibi_slopes=slopes, lib=lib)
        for b in range(B):
            for h in range(H):
                r = math.exp(-slopes[b, h])
                for i in range(M):
                    left = (1 - r ** (i + 1)) / (1 - r)
                    right = 0.0 if causal else r * (1 - r ** (N - 1 - i)) / (1 - r)
                    z = left + right
                    want = np.array([r ** abs(i - j) / z if (j <= i or not causal) else 0.0
                                     for j in range(N)])
                    if not (same(o[b, h, i], want, 1e-14) and abs(lse[b, h, i] - math.log(z)) <= 1e-14):
                        errs.append(f"ALiBi closed form b={b} h={h} i={i} causal={causal}")
    # softcap c = 2 on the scores (ln 3, 0): 2 tanh(ln(3)/2) = 1 exactly, so the
    # capped scores are (1, 0): O = (e v0 + v1) / (e + 1), L = ln(e + 1).  With
    # ALiBi slope 1 on top (row 0 sees key 1 at distance 1): scores (1, -1).
    q = np.full((1, 1, 1, 1), math.log(3.0))
    k = np.array([1.0, 0.0]).reshape(1, 1, 2, 1)
    v = np.array([3.0, -5.0]).reshape(1, 1, 2, 1)
    e = math.e
    o, lse = oracle.attn_fwd_mod(q, k, v, 1.0, False, softcap=2.0, lib=lib)
    if abs(o.item() - (3 * e - 5) / (e + 1)) > 1e-14 or abs(lse.item() - math.log(e + 1)) > 1e-14:
        errs.append("softcap closed form")
    o, lse = oracle.attn_fwd_mod(q, k, v, 1.0, False, softcap=2.0, alibi_slopes=np.ones(1), lib=lib)
    if abs(o.item() - (3 * e - 5 / e) / (e + 1 / e)) > 1e-14 or abs(lse.item() - math.log(e + 1 / e)) > 1e-14:
        errs.append("softcap then ALiBi closed form")
    # saturated softcap: scores 100 and 200 both cap to 5: mean of V, L = 5 + ln 2
    o, lse = oracle.attn_fwd_mod(np.full((1, 1, 1, 1), 100.0), np.array([1.0, 2.0]).reshape(1, 1, 2, 1),
                                 v, 1.0, False, softcap=5.0, lib=lib)
    if abs(o.item() + 1.0) > 1e-14 or abs(lse.item() - (5 + math.log(2))) > 1e-14:
        errs.append("saturated softcap")
    return errs


def bwd_inputs(seed, B, H, Hkv, M, N, D, dtype=si.FP64):
    q = si.normal(seed, 1, (B, H, M, D), 1.0, dtype)
    k = si.normal(seed, 2, (B, Hkv, N, D), 1.0, dtype)
    v = si.normal(seed, 3, (B, Hkv, N, D), 1.0, dtype)
    do = si.normal(seed, 4, (B, H, M, D), 1.0, dtype)
    return q, k, v, do


def bwd_finite_difference_errors(lib):
    """The backward is the gradient of f(Q, K, V) = sum(dO o O(Q, K, V)) with O
    from the (separately pinned) forward oracle: central differences on sampled
    elements of Q, K and V, step 1e-5, relative error <= 1e-6."""
    errs = []
    for n, (B, H, Hkv, M, N, D, causal) in enumerate([(1, 2, 1, 6, 9, 4, False), (2, 2, 2, 7, 5, 3, True),
                                                       (1, 4, 2, 9, 9, 2, True)]):
        q, k, v, do = bwd_inputs(120 + n, B, H, Hkv, M, N, D)
        scale = 0.45
        grads = oracle.attn_bwd(q, k, v, do, scale, causal, lib=lib)

        def f(qq, kk, vv):
            o, _ = oracle.attn_fwd_gqa(qq, kk, vv, scale, causal, lib=lib)
            return float(np.sum(do * o))

        rng = np.random.default_rng(n)
        for which, (x, g) in enumerate(zip((q, k, v), grads)):
            gmax = float(np.max(np.abs(g))) + 1e-300
            for _ in range(6):
                idx = tuple(int(rng.integers(0, s)) for s in x.shape)
                xp, xm = x.copy(), x.copy()
                xp[idx] += 1e-5
                xm[idx] -= 1e-5
                args_p = [q, k, v]
                args_m = [q, k, v]
                args_p[which], args_m[which] = xp, xm
                fd = (f(*args_p) - f(*args_m)) / 2e-5
                if abs(fd - g[idx]) > 1e-6 * gmax:
                    errs.append(f"bwd finite difference case {n} {'qkv'[which]}{idx}: {fd} vs {g[idx]}")
    return errs


def bwd_closed_form_errors(lib):
    errs = []
    B, H, Hkv, M, N, D = 2, 4, 2, 11, 7, 5
    q, k, v, do = bwd_inputs(130, B, H, Hkv, M, N, D)
    g = H // Hkv
    for causal in (False, True):
        # one key: O = V_0 whatever Q and K are, so dQ = dK = 0 and dV_0 = sum of dO
        dq, dk, dv = oracle.attn_bwd(q, k[:, :, :1], v[:, :, :1], do, 0.5, causal, lib=lib)
        want = do.reshape(B, Hkv, g, M, D).sum(axis=(2, 3))
        if max_err(dq, 0) > 1e-14 or max_err(dk, 0) > 1e-14 or max_err(dv[:, :, 0], want) > 1e-12:
            errs.append(f"bwd N=1 causal={causal}")
        # K = 0: uniform weights, dV_j = sum over rows that see j of dO_i / #visible(i)
        dq, dk, dv = oracle.attn_bwd(q, np.zeros_like(k), v, do, 0.5, causal, lib=lib)
        nvis = np.minimum(np.arange(M) + 1, N) if causal else np.full(M, N)
        w = np.array([[1.0 / nvis[i] if (j < nvis[i]) else 0.0 for j in range(N)] for i in range(M)])
        want = np.einsum("ij,bkgid->bkjd", w, do.reshape(B, Hkv, g, M, D))
        if max_err(dv, want) > 1e-12:
            errs.append(f"bwd K=0 dV causal={causal}")
        # rows of dS sum to zero, so the dK of every key/value head sums to zero over keys
        dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.5, causal, lib=lib)
        if max_err(dk.sum(axis=2), 0) > 1e-12:
            errs.append(f"bwd sum_j dK_j != 0 causal={causal}")
    return errs


def bwd_torch_errors(lib):
    """PyTorch CPU autograd in fp64 (K/V heads repeated for grouped-query)."""
    try:
        import torch
    except ImportError:
        return []
    errs = []
    for n, (B, H, Hkv, M, N, D) in enumerate([(2, 4, 2, 13, 17, 8), (1, 3, 3, 20, 9, 16), (1, 2, 1, 1, 4, 4)]):
        for dtype in (si.FP64, si.BF16):
            q, k, v, do = bwd_inputs(140 + n, B, H, Hkv, M, N, D, dtype)
            for causal in (False, True):
                dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.3, causal, lib=lib)
                tq, tk, tv = (torch.from_numpy(widen(x)).requires_grad_() for x in (q, k, v))
                rk, rv = (t.repeat_interleave(H // Hkv, dim=1) for t in (tk, tv))
                sc = 0.3 * tq @ rk.transpose(-1, -2)
                if causal:
                    sc = sc.masked_fill(~torch.ones(M, N, dtype=torch.bool).tril(), float("-inf"))
                (torch.softmax(sc, -1) @ rv).backward(torch.from_numpy(widen(do)))
                e = max(max_err(dq, tq.grad.numpy()), max_err(dk, tk.grad.numpy()),
                        max_err(dv, tv.grad.numpy()))
                if not e <= 1e-12:
                    errs.append(f"bwd torch {(B, H, Hkv, M, N, D)} {dtype} causal={causal}: {e}")
    return errs


def all_pin_errors(lib):
    errs = []
    for check in (golden_errors, brute_errors, large_score_errors, invariant_errors,
                  rows_errors, tiled_errors, gqa_errors, mod_brute_errors, mod_reduction_errors,
                  mod_closed_form_errors, bwd_finite_difference_errors, bwd_closed_form_errors,
                  bwd_torch_errors):
        try:
            errs += check(lib)
        except Exception as exc:  # a mutant may also crash or return an error code
            errs.append(f"{check.__name__} raised {exc!r}")
    return errs


# ---------------------------------------------------------------- tests
def test_generator_is_counter_based_and_deterministic():
    a = si.normal(9, 2, (1000,), 1.0, si.FP64)
    b = si.normal(9, 2, (400,), 1.0, si.FP64, offset=600)
    assert np.array_equal(a[600:], b)
    assert np.array_equal(a, si.normal(9, 2, (1000,), 1.0, si.FP64))
    assert not np.array_equal(a, si.normal(9, 3, (1000,), 1.0, si.FP64))
    big = si.normal(1, 1, (200000,), 1.0, si.FP64)
    assert abs(big.mean()) < 0.01 and abs(big.std() - 1.0) < 0.01
    bits = si.normal(9, 2, (1000,), 1.0, si.BF16)
    f32 = si.normal(9, 2, (1000,), 1.0, si.FP32)
    # bf16 = RNE of the fp32 value: within half a bf16 ulp
    w = si.bf16_bits_to_f32(bits)
    assert np.all(np.abs(w - f32) <= np.abs(f32) * 2.0 ** -8 + 1e-30)
    assert np.array_equal(si.f64_to_bf16_bits(f32.astype(np.float64)), bits)


def test_golden_worked_examples(oracle_lib):
    assert golden_errors(oracle_lib) == []


def test_matches_brute_force(oracle_lib):
    assert brute_errors(oracle_lib) == []


def test_large_scores_stable(oracle_lib):
    assert large_score_errors(oracle_lib) == []


def test_invariants(oracle_lib):
    assert invariant_errors(oracle_lib) == []


def test_row_sampled_entry_matches_full(oracle_lib):
    assert rows_errors(oracle_lib) == []


def test_tiled_recurrence_equals_two_pass(oracle_lib):
    assert tiled_errors(oracle_lib) == []


def test_grouped_query_attention_matches_repeated_heads(oracle_lib):
    assert gqa_errors(oracle_lib) == []


def test_score_modifiers_match_brute_force(oracle_lib):
    assert mod_brute_errors(oracle_lib) == []


def test_score_modifiers_reduce_to_plain_attention(oracle_lib):
    assert mod_reduction_errors(oracle_lib) == []


def test_score_modifiers_closed_forms(oracle_lib):
    assert mod_closed_form_errors(oracle_lib) == []


def test_backward_is_the_gradient_of_the_forward(oracle_lib):
    assert bwd_finite_difference_errors(oracle_lib) == []


def test_backward_closed_forms(oracle_lib):
    assert bwd_closed_form_errors(oracle_lib) == []


def test_backward_matches_torch_autograd_fp64(oracle_lib):
    pytest.importorskip("torch")
    assert bwd_torch_errors(oracle_lib) == []


def test_matches_torch_sdpa_fp64():
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    for n, (B, H, M, N, D) in enumerate([(2, 3, 17, 17, 32), (1, 2, 40, 24, 64), (1, 1, 24, 40, 8)]):
        q, k, v = rand_inputs(60 + n, B, H, M, N, D, si.FP32)
        for causal in (False, True):
            o, lse = oracle.attn_fwd(q, k, v, 1.0 / math.sqrt(D), causal)
            tq, tk, tv = (torch.from_numpy(widen(t)) for t in (q, k, v))
            to = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)
            s = tq @ tk.transpose(-1, -2) / math.sqrt(D)
            if causal:
                s = s.masked_fill(~torch.ones(M, N, dtype=torch.bool).tril(), float("-inf"))
            tl = torch.logsumexp(s, dim=-1)
            assert max_err(o, to.numpy()) < 1e-12
            assert max_err(lse, tl.numpy()) < 1e-12


def test_rejects_bad_sizes(oracle_lib):
    q = np.zeros((1, 1, 4, 8))
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, np.zeros((1, 1, 4, 7)), np.zeros((1, 1, 4, 7)), 1.0, False)
    with pytest.raises(RuntimeError):
        oracle.attn_fwd(q, np.zeros((1, 1, 0, 8)), np.zeros((1, 1, 0, 8)), 1.0, False)


# Each mutant: (name, original snippet, replacement, count). The snippets are
# taken from fa2_oracle.c; the test fails loudly if one no longer matches.
MUTANTS = [
    ("causal excludes the diagonal", "return (i + 1 < N) ? i + 1 : N;", "return (i < N) ? i : N;", 1),
    ("causal one key too many", "return (i + 1 < N) ? i + 1 : N;", "return (i + 2 < N) ? i + 2 : N;", 1),
    ("causal ignored", "if (!causal) return N;", "if (1) return N;", 1),
    ("scale dropped", "w[j] = scale * dot;", "w[j] = dot;", 1),
    ("K read transposed", "widen(k, kvoff + j * D + d, dtype);\n    w[j]",
     "widen(k, kvoff + d * N + j, dtype);\n    w[j]", 1),
    ("exp sign flipped", "w[j] = exp(w[j] - m);", "w[j] = exp(m - w[j]);", 1),
    ("max not subtracted", "w[j] = exp(w[j] - m);", "w[j] = exp(w[j]);", 1),
    ("no final divide", "o_row[d] = acc / l;", "o_row[d] = acc;", 1),
    ("L without log", "*lse = m + log(l);", "*lse = m + l;", 1),
    ("L in log2", "*lse = m + log(l);", "*lse = m + log2(l);", 1),
    ("L missing max", "*lse = m + log(l);", "*lse = log(l);", 1),
    ("V always row 0", "acc += w[j] * widen(v, kvoff + j * D + d, dtype);",
     "acc += w[j] * widen(v, kvoff + d, dtype);", 1),
    ("Q row offset dropped", "const int64_t qoff = (bh * M + i) * (int64_t)D;\n  const int64_t kvoff = kvh",
     "const int64_t qoff = (bh * M) * (int64_t)D;\n  const int64_t kvoff = kvh", 1),
    ("K/V head offset dropped", "const int64_t kvoff = kvh * (int64_t)N * D;\n  const int64_t nvis",
     "const int64_t kvoff = 0;\n  const int64_t nvis", 1),
    ("GQA: query head mapped modulo Hkv", "return (bh / H) * Hkv + (bh % H) / (H / Hkv);",
     "return (bh / H) * Hkv + (bh % H) % Hkv;", 1),
    ("GQA: batch offset of the K/V head dropped", "return (bh / H) * Hkv + (bh % H) / (H / Hkv);",
     "return (bh % H) / (H / Hkv);", 1),
    ("window: left bound one key short", "if (wl >= 0 && i - wl > lo) lo = i - wl;",
     "if (wl >= 0 && i - wl > lo) lo = i - wl + 1;", 1),
    ("window: right bound one key long", "if (wr >= 0 && i + wr < hi) hi = i + wr;",
     "if (wr >= 0 && i + wr < hi) hi = i + wr + 1;", 1),
    ("window: causal ignored", "if (causal && i < hi) hi = i;", "if (0 && i < hi) hi = i;", 1),
    ("window: V rows read from the window start", "acc += w[j - lo] * widen(v, kvoff + j * D + d, dtype);",
     "acc += w[j - lo] * widen(v, kvoff + (j - lo) * D + d, dtype);", 1),
    ("window: empty row L = 0", "    *lse = -INFINITY;\n    return 0;", "    *lse = 0.0;\n    return 0;", 1),
    ("softcap: inner divide dropped", "s = softcap * tanh(s / softcap);", "s = softcap * tanh(s);", 1),
    ("softcap: outer multiply dropped", "s = softcap * tanh(s / softcap);", "s = tanh(s / softcap);", 1),
    ("ALiBi: sign flipped", "s -= slope * fabs((double)(i - j));", "s += slope * fabs((double)(i - j));", 1),
    ("ALiBi: signed distance", "s -= slope * fabs((double)(i - j));", "s -= slope * (double)(i - j);", 1),
    ("ALiBi: every head uses slope 0", "slopes[(bh / H) * slope_bstride + bh % H]",
     "slopes[(bh / H) * slope_bstride]", 1),
    ("ALiBi: batch stride ignored", "slopes[(bh / H) * slope_bstride + bh % H]", "slopes[bh % H]", 1),
    ("ALiBi: added before the softcap", "    if (softcap > 0.0) s = softcap * tanh(s / softcap);\n"
     "    s -= slope * fabs((double)(i - j));",
     "    s -= slope * fabs((double)(i - j));\n    if (softcap > 0.0) s = softcap * tanh(s / softcap);", 1),
    ("mod: Q row offset dropped", "const int64_t qoff = (bh * M + i) * (int64_t)D;\n  int64_t lo",
     "const int64_t qoff = (bh * M) * (int64_t)D;\n  int64_t lo", 1),
    ("mod: K/V head offset dropped", "const int64_t kvoff = kvh * (int64_t)N * D;\n  const int64_t qoff",
     "const int64_t kvoff = 0;\n  const int64_t qoff", 1),
    ("mod: no final divide", "o_row[d] = acc / lsum;", "o_row[d] = acc;", 1),
    ("mod: L missing max", "*lse = m + log(lsum);", "*lse = log(lsum);", 1),
    ("mod: max not subtracted", "w[j - lo] = exp(w[j - lo] - m);", "w[j - lo] = exp(w[j - lo]);", 1),
    ("bwd: dQ scale dropped", "dq[qoff + d] = scale * acc;", "dq[qoff + d] = acc;", 1),
    ("bwd: dK scale dropped", "dk_t[j * D + d] += scale * ds[j] * widen(q, qoff + d, dtype);",
     "dk_t[j * D + d] += ds[j] * widen(q, qoff + d, dtype);", 1),
    ("bwd: D_i added instead of subtracted", "ds[j] = p[j] * (dp - Di);", "ds[j] = p[j] * (dp + Di);", 1),
    ("bwd: D_i dropped", "ds[j] = p[j] * (dp - Di);", "ds[j] = p[j] * dp;", 1),
    ("bwd: dS without P", "ds[j] = p[j] * (dp - Di);", "ds[j] = dp - Di;", 1),
    ("bwd: D_i from dO . dO", "Di += widen(dout, qoff + d, dtype) * acc;",
     "Di += widen(dout, qoff + d, dtype) * widen(dout, qoff + d, dtype);", 1),
    ("bwd: dV from dS", "dv_t[j * D + d] += p[j] * widen(dout, qoff + d, dtype);",
     "dv_t[j * D + d] += ds[j] * widen(dout, qoff + d, dtype);", 1),
    ("bwd: dK from K", "dk_t[j * D + d] += scale * ds[j] * widen(q, qoff + d, dtype);",
     "dk_t[j * D + d] += scale * ds[j] * widen(k, kvoff + j * D + d, dtype);", 1),
    ("bwd: thread partials of dK dropped", "dk[kvoff + e] += dk_t[e];", "dk[kvoff + e] = dk_t[e];", 1),
    ("bwd: P not normalised", "for (int64_t j = 0; j < nvis; ++j) p[j] = exp(p[j] - L);",
     "for (int64_t j = 0; j < nvis; ++j) p[j] = exp(p[j] - m);", 1),
    ("bwd: query heads of a group interleaved", "const int64_t bh = (kvh / Hkv) * H + (kvh % Hkv) * group + g;",
     "const int64_t bh = (kvh / Hkv) * H + g * Hkv + (kvh % Hkv);", 1),
    ("bwd: causal ignored", "const int64_t nvis = visible_keys(i, N, causal);\n          /* scores",
     "const int64_t nvis = visible_keys(i, N, 0);\n          /* scores", 1),
    ("tiled: O not rescaled", "acc[(int64_t)r * D + d] = alpha * acc[(int64_t)r * D + d] + pv;",
     "acc[(int64_t)r * D + d] = acc[(int64_t)r * D + d] + pv;", 1),
    ("tiled: l not rescaled", "l_run[r] = alpha * l_run[r] + rowsum;", "l_run[r] = l_run[r] + rowsum;", 1),
    ("tiled: alpha sign flipped", "const double alpha = exp(m_run[r] - m_new);",
     "const double alpha = exp(m_new - m_run[r]);", 1),
    ("tiled: causal mask off by one", "if (causal && j > i) {", "if (causal && j >= i) {", 1),
    ("tiled: ragged last key tile dropped", "for (int64_t j0 = 0; j0 < N; j0 += BN) {",
     "for (int64_t j0 = 0; j0 + BN <= N; j0 += BN) {", 1),
]


def test_planted_mistakes_are_caught():
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(oracle._SRC).read()
    assert all_pin_errors(oracle.load()) == [], "the unmodified oracle must pass every pin"
    survived = []
    with tempfile.TemporaryDirectory() as tmp:
        for n, (name, old, new, count) in enumerate(MUTANTS):
            assert src.count(old) == count, f"mutant {name!r}: snippet not found in the oracle source"
            msrc = os.path.join(tmp, f"m{n}.c")
            mlib = os.path.join(tmp, f"m{n}.so")
            with open(msrc, "w") as f:
                f.write(src.replace(old, new))
            subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", "-fopenmp", "-o", mlib, msrc, "-lm"])
            errs = all_pin_errors(oracle.load(mlib))
            if not errs:
                survived.append(name)
    assert survived == [], f"mutants not caught by any pin: {survived}"
