"""CPU checks of two readings the kernels rely on.  (1) The online softmax
recurrence gives the plain softmax result for any exponent base, so the base may
lag the running row max.  (2) The split-KV slices' partials, merged by their
logsumexp, give the plain result (end of the file).

"From FlashAttention to FlashAttention 2" (FlashAttention 2: What Changed) and
"Writing FlashAttention 2 in Triton" (Step 3) move the running max m on every key
tile and rescale the accumulator by exp(m_old - m_new).  The kernels move a row's
base only when its max has grown past the base by more than 4 in log2 units (a
factor of 2^4).
Here that lagging recurrence, written out in fp64 over 128-key tiles, is compared
with the fp64 oracle (the two-pass definition) on rows whose max climbs over the
tiles, so the base both lags and moves.  Two broken variants (no rescale of
what was summed when the base moves; L without the base) must miss the oracle by
far more than the 1e-12 the correct one meets, so the check can tell them apart.
"""
import math

import numpy as np
import pytest

import oracle

LAG_LOG2 = 4.0  # the kernels' bound (kBaseLagLog2)
BN = 128


def lagging_recurrence(q, k, v, scale, causal, rescale=True, base_in_l=True):
    """O and L (natural log) of one head, tile by tile, with a lagging base.
    ``rescale=False`` or ``base_in_l=False`` drop one step (test mutants)."""
    M, D = q.shape
    N = k.shape[0]
    c = scale / math.log(2.0)  # scores in log2 units
    o = np.zeros((M, D))
    lse = np.zeros(M)
    moves = 0
    for i in range(M):
        base, l, acc = -math.inf, 0.0, np.zeros(D)
        for j0 in range(0, N, BN):
            j1 = min(N, j0 + BN) if not causal else min(N, j0 + BN, i + 1)
            if j1 <= j0:
                break
            s = (k[j0:j1] @ q[i]) * c
            m_tile = float(s.max())
            if m_tile - base > LAG_LOG2:  # move the base; rescale what was summed
                alpha = 0.0 if base == -math.inf else 2.0 ** (base - m_tile)
                if rescale:
                    acc *= alpha
                    l *= alpha
                base = m_tile
                moves += 1
            p = 2.0 ** (s - base)
            l += float(p.sum())
            acc += p @ v[j0:j1]
        o[i] = acc / l
        lse[i] = ((base if base_in_l else 0.0) + math.log2(l)) * math.log(2.0)
    return o, lse, moves


@pytest.mark.parametrize("causal", [False, True])
def test_lagging_base_matches_two_pass(causal):
    rng = np.random.default_rng(11)
    # causal rows see keys up to their own index only, so they need M = N to
    # span several key tiles
    M, N, D = (520, 520, 32) if causal else (40, 700, 32)
    q = rng.standard_normal((M, D)) * 2.0
    # keys scaled up along the key axis: each row's max climbs over the tiles
    k = rng.standard_normal((N, D)) * 2.0 * np.linspace(0.1, 3.0, N)[:, None]
    v = rng.standard_normal((N, D))
    scale = D ** -0.5
    o, lse, moves = lagging_recurrence(q, k, v, scale, causal)
    o_ref, l_ref = oracle.attn_fwd(q[None, None], k[None, None], v[None, None], scale, causal)
    assert moves > M  # some rows moved their base after the first tile
    assert np.max(np.abs(o - o_ref[0, 0])) < 1e-12
    assert np.max(np.abs(lse - l_ref[0, 0])) < 1e-12
    # a recurrence that forgets to rescale, or an L without the base, is caught
    o_bad, l_bad, _ = lagging_recurrence(q, k, v, scale, causal, rescale=False)
    assert max(np.max(np.abs(o_bad - o_ref[0, 0])), np.max(np.abs(l_bad - l_ref[0, 0]))) > 1e-3
    o_bad, l_bad, _ = lagging_recurrence(q, k, v, scale, causal, base_in_l=False)
    assert np.max(np.abs(l_bad - l_ref[0, 0])) > 1.0


def split_partials(q, k, v, scale, causal, num_splits):
    """Per-slice partials of one head, as the split-KV kernels write them: slice s
    holds whole 128-key tiles [s*tps, (s+1)*tps) and gives O_s = (its P V) / l_s
    and L_s = m_s + ln l_s; a row without a visible key in the slice gets O_s = 0
    and L_s = -inf."""
    M, D = q.shape
    N = k.shape[0]
    n_kv = -(-N // BN)
    tps = -(-n_kv // num_splits)
    parts = []
    for j0 in range(0, N, tps * BN):
        j1 = min(N, j0 + tps * BN)
        s = (q @ k[j0:j1].T) * scale
        if causal:
            s = np.where(np.arange(j0, j1)[None, :] <= np.arange(M)[:, None], s, -np.inf)
        m = s.max(1)
        seen = np.isfinite(m)
        w = np.exp(s - np.where(seen, m, 0.0)[:, None])
        l = w.sum(1)
        o = np.where(seen[:, None], (w @ v[j0:j1]) / np.where(seen, l, 1.0)[:, None], 0.0)
        parts.append((o, np.where(seen, m + np.log(np.where(seen, l, 1.0)), -np.inf)))
    return parts


def merge(parts, weights="lse"):
    """The combine: L = ln sum_s exp(L_s), O = sum_s exp(L_s - L) O_s.
    ``weights`` "mean" or "max" are broken merges (test mutants)."""
    o_s = np.stack([o for o, _ in parts])
    l_s = np.stack([l for _, l in parts])
    lmax = l_s.max(0)
    if weights == "mean":
        w = np.isfinite(l_s).astype(np.float64)
    else:
        w = np.exp(l_s - lmax)
    denom = w.sum(0)
    o = (w[:, :, None] * o_s).sum(0) / denom[:, None]
    lse = lmax if weights == "max" else lmax + np.log(denom)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("num_splits", [2, 3, 7])
def test_split_kv_merge_matches_two_pass(causal, num_splits):
    """The reading of the split-KV dispatch ("From FlashAttention to FlashAttention
    2", Layer 2): merging the slices' (O_s, L_s) by their logsumexp gives the plain
    result.  Causal rows see no key of the later slices (L_s = -inf), so those
    slices must add nothing."""
    rng = np.random.default_rng(23 + num_splits)
    # causal rows see keys up to their own index: M = N lets late rows span slices
    M, N, D = (900, 900, 16) if causal else (300, 900, 16)
    q = rng.standard_normal((M, D)) * 1.5
    k = rng.standard_normal((N, D)) * 1.5
    v = rng.standard_normal((N, D))
    scale = D ** -0.5
    parts = split_partials(q, k, v, scale, causal, num_splits)
    assert len(parts) > 1
    if causal:
        assert np.isinf(parts[-1][1][:128]).all()  # early rows: the last slice is empty
    o, lse = merge(parts)
    o_ref, l_ref = oracle.attn_fwd(q[None, None], k[None, None], v[None, None], scale, causal)
    assert np.max(np.abs(o - o_ref[0, 0])) < 1e-12
    assert np.max(np.abs(lse - l_ref[0, 0])) < 1e-12
    # equal weights per slice, or L without the log-sum, miss the oracle by far more
    o_bad, _ = merge(parts, "mean")
    assert np.max(np.abs(o_bad - o_ref[0, 0])) > 1e-3
    _, l_bad = merge(parts, "max")
    assert np.max(np.abs(l_bad - l_ref[0, 0])) > 1e-3
