"""CPU check of a reading the kernels rely on: the online softmax recurrence gives
the plain softmax result for any exponent base, so the base may lag the running
row max.

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
