"""Host-side pins for the parity comparison itself (no GPU)."""
import numpy as np

import seeded_inputs as si
from gpu_helpers import half_ulp_bf16, sample_rows


def test_half_ulp_bf16_values():
    x = np.array([1.0, 1.99, 2.0, 3.5, 4.0, 7.9, 0.5, -4.5, 0.0])
    want = np.array([2 ** -8, 2 ** -8, 2 ** -7, 2 ** -7, 2 ** -6, 2 ** -6, 2 ** -9, 2 ** -6, 0.0])
    assert np.array_equal(half_ulp_bf16(x), want)


def test_half_ulp_bounds_bf16_rounding():
    x = si.normal(3, 1, (200000,), 3.0, si.FP64)
    r = si.bf16_bits_to_f32(si.f64_to_bf16_bits(x)).astype(np.float64)
    # fp64 -> fp32 -> bf16 double rounding may exceed half an ulp by half an fp32 ulp
    assert np.all(np.abs(r - x) <= half_ulp_bf16(x) * (1 + 2 ** -14))
    # the bound is reached: rounding error of the exact value can exceed 1e-2 for |x| >= 4
    big = np.abs(x) >= 4
    assert np.max(np.abs(r - x)[big]) > 1e-2


def test_sample_rows_cover_edges_and_stay_in_range():
    B, H, M, N = 2, 3, 1000, 3000
    rows = sample_rows(B, H, M, N, causal=False, n_random=100)
    assert rows.min() >= 0 and rows.max() < B * H * M
    assert set(range(M)) <= set(rows.tolist())                 # first head in full
    assert set(range((B * H - 1) * M, B * H * M)) <= set(rows.tolist())  # last head in full
    for bh in range(B * H):
        for i in (0, M - 1, 127, 128, 895, 896, 999):
            assert bh * M + i in set(rows.tolist())
