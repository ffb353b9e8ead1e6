"""Host-side pins for the parity comparison itself (no GPU)."""
import numpy as np

import seeded_inputs as si
from gpu_helpers import TOL, compare, compare_stats, half_ulp_bf16, o_bound


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


def test_o_bound_is_flat_below_two_and_adds_half_an_ulp_above():
    o = np.array([0.0, 0.3, -1.0, 1.999, -1.999, 2.0, -3.0, 4.0, 7.5])
    b = o_bound(o, si.BF16)
    assert np.all(b[:5] == 1e-2)                       # the flat bound where it is attainable
    assert np.array_equal(b[5:], 1e-2 + np.array([2 ** -7, 2 ** -7, 2 ** -6, 2 ** -6]))
    assert np.all(o_bound(o, si.FP32) == 5e-3)          # fp32 outputs: flat everywhere


def test_compare_rejects_an_error_over_the_flat_bound_below_two():
    o_ref = np.array([[1.5, 0.25], [3.0, -5.0]])
    l_ref = np.array([0.1, 0.2])
    # 0.0101 on an element with |O_ref| < 2: over 1e-2, though within 1e-2 + half an ulp
    o_gpu = o_ref + np.array([[0.0101, 0.0], [0.0, 0.0]])
    assert compare(o_gpu, l_ref, o_ref, l_ref, si.BF16)[2] > 0
    # the same error at |O_ref| = 3 is inside 1e-2 + 2^-7
    o_gpu = o_ref + np.array([[0.0, 0.0], [0.0101, 0.0]])
    assert compare(o_gpu, l_ref, o_ref, l_ref, si.BF16)[2] <= 0
    # and 0.0101 + 2^-6 at |O_ref| = 5 is over 1e-2 + 2^-6
    o_gpu = o_ref + np.array([[0.0, 0.0], [0.0, -(0.0101 + 2 ** -6)]])
    assert compare(o_gpu, l_ref, o_ref, l_ref, si.BF16)[2] > 0


def test_compare_stats_split_by_magnitude():
    o_ref = np.array([[1.0, 2.5], [-0.5, -4.0]])
    o_gpu = o_ref + np.array([[0.004, 0.012], [-0.001, 0.0]])
    l = np.zeros(2)
    st = compare_stats(o_gpu, l + 0.003, o_ref, l, si.BF16)
    assert np.isclose(st["max_do_small"], 0.004) and np.isclose(st["max_do_large"], 0.012)
    assert st["n_large"] == 2 and np.isclose(st["max_dl"], 0.003) and st["max_abs_oref"] == 4.0
    assert st["tol"] == TOL[si.BF16]
