"""The allocation-free split-KV entry point, fa2_fwd_splitkv_noalloc.

It exists for callers that cannot obtain device memory themselves (an exhausted
or locked-down allocator, a host framework that owns every allocation, code that
must not call cudaMalloc/cudaFree): its scratch is a buffer built into the
library.  This file is named so that pytest collects it last.

The test calls the entry point through the C ABI (ctypes) on several problems in
a row, each call reusing the buffer the previous one left behind, and checks
every result against the fp64 oracle at the parity bound and against
fa2_fwd_splitkv (the same computation with a caller-provided workspace).  The
problems cover an explicit split count, the automatic count (num_splits = 0),
and a count above the 64-slice cap whose lowered count fits in the buffer.
"""
import ctypes

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import TOL, compare, to_device, to_host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DEV = "cuda:0"
BUFFER_BYTES = 32 << 20  # the built-in buffer's size


@pytest.fixture(scope="module")
def fa2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_fa2_gb300 as m
    m.lib()
    return m


def call_noalloc(fa2, tq, tk, tv, o, lse, scale, causal, num_splits):
    B, H, M, D = tq.shape
    H_kv, N = tk.shape[1], tk.shape[2]
    dtype = fa2.FA2_BF16 if tq.dtype == torch.bfloat16 else fa2.FA2_FP32
    stream = torch.cuda.current_stream().cuda_stream
    return fa2.lib().fa2_fwd_splitkv_noalloc(
        tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, H_kv, M, N,
        D, ctypes.c_float(scale), 1 if causal else 0, dtype, num_splits, stream)


CASES = [  # (seed, B, H, H_kv, M, N, D, causal, num_splits, dtype)
    (41, 1, 8, 2, 128, 8192, 128, False, 4, si.BF16),
    (42, 2, 4, 4, 200, 3000, 64, True, 3, si.FP32),
    # 128 slices asked for: 67.6 MB of partials, but the call runs 32 slices
    # (one per key tile), 16.9 MB, which fit
    (43, 1, 8, 2, 128, 4096, 128, False, 128, si.BF16),
    # the library's own split count
    (44, 2, 8, 8, 64, 6000, 128, False, 0, si.BF16),
]


def test_calls_in_a_row_match_the_oracle_and_the_workspace_entry(fa2):
    assert fa2.fa2_device_status(reset=True) == 0
    assert fa2.fa2_splitkv_workspace_bytes(1, 8, 128, 128, 128) > BUFFER_BYTES
    results = []
    for seed, B, H, Hkv, M, N, D, causal, splits, dtype in CASES:
        q = si.normal(seed, 1, (B, H, M, D), 1.0, dtype)
        k = si.normal(seed, 2, (B, Hkv, N, D), 1.0, dtype)
        v = si.normal(seed, 3, (B, Hkv, N, D), 1.0, dtype)
        tq, tk, tv = (to_device(a, DEV) for a in (q, k, v))
        o = torch.empty_like(tq)
        lse = torch.empty((B, H, M), dtype=torch.float32, device=DEV)
        rc = call_noalloc(fa2, tq, tk, tv, o, lse, D ** -0.5, causal, splits)
        assert rc == fa2.FA2_OK, fa2.fa2_strerror(rc)
        results.append((q, k, v, tq, tk, tv, o, lse, D, causal, splits, dtype))
    torch.cuda.synchronize()
    for q, k, v, tq, tk, tv, o, lse, D, causal, splits, dtype in results:
        og, lg = to_host_f64(o), lse.cpu().numpy().astype(np.float64)
        o_ref, l_ref = oracle.attn_fwd_gqa(q, k, v, D ** -0.5, causal)
        eo, el, excess = compare(og, lg, o_ref, l_ref, dtype)
        assert excess <= 0 and el <= TOL[dtype], (splits, eo, el)
        o_ws, l_ws = fa2.fa2_fwd_splitkv(tq, tk, tv, scale=D ** -0.5, causal=causal, num_splits=splits)
        torch.cuda.synchronize()
        d_o = float(np.max(np.abs(og - to_host_f64(o_ws))))
        d_l = float((lse - l_ws).abs().max())
        assert d_o <= TOL[dtype] and d_l <= TOL[dtype], (splits, d_o, d_l)
    assert fa2.fa2_device_status(reset=True) == 0


def test_rejects_a_problem_larger_than_the_built_in_buffer(fa2):
    # 64 slices of 16 * 4096 rows of 129 fp32 values need about 2 GB, far beyond 32 MiB
    B, H, M, N, D = 1, 16, 4096, 65536, 128
    need = fa2.fa2_splitkv_workspace_bytes(B, H, M, D, 64)
    assert need > BUFFER_BYTES
    t = torch.empty(16, dtype=torch.bfloat16, device=DEV)  # never read: the call refuses first
    rc = fa2.lib().fa2_fwd_splitkv_noalloc(t.data_ptr(), t.data_ptr(), t.data_ptr(), t.data_ptr(),
                                           t.data_ptr(), B, H, H, M, N, D, ctypes.c_float(0.1), 0,
                                           fa2.FA2_BF16, 64, None)
    assert rc == fa2.FA2_ERR_WORKSPACE
