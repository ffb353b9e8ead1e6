"""The failure path on the GPU, without a fault or a hang: a bounded wait that
nothing completes runs out after 20 ms (fa2_selftest_wait_timeout uses the same
bounded wait as every pipeline wait of the kernels) and records its code in the
device status word; while the word is set, a forward launch returns without
computing (its output keeps a canary value); once the word is cleared the same
call computes the right answer again and the context stayed usable throughout."""
import ctypes

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import TOL, compare, to_device, to_host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fa2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_fa2_gb300 as m
    m.lib()
    return m


def test_wait_that_runs_out_is_reported_and_later_launches_skip(fa2):
    assert fa2.fa2_device_status(reset=True) == 0
    B, H, M, N, D = 1, 2, 200, 300, 128
    q, k, v = (si.normal(600, s, (B, H, M if s == 1 else N, D), 1.0, si.BF16) for s in (1, 2, 3))
    tq, tk, tv = (to_device(a, "cuda:0") for a in (q, k, v))

    fa2.fa2_selftest_wait_timeout(20)
    torch.cuda.synchronize()
    raw = ctypes.c_int(-1)
    assert fa2.lib().fa2_device_status(0, ctypes.byref(raw)) == fa2.FA2_ERR_DEVICE_TIMEOUT
    assert raw.value == 99

    # while the word is set a forward launch is accepted but computes nothing
    o = torch.full((B, H, M, D), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, M), 7.0, dtype=torch.float32, device="cuda")
    fa2.fa2_fwd(tq, tk, tv, o=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(o == 7.0) and torch.all(lse == 7.0)

    # reading with reset clears it; the context is usable and the call computes again
    assert fa2.fa2_device_status(reset=True) == 99
    assert fa2.fa2_device_status(reset=True) == 0
    o, lse = fa2.fa2_fwd(tq, tk, tv, o=o, lse=lse)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attn_fwd(q, k, v, D ** -0.5, False)
    eo, el, excess = compare(to_host_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, l_ref, si.BF16)
    assert excess <= 0 and el <= TOL[si.BF16]
    assert fa2.fa2_device_status(reset=True) == 0
