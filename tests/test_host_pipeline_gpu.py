"""The host-buffer entries fa2_fwd_host and fa2_bwd_host: copies in slices of
heads overlapped with the compute of other slices.  Each slice is computed by the
same kernels as a whole-problem call, so the outputs must equal fa2_fwd's (and
fa2_bwd's) bitwise, for any number of slices, grouped-query heads and page-locked
or pageable host memory -- except the backward's dQ at head dim 128, formed by
fp32 reductions whose order varies from run to run; one forward case is also
checked against the oracle."""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import TOL, compare, to_host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fa2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_fa2_gb300 as m
    m.lib()
    return m


@pytest.fixture(autouse=True)
def device_status_clean(fa2):
    assert fa2.fa2_device_status(reset=True) == 0
    yield
    assert fa2.fa2_device_status(reset=True) == 0


def host(a, pin=True):
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
    return t.pin_memory() if pin else t.clone()


CASES = [  # (B, H, H_kv, M, N, D, dtype, causal)
    (2, 4, 4, 300, 500, 128, si.BF16, True),
    (1, 8, 2, 257, 257, 64, si.BF16, False),
    (3, 6, 3, 130, 700, 128, si.FP32, True),
    (1, 1, 1, 1, 1, 64, si.BF16, False),
]


@pytest.mark.parametrize("chunks", [0, 1, 3, 99])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_host_entry_equals_device_entry(fa2, case, chunks):
    B, H, Hkv, M, N, D, dtype, causal = case
    q = si.normal(500, 1, (B, H, M, D), 1.0, dtype)
    k = si.normal(500, 2, (B, Hkv, N, D), 1.0, dtype)
    v = si.normal(500, 3, (B, Hkv, N, D), 1.0, dtype)
    hq, hk, hv = host(q), host(k), host(v)
    o_h, l_h = fa2.fa2_fwd_host(hq, hk, hv, causal=causal, chunks=chunks)
    torch.cuda.synchronize()
    o_d, l_d = fa2.fa2_fwd(hq.cuda(), hk.cuda(), hv.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())


def test_host_entry_pageable_memory_and_oracle(fa2):
    B, H, Hkv, M, N, D = 2, 8, 2, 200, 333, 128
    q = si.normal(510, 1, (B, H, M, D), 1.0, si.BF16)
    k = si.normal(510, 2, (B, Hkv, N, D), 1.0, si.BF16)
    v = si.normal(510, 3, (B, Hkv, N, D), 1.0, si.BF16)
    o_h, l_h = fa2.fa2_fwd_host(host(q, False), host(k, False), host(v, False), causal=True, chunks=3,
                                o_host=torch.empty((B, H, M, D), dtype=torch.bfloat16),
                                lse_host=torch.empty((B, H, M), dtype=torch.float32))
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attn_fwd_gqa(q, k, v, float(np.float32(D ** -0.5)), True)
    eo, el, excess = compare(to_host_f64(o_h), l_h.numpy().astype(np.float64), o_ref, l_ref, si.BF16)
    assert excess <= 0 and el <= TOL[si.BF16], (eo, el)


def test_host_entry_back_to_back_calls(fa2):
    """Consecutive calls reuse the device buffers: the second call's copies must
    wait for the first call's kernels and copies back."""
    B, H, M, N, D = 2, 8, 256, 256, 128
    ins = [[si.normal(520 + i, s, (B, H, M if s == 1 else N, D), 1.0, si.BF16) for s in (1, 2, 3)]
           for i in range(2)]
    bufs = [torch.empty((B, H, M, D), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    lse = torch.empty((B, H, M), dtype=torch.float32, device="cuda")
    outs = []
    for q, k, v in ins:
        outs.append(fa2.fa2_fwd_host(host(q), host(k), host(v), q=bufs[0], k=bufs[1], v=bufs[2], o=bufs[3],
                                     lse=lse, chunks=4))
    torch.cuda.synchronize()
    for (q, k, v), (o_h, l_h) in zip(ins, outs):
        o_d, l_d = fa2.fa2_fwd(host(q).cuda(), host(k).cuda(), host(v).cuda())
        torch.cuda.synchronize()
        assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())


BWD_CASES = [  # (B, H, H_kv, M, N, D, causal)
    (2, 4, 4, 300, 500, 128, True),
    (1, 8, 2, 257, 257, 64, False),
    (2, 6, 3, 130, 700, 128, True),
    (1, 1, 1, 1, 1, 64, False),
]


@pytest.mark.parametrize("chunks", [0, 1, 3, 99])
@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: "x".join(map(str, c)))
def test_host_backward_equals_device_backward(fa2, case, chunks):
    """fa2_bwd_host: the same kernels per slice of heads, so dk, dv (and dq at
    head dim 64) equal fa2_bwd's bitwise for any number of slices; dq at head dim
    128 (by reduction) to within one bf16 ulp of its largest entry."""
    B, H, Hkv, M, N, D, causal = case
    q = si.normal(510, 1, (B, H, M, D), 1.0, si.BF16)
    k = si.normal(510, 2, (B, Hkv, N, D), 1.0, si.BF16)
    v = si.normal(510, 3, (B, Hkv, N, D), 1.0, si.BF16)
    do = si.normal(510, 4, (B, H, M, D), 1.0, si.BF16)
    hq, hk, hv, hdo = host(q), host(k), host(v), host(do)
    o, lse = fa2.fa2_fwd(hq.cuda(), hk.cuda(), hv.cuda(), causal=causal)
    torch.cuda.synchronize()
    ho, hl = o.cpu().pin_memory(), lse.cpu().pin_memory()
    dq_h, dk_h, dv_h = fa2.fa2_bwd_host(hq, hk, hv, ho, hl, hdo, causal=causal, chunks=chunks)
    torch.cuda.synchronize()
    dq, dk, dv = fa2.fa2_bwd(hq.cuda(), hk.cuda(), hv.cuda(), o, lse, hdo.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(dk_h, dk.cpu()) and torch.equal(dv_h, dv.cpu())
    if D == 64:
        assert torch.equal(dq_h, dq.cpu())
    else:
        ulp = float(dq.float().abs().max()) * 2.0 ** -8
        assert float((dq_h.float() - dq.cpu().float()).abs().max()) <= ulp
