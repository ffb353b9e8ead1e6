"""GPU parity of the backward pass against the fp64 oracle's attn_bwd, for both
ways of forming dQ: by reduction into an fp32 accumulator (fa2_bwd at head dim
128) and by a second pass (fa2_bwd_deterministic, and fa2_bwd at head dim 64).

The GPU backward gets the GPU forward's own O (bf16) and L, as it would in
training; the oracle recomputes everything from Q, K, V and dO in fp64 (the exact
gradient).  Bar, per gradient tensor: max |GPU - oracle| <= 1e-2 * max |oracle|
+ 1e-5.  Gradients have no fixed scale (dV_j sums P_ij dO_i over the queries
that see key j), so the bound is relative to the tensor's largest entry; the
rounding of the exact answer to bf16 alone is 2^-9 of an entry.  The 1e-5 floor
is for gradients that are exactly zero (one visible key: dQ = dK = 0), where the
fp32 difference dP - D leaves ~1e-6.  Shapes span several tiles with ragged
tails on both axes, M < N and M > N causal, grouped-query and multi-query
heads, both head dims.
"""
import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import to_device, to_host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DEV = "cuda:0"
REL_TOL = 1e-2
ABS_FLOOR = 1e-5


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
    assert fa2.fa2_device_status(reset=True) == 0, "a kernel pipeline wait ran out"


def inputs(seed, B, H, Hkv, M, N, D):
    q = si.normal(seed, 1, (B, H, M, D), 1.0, si.BF16)
    k = si.normal(seed, 2, (B, Hkv, N, D), 1.0, si.BF16)
    v = si.normal(seed, 3, (B, Hkv, N, D), 1.0, si.BF16)
    do = si.normal(seed, 4, (B, H, M, D), 1.0, si.BF16)
    return q, k, v, do


def gpu_grads(fa2, q, k, v, do, scale, causal, deterministic=False):
    tq, tk, tv, tdo = (to_device(a, DEV) for a in (q, k, v, do))
    o, lse = fa2.fa2_fwd(tq, tk, tv, scale=scale, causal=causal)
    dq, dk, dv = fa2.fa2_bwd(tq, tk, tv, o, lse, tdo, scale=scale, causal=causal, deterministic=deterministic)
    torch.cuda.synchronize()
    return tuple(to_host_f64(t) for t in (dq, dk, dv))


def check(got, want, what):
    for name, g, w in zip(("dQ", "dK", "dV"), got, want):
        assert np.all(np.isfinite(g)), f"{what}: non-finite {name}"
        err = float(np.max(np.abs(g - w)))
        ref = float(np.max(np.abs(w)))
        assert err <= REL_TOL * ref + ABS_FLOOR, f"{what}: {name} max err {err:.3g} vs max |ref| {ref:.3g}"


CASES = [  # (B, H, Hkv, M, N, D)
    (1, 1, 1, 128, 128, 128),
    (1, 2, 2, 256, 384, 64),
    (2, 2, 2, 200, 333, 128),   # ragged on both axes
    (1, 4, 2, 257, 190, 128),   # grouped-query, M > N
    (2, 4, 1, 130, 520, 64),    # multi-query, M < N
    (1, 2, 2, 64, 700, 128),    # one query step per head
    (1, 2, 2, 700, 64, 64),     # one key tile
    (1, 1, 1, 1, 1, 128),       # a single query and key
    (1, 3, 3, 1, 300, 64),      # a single query
    (1, 3, 3, 300, 1, 128),     # a single key
]


@pytest.mark.parametrize("deterministic", [False, True], ids=["reduce", "two_pass"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_backward_all_elements(fa2, case, causal, deterministic):
    B, H, Hkv, M, N, D = case
    q, k, v, do = inputs(400 + CASES.index(case), B, H, Hkv, M, N, D)
    scale = 1.0 / math.sqrt(D)
    got = gpu_grads(fa2, q, k, v, do, scale, causal, deterministic)
    want = oracle.attn_bwd(q, k, v, do, float(np.float32(scale)), causal)
    check(got, want, f"{case} causal={causal} deterministic={deterministic}")


def test_backward_other_scale(fa2):
    B, H, Hkv, M, N, D = 1, 2, 2, 190, 260, 128
    q, k, v, do = inputs(450, B, H, Hkv, M, N, D)
    for scale in (0.03, 0.2):
        got = gpu_grads(fa2, q, k, v, do, scale, True)
        want = oracle.attn_bwd(q, k, v, do, float(np.float32(scale)), True)
        check(got, want, f"scale {scale}")


def test_backward_deterministic(fa2):
    """fa2_bwd_deterministic forms dQ by a second pass, not by reduction:
    repeated calls agree bitwise."""
    B, H, Hkv, M, N, D = 2, 4, 2, 300, 500, 128
    q, k, v, do = (to_device(a, DEV) for a in inputs(460, B, H, Hkv, M, N, D))
    o, lse = fa2.fa2_fwd(q, k, v, causal=True)
    first = fa2.fa2_bwd(q, k, v, o, lse, do, causal=True, deterministic=True)
    for _ in range(3):
        again = fa2.fa2_bwd(q, k, v, o, lse, do, causal=True, deterministic=True)
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(first, again))


def test_backward_reduction_repeats(fa2):
    """dQ by reduction: dK and dV are still bitwise reproducible; dQ varies from
    call to call only by the order of its fp32 adds (within one bf16 ulp of its
    largest entry), and all three agree with the second-pass path as closely."""
    B, H, Hkv, M, N, D = 2, 4, 2, 700, 900, 128
    q, k, v, do = (to_device(a, DEV) for a in inputs(465, B, H, Hkv, M, N, D))
    o, lse = fa2.fa2_fwd(q, k, v, causal=True)
    first = fa2.fa2_bwd(q, k, v, o, lse, do, causal=True)
    two_pass = fa2.fa2_bwd(q, k, v, o, lse, do, causal=True, deterministic=True)
    torch.cuda.synchronize()
    for a, b in zip(first, two_pass):  # same sums in another order: at most one bf16 ulp apart
        assert float((a.float() - b.float()).abs().max()) <= float(b.float().abs().max()) * 2.0 ** -8
    ulp = float(first[0].float().abs().max()) * 2.0 ** -8
    for _ in range(3):
        again = fa2.fa2_bwd(q, k, v, o, lse, do, causal=True)
        torch.cuda.synchronize()
        assert float((first[0].float() - again[0].float()).abs().max()) <= ulp
        assert torch.equal(first[1], again[1]) and torch.equal(first[2], again[2])


def test_backward_writes_stay_inside_outputs(fa2):
    """Canary rows around dq, dk, dv: the TMA stores are clipped at M and N."""
    B, H, Hkv, M, N, D = 1, 2, 1, 130, 70, 128
    q, k, v, do = (to_device(a, DEV) for a in inputs(470, B, H, Hkv, M, N, D))
    o, lse = fa2.fa2_fwd(q, k, v)
    pad = 4096
    bufs = [torch.full((t.numel() + 2 * pad,), 7.0, dtype=torch.bfloat16, device=DEV) for t in (q, k, v)]
    dq, dk, dv = (b[pad:pad + t.numel()].view(t.shape) for b, t in zip(bufs, (q, k, v)))
    for deterministic in (False, True):
        fa2.fa2_bwd(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, deterministic=deterministic)
        torch.cuda.synchronize()
        for b in bufs:
            assert torch.all(b[:pad] == 7.0) and torch.all(b[-pad:] == 7.0)


def test_backward_at_bench_size_one_head(fa2):
    """2 x 16 x 8192 x 8192, D = 128, causal (the headline forward workload):
    every gradient of the first and the last head against the oracle run on
    that head alone."""
    w = si.WORKLOADS["bf16_2x16x8192x8192x128_causal"]
    q, k, v = si.make_qkv(w)
    do = si.normal(w.seed, 4, q.shape, 1.0, si.BF16)
    got = gpu_grads(fa2, q, k, v, do, w.scale, True)
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        want = oracle.attn_bwd(q[sl], k[sl], v[sl], do[sl], float(np.float32(w.scale)), True)
        check(tuple(g[sl] for g in got), want, f"head ({b}, {h})")
