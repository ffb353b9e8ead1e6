"""Problems with more than 2^31 elements in one tensor.

q, o, dO and dQ of 1 x 2 x (2^23 + 77) x 128 bf16 hold 2.15e9 elements each
(4.3 GB), so every flat offset the kernels, the tensor maps and the host code
form past 2^31 must be 64-bit.  The inputs are drawn on the device with a
seeded torch generator (the host generator would take minutes at this size);
the oracle gets the exact bf16 values of the rows it checks, copied back.

- Forward: sampled rows (the first and last rows of each head, the rows on
  both sides of the 2^30- and 2^31-element offsets, seeded random rows)
  against the oracle run on those rows alone.  The problem is non-causal, so a
  row's output depends only on its own query and the head's keys and values.
- Backward: dO is zero except on the sampled rows.  A query row with dO = 0
  adds exactly nothing to dK and dV (its dP and D are 0, so is its dS), so the
  backward of the sub-problem made of the sampled rows gives the exact dK and
  dV of the whole problem, and its dQ on those rows: all three are checked
  against the oracle's attn_bwd on that sub-problem, while the kernels still
  stream all 8.4M query rows.  (With a dO that is nonzero everywhere, dK and dV
  are sums of 8.4M terms and came out ~1% of their size from a chunked fp32
  reference: an effect of the accumulation length, which is not what this test
  is about.)  Bar: max |GPU - oracle| <= 1e-2 max |oracle| + 1e-5,
  as in the backward parity tests; rows without dO must get dQ = 0 exactly.
"""
import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import TOL, compare, to_host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DEV = "cuda:0"
B, H, M, N, D = 1, 2, (1 << 23) + 77, 200, 128
REL_TOL = 1e-2


@pytest.fixture(scope="module")
def fa2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_fa2_gb300 as m
    m.lib()
    return m


@pytest.fixture(scope="module")
def problem(fa2):
    g = torch.Generator(device=DEV).manual_seed(2024)
    q = torch.randn((B, H, M, D), generator=g, device=DEV, dtype=torch.bfloat16)
    k = torch.randn((B, H, N, D), generator=g, device=DEV, dtype=torch.bfloat16)
    v = torch.randn((B, H, N, D), generator=g, device=DEV, dtype=torch.bfloat16)
    do = torch.zeros((B, H, M, D), device=DEV, dtype=torch.bfloat16)
    for h in range(H):
        idx = torch.from_numpy(rows_of_head(h)).to(DEV)
        do[0, h].index_copy_(0, idx, torch.randn((idx.numel(), D), generator=g, device=DEV,
                                                 dtype=torch.bfloat16))
    assert q.numel() > 2 ** 31
    scale = 1.0 / math.sqrt(D)
    o, lse = fa2.fa2_fwd(q, k, v, scale=scale)
    dq, dk, dv = fa2.fa2_bwd(q, k, v, o, lse, do, scale=scale)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 0
    yield dict(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv, scale=scale)


def rows_of_head(h):
    """Row indices i of head h to check."""
    rows = {0, 1, 127, 128, M - 1, M - 2, M - 77, M - 78}
    for elems in (1 << 30, 1 << 31):  # flat element offsets (h*M + i)*D
        flat = elems // D - h * M
        rows.update(i for i in range(flat - 3, flat + 3) if 0 <= i < M)
    rng = np.random.default_rng(7 + h)
    rows.update(rng.integers(0, M, size=128).tolist())
    return np.array(sorted(rows), np.int64)


def bits(t):
    """Device bf16 tensor -> host uint16 bf16 bits (the oracle's input type)."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def test_forward_rows_past_2_31_elements(problem):
    P = problem
    for h in range(H):
        rows = rows_of_head(h)
        idx = torch.from_numpy(rows).to(DEV)
        q_s = bits(P["q"][0, h].index_select(0, idx))[None, None]
        k_h, v_h = bits(P["k"][:, h:h + 1]), bits(P["v"][:, h:h + 1])
        o_ref, l_ref = oracle.attn_fwd(q_s, k_h, v_h, float(np.float32(P["scale"])), False)
        o_got = to_host_f64(P["o"][0, h].index_select(0, idx))
        l_got = P["lse"][0, h].index_select(0, idx).cpu().numpy().astype(np.float64)
        eo, el, excess = compare(o_got, l_got, o_ref[0, 0], l_ref[0, 0], si.BF16)
        assert excess <= 0 and el <= TOL[si.BF16], (h, eo, el)


def test_backward_past_2_31_elements(problem):
    P = problem
    scale = float(np.float32(P["scale"]))
    for h in range(H):
        rows = rows_of_head(h)
        idx = torch.from_numpy(rows).to(DEV)
        q_s = bits(P["q"][0, h].index_select(0, idx))[None, None]
        do_s = bits(P["do"][0, h].index_select(0, idx))[None, None]
        k_h, v_h = bits(P["k"][:, h:h + 1]), bits(P["v"][:, h:h + 1])
        dq_ref, dk_ref, dv_ref = oracle.attn_bwd(q_s, k_h, v_h, do_s, scale, False)
        got = (to_host_f64(P["dq"][0, h].index_select(0, idx)), to_host_f64(P["dk"][0, h]),
               to_host_f64(P["dv"][0, h]))
        for name, g, w in zip(("dQ", "dK", "dV"), got, (dq_ref[0, 0], dk_ref[0, 0], dv_ref[0, 0])):
            err = float(np.max(np.abs(g - w)))
            assert err <= REL_TOL * float(np.max(np.abs(w))) + 1e-5, (h, name, err)
        # rows without dO: dQ is exactly zero, including past the 2^31-element offset
        others = torch.tensor([2, 129, M // 2, M - 3, M - 79], device=DEV)
        others = others[~torch.isin(others, idx)]
        assert torch.count_nonzero(P["dq"][0, h].index_select(0, others)) == 0
