"""Measurement aids on the GPU: the ex2 throughput probe (C ABI fa2_probe_ex2)
returns a rate the special-function pipe can deliver, and its chains stay
finite (the values it writes are read back)."""
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fa2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_forward_fa2_gb300 as m
    m.lib()
    return m


def test_ex2_probe_rate_is_plausible(fa2):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rate = fa2.fa2_probe_ex2(iters=2048)
    # 8 to 64 exponentials per clock per SM, at a clock between 0.5 and 3 GHz
    assert 8 * sms * 0.5e9 < rate < 64 * sms * 3.0e9


def test_ex2_probe_values_stay_finite(fa2):
    out = torch.full((4 * 256,), float("nan"), dtype=torch.float32, device="cuda")
    rc = fa2.lib().fa2_probe_ex2(out.data_ptr(), 4, 1000, None)
    assert rc == fa2.FA2_OK
    torch.cuda.synchronize()
    # each chain settles in (-0.75, -0.25); a thread writes the sum of its 8 chains
    assert torch.isfinite(out).all()
    assert (out > -6.0).all() and (out < -2.0).all()
