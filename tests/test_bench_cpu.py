"""CPU checks of the bench's work and byte counts and of its profile lookup.

The FLOP count is the pages' metric ("FlashAttention-2 from PyTorch to Triton",
the bench harness: 4*B*H*M*N*D, halved for causal); the algorithmic HBM bytes
read every input and write every output once.  The expected values are worked
out by hand in the comments, not by the functions under test.
"""
import bench
import seeded_inputs as si

HEADLINE = si.WORKLOADS["bf16_2x16x8192x8192x128_causal"]


def test_headline_flops_are_the_pages_metric():
    # 4 * 2 * 16 * 8192 * 8192 * 128 / 2 = 549755813888
    assert HEADLINE.flops == 549755813888
    full = si.WORKLOADS["bf16_2x16x8192x8192x128"]
    assert full.flops == 2 * 549755813888


def test_forward_bytes():
    # Q and O: 32 heads x 2 x 8192 x 128 x 2 B = 134217728, L: 32 x 8192 x 4 B = 1048576,
    # K and V: 32 heads x 2 x 8192 x 128 x 2 B = 134217728
    assert HEADLINE.io_bytes() == 134217728 + 1048576 + 134217728


def test_backward_bytes():
    # Q, O, dO, dQ: 32 x 4 x 8192 x 128 x 2 B = 268435456, L: 1048576,
    # K, V, dK, dV: 32 x 4 x 8192 x 128 x 2 B = 268435456
    assert bench.bwd_io_bytes(HEADLINE) == 268435456 + 1048576 + 268435456
    gqa = si.WORKLOADS["bf16_2x32x8192x8192x128_gqa8_causal"]
    # B = 2, H = 32, H_kv = 8: 64 query heads x (4 x 8192 x 128 x 2 + 8192 x 4) =
    # 538968064; 16 key/value heads x 4 x 8192 x 128 x 2 = 134217728
    assert bench.bwd_io_bytes(gqa) == 538968064 + 134217728


def test_traffic_is_dropped_once_the_sources_change(monkeypatch):
    """A profile summary counts only while its recorded source hash matches."""
    monkeypatch.setattr(bench, "kernel_source_hash", lambda pass_="fwd": "0" * 16)
    assert bench.dram_traffic_per_launch(HEADLINE.name, "fwd") is None
    assert bench.dram_traffic_per_launch(HEADLINE.name, "bwd") is None


def test_split_kv_profiles_depend_on_the_combine_source():
    """Workloads measured through the split-KV entry also run the combine kernel,
    so their profile summaries are keyed to a source list that includes it."""
    assert bench.source_key("bf16_1x32x128x32768x128_gqa8_splitkv", "fwd") == "splitkv"
    assert bench.source_key("bf16_16x32x1x8192x128_gqa8_decode", "fwd") == "splitkv"
    assert bench.source_key(HEADLINE.name, "fwd") == "fwd"
    assert bench.source_key(HEADLINE.name, "bwd") == "bwd"
    assert set(bench.PASS_SOURCES["fwd"]) < set(bench.PASS_SOURCES["splitkv"])
    assert "fa2_combine.cu" in bench.PASS_SOURCES["splitkv"]
