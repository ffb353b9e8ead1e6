"""The C-ABI library without a GPU: it loads, exports every symbol that
include/fa2.h declares, and rejects bad arguments before any CUDA work.
No compute call is made here."""
import ctypes
import os
import re

import pytest

import exact_attention_forward_fa2_gb300 as fa2

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fa2.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa2_\w+)\s*\(", text, flags=re.M)))


def declared_codes():
    return {m.group(1): int(m.group(2)) for m in
            re.finditer(r"#define\s+(FA2_\w+)\s+\(?(-?\d+)\)?", open(HEADER).read())}


@pytest.fixture(scope="module")
def lib():
    from exact_attention_forward_fa2_gb300 import _build
    _build.build()
    return fa2.lib()


def test_header_declares_the_api():
    assert declared_functions() == ["fa2_bwd", "fa2_bwd_deterministic", "fa2_bwd_host", "fa2_bwd_workspace_bytes",
                                    "fa2_device_status", "fa2_fwd",
                                    "fa2_fwd_ext", "fa2_fwd_gqa", "fa2_fwd_host", "fa2_fwd_splitkv",
                                    "fa2_fwd_splitkv_noalloc", "fa2_probe_ex2", "fa2_selftest_wait_timeout",
                                    "fa2_splitkv_num_splits", "fa2_splitkv_workspace_bytes", "fa2_strerror",
                                    "fa2_version"]


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in fa2.SIGNATURES


def test_binding_constants_match_header():
    for name, value in declared_codes().items():
        assert getattr(fa2, name) == value, name


def test_strerror_names_every_code(lib):
    codes = declared_codes()
    msgs = set()
    for name, value in codes.items():
        if name in ("FA2_BF16", "FA2_FP32"):
            continue
        msg = fa2.fa2_strerror(value)
        assert msg and msg != "unknown status", name
        msgs.add(msg)
    assert fa2.fa2_strerror(12345) == "unknown status"
    assert fa2.fa2_version() >= 100


# Fake, 16-byte aligned addresses: validation must fail before anything touches them.
P = 0x10000


def call(lib, q=P, k=P, v=P, o=P, lse=P, B=1, H=1, M=8, N=8, D=64, scale=0.125, causal=0, dtype=0):
    return lib.fa2_fwd(q, k, v, o, lse, B, H, M, N, D, scale, causal, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa2.FA2_ERR_NULL), (dict(k=None), fa2.FA2_ERR_NULL), (dict(v=None), fa2.FA2_ERR_NULL),
    (dict(o=None), fa2.FA2_ERR_NULL), (dict(lse=None), fa2.FA2_ERR_NULL),
    (dict(B=0), fa2.FA2_ERR_SHAPE), (dict(H=-1), fa2.FA2_ERR_SHAPE), (dict(M=0), fa2.FA2_ERR_SHAPE),
    (dict(N=0), fa2.FA2_ERR_SHAPE),
    (dict(D=32), fa2.FA2_ERR_HEADDIM), (dict(D=96), fa2.FA2_ERR_HEADDIM), (dict(D=256), fa2.FA2_ERR_HEADDIM),
    (dict(dtype=2), fa2.FA2_ERR_DTYPE), (dict(dtype=-1), fa2.FA2_ERR_DTYPE),
    (dict(scale=0.0), fa2.FA2_ERR_SCALE), (dict(scale=-1.0), fa2.FA2_ERR_SCALE),
    (dict(scale=float("inf")), fa2.FA2_ERR_SCALE), (dict(scale=float("nan")), fa2.FA2_ERR_SCALE),
    (dict(q=P + 8), fa2.FA2_ERR_ALIGN), (dict(o=P + 2), fa2.FA2_ERR_ALIGN), (dict(lse=P + 2), fa2.FA2_ERR_ALIGN),
    (dict(B=65536, H=65536), fa2.FA2_ERR_TOO_LARGE),
])
def test_rejects_bad_arguments(lib, kw, code):
    assert call(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa2.FA2_ERR_NULL), (dict(lse=None), fa2.FA2_ERR_NULL), (dict(B=0), fa2.FA2_ERR_SHAPE),
    (dict(D=96), fa2.FA2_ERR_HEADDIM), (dict(dtype=2), fa2.FA2_ERR_DTYPE), (dict(scale=0.0), fa2.FA2_ERR_SCALE),
    (dict(o=P + 2), fa2.FA2_ERR_ALIGN),
])
def test_noalloc_validates_before_any_cuda_call(lib, kw, code):
    """The allocation-free split-KV entry checks its arguments like fa2_fwd before
    it looks up its built-in buffer (a CUDA call): same codes, here without a GPU."""
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, M=8, N=8, D=64, scale=0.125, dtype=0)
    a.update(kw)
    assert lib.fa2_fwd_splitkv_noalloc(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], 2, 1, a["M"], a["N"],
                                       a["D"], a["scale"], 0, a["dtype"], 4, None) == code


def call_gqa(lib, H=8, H_kv=2, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, M=8, N=8, D=64, scale=0.125, causal=0, dtype=0)
    a.update(kw)
    return lib.fa2_fwd_gqa(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], H, H_kv, a["M"], a["N"],
                           a["D"], a["scale"], a["causal"], a["dtype"], None)


@pytest.mark.parametrize("H,H_kv", [(8, 0), (8, -1), (8, 3), (4, 8)])
def test_gqa_rejects_bad_head_grouping(lib, H, H_kv):
    assert call_gqa(lib, H=H, H_kv=H_kv) == fa2.FA2_ERR_SHAPE


def test_gqa_validates_like_fa2_fwd(lib):
    assert call_gqa(lib, q=None) == fa2.FA2_ERR_NULL
    assert call_gqa(lib, D=96) == fa2.FA2_ERR_HEADDIM
    assert call_gqa(lib, k=P + 4) == fa2.FA2_ERR_ALIGN


def test_splitkv_workspace_bytes(lib):
    B, H, M, D, S = 2, 3, 100, 128, 5
    o_bytes = S * B * H * M * D * 4
    want = ((o_bytes + 255) // 256) * 256 + S * B * H * M * 4
    assert lib.fa2_splitkv_workspace_bytes(B, H, M, D, S) == want
    assert lib.fa2_splitkv_workspace_bytes(B, H, M, D, 1) == 0
    assert lib.fa2_splitkv_workspace_bytes(B, H, M, 96, S) == 0


def call_split(lib, num_splits=4, ws=P, ws_bytes=1 << 30, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, H=8, H_kv=2, M=8, N=4096, D=64, scale=0.125, causal=0,
             dtype=0)
    a.update(kw)
    return lib.fa2_fwd_splitkv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["H_kv"],
                               a["M"], a["N"], a["D"], a["scale"], a["causal"], a["dtype"], num_splits,
                               ws, ws_bytes, None)


@pytest.mark.parametrize("kw", [dict(ws=None), dict(ws=P + 16), dict(ws_bytes=1024)])
def test_splitkv_rejects_bad_workspace(lib, kw):
    assert call_split(lib, **kw) == fa2.FA2_ERR_WORKSPACE


def test_splitkv_validates_like_fa2_fwd(lib):
    assert call_split(lib, q=None) == fa2.FA2_ERR_NULL
    assert call_split(lib, H_kv=3) == fa2.FA2_ERR_SHAPE
    assert call_split(lib, D=32) == fa2.FA2_ERR_HEADDIM


def call_ext(lib, window=(-1, -1), softcap=0.0, slopes=None, stride=0, num_splits=1, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=2, H=4, H_kv=2, M=8, N=300, D=64, scale=0.125, causal=0,
             dtype=0)
    a.update(kw)
    return lib.fa2_fwd_ext(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["H_kv"], a["M"],
                           a["N"], a["D"], a["scale"], a["causal"], window[0], window[1], softcap,
                           slopes, stride, a["dtype"], num_splits, None, 0, None)


@pytest.mark.parametrize("kw,code", [
    (dict(softcap=-1.0), fa2.FA2_ERR_MODIFIER), (dict(softcap=float("inf")), fa2.FA2_ERR_MODIFIER),
    (dict(softcap=float("nan")), fa2.FA2_ERR_MODIFIER),
    (dict(slopes=P, stride=3), fa2.FA2_ERR_MODIFIER), (dict(slopes=P, stride=-4), fa2.FA2_ERR_MODIFIER),
    (dict(slopes=P + 2), fa2.FA2_ERR_ALIGN),
    (dict(window=(5, 5), M=(1 << 30) + 1), fa2.FA2_ERR_TOO_LARGE),
    (dict(window=(5, 5), q=None), fa2.FA2_ERR_NULL), (dict(softcap=30.0, D=96), fa2.FA2_ERR_HEADDIM),
    (dict(window=(5, 5), num_splits=4), fa2.FA2_ERR_WORKSPACE),
])
def test_ext_rejects_bad_arguments(lib, kw, code):
    assert call_ext(lib, **kw) == code


def call_bwd(lib, ws=P, ws_bytes=1 << 30, entry="fa2_bwd", **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, do=P, dq=P, dk=P, dv=P, B=2, H=4, H_kv=2, M=100, N=300, D=128,
             scale=0.125, causal=1, dtype=0)
    a.update(kw)
    return getattr(lib, entry)(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"],
                               a["B"], a["H"], a["H_kv"], a["M"], a["N"], a["D"], a["scale"], a["causal"],
                               a["dtype"], ws, ws_bytes, None)


def test_bwd_workspace_bytes(lib):
    # two fp32 vectors per padded query row, then the fp32 dQ accumulator (128 per row)
    assert lib.fa2_bwd_workspace_bytes(2, 3, 100) == 130 * 2 * 3 * 128 * 4
    assert lib.fa2_bwd_workspace_bytes(1, 1, 129) == 130 * 256 * 4
    assert lib.fa2_bwd_workspace_bytes(0, 1, 1) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(do=None), fa2.FA2_ERR_NULL), (dict(dv=None), fa2.FA2_ERR_NULL), (dict(lse=None), fa2.FA2_ERR_NULL),
    (dict(M=0), fa2.FA2_ERR_SHAPE), (dict(H_kv=3), fa2.FA2_ERR_SHAPE), (dict(D=96), fa2.FA2_ERR_HEADDIM),
    (dict(dtype=1), fa2.FA2_ERR_DTYPE), (dict(scale=0.0), fa2.FA2_ERR_SCALE),
    (dict(dq=P + 8), fa2.FA2_ERR_ALIGN), (dict(do=P + 4), fa2.FA2_ERR_ALIGN),
    (dict(ws=None), fa2.FA2_ERR_WORKSPACE), (dict(ws=P + 128), fa2.FA2_ERR_WORKSPACE),
    (dict(ws_bytes=1024), fa2.FA2_ERR_WORKSPACE), (dict(N=(1 << 30) + 1), fa2.FA2_ERR_TOO_LARGE),
])
@pytest.mark.parametrize("entry", ["fa2_bwd", "fa2_bwd_deterministic"])
def test_bwd_rejects_bad_arguments(lib, kw, code, entry):
    assert call_bwd(lib, entry=entry, **kw) == code


def call_host(lib, **kw):
    a = dict(qh=P, kh=P, vh=P, oh=P, lh=P, q=P, k=P, v=P, o=P, lse=P, B=2, H=4, H_kv=2, M=64, N=64, D=64,
             scale=0.125, causal=0, dtype=0, chunks=0)
    a.update(kw)
    return lib.fa2_fwd_host(a["qh"], a["kh"], a["vh"], a["oh"], a["lh"], a["q"], a["k"], a["v"], a["o"],
                            a["lse"], a["B"], a["H"], a["H_kv"], a["M"], a["N"], a["D"], a["scale"],
                            a["causal"], a["dtype"], a["chunks"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(qh=None), fa2.FA2_ERR_NULL), (dict(lh=None), fa2.FA2_ERR_NULL), (dict(o=None), fa2.FA2_ERR_NULL),
    (dict(H_kv=3), fa2.FA2_ERR_SHAPE), (dict(D=32), fa2.FA2_ERR_HEADDIM), (dict(dtype=5), fa2.FA2_ERR_DTYPE),
    (dict(scale=-1.0), fa2.FA2_ERR_SCALE), (dict(v=P + 4), fa2.FA2_ERR_ALIGN),
])
def test_host_entry_rejects_bad_arguments(lib, kw, code):
    assert call_host(lib, **kw) == code


def call_bwd_host(lib, **kw):
    a = dict(h=P, q=P, B=2, H=4, H_kv=2, M=64, N=64, D=64, scale=0.125, causal=0, dtype=0, ws=P, ws_bytes=1 << 20,
             chunks=0, lh=P, dqh=P)
    a.update(kw)
    return lib.fa2_bwd_host(a["h"], a["h"], a["h"], a["h"], a["lh"], a["h"], a["dqh"], a["h"], a["h"],
                            a["q"], P, P, P, P, P, P, P, P, a["B"], a["H"], a["H_kv"], a["M"], a["N"], a["D"],
                            a["scale"], a["causal"], a["dtype"], a["ws"], a["ws_bytes"], a["chunks"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(h=None), fa2.FA2_ERR_NULL), (dict(lh=None), fa2.FA2_ERR_NULL), (dict(dqh=None), fa2.FA2_ERR_NULL),
    (dict(q=None), fa2.FA2_ERR_NULL), (dict(H_kv=3), fa2.FA2_ERR_SHAPE), (dict(D=32), fa2.FA2_ERR_HEADDIM),
    (dict(dtype=1), fa2.FA2_ERR_DTYPE), (dict(scale=-1.0), fa2.FA2_ERR_SCALE), (dict(q=P + 4), fa2.FA2_ERR_ALIGN),
    (dict(ws=None), fa2.FA2_ERR_WORKSPACE), (dict(ws_bytes=1024), fa2.FA2_ERR_WORKSPACE),
])
def test_bwd_host_entry_rejects_bad_arguments(lib, kw, code):
    assert call_bwd_host(lib, **kw) == code


@pytest.mark.parametrize("limit", [0, -5, 2001])
def test_selftest_rejects_limits_out_of_range(lib, limit):
    assert lib.fa2_selftest_wait_timeout(limit, None) == fa2.FA2_ERR_SHAPE


@pytest.mark.parametrize("out,blocks,iters,code", [
    (None, 8, 16, fa2.FA2_ERR_NULL),
    (256, 0, 16, fa2.FA2_ERR_SHAPE),
    (256, 65537, 16, fa2.FA2_ERR_SHAPE),
    (256, 8, 0, fa2.FA2_ERR_SHAPE),
    (256, 8, (1 << 20) + 1, fa2.FA2_ERR_SHAPE),
    (258, 8, 16, fa2.FA2_ERR_ALIGN),
])
def test_ex2_probe_rejects_bad_arguments(lib, out, blocks, iters, code):
    # checked before any CUDA call, so no device is needed
    assert lib.fa2_probe_ex2(out, blocks, iters, None) == code


def test_no_gpu_means_an_error_not_a_fallback(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call(lib) in (fa2.FA2_ERR_CUDA, fa2.FA2_ERR_ARCH)
