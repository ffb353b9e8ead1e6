"""FlashAttention-2 forward pass on GB300 (sm_103a).

Thin Python binding of the C ABI in ``include/fa2.h`` (library
``libfa2_gb300.so``, built in-tree by ``_build.build()``).  This module only
marshals arguments: every step of the forward pass runs in the library's CUDA
kernels.  There is no fallback: if the library is missing, every call raises.

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

FA2_BF16 = 0
FA2_FP32 = 1

FA2_OK = 0
FA2_ERR_NULL = -1
FA2_ERR_SHAPE = -2
FA2_ERR_HEADDIM = -3
FA2_ERR_DTYPE = -4
FA2_ERR_ALIGN = -5
FA2_ERR_SCALE = -6
FA2_ERR_TOO_LARGE = -7
FA2_ERR_ARCH = -8
FA2_ERR_CUDA = -9
FA2_ERR_DEVICE_TIMEOUT = -10
FA2_ERR_WORKSPACE = -11
FA2_ERR_MODIFIER = -12

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa2_gb300.so")

# Every symbol include/fa2.h declares, with its ctypes signature.
_VP, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "fa2_fwd": ([_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _I, _I, _VP], _I),
    "fa2_fwd_gqa": ([_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _I, _I, _VP], _I),
    "fa2_fwd_splitkv": ([_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _VP, _SZ,
                         _VP], _I),
    "fa2_fwd_splitkv_noalloc": ([_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I,
                                 _VP], _I),
    "fa2_fwd_ext": ([_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _F, _VP, _I, _I,
                     _I, _VP, _SZ, _VP], _I),
    "fa2_bwd": ([_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _I, _I, _VP, _SZ,
                 _VP], _I),
    "fa2_bwd_deterministic": ([_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _I, _I,
                               _VP, _SZ, _VP], _I),
    "fa2_bwd_workspace_bytes": ([_I, _I, _I], _SZ),
    "fa2_bwd_host": ([_VP] * 18 + [_I, _I, _I, _I, _I, _I, _F, _I, _I, _VP, _SZ, _I, _VP], _I),
    "fa2_fwd_host": ([_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _I, _I,
                      _I, _VP], _I),
    "fa2_splitkv_num_splits": ([_I, _I, _I, _I, _I, _I, _I], _I),
    "fa2_splitkv_workspace_bytes": ([_I, _I, _I, _I, _I], _SZ),
    "fa2_selftest_wait_timeout": ([_I, _VP], _I),
    "fa2_strerror": ([_I], ctypes.c_char_p),
    "fa2_device_status": ([_I, ctypes.POINTER(_I)], _I),
    "fa2_probe_ex2": ([_VP, _I, _I, _VP], _I),
    "fa2_version": ([], _I),
}

_lock = threading.Lock()
_lib = None


class Fa2Error(RuntimeError):
    """A nonzero status returned by the library."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {fa2_strerror(code)} ({code})")


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build()")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = args
                fn.restype = res
            _lib = handle
    return _lib


def fa2_strerror(code: int) -> str:
    return lib().fa2_strerror(int(code)).decode()


def fa2_version() -> int:
    return lib().fa2_version()


def fa2_device_status(reset: bool = True) -> int:
    """Raw device status word (0 = no pipeline wait ran out); clears it if ``reset``."""
    raw = ctypes.c_int(0)
    rc = lib().fa2_device_status(1 if reset else 0, ctypes.byref(raw))
    if rc not in (FA2_OK, FA2_ERR_DEVICE_TIMEOUT):
        raise Fa2Error(rc, "fa2_device_status")
    return raw.value


def fa2_selftest_wait_timeout(limit_ms: int = 20, stream=None) -> None:
    """Run the failure-path self-test (C ABI ``fa2_selftest_wait_timeout``): a
    bounded wait that runs out after ``limit_ms`` and sets the device status word
    to 99.  Read and clear it with fa2_device_status()."""
    import torch
    handle = _stream_handle(torch.empty(0, device="cuda"), stream)
    rc = lib().fa2_selftest_wait_timeout(int(limit_ms), handle)
    if rc != FA2_OK:
        raise Fa2Error(rc, "fa2_selftest_wait_timeout")


def fa2_probe_ex2(blocks: int | None = None, iters: int = 4096, reps: int = 5, stream=None) -> float:
    """Exponentials per second of the special-function pipe's ex2 on the current
    device (C ABI ``fa2_probe_ex2``): the median over ``reps`` launches of
    ``blocks`` CTAs (default 8 per SM, full occupancy), each timed with CUDA
    events on ``stream``.  A measurement aid for the softmax's ceiling."""
    import torch
    dev = torch.cuda.current_device()
    if blocks is None:
        blocks = 8 * torch.cuda.get_device_properties(dev).multi_processor_count
    out = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    handle = _stream_handle(out, stream)
    s = torch.cuda.current_stream(dev) if stream is None else stream
    times = []
    for i in range(reps + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        rc = lib().fa2_probe_ex2(out.data_ptr(), int(blocks), int(iters), handle)
        if rc != FA2_OK:
            raise Fa2Error(rc, "fa2_probe_ex2")
        e1.record(s)
        e1.synchronize()
        if i > 0:  # the first launch is a warm-up
            times.append(e0.elapsed_time(e1) / 1e3)
    times.sort()
    return blocks * 256 * 8 * iters / times[len(times) // 2]


def _check_qkv(q, k, v):
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape or q.shape[0] != k.shape[0] \
            or q.shape[3] != k.shape[3] or k.shape[1] == 0 or q.shape[1] % k.shape[1] != 0:
        raise ValueError("expected q [B,H,M,D] and k, v [B,H_kv,N,D] with H_kv dividing H")
    if q.dtype == torch.bfloat16:
        dtype = FA2_BF16
    elif q.dtype == torch.float32:
        dtype = FA2_FP32
    else:
        raise TypeError(f"unsupported dtype {q.dtype}")
    for t in (q, k, v):
        if t.dtype != q.dtype or t.device != q.device or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("q, k, v must be contiguous CUDA tensors of one dtype and device")
    return dtype


def _outputs(q, o, lse):
    import torch
    B, H, M, _ = q.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, M), dtype=torch.float32, device=q.device)
    if o.shape != q.shape or o.dtype != q.dtype or not o.is_contiguous() or o.device != q.device:
        raise ValueError("o must be a contiguous tensor like q")
    if lse.shape != (B, H, M) or lse.dtype != torch.float32 or not lse.is_contiguous() \
            or lse.device != q.device:
        raise ValueError("lse must be a contiguous fp32 tensor of shape [B,H,M]")
    return o, lse


def _stream_handle(q, stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def fa2_splitkv_num_splits(B: int, H: int, H_kv: int, M: int, N: int, D: int, dtype: int) -> int:
    """Split count chosen by the library for the current device."""
    rc = lib().fa2_splitkv_num_splits(B, H, H_kv, M, N, D, dtype)
    if rc < 0:
        raise Fa2Error(rc, "fa2_splitkv_num_splits")
    return rc


def fa2_splitkv_workspace_bytes(B: int, H: int, M: int, D: int, num_splits: int) -> int:
    return lib().fa2_splitkv_workspace_bytes(B, H, M, D, num_splits)


def fa2_fwd_splitkv(q, k, v, o=None, lse=None, scale: float | None = None, causal: bool = False,
                    num_splits: int = 0, workspace=None, stream=None):
    """Split-KV forward (same result as fa2_fwd): the key range is cut into
    ``num_splits`` slices (0 = the library's choice) whose partial results are
    merged by a combine kernel.  ``workspace`` (a CUDA uint8 tensor) is allocated
    with torch when not given."""
    import torch

    dtype = _check_qkv(q, k, v)
    B, H, M, D = q.shape
    H_kv, N = k.shape[1], k.shape[2]
    o, lse = _outputs(q, o, lse)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        if num_splits <= 0:
            num_splits = fa2_splitkv_num_splits(B, H, H_kv, M, N, D, dtype)
        need = fa2_splitkv_workspace_bytes(B, H, M, D, num_splits)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
        rc = lib().fa2_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, H_kv, M, N, D, float(scale),
                                   1 if causal else 0, dtype, num_splits, ws_ptr, ws_len,
                                   _stream_handle(q, stream))
    if rc != FA2_OK:
        raise Fa2Error(rc, "fa2_fwd_splitkv")
    return o, lse


def fa2_fwd_ext(q, k, v, o=None, lse=None, scale: float | None = None, causal: bool = False,
                window=(-1, -1), softcap: float = 0.0, alibi_slopes=None, num_splits: int = 1,
                workspace=None, stream=None):
    """Forward with score modifiers (C ABI ``fa2_fwd_ext``): ``window`` =
    (left, right) keys a row may see before / after its diagonal, negative =
    unbounded; ``softcap`` > 0 caps scores at softcap * tanh(s / softcap);
    ``alibi_slopes`` (fp32 CUDA tensor [H] or [B, H]) subtracts slope * |i - j|.
    ``num_splits`` as in fa2_fwd_splitkv (1 = no key split, 0 = the library's
    choice); the workspace is allocated with torch when needed and not given."""
    import torch

    dtype = _check_qkv(q, k, v)
    B, H, M, D = q.shape
    H_kv, N = k.shape[1], k.shape[2]
    o, lse = _outputs(q, o, lse)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    slopes_ptr, stride = None, 0
    if alibi_slopes is not None:
        if alibi_slopes.dtype != torch.float32 or not alibi_slopes.is_contiguous() \
                or alibi_slopes.device != q.device:
            raise ValueError("alibi_slopes must be a contiguous fp32 tensor on q's device")
        if tuple(alibi_slopes.shape) == (H,):
            stride = 0
        elif tuple(alibi_slopes.shape) == (B, H):
            stride = H
        else:
            raise ValueError("alibi_slopes must have shape [H] or [B, H]")
        slopes_ptr = alibi_slopes.data_ptr()
    wl, wr = (int(x) for x in window)
    with torch.cuda.device(q.device):
        if num_splits <= 0:
            num_splits = fa2_splitkv_num_splits(B, H, H_kv, M, N, D, dtype)
        need = fa2_splitkv_workspace_bytes(B, H, M, D, num_splits)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
        rc = lib().fa2_fwd_ext(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), B, H, H_kv, M, N, D, float(scale),
                               1 if causal else 0, wl, wr, float(softcap), slopes_ptr, stride,
                               dtype, num_splits, ws_ptr, ws_len, _stream_handle(q, stream))
    if rc != FA2_OK:
        raise Fa2Error(rc, "fa2_fwd_ext")
    return o, lse


def fa2_fwd_host(q_host, k_host, v_host, o_host=None, lse_host=None, q=None, k=None, v=None, o=None,
                 lse=None, scale: float | None = None, causal: bool = False, chunks: int = 0,
                 device=None, stream=None):
    """Forward for host tensors (C ABI ``fa2_fwd_host``): copies in, computes and
    copies out in slices of heads that overlap one another.  ``q_host`` etc. are
    CPU tensors (page-locked for overlap); the device buffers ``q, k, v, o, lse``
    are allocated on ``device`` (default: the current CUDA device) when not given.
    Returns (o_host, lse_host); they are valid once ``stream`` is synchronised."""
    import torch

    if q_host.is_cuda or k_host.is_cuda or v_host.is_cuda:
        raise ValueError("q_host, k_host, v_host must be host tensors")
    if q_host.dim() != 4 or k_host.dim() != 4 or v_host.shape != k_host.shape \
            or q_host.shape[0] != k_host.shape[0] or q_host.shape[3] != k_host.shape[3] \
            or q_host.shape[1] % k_host.shape[1] != 0:
        raise ValueError("expected q [B,H,M,D] and k, v [B,H_kv,N,D] with H_kv dividing H")
    if q_host.dtype not in (torch.bfloat16, torch.float32) or k_host.dtype != q_host.dtype \
            or v_host.dtype != q_host.dtype:
        raise TypeError("q, k, v must share one dtype, bf16 or fp32")
    for t in (q_host, k_host, v_host):
        if not t.is_contiguous():
            raise ValueError("host tensors must be contiguous")
    dtype = FA2_BF16 if q_host.dtype == torch.bfloat16 else FA2_FP32
    B, H, M, D = q_host.shape
    H_kv, N = k_host.shape[1], k_host.shape[2]
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if o_host is None:
        o_host = torch.empty(q_host.shape, dtype=q_host.dtype).pin_memory()
    if lse_host is None:
        lse_host = torch.empty((B, H, M), dtype=torch.float32).pin_memory()
    q = torch.empty(q_host.shape, dtype=q_host.dtype, device=dev) if q is None else q
    k = torch.empty(k_host.shape, dtype=k_host.dtype, device=dev) if k is None else k
    v = torch.empty(v_host.shape, dtype=v_host.dtype, device=dev) if v is None else v
    o = torch.empty(q_host.shape, dtype=q_host.dtype, device=dev) if o is None else o
    lse = torch.empty((B, H, M), dtype=torch.float32, device=dev) if lse is None else lse
    for t, like in ((q, q_host), (k, k_host), (v, v_host), (o, q_host), (o_host, q_host)):
        if t.shape != like.shape or t.dtype != like.dtype or not t.is_contiguous():
            raise ValueError("buffers must match the shapes and dtype of q_host / k_host")
    if lse.shape != (B, H, M) or lse_host.shape != (B, H, M) or lse.dtype != torch.float32 \
            or lse_host.dtype != torch.float32:
        raise ValueError("lse buffers must be fp32 [B,H,M]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        rc = lib().fa2_fwd_host(q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(), o_host.data_ptr(),
                                lse_host.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr(), B, H, H_kv, M, N, D, float(scale), 1 if causal else 0, dtype,
                                int(chunks), _stream_handle(q, stream))
    if rc != FA2_OK:
        raise Fa2Error(rc, "fa2_fwd_host")
    return o_host, lse_host


def fa2_fwd(q, k, v, o=None, lse=None, scale: float | None = None, causal: bool = False,
            stream=None):
    """FlashAttention-2 forward on torch CUDA tensors.

    q [B,H,M,D], k and v [B,H_kv,N,D] (bf16 or fp32, contiguous, same
    device); H_kv == H is multi-head attention, a divisor of H grouped-query
    attention (``fa2_fwd_gqa`` in the C ABI).  o [B,H,M,D] and lse [B,H,M] fp32
    are allocated when not given.  ``scale`` defaults to 1/sqrt(D).  Launches on
    ``stream`` (default: torch's current stream) and returns (o, lse) without
    synchronising.
    """
    import torch

    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape or q.shape[0] != k.shape[0] \
            or q.shape[3] != k.shape[3] or k.shape[1] == 0 or q.shape[1] % k.shape[1] != 0:
        raise ValueError("expected q [B,H,M,D] and k, v [B,H_kv,N,D] with H_kv dividing H")
    B, H, M, D = q.shape
    H_kv = k.shape[1]
    N = k.shape[2]
    if q.dtype == torch.bfloat16:
        dtype = FA2_BF16
    elif q.dtype == torch.float32:
        dtype = FA2_FP32
    else:
        raise TypeError(f"unsupported dtype {q.dtype}")
    for t in (q, k, v):
        if t.dtype != q.dtype or t.device != q.device or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("q, k, v must be contiguous CUDA tensors of one dtype and device")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, M), dtype=torch.float32, device=q.device)
    if o.shape != q.shape or o.dtype != q.dtype or not o.is_contiguous() or o.device != q.device:
        raise ValueError("o must be a contiguous tensor like q")
    if lse.shape != (B, H, M) or lse.dtype != torch.float32 or not lse.is_contiguous() \
            or lse.device != q.device:
        raise ValueError("lse must be a contiguous fp32 tensor of shape [B,H,M]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    with torch.cuda.device(q.device):
        if H_kv == H:
            rc = lib().fa2_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), B, H, M, N, D, float(scale), 1 if causal else 0,
                               dtype, handle)
        else:
            rc = lib().fa2_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, H_kv, M, N, D, float(scale),
                                   1 if causal else 0, dtype, handle)
    if rc != FA2_OK:
        raise Fa2Error(rc, "fa2_fwd")
    return o, lse


def fa2_bwd(q, k, v, o, lse, dout, dq=None, dk=None, dv=None, scale: float | None = None,
            causal: bool = False, workspace=None, stream=None, deterministic: bool = False):
    """Backward pass (C ABI ``fa2_bwd``, or ``fa2_bwd_deterministic`` when
    ``deterministic``): gradients (dq, dk, dv) for upstream gradient ``dout``,
    from the forward's inputs and its outputs ``o`` and ``lse``.  bf16 CUDA
    tensors; dq like q, dk and dv like k.  The workspace is allocated with torch
    when not given.  Returns (dq, dk, dv) without synchronising."""
    import torch

    dtype = _check_qkv(q, k, v)
    B, H, M, D = q.shape
    H_kv, N = k.shape[1], k.shape[2]
    for t in (o, dout):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous() or t.device != q.device:
            raise ValueError("o and dout must be contiguous tensors like q")
    if lse.shape != (B, H, M) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor of shape [B,H,M]")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, like in ((dq, q), (dk, k), (dv, v)):
        if t.shape != like.shape or t.dtype != like.dtype or not t.is_contiguous() or t.device != q.device:
            raise ValueError("dq must be like q, dk and dv like k")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        need = lib().fa2_bwd_workspace_bytes(B, H, M)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        entry = lib().fa2_bwd_deterministic if deterministic else lib().fa2_bwd
        rc = entry(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                   dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, H_kv, M, N, D, float(scale),
                   1 if causal else 0, dtype, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                   _stream_handle(q, stream))
    if rc != FA2_OK:
        raise Fa2Error(rc, "fa2_bwd_deterministic" if deterministic else "fa2_bwd")
    return dq, dk, dv


def fa2_bwd_host(q_host, k_host, v_host, o_host, lse_host, dout_host, dq_host=None, dk_host=None,
                 dv_host=None, scale: float | None = None, causal: bool = False, chunks: int = 0,
                 device=None, workspace=None, buffers=None, stream=None):
    """Backward for host tensors (C ABI ``fa2_bwd_host``): copies q, k, v, o, lse
    and dout in, computes and copies dq, dk, dv out in slices of heads that overlap
    one another.  Host tensors (page-locked for overlap) of the ``fa2_bwd`` shapes;
    the device buffers (``buffers``: q, k, v, o, lse, dout, dq, dk, dv) and the
    workspace are allocated on ``device`` (default: the current CUDA device) when
    not given.  Returns (dq_host, dk_host, dv_host); they are valid once ``stream``
    is synchronised."""
    import torch

    host_in = (q_host, k_host, v_host, o_host, lse_host, dout_host)
    if any(t.is_cuda for t in host_in):
        raise ValueError("inputs must be host tensors")
    if q_host.dtype != torch.bfloat16 or any(t.dtype != torch.bfloat16 for t in (k_host, v_host, o_host, dout_host)):
        raise TypeError("q, k, v, o, dout must be bf16")
    if q_host.dim() != 4 or k_host.dim() != 4 or v_host.shape != k_host.shape \
            or q_host.shape[0] != k_host.shape[0] or q_host.shape[3] != k_host.shape[3] \
            or q_host.shape[1] % k_host.shape[1] != 0:
        raise ValueError("expected q [B,H,M,D] and k, v [B,H_kv,N,D] with H_kv dividing H")
    B, H, M, D = q_host.shape
    H_kv, N = k_host.shape[1], k_host.shape[2]
    if o_host.shape != q_host.shape or dout_host.shape != q_host.shape:
        raise ValueError("o and dout must be like q")
    if lse_host.shape != (B, H, M) or lse_host.dtype != torch.float32:
        raise ValueError("lse must be fp32 [B,H,M]")
    for t in host_in:
        if not t.is_contiguous():
            raise ValueError("host tensors must be contiguous")
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    dq_host = torch.empty(q_host.shape, dtype=torch.bfloat16).pin_memory() if dq_host is None else dq_host
    dk_host = torch.empty(k_host.shape, dtype=torch.bfloat16).pin_memory() if dk_host is None else dk_host
    dv_host = torch.empty(k_host.shape, dtype=torch.bfloat16).pin_memory() if dv_host is None else dv_host
    for t, like in ((dq_host, q_host), (dk_host, k_host), (dv_host, k_host)):
        if t.shape != like.shape or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.is_cuda:
            raise ValueError("dq_host must be like q_host, dk_host and dv_host like k_host")
    if buffers is None:
        dbuf = [torch.empty(t.shape, dtype=t.dtype, device=dev) for t in host_in]
        dq, dk, dv = (torch.empty(t.shape, dtype=torch.bfloat16, device=dev) for t in (q_host, k_host, k_host))
    else:
        if len(buffers) != 9:
            raise ValueError("buffers: q, k, v, o, lse, dout, dq, dk, dv")
        dbuf, (dq, dk, dv) = list(buffers[:6]), buffers[6:]
        for t, like in zip(list(buffers), list(host_in) + [q_host, k_host, k_host]):
            if not t.is_cuda or t.shape != like.shape or t.dtype != like.dtype or not t.is_contiguous():
                raise ValueError("device buffers must be contiguous CUDA tensors like the host ones")
        dev = dbuf[0].device
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(dev):
        need = lib().fa2_bwd_workspace_bytes(B, H, M)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        rc = lib().fa2_bwd_host(*(t.data_ptr() for t in host_in), dq_host.data_ptr(), dk_host.data_ptr(),
                                dv_host.data_ptr(), *(t.data_ptr() for t in dbuf), dq.data_ptr(), dk.data_ptr(),
                                dv.data_ptr(), B, H, H_kv, M, N, D, float(scale), 1 if causal else 0, FA2_BF16,
                                workspace.data_ptr(), workspace.numel() * workspace.element_size(), int(chunks),
                                _stream_handle(dbuf[0], stream))
    if rc != FA2_OK:
        raise Fa2Error(rc, "fa2_bwd_host")
    return dq_host, dk_host, dv_host


# The grouped-query entry has the same Python signature: k and v carry H_kv heads.
fa2_fwd_gqa = fa2_fwd
