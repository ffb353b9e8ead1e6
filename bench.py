"""Bench: FlashAttention-2 forward TFLOP/s on GB300 and its fraction of the
dense bf16 tensor-core peak.

One step = one fa2_fwd call (the whole forward: every row of the hot path) over
the workload below, inputs resident in HBM.  Prints ONE JSON line.

Workload: bf16, B=2, H=16, M=N=8192, D=128, causal, scale 1/sqrt(128) (the
configuration the >= 50%-of-peak target is stated on); FLOP = 4*B*H*M*N*D / 2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--pass fwd|bwd]

--pass bwd times the backward (fa2_bwd: dQ, dK, dV from dO, with the forward's O
and L resident) on the same workload; its FLOP count is the usual 2.5x the
forward's (five GEMMs of 2*M*N*D per head against the forward's two).  At head
dim 128 fa2_bwd forms dQ by fp32 reductions (not bitwise reproducible);
fa2_bwd_deterministic is the two-pass alternative.

--impl reference times the fp64 CPU oracle on the host cores (a bounded sample
of the same workload per step): the method has no runnable reference
implementation, so the oracle is the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import seeded_inputs as si  # noqa: E402

WORKLOAD = "bf16_2x16x8192x8192x128_causal"
METRIC = "FA2 fwd TFLOP/s (4BHMND, 1/2 causal) and % of GB300 dense tensor peak"
METRIC_BWD = "FA2 bwd TFLOP/s (10BHMND, 1/2 causal) and % of GB300 dense tensor peak"
BWD_FLOPS_OVER_FWD = 2.5
REFERENCE_BUDGET_S = 120.0  # CPU seconds of oracle work for a whole --impl reference run
UNIT = "TFLOP/s"
KERNEL = "fa2_fwd_kernel"
def profile_summary(workload: str, pass_: str = "fwd") -> str:
    name = f"fa2_fwd_kernel_{workload}.md" if pass_ == "fwd" else f"fa2_bwd_{workload}.md"
    return os.path.join(ROOT, "profiles", name)
L2_FLUSH_BYTES = 256 << 20
# Timing protocol of the measurement plan: median of PROTOCOL_REPS event-timed
# launches after PROTOCOL_WARMUP warm-ups (L2 flushed between launches).
PROTOCOL_WARMUP = 25
PROTOCOL_REPS = 100
# The pages' own numbers for this shape, as context: "FlashAttention-2" (the
# drew-chen README), Results table, on an RTX 4080 in fp32 (CUDA cores; 5
# warm-ups, 10 reps), B=4, H=12, M=N=2048, D=64, non-causal.
PAGES_CONTEXT_WORKLOAD = "tf32_4x12x2048x2048x64"
PAGES_CONTEXT = {
    "pages_shape": "fp32, B=4, H=12, M=N=2048, D=64, non-causal",
    "hardware": "RTX 4080, fp32",
    "source": "\"FlashAttention-2\" (drew-chen README), Results",
    "v4_best_cuda_kernel_us": 3810.30,
    "pytorch_sdpa_us": 5507.07,
}
TF32_OVER_BF16 = 1.1 / 2.25  # nominal dense tensor rates per GPU


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bf16_tflops"), d.get("hbm_gbs"), "measured"
    return 1900.0, 6800.0, "fallback"


def peak_sustained():
    """The bf16 sustained peak (seconds-long cuBLAS loop) from MEASURED_PEAKS.json,
    or None."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f).get("bf16_tflops_sustained")
    return None


# Sources each timed pass is built from: a profile summary stays valid while these are unchanged.
PASS_SOURCES = {
    "fwd": ("fa2_fwd_kernel.cuh", "fa2_launch.cuh", "fa2_config.h", "sm103_ptx.cuh",
            "fa2_fwd_bf16_d64.cu", "fa2_fwd_bf16_d128.cu", "fa2_fwd_fp32_d64.cu", "fa2_fwd_fp32_d128.cu"),
    "bwd": ("fa2_bwd_kernel.cuh", "fa2_bwd.cu", "fa2_fwd_kernel.cuh", "sm103_ptx.cuh"),
}
# workloads measured through the split-KV entry also run the combine kernel
PASS_SOURCES["splitkv"] = PASS_SOURCES["fwd"] + ("fa2_combine.cu",)


def source_key(workload: str, pass_: str) -> str:
    """Which source list a profile summary of ``workload`` depends on."""
    w = si.WORKLOADS.get(workload)
    return "splitkv" if pass_ == "fwd" and w is not None and w.split_kv else pass_


def bwd_io_bytes(w) -> int:
    """Algorithmic HBM bytes of one backward step: read Q, K, V, O, dO and the
    fp32 L once, write dQ, dK and dV once."""
    e = 2 if w.dtype == si.BF16 else 4
    per_q_head = 4 * w.M * w.D * e + 4 * w.M      # Q, O, dO, dQ and L
    per_kv_head = 4 * w.N * w.D * e               # K, V, dK, dV
    return w.B * w.H * per_q_head + w.B * w.Hkv * per_kv_head


def kernel_source_hash(pass_: str = "fwd") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_forward_fa2_gb300", "csrc")
    for name in sorted(PASS_SOURCES[pass_]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def dram_traffic_per_launch(workload: str = WORKLOAD, pass_: str = "fwd"):
    """DRAM bytes per launch (per step, for the backward's kernels together) from
    the committed ncu summary of ``workload``, if it was taken on the current
    kernel source (its recorded source hash matches)."""
    path = profile_summary(workload, pass_)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash(source_key(workload, pass_)):
        return None
    return float(m_bytes.group(1))


class ClockSampler:
    """Samples the GPU's SM clock, power and clock-event (throttle) reasons
    through NVML every 2 ms on a background thread while the timed region runs
    (NVML is called through ctypes; nvidia-smi's 200 ms period is longer than
    the whole timed region)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, log_path: str | None = None):
        self.index = device_index
        self.log_path = log_path
        self.samples = []
        self.nvml = None

    def _open(self):
        import ctypes
        try:
            nvml = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return None
        if nvml.nvmlInit_v2() != 0:
            return None
        handle = ctypes.c_void_p()
        ok = False
        try:
            import torch
            props = torch.cuda.get_device_properties(self.index)
            bus = getattr(props, "pci_bus_id", None)
            if bus is not None:
                pci = f"{getattr(props, 'pci_domain_id', 0):08X}:{bus:02X}:{getattr(props, 'pci_device_id', 0):02X}.0"
                ok = nvml.nvmlDeviceGetHandleByPciBusId_v2(pci.encode(), ctypes.byref(handle)) == 0
        except Exception:
            ok = False
        if not ok and nvml.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(handle)) != 0:
            return None
        self.handle = handle
        self.reason_fn = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint(0)
        nvml.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx))
        self.max_mhz = float(mx.value)
        return nvml

    def _run(self):
        import ctypes
        mhz, reasons, mw = ctypes.c_uint(0), ctypes.c_ulonglong(0), ctypes.c_uint(0)
        while not self._stop.is_set():
            self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz))
            self.reason_fn(self.handle, ctypes.byref(reasons))
            self.nvml.nvmlDeviceGetPowerUsage(self.handle, ctypes.byref(mw))
            self.samples.append((time.perf_counter(), float(mhz.value), int(reasons.value), mw.value / 1e3))
            time.sleep(0.002)

    def __enter__(self):
        import threading
        self.nvml = self._open()
        if self.nvml is not None:
            self._stop = threading.Event()
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        if self.nvml is not None:
            self._stop.set()
            self._thread.join()
            # one more sample after the region, so even a region shorter than the
            # period has its closing sample
            if self.log_path:
                with open(self.log_path, "w") as f:
                    f.write("t_s,sm_mhz,reasons_mask,power_w\n")
                    for t, m, r, w in self.samples:
                        f.write(f"{t:.6f},{m:.0f},{r:#x},{w:.1f}\n")

    def summary(self):
        if not self.samples:
            return None
        reasons = set()
        for _, _, mask, _ in self.samples:
            for bit, name in self.REASONS.items():
                if mask & bit:
                    reasons.add(name)
        return {"sm_mhz": float(np.median([m for _, m, _, _ in self.samples])),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "power_w_max": max(w for _, _, _, w in self.samples),
                "samples": len(self.samples), "source": "NVML, 2 ms period"}


def dist_setup(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle
def cpu_model() -> str:
    """Best-effort name of the host CPU (x86 lists a model name; Arm lists the
    implementer and part numbers)."""
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return platform.machine()
    for key in ("model name", "Model Name", "Hardware"):
        m = re.search(rf"^{key}\s*:\s*(.+)$", info, flags=re.M)
        if m:
            return m.group(1).strip()
    imp = re.search(r"^CPU implementer\s*:\s*(\S+)", info, flags=re.M)
    part = re.search(r"^CPU part\s*:\s*(\S+)", info, flags=re.M)
    if imp and part:
        return f"{platform.machine()} (CPU implementer {imp.group(1)}, part {part.group(1)})"
    return platform.machine()


def oracle_sample(w, q, k, v, seconds_target: float, seed: int = 0, n_start: int = 64):
    """Time the fp64 oracle on a bounded, seeded sample of the workload's rows,
    growing the sample from ``n_start`` rows until it takes ``seconds_target``.
    Returns (TFLOP/s, rows, seconds, cores)."""
    import oracle
    rng = np.random.default_rng(seed)
    total_rows = w.B * w.H * w.M

    def run(rows):
        if w.modified:
            oracle.attn_fwd_mod(q, k, v, w.scale, w.causal, w.window, w.softcap,
                                si.alibi_slopes(w.H).astype(np.float64) if w.alibi else None,
                                rows=rows)
        else:
            oracle.attn_fwd_gqa_rows(q, k, v, w.scale, w.causal, rows)

    rows = np.sort(rng.choice(total_rows, size=64, replace=False))
    run(rows[:8])  # warm (build, pages)
    n = max(8, min(total_rows, n_start))
    while True:
        rows = np.sort(rng.choice(total_rows, size=n, replace=False))
        t0 = time.perf_counter()
        run(rows)
        dt = time.perf_counter() - t0
        if dt >= seconds_target or n >= total_rows:
            break
        n = min(total_rows, int(n * max(2.0, 1.2 * seconds_target / max(dt, 1e-3))))
    flops = float(np.sum(4.0 * w.D * w.visible_keys(rows % w.M)))
    cores = oracle.omp_threads()
    return flops / dt / 1e12, int(n), dt, cores


def oracle_sample_bwd(w, q, k, v, seconds_target: float, seed: int = 0):
    """Time the fp64 oracle backward on whole heads of the workload (one key/value
    head with its query heads at a time, seeded order) until ~seconds_target.
    Returns (TFLOP/s, heads, seconds, cores)."""
    import oracle
    rng = np.random.default_rng(seed)
    group = w.H // w.Hkv
    units = rng.permutation(w.B * w.Hkv)
    flops_per_unit = BWD_FLOPS_OVER_FWD * w.flops / (w.B * w.Hkv)
    dt, n = 0.0, 0
    for u in units:
        b, hk = divmod(int(u), w.Hkv)
        sq = (slice(b, b + 1), slice(hk * group, (hk + 1) * group))
        skv = (slice(b, b + 1), slice(hk, hk + 1))
        do = si.normal(w.seed, 4, (1, group, w.M, w.D), 1.0, w.dtype)
        t0 = time.perf_counter()
        oracle.attn_bwd(q[sq], k[skv], v[skv], do, w.scale, w.causal)
        dt += time.perf_counter() - t0
        n += 1
        if dt >= seconds_target:
            break
    cores = oracle.omp_threads()
    return n * flops_per_unit / dt / 1e12, n * group, dt, cores


def cpu_extrapolation(w, flops, tflops, rows, seconds) -> dict:
    """The oracle's time for the whole workload, extrapolated from the sample's
    rate (labelled as such), with the host's core count beside the threads the
    oracle ran with."""
    aff = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    out = {"omp_threads": cores_of_oracle(), "host_cores": aff,
           "full_workload_s_extrapolated": flops / (tflops * 1e12) if tflops > 0 else None}
    if rows:
        out["ms_per_row"] = seconds / rows * 1e3
    return out


def cores_of_oracle() -> int:
    import oracle
    return oracle.omp_threads()


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = si.WORKLOADS[args.workload]
    q, k, v = si.make_qkv(w)
    bwd = args.pass_ == "bwd"
    # each step is a bounded sample, sized so that the whole run stays near
    # REFERENCE_BUDGET_S of CPU work (at most 2 s per step)
    per_step_s = max(0.05, min(2.0, REFERENCE_BUDGET_S / (args.warmup + args.steps)))
    per_step = []
    n_rows = 64
    for step in range(args.warmup + args.steps):
        if bwd:
            tf, n, dt, cores = oracle_sample_bwd(w, q, k, v, seconds_target=per_step_s, seed=step)
        else:  # start each step's sample at the size the previous step reached
            tf, n, dt, cores = oracle_sample(w, q, k, v, seconds_target=per_step_s, seed=step, n_start=n_rows)
            n_rows = n
        if step >= args.warmup:
            per_step.append((tf, n, dt))
    value = float(np.mean([p[0] for p in per_step]))
    ms = float(np.mean([p[2] for p in per_step])) * 1e3
    line = {
        "impl": "reference", "metric": METRIC_BWD if bwd else METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "pass": args.pass_, "B": w.B, "H": w.H, "H_kv": w.Hkv, "M": w.M,
                   "N": w.N, "D": w.D, "causal": w.causal},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "cpu": cpu_model(), "kind": "oracle",
                         "sample": (f"per step: {per_step[-1][1]} whole query heads of the workload "
                                    f"(fp64 backward), >= {per_step_s:.2f} s of CPU work" if bwd else
                                    f"per step: {per_step[-1][1]} seeded random query rows of the "
                                    f"workload (fp64, all their visible keys), ~{per_step_s:.2f} s of "
                                    f"CPU work")},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def measure_e2e(args, flops, step, stream, world, ins, outs, host_step=None):
    """Same metric end to end: each step copies the step's inputs from pinned host
    memory (``ins``: pairs of host array and its device tensor), runs the pass
    through the C ABI and copies the results (``outs``) back to pinned host
    memory, all inside the timed region.  ``host_step(host_ins, host_outs)``, when
    given, is one call of the library's host-buffer entry doing all three."""
    import torch

    def raw(t):
        return t.view(torch.int16) if t.dtype == torch.bfloat16 else t

    pairs = []
    for a, t in ins:
        h = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).pin_memory()
        pairs.append((h, raw(t)))
    houts = [(torch.empty(t.shape, dtype=raw(t).dtype).pin_memory(), raw(t)) for t in outs]

    def e2e_step():
        if host_step is not None:
            host_step([h for h, _ in pairs], [h for h, _ in houts])
            return
        for h, d in pairs:
            d.copy_(h, non_blocking=True)
        step()
        for h, d in houts:
            h.copy_(d, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    return {"value": flops * args.steps * world / t_e2e / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": int(sum(a.nbytes for a, _ in ins)),
            "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in outs)),
            "ms_per_step": t_e2e / args.steps * 1e3}


# ------------------------------------------------------------------ GPU path
def time_launches(step, flush, stream, warmup: int, reps: int) -> list:
    """Per-launch times in ms: ``warmup`` untimed launches, then ``reps`` launches
    each bracketed by CUDA events on the launching stream, with the L2 flushed
    (outside the events) before every launch."""
    import torch
    for _ in range(warmup):
        flush.zero_()
        step()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
    torch.cuda.synchronize()
    for i in range(reps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


def sdpa_same_gpu(w, tq, tk, tv, flush, stream, flops):
    """PyTorch's scaled_dot_product_attention (the backend torch picks) on the same
    device tensors and GPU, timed like the forward: the median of 30 launches
    after 5 warm-ups, the L2 flushed before each.  Context, not a baseline; None
    for fp32 and score-modified workloads, which it does not express alike."""
    import torch
    import torch.nn.functional as F
    if w.dtype != si.BF16 or w.modified:
        return None
    kw = {"is_causal": bool(w.causal), "scale": float(w.scale)}
    if w.Hkv != w.H:
        kw["enable_gqa"] = True
    try:
        def step():
            F.scaled_dot_product_attention(tq, tk, tv, **kw)
        with torch.cuda.stream(stream):
            ts = sorted(time_launches(step, flush, stream, 5, 30))
        med = ts[len(ts) // 2]
        return {"value": flops / (med * 1e-3) / 1e12, "unit": UNIT, "median_ms": med,
                "torch": torch.__version__, "what": "torch.nn.functional.scaled_dot_product_attention, "
                "same inputs and GPU, median of 30 launches, L2 flushed before each"}
    except Exception as e:  # a backend that does not run here is reported, not fatal
        return {"unavailable": f"{type(e).__name__}: {str(e)[:160]}"}


def measure_sustained(seconds, flops, step, stream, local, launch_s):
    """Back-to-back launches for about ``seconds`` on the launching stream, with
    no L2 flush between them: the rate a long run settles at under the power cap
    (timed with one CUDA event pair around the whole run)."""
    import torch
    n = max(3, min(200000, int(seconds / max(launch_s, 1e-6))))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        e0.record(stream)
        for _ in range(n):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    dt = e0.elapsed_time(e1) / 1e3
    return {"value": flops * n / dt / 1e12, "unit": UNIT, "seconds": dt, "launches": n,
            "l2": "not flushed (back-to-back launches)", "clocks": clocks.summary()}


def tf32_matmul_peak(dev, n: int = 8192, reps: int = 10) -> float:
    """Dense TF32 tensor throughput of this GPU, measured here: the best of
    ``reps`` cuBLAS fp32 matmuls of n^3 with TF32 allowed (2 n^3 FLOP each)."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        a = torch.randn(n, n, device=dev)
        b = torch.randn(n, n, device=dev)
        c = torch.empty(n, n, device=dev)
        best = float("inf")
        for i in range(reps + 3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            e1.synchronize()
            if i >= 3:
                best = min(best, e0.elapsed_time(e1) / 1e3)
        del a, b, c
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / best / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def sfu_probe(fa2, local, flops_per_exp: float, peak_tflops: float):
    """The special-function pipe's ex2 rate (the library's probe kernel) against
    the exponentials the softmax needs at the tensor peak: one per score element,
    i.e. peak / (4 D) per second in the forward."""
    import torch
    with ClockSampler(local) as clocks:
        rate = fa2.fa2_probe_ex2()
    summ = clocks.summary()
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    out = {"ex2_per_s": rate, "demand_at_peak_per_s": peak_tflops * 1e12 / flops_per_exp}
    out["demand_frac"] = out["demand_at_peak_per_s"] / rate
    if summ and summ["sm_mhz"] > 0:
        out["ex2_per_clk_per_sm"] = rate / (sms * summ["sm_mhz"] * 1e6)
        out["sm_mhz"] = summ["sm_mhz"]
    return out


def run_ours(args, rank, local, world):
    import torch
    import exact_attention_forward_fa2_gb300 as fa2

    w = si.WORKLOADS[args.workload]
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    q, k, v = si.make_qkv(w)

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    o = torch.empty_like(tq)
    lse = torch.empty((w.B, w.H, w.M), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    launches_per_step = 1
    flops = w.flops
    bwd = args.pass_ == "bwd"
    e2e_ins, e2e_outs = [(q, tq), (k, tk), (v, tv)], [o, lse]
    if bwd:
        if w.modified or w.split_kv or w.dtype != si.BF16:
            raise SystemExit(f"--pass bwd: workload {w.name} is not a plain bf16 one")
        do = si.normal(w.seed, 4, q.shape, 1.0, w.dtype)
        tdo = to_dev(do)
        fa2.fa2_fwd(tq, tk, tv, o=o, lse=lse, scale=w.scale, causal=w.causal, stream=stream)
        dq, dk, dv = torch.empty_like(tq), torch.empty_like(tk), torch.empty_like(tv)
        ws = torch.empty(fa2.lib().fa2_bwd_workspace_bytes(w.B, w.H, w.M), dtype=torch.uint8, device=dev)
        flops = BWD_FLOPS_OVER_FWD * w.flops
        # preprocess, dK/dV pass with dQ by reduction, dQ convert (head dim 128);
        # preprocess, dK/dV pass, dQ pass (head dim 64)
        launches_per_step = 3

        def step():
            fa2.fa2_bwd(tq, tk, tv, o, lse, tdo, dq=dq, dk=dk, dv=dv, scale=w.scale, causal=w.causal,
                        workspace=ws, stream=stream, deterministic=args.deterministic)
    elif w.modified:
        slopes = torch.from_numpy(si.alibi_slopes(w.H)).to(dev) if w.alibi else None

        def step():
            fa2.fa2_fwd_ext(tq, tk, tv, o=o, lse=lse, scale=w.scale, causal=w.causal, window=w.window,
                            softcap=w.softcap, alibi_slopes=slopes, num_splits=1, stream=stream)
    elif w.split_kv:
        dcode = fa2.FA2_BF16 if w.dtype == si.BF16 else fa2.FA2_FP32
        n_split = fa2.fa2_splitkv_num_splits(w.B, w.H, w.Hkv, w.M, w.N, w.D, dcode)
        ws = torch.empty(max(256, fa2.fa2_splitkv_workspace_bytes(w.B, w.H, w.M, w.D, n_split)),
                         dtype=torch.uint8, device=dev)
        launches_per_step = 2 if n_split > 1 else 1  # forward slices + combine

        def step():
            fa2.fa2_fwd_splitkv(tq, tk, tv, o=o, lse=lse, scale=w.scale, causal=w.causal,
                                num_splits=n_split, workspace=ws, stream=stream)
    else:
        def step():
            fa2.fa2_fwd(tq, tk, tv, o=o, lse=lse, scale=w.scale, causal=w.causal, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if fa2.fa2_device_status(reset=True) != 0:
        raise RuntimeError("device status set during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local, args.clock_log) as clocks:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()  # L2 flush between timed steps (outside the event pair)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    barrier(world)
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    status = fa2.fa2_device_status(reset=True)
    t_total = max_over_ranks(sum(kernel_ms) / 1e3, world)
    value = flops * args.steps * world / t_total / 1e12
    ms_per_step = t_total / args.steps * 1e3

    if args.e2e and bwd:
        o_host = o.view(torch.int16).cpu().numpy().view(np.uint16)
        e2e_ins = [(q, tq), (k, tk), (v, tv), (o_host, o), (lse.cpu().numpy(), lse), (do, tdo)]
        e2e_outs = [dq, dk, dv]
    host_step = None
    if bwd and args.e2e and not args.deterministic:  # fa2_bwd_host runs fa2_bwd
        def host_step(hin, hout):
            bf = [t.view(torch.bfloat16) if t.dtype == torch.int16 else t for t in hin + hout]
            fa2.fa2_bwd_host(*bf[:6], dq_host=bf[6], dk_host=bf[7], dv_host=bf[8], scale=w.scale,
                             causal=w.causal, chunks=args.e2e_chunks, workspace=ws,
                             buffers=(tq, tk, tv, o, lse, tdo, dq, dk, dv), stream=stream)
    elif not (bwd or w.modified or w.split_kv):
        def host_step(hin, hout):
            as_dt = (lambda t: t.view(torch.bfloat16)) if w.dtype == si.BF16 else (lambda t: t)
            fa2.fa2_fwd_host(as_dt(hin[0]), as_dt(hin[1]), as_dt(hin[2]), o_host=as_dt(hout[0]),
                             lse_host=hout[1], q=tq, k=tk, v=tv, o=o, lse=lse, scale=w.scale,
                             causal=w.causal, chunks=args.e2e_chunks, stream=stream)
    e2e = measure_e2e(args, flops, step, stream, world, e2e_ins, e2e_outs, host_step) if args.e2e else None
    if e2e is not None:
        e2e["api"] = (("fa2_bwd_host" if bwd else "fa2_fwd_host") + " (pipelined copies)") if host_step \
            else "copies + device-buffer call"

    launch_s = sum(kernel_ms) / len(kernel_ms) / 1e3
    # the measurement plan's protocol: the median of >= 100 event-timed launches
    # after >= 25 warm-ups; the timed steps serve when there are enough of them
    if args.steps >= PROTOCOL_REPS and args.warmup >= PROTOCOL_WARMUP:
        proto_ms, proto_src = kernel_ms, "the timed steps above"
    else:
        proto_ms = time_launches(step, flush, stream, PROTOCOL_WARMUP, PROTOCOL_REPS)
        proto_src = (f"{PROTOCOL_REPS} more launches after {PROTOCOL_WARMUP} warm-ups "
                     "(the timed steps were fewer)")
    protocol = {"median_ms": float(np.median(proto_ms)), "mean_ms": float(np.mean(proto_ms)),
                "p10_ms": float(np.percentile(proto_ms, 10)), "p90_ms": float(np.percentile(proto_ms, 90)),
                "reps": len(proto_ms), "from": proto_src,
                "value_median": flops / (float(np.median(proto_ms)) / 1e3) / 1e12, "unit": UNIT,
                "l2": "flushed between launches (256 MiB write, outside the events)"}
    sustained = None
    if args.sustained_s > 0 and launch_s < 100e-6:
        sustained = {"skipped": "launches shorter than 100 us: a back-to-back loop issued from Python "
                                "would measure the host, not the GPU"}
    elif args.sustained_s > 0:
        sustained = measure_sustained(args.sustained_s, flops, step, stream, local, launch_s)
    if fa2.fa2_device_status(reset=True) != 0:
        raise RuntimeError("device status set during the sustained run")

    if rank != 0:
        return
    peak, hbm_peak, peak_kind = measured_peaks()
    peak_kind = f"bf16 dense burst, {peak_kind}"
    tf32_probe = None
    if w.dtype != si.BF16 and not args.probes:
        peak = TF32_OVER_BF16 * peak
        peak_kind = "tf32 dense, nominal ratio x measured bf16 burst (the TF32 probe was skipped)"
    elif w.dtype != si.BF16:
        # TF32 contraction: this GPU's TF32 rate, measured by a cuBLAS matmul probe
        tf32_probe = tf32_matmul_peak(dev)
        peak = tf32_probe
        peak_kind = ("tf32 dense burst, measured in this run (cuBLAS fp32 8192^3 matmul with TF32, "
                     f"best of 10); nominal ratio would give {TF32_OVER_BF16 * measured_peaks()[0]:.1f}")
    sus_peak = peak_sustained() if w.dtype == si.BF16 else None
    if sustained is not None and "value" in sustained and sus_peak:
        sustained["peak"] = sus_peak
        sustained["frac"] = sustained["value"] / sus_peak
        sustained["peak_kind"] = "bf16 dense sustained (4 s back-to-back cuBLAS), measured"
    achieved = flops / launch_s / 1e12
    io = bwd_io_bytes(w) if bwd else w.io_bytes()
    # below the ridge (peak FLOP/s over peak HBM bytes/s) the launch is bound by
    # reading Q, K, V and writing O, L once: decode-shaped workloads
    hbm_bound = (not bwd) and flops / io < peak * 1e12 / (hbm_peak * 1e9)
    if hbm_bound:
        roof = {"bound": "hbm", "achieved": io / launch_s / 1e9, "peak": hbm_peak, "unit": "GB/s",
                "frac": io / launch_s / 1e9 / hbm_peak, "peak_kind": "HBM copy, measured",
                "tensor_tflops": achieved, "tensor_peak_tflops": peak}
    else:
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_kind": peak_kind}
    line = {
        "metric": METRIC_BWD if bwd else METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == si.BF16 else "tf32", "data": "synthetic",
        "config": {"workload": w.name, "pass": args.pass_, "B": w.B, "H": w.H, "H_kv": w.Hkv, "M": w.M,
                   "N": w.N, "D": w.D, "causal": w.causal, "scale": w.scale,
                   "l2": "flushed between timed steps (256 MiB write, outside the events)",
                   "parallelism": f"replicas x{world}",
                   **({"num_splits": n_split} if w.split_kv else {}),
                   **({"window": list(w.window), "softcap": w.softcap, "alibi": w.alibi}
                      if w.modified else {})},
        "frac_of_peak": roof["frac"],
        "roofline": {**roof,
                     "traffic": dram_traffic_per_launch(w.name, args.pass_),
                     "kernel": ("fa2_bwd (preprocess + dK/dV/dQ-by-reduction + dQ convert kernels)"
                                if w.D == 128 and not args.deterministic
                                else "fa2_bwd%s (preprocess + dK/dV + dQ kernels)"
                                % ("_deterministic" if args.deterministic else "")) if bwd else KERNEL,
                     "algorithmic_flops_per_launch": flops,
                     "hbm_algorithmic_bytes_per_launch": io,
                     "hbm_gbs_at_this_time": io / (sum(kernel_ms) / len(kernel_ms) / 1e3) / 1e9,
                     "hbm_peak_gbs": hbm_peak},
        "timing": {"value_from": "mean of the timed steps (sum of their event times)",
                   "median_ms_timed_steps": float(np.median(kernel_ms)),
                   "mean_ms_timed_steps": float(np.mean(kernel_ms)),
                   "protocol_median_of_100": protocol},
        "e2e": e2e,
        "sustained": sustained,
        "sfu": None if bwd or w.dtype != si.BF16 or not args.probes else sfu_probe(fa2, local, 4.0 * w.D, peak),
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks.summary(),
        "device_status": status,
        "wall_s_timed_region": wall,
    }
    if args.cpu_baseline and bwd:
        tf, n, dt, cores = oracle_sample_bwd(w, q, k, v, seconds_target=args.cpu_seconds)
        line["cpu_baseline"] = {"value": tf, "unit": UNIT, "cores": cores, "cpu": cpu_model(), "kind": "oracle",
                                "sample": f"fp64 backward of {n} whole query heads of the workload "
                                          f"in {dt:.1f} s",
                                **cpu_extrapolation(w, flops, tf, None, dt)}
    elif args.cpu_baseline:
        tf, n, dt, cores = oracle_sample(w, q, k, v, seconds_target=args.cpu_seconds)
        line["cpu_baseline"] = {"value": tf, "unit": UNIT, "cores": cores, "cpu": cpu_model(), "kind": "oracle",
                                "sample": f"{n} seeded random query rows of the workload (fp64, all "
                                          f"their visible keys) in {dt:.1f} s",
                                **cpu_extrapolation(w, flops, tf, n, dt)}
    # the pages' own timings, quoted as context on every line (their shape is the
    # TF32 workload's); this run's median sits beside them only on that workload
    ctx = dict(PAGES_CONTEXT)
    if w.name == PAGES_CONTEXT_WORKLOAD and not bwd:
        ctx["this_run_median_us"] = protocol["median_ms"] * 1e3
    else:
        ctx["this_run"] = f"another workload ({w.name}); the pages' shape is bench.py --workload {PAGES_CONTEXT_WORKLOAD}"
    ctx["note"] = "other hardware and precision: context, not a target or a baseline"
    if args.probes and not bwd:
        sd = sdpa_same_gpu(w, tq, tk, tv, flush, stream, flops)
        if sd is not None:
            ctx["pytorch_sdpa_same_gpu"] = sd
    line["context"] = ctx
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=PROTOCOL_WARMUP)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(si.WORKLOADS), default=WORKLOAD,
                    help="workload to measure (default: the headline bf16 D=128 causal one)")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="time the forward (default) or the backward pass")
    ap.add_argument("--deterministic", action="store_true",
                    help="--pass bwd: time fa2_bwd_deterministic (dQ by a second pass)")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-probes", dest="probes", action="store_false",
                    help="skip the ex2-rate and TF32-peak probes after the timed steps (for launch lists)")
    ap.add_argument("--sustained-s", type=float, default=4.0,
                    help="seconds of back-to-back launches after the timed steps (0: skip)")
    ap.add_argument("--e2e-chunks", type=int, default=0,
                    help="head slices of the host-buffer pipeline (0: the library's choice)")
    ap.add_argument("--clock-log", default=None, help="write the NVML clock samples here (CSV)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    rank, local, world = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, local, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
