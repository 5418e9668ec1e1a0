#!/usr/bin/env python
"""Benchmark of the fused attention forward on GB300.

One step = one fmha_fwd launch over the whole workload (every query row of
every head).  Default workload: dense, batch 1, heads 16, seq 2225,
head_dim 128, non-causal (the shape of the pages' 77_blackwell_fmha /
fmha.py comparison).  Inputs are seeded synthetic bf16 N(0, 1) tensors.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-cpu-baseline]

Multi-GPU (torchrun, one rank per GPU): every rank runs an independent
replica of the workload on its own GPU (the forward has no exchange step);
value = units of all ranks / max-over-ranks time.  --impl reference times the
CPU oracle (fp64) on a bounded row sample on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from attention_forward_mbarrier_gb300 import workloads as wl  # noqa: E402

METRIC = "FMHA fwd TFLOP/s (bf16, d=128) and % of GB300 dense bf16 tensor peak"
UNIT = "TFLOP/s"
L2_BYTES = 126 * 1024 * 1024


class L2Flusher:
    """Evicts the inputs from L2 between timed steps (outside the events).

    "write+read" (default): write a 504 MiB buffer, then read another 504 MiB
    buffer, so L2 holds neither input bytes nor the dirty lines of the write
    (whose write-back would otherwise be charged to the timed kernel; measured
    ~1.9 us on the dense workload).  "write": the write pass alone.
    """

    def __init__(self, dev, mode: str):
        self.mode = mode
        self.scratch = torch.empty(L2_BYTES, dtype=torch.float32, device=dev)
        self.reader = None
        if mode == "write+read":
            self.reader = torch.zeros(L2_BYTES, dtype=torch.float32, device=dev)
            self.sink = torch.empty(1, dtype=torch.float32, device=dev)

    def flush(self):
        self.scratch.zero_()
        if self.reader is not None:
            self.sink.copy_(self.reader.sum().reshape(1))

    DESCRIBE = {
        "write+read": "flushed between steps: 504 MiB written, then 504 MiB read (no input and no dirty lines in L2)",
        "write": "flushed between steps: 504 MiB written",
    }

    def describe(self) -> str:
        return self.DESCRIBE[self.mode]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = ("fmha_api.cu", "fmha_fwd_kernel.cuh", "sm103_ptx.cuh")


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_forward_mbarrier_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name in KERNEL_SOURCES:
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches this kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(workload_name)
    if not rec or rec.get("kernel_sha") != kernel_source_sha():
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_baseline(w: wl.Workload, inp, budget_s: float = 15.0):
    """Time the oracle (as it stands) on a bounded seeded row sample; TFLOP/s."""
    import oracle

    oracle.build()
    rng = np.random.default_rng(123)
    # cost of a row ~ its visible keys; start small, grow to the time budget
    n = 64
    rows = None
    elapsed = 0.0
    while True:
        toks = rng.integers(0, w.total_q, size=n)
        hs = rng.integers(0, w.heads, size=n)
        rows = (toks * w.heads + hs).astype(np.int64)
        t0 = time.perf_counter()
        oracle.oracle_fwd(*inp.oracle_args(), rows=rows)
        elapsed = time.perf_counter() - t0
        if elapsed >= budget_s / 3 or n >= w.total_q * w.heads:
            break
        n = int(min(n * max(2.0, budget_s / 3 / max(elapsed, 1e-3)), w.total_q * w.heads))
    flops = sample_flops(w, rows)
    return {"value": flops / elapsed / 1e12, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{len(rows)} random (token, head) rows of {w.name}, fp64, "
                      f"{elapsed:.1f} s, {flops / 1e9:.2f} algorithmic GFLOP"}


def sample_flops(w: wl.Workload, rows: np.ndarray) -> float:
    """Algorithmic FLOPs of the sampled rows: 4 * head_dim * visible keys per row."""
    cq, ck = w.cu_seqlens()
    tok = rows // w.heads
    b = np.searchsorted(cq, tok, side="right") - 1
    i = tok - cq[b]
    lq = np.diff(cq)[b]
    lk = np.diff(ck)[b]
    vis = np.minimum(lk, np.maximum(0, i + lk - lq + 1)) if w.causal else lk
    return float(4.0 * w.head_dim * vis.sum())


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    inp = wl.make_inputs(w, seed=0)
    for _ in range(args.warmup):
        pass  # the oracle has no state to warm
    vals = []
    base = None
    for _ in range(args.steps):
        base = cpu_baseline(w, inp, budget_s=args.ref_budget)
        vals.append(base["value"])
    value = statistics.median(vals)
    base["value"] = value
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, world, args.flush),
            "note": "CPU oracle: config.l2 describes the GPU arm's flush",
            "impl": "reference", "cpu_baseline": base,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def input_bytes(w: wl.Workload) -> int:
    return 2 * w.head_dim * (w.total_q * w.heads + 2 * w.total_k * w.n_kv_heads)


def l2_policy(w: wl.Workload, flush_mode: str) -> str:
    """How the GPU arm keeps L2 from carrying inputs between timed steps."""
    if input_bytes(w) < 2 * L2_BYTES:
        return L2Flusher.DESCRIBE[flush_mode]
    return "inputs larger than L2"


def workload_config(w: wl.Workload, world: int, flush_mode: str) -> dict:
    """The workload description both arms print (identical for the same workload)."""
    return {"workload": w.name, "description": w.description, "heads": w.heads, "total_q": w.total_q,
            "max_seqlen": w.max_seqlen_q, "causal": w.causal, "gflop_per_step": w.flops() / 1e9,
            "l2": l2_policy(w, flush_mode), "parallelism": f"replicas x{world}"}


def call_fwd(binding, w: wl.Workload, q, k, v, out, lse, cq, ck, stream) -> int:
    """One launch through the C ABI (the grouped-K/V entry when w has kv_heads)."""
    if w.kv_heads is None:
        return binding.fmha_fwd(q, k, v, out, lse, cq, ck, w.batch, w.total_q, w.total_k, w.max_seqlen_q,
                                w.max_seqlen_k, w.heads, w.head_dim, w.softmax_scale, int(w.causal), stream)
    return binding.fmha_fwd_gqa(q, k, v, out, lse, cq, ck, w.batch, w.total_q, w.total_k, w.max_seqlen_q,
                                w.max_seqlen_k, w.heads, w.n_kv_heads, w.head_dim, w.softmax_scale,
                                int(w.causal), stream)


def kernel_only(w: wl.Workload, dev, peak: float, steps: int = 5, warmup: int = 3, flush_mode: str = "write+read"):
    """Kernel time of another workload (inputs resident, CUDA events), for context."""
    from attention_forward_mbarrier_gb300 import binding

    inp = wl.make_inputs(w, seed=0)
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    cq = None if inp.cu_seqlens_q is None else inp.cu_seqlens_q.to(dev)
    ck = None if inp.cu_seqlens_k is None else inp.cu_seqlens_k.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.heads, w.total_q), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    flusher = L2Flusher(dev, flush_mode) if in_bytes < 2 * L2_BYTES else None
    def launch():
        st = call_fwd(binding, w, q, k, v, out, lse, cq, ck, stream)
        if st != binding.FMHA_OK:
            raise RuntimeError(binding.status_string(st))

    ms = []
    if flusher is not None:
        # the flush before each step keeps the GPU busy while the host enqueues
        for i in range(warmup + steps):
            flusher.flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch()
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= warmup:
                ms.append(e0.elapsed_time(e1))
    else:
        # inputs larger than 2x L2: back-to-back launches between one pair of
        # events, so no host enqueue time is inside the region
        for _ in range(warmup):
            launch()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            launch()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = [e0.elapsed_time(e1) / steps]
    mean = statistics.mean(ms)
    tf = w.flops() / (mean * 1e-3) / 1e12
    del q, k, v, out, lse, flusher
    torch.cuda.empty_cache()
    return {"tflops": tf, "frac_of_peak": tf / peak, "ms": mean, "gflop": w.flops() / 1e9,
            "causal": w.causal}


def backward_only(w: wl.Workload, dev, peak: float, steps: int = 5, warmup: int = 3,
                  flush_mode: str = "write+read"):
    """Time fmha_bwd (both of its kernels) with inputs, O and LSE resident, for
    context.  Algorithmic FLOPs of the backward: five GEMM families (S, dP, dV,
    dK, dQ) = 2.5x the forward's; the kernels' recomputation of S and dP for
    dQ is not credited.  Also times one forward + backward step."""
    from attention_forward_mbarrier_gb300 import binding

    inp = wl.make_inputs(w, seed=0)
    dO = wl.make_dout(w, seed=0)
    q, k, v, g = (t.to(dev) for t in (inp.q, inp.k, inp.v, dO))
    cq = None if inp.cu_seqlens_q is None else inp.cu_seqlens_q.to(dev)
    ck = None if inp.cu_seqlens_k is None else inp.cu_seqlens_k.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.heads, w.total_q), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(max(1, binding.fmha_bwd_workspace_size(w.heads, w.total_q) // 4), dtype=torch.float32,
                     device=dev)
    stream = torch.cuda.current_stream(dev)
    flusher = L2Flusher(dev, flush_mode) if input_bytes(w) < 2 * L2_BYTES else None

    def fwd():
        st = call_fwd(binding, w, q, k, v, out, lse, cq, ck, stream)
        if st != binding.FMHA_OK:
            raise RuntimeError(binding.status_string(st))

    def bwd():
        st = binding.fmha_bwd(q, k, v, out, g, lse, dq, dk, dv, ws, cq, ck, w.batch, w.total_q, w.total_k,
                              w.max_seqlen_q, w.max_seqlen_k, w.heads, w.n_kv_heads, w.head_dim,
                              w.softmax_scale, int(w.causal), stream)
        if st != binding.FMHA_OK:
            raise RuntimeError(binding.status_string(st))

    def timed(fn):
        ms = []
        for i in range(warmup + steps):
            if flusher is not None:
                flusher.flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= warmup:
                ms.append(e0.elapsed_time(e1))
        return statistics.mean(ms)

    fwd()
    bwd_ms = timed(bwd)
    step_ms = timed(lambda: (fwd(), bwd()))
    st, detail = binding.fmha_get_device_status(stream)
    if st != binding.FMHA_OK:
        raise RuntimeError(f"device status {binding.status_string(st)} detail {detail}")
    flops = 2.5 * w.flops()
    tf = flops / (bwd_ms * 1e-3) / 1e12
    del q, k, v, g, out, lse, dq, dk, dv, ws, flusher
    torch.cuda.empty_cache()
    return {"tflops": tf, "frac_of_peak": tf / peak, "ms": bwd_ms, "gflop": flops / 1e9, "causal": w.causal,
            "launches": 3, "fwd_bwd_ms": step_ms,
            "fwd_bwd_tflops": 3.5 * w.flops() / (step_ms * 1e-3) / 1e12}


def fp8_call(w: wl.Workload, dev, peak: float, steps: int = 5, warmup: int = 3, flush_mode: str = "write+read"):
    """Time the whole fmha_fwd_fp8pv call (V quantisation pre-pass + attention),
    inputs resident, for context.  FLOPs are the forward's; the peak is the mixed
    one (QK^T at the bf16 rate, PV at twice it: 4/3 of the bf16 peak)."""
    from attention_forward_mbarrier_gb300 import binding

    inp = wl.make_inputs(w, seed=0)
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    cq = None if inp.cu_seqlens_q is None else inp.cu_seqlens_q.to(dev)
    ck = None if inp.cu_seqlens_k is None else inp.cu_seqlens_k.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.heads, w.total_q), dtype=torch.float32, device=dev)
    ws = torch.empty(binding.fmha_fwd_fp8pv_workspace_size(w.batch, w.total_k, w.n_kv_heads, w.head_dim),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    flusher = L2Flusher(dev, flush_mode) if input_bytes(w) < 2 * L2_BYTES else None
    ms = []
    for i in range(warmup + steps):
        if flusher is not None:
            flusher.flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        st = binding.fmha_fwd_fp8pv(q, k, v, out, lse, ws, cq, ck, w.batch, w.total_q, w.total_k, w.max_seqlen_q,
                                    w.max_seqlen_k, w.heads, w.n_kv_heads, w.head_dim, w.softmax_scale,
                                    int(w.causal), stream)
        e1.record(stream)
        if st != binding.FMHA_OK:
            raise RuntimeError(binding.status_string(st))
        torch.cuda.synchronize()
        if i >= warmup:
            ms.append(e0.elapsed_time(e1))
    mean = statistics.mean(ms)
    tf = w.flops() / (mean * 1e-3) / 1e12
    mixed_peak = peak * 4.0 / 3.0
    del q, k, v, out, lse, ws, flusher
    torch.cuda.empty_cache()
    return {"tflops": tf, "frac_of_mixed_peak": tf / mixed_peak, "mixed_peak": mixed_peak, "ms": mean,
            "launches": 3, "includes": "V max + e4m3 quantise/transpose pre-pass + attention"}


def run_ours(args, w, rank, world, local):
    from attention_forward_mbarrier_gb300 import binding
    from attention_forward_mbarrier_gb300 import build as _build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    _build.build()
    binding.lib()
    dev = torch.device("cuda", local)
    inp = wl.make_inputs(w, seed=0)
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    cq = None if inp.cu_seqlens_q is None else inp.cu_seqlens_q.to(dev)
    ck = None if inp.cu_seqlens_k is None else inp.cu_seqlens_k.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.heads, w.total_q), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = input_bytes(w) < 2 * L2_BYTES
    flusher = L2Flusher(dev, args.flush) if flush else None

    def launch():
        st = call_fwd(binding, w, q, k, v, out, lse, cq, ck, stream)
        if st != binding.FMHA_OK:
            raise RuntimeError(binding.status_string(st))

    for _ in range(max(3, args.warmup)):
        if flush:
            flusher.flush()
        launch()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        # keep the GPU busy for ~1 s right before the timed region so the
        # 100 ms clock samples cover the clocks the timed steps run at
        t_busy = time.perf_counter()
        while time.perf_counter() - t_busy < args.clock_window:
            for _ in range(50):
                if flush:
                    flusher.flush()
                launch()
            torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            if flush:
                flusher.flush()  # L2 flush, outside the timed events
            starts[i].record(stream)
            launch()
            ends[i].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        t_wall = time.perf_counter() - t_wall
    st, detail = binding.fmha_get_device_status(stream)
    if st != binding.FMHA_OK:
        raise RuntimeError(f"device status {binding.status_string(st)} detail {detail}")
    times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = statistics.mean(times_ms)
    ms_max = max_over_ranks(ms, world)
    flops = w.flops()
    value = world * flops / (ms_max * 1e-3) / 1e12

    # context only: the same launch with its inputs resident in L2 (back-to-back
    # launches between one pair of events, no flush)
    warm_ms = None
    if flush:
        for _ in range(3):
            launch()
        torch.cuda.synchronize()
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        for _ in range(args.steps):
            launch()
        w1.record(stream)
        torch.cuda.synchronize()
        warm_ms = w0.elapsed_time(w1) / args.steps

    # end to end through the public API: pinned host buffers, every step's
    # host->device copies of q, k, v and device->host copies of O and LSE
    # inside the timed region.  Double-buffered as a streaming caller would
    # run it: step i+1's input copies (copy stream) overlap step i's kernel
    # (compute stream) and its result read-back (read-back stream); events
    # keep each buffer slot's copy -> kernel -> read-back order.
    hq, hk, hv = (t.pin_memory() for t in (inp.q, inp.k, inp.v))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    slots = [dict(q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v), out=torch.empty_like(out),
                  lse=torch.empty_like(lse)) for _ in range(2)]
    s_in, s_back = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]    # slot inputs copied
    ev_run = [torch.cuda.Event() for _ in range(2)]   # slot kernel done
    ev_back = [torch.cuda.Event() for _ in range(2)]  # slot outputs read back
    e_steps = max(3, min(args.steps, 20))

    def e2e_step(i):
        sl, j = slots[i % 2], i % 2
        if i >= 2:
            s_in.wait_event(ev_run[j])  # the kernel that read this slot's inputs is done
        with torch.cuda.stream(s_in):
            sl["q"].copy_(hq, non_blocking=True)
            sl["k"].copy_(hk, non_blocking=True)
            sl["v"].copy_(hv, non_blocking=True)
        ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        if i >= 2:
            stream.wait_event(ev_back[j])  # this slot's previous outputs were read back
        st2 = call_fwd(binding, w, sl["q"], sl["k"], sl["v"], sl["out"], sl["lse"], cq, ck, stream)
        if st2 != binding.FMHA_OK:
            raise RuntimeError(binding.status_string(st2))
        ev_run[j].record(stream)
        s_back.wait_event(ev_run[j])
        with torch.cuda.stream(s_back):
            hout.copy_(sl["out"], non_blocking=True)
            hlse.copy_(sl["lse"], non_blocking=True)
        ev_back[j].record(s_back)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_back.wait_event(e0)
    for i in range(e_steps):
        e2e_step(i)
    stream.wait_stream(s_in)
    stream.wait_stream(s_back)
    e1.record(stream)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, world)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = hout.numel() * hout.element_size() + hlse.numel() * hlse.element_size()

    if rank != 0:
        return
    pk, pk_src = peaks()
    peak = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = flops / (ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, world, args.flush),
        "pct_of_peak": 100.0 * achieved / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak, "peak_source": f"bf16_tflops (burst) of {pk_src}",
                     "traffic": recorded_traffic(w.name)},
        "e2e": {"value": world * flops / (e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
                "schedule": "pinned host buffers, two device buffer slots: step i+1's host-to-device copies "
                            "overlap step i's kernel and device-to-host copies"},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "wall_s": t_wall,
        "kernel_ms": {"mean": ms, "min": min(times_ms), "median": statistics.median(times_ms)},
        "median": {"value": flops / (statistics.median(times_ms) * 1e-3) / 1e12, "unit": UNIT,
                   "note": "median of the timed steps (value uses their mean, the more conservative)"},
    }
    if warm_ms is not None:
        line["warm_l2"] = {"value": flops / (warm_ms * 1e-3) / 1e12, "unit": UNIT, "ms": warm_ms,
                           "note": "inputs resident in L2, back-to-back launches; context only"}
    if not args.no_secondary:
        known = {**wl.CONFIGS, **wl.EXTRA}
        line["secondary"] = {x: kernel_only(known[x], dev, peak, flush_mode=args.flush)
                             for x in args.secondary.split(",") if x}
    if not args.no_secondary and args.secondary_bwd:
        known = {**wl.CONFIGS, **wl.EXTRA}
        line["secondary_bwd"] = {x: backward_only(known[x], dev, peak, flush_mode=args.flush)
                                 for x in args.secondary_bwd.split(",") if x}
    if not args.no_secondary and args.secondary_fp8:
        known = {**wl.CONFIGS, **wl.EXTRA}
        line["secondary_fp8pv"] = {x: fp8_call(known[x], dev, peak, flush_mode=args.flush)
                                   for x in args.secondary_fp8.split(",") if x}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp, budget_s=args.ref_budget)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=wl.C2.name, choices=sorted({**wl.CONFIGS, **wl.EXTRA}))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--flush", choices=["write+read", "write"], default="write+read",
                    help="L2 flush between timed steps (see L2Flusher)")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--secondary", default=",".join([wl.C3.name, wl.C4.name, wl.C5.name, wl.GQA_C3.name,
                                                     wl.D64_C5.name, wl.D256_C2.name, wl.D256_C3.name]),
                    help="comma-separated workloads timed kernel-only after the main line")
    ap.add_argument("--secondary-bwd", default=",".join([wl.C2.name, wl.C3.name, wl.C4.name, wl.C5.name]),
                    help="comma-separated workloads whose backward pass (fmha_bwd) is timed after the main line")
    ap.add_argument("--secondary-fp8", default=",".join([wl.C2.name, wl.C3.name, wl.C5.name]),
                    help="comma-separated workloads timed through fmha_fwd_fp8pv after the main line")
    ap.add_argument("--clock-window", type=float, default=1.0,
                    help="seconds of back-to-back launches before the timed region")
    ap.add_argument("--ref-budget", type=float, default=15.0, help="seconds of oracle work per sample")
    args = ap.parse_args()
    w = {**wl.CONFIGS, **wl.EXTRA}[args.workload]
    rank, world, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, w, rank, world)
        else:
            run_ours(args, w, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
