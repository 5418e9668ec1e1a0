"""Coarse pipeline trace of the attention kernel (opt-in trace build).

Builds ``libfmha_trace.so`` (the kernel compiled with -DFMHA_TRACE), runs one
workload, and summarises the %clock64 stamps the CTAs of head 0 / sequence 0
record at role hand-off points: per KV step, how long the softmax warpgroups
spend loading S from tensor memory, reducing the max, exponentiating and
storing P, how long the MMA warp takes to notice P and to issue the next
MMAs, and the step period.  This is the coarse mode of "Kernel Bottleneck
Tuning", section "2. Trace the real pipeline, coarsely": stamps only at
hand-offs, numbers in SM cycles.

  python -m attention_forward_mbarrier_gb300.trace [--workload NAME] [--row R]
         [--flags "-DNAME=VALUE ..."] [--raw stamps.npy]
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics

import numpy as np
import torch

from . import build as _build
from . import workloads as wl

TRACE_LIB = os.path.join(_build.PKG, "libfmha_trace.so")
SLOTS = 2048
TR_SOFTMAX, TR_MMA, TR_CORR, TR_LOAD = 16, 1040, 1300, 1600


def load_trace_lib(flags=()):
    _build.build(force=True, extra_flags=["-DFMHA_TRACE", *flags], out=TRACE_LIB)
    L = ctypes.CDLL(TRACE_LIB)
    L.fmha_fwd.restype = ctypes.c_int
    L.fmha_fwd.argtypes = ([ctypes.c_void_p] * 7 + [ctypes.c_int] * 7
                           + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p])
    L.fmha_debug_set_trace.restype = ctypes.c_int
    L.fmha_debug_set_trace.argtypes = [ctypes.c_void_p]
    L.fmha_debug_set_cta_trace.restype = ctypes.c_int
    L.fmha_debug_set_cta_trace.argtypes = [ctypes.c_void_p]
    return L


def run(w: wl.Workload, repeats: int = 3, flags=(), flush_l2: bool = True):
    """Stamps of the last of `repeats` launches: [query blocks, SLOTS] int64."""
    L = load_trace_lib(flags)
    dev = torch.device("cuda:0")
    inp = wl.make_inputs(w, seed=0)
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    cq = None if inp.cu_seqlens_q is None else inp.cu_seqlens_q.to(dev)
    ck = None if inp.cu_seqlens_k is None else inp.cu_seqlens_k.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.heads, w.total_q), dtype=torch.float32, device=dev)
    pairs = (w.max_seqlen_q + 255) // 256
    buf = torch.zeros((pairs, SLOTS), dtype=torch.int64, device=dev)
    ctas = torch.zeros((w.heads * pairs * w.batch, 4), dtype=torch.int64, device=dev)
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream

    def ptr(t):
        return None if t is None else t.data_ptr()

    if L.fmha_debug_set_trace(buf.data_ptr()) != 0 or L.fmha_debug_set_cta_trace(ctas.data_ptr()) != 0:
        raise RuntimeError("fmha_debug_set_trace failed")
    try:
        for _ in range(repeats):
            buf.zero_()
            ctas.zero_()
            if flush_l2:
                flush.zero_()  # the benchmark's L2 flush precedes every launch
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            st = L.fmha_fwd(ptr(q), ptr(k), ptr(v), ptr(out), ptr(lse), ptr(cq), ptr(ck), w.batch,
                            w.total_q, w.total_k, w.max_seqlen_q, w.max_seqlen_k, w.heads,
                            w.head_dim, w.softmax_scale, int(w.causal), stream)
            e1.record()
            if st != 0:
                raise RuntimeError(f"fmha_fwd returned {st}")
            torch.cuda.synchronize()
            run.last_event_ns = int(e0.elapsed_time(e1) * 1e6)
    finally:
        L.fmha_debug_set_trace(None)
        L.fmha_debug_set_cta_trace(None)
    return buf.cpu().numpy(), ctas.cpu().numpy()


def summarize_ctas(ctas: np.ndarray) -> dict:
    """Spread of CTA entry / set-up / exit times (ns, relative to the first entry)."""
    live = ctas[ctas[:, 0] > 0]
    t0 = live[:, 0].min()
    ent, setup, ext = live[:, 0] - t0, live[:, 1] - t0, live[:, 2] - t0
    q = lambda a: [int(np.percentile(a, x)) for x in (0, 50, 100)]  # noqa: E731
    return {"ctas": int(len(live)), "sms": int(len(np.unique(live[:, 3]))),
            "entry_ns_min_med_max": q(ent), "setup_done_ns_min_med_max": q(setup),
            "exit_ns_min_med_max": q(ext), "lifetime_ns_min_med_max": q(ext - ent)}


def summarize(row: np.ndarray) -> dict:
    """Median cycles per KV step of each phase, over both tiles and all steps."""
    t0 = row[0]

    def sm(t, j, e):
        return int(row[TR_SOFTMAX + t * 512 + j * 8 + e])

    def mma(j, e):
        return int(row[TR_MMA + j * 8 + e])

    nblk = 0
    while nblk < 32 and (sm(0, nblk, 0) or sm(1, nblk, 0)):
        nblk += 1
    ph = {k: [] for k in ("ld", "max", "exp", "store_arrive", "wait_S", "period", "mma_notice",
                          "mma_issue_span")}
    for t in (0, 1):
        for j in range(nblk):
            if not sm(t, j, 0):
                continue
            ph["ld"].append(sm(t, j, 1) - sm(t, j, 0))
            ph["max"].append(sm(t, j, 2) - sm(t, j, 1))
            ph["exp"].append(sm(t, j, 3) - sm(t, j, 2))
            ph["store_arrive"].append(sm(t, j, 4) - sm(t, j, 3))
            if j + 1 < nblk and sm(t, j + 1, 0):
                ph["wait_S"].append(sm(t, j + 1, 0) - sm(t, j, 4))
                ph["period"].append(sm(t, j + 1, 0) - sm(t, j, 0))
            acq, issued = mma(j, 1 + 2 * t), mma(j, 2 + 2 * t)
            if acq:
                ph["mma_notice"].append(acq - sm(t, j, 4))
                if issued:
                    ph["mma_issue_span"].append(issued - acq)
    out = {k: (statistics.median(v) if v else None) for k, v in ph.items()}
    out["blocks"] = nblk
    out["first_S_ready"] = sm(0, 0, 0) - int(t0) if sm(0, 0, 0) else None
    out["cta_end"] = int(row[1] - t0) if row[1] else None
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default=wl.C2.name, choices=sorted(wl.CONFIGS))
    ap.add_argument("--row", type=int, default=0, help="query block (256 rows) of head 0 to show")
    ap.add_argument("--raw", default=None, help="save the raw stamps (.npy)")
    ap.add_argument("--flags", default="", help="extra -D flags for the trace build (tuning variants)")
    ap.add_argument("--no-flush", action="store_true", help="skip the L2 flush before each launch")
    args = ap.parse_args()
    w = wl.CONFIGS[args.workload]
    stamps, ctas = run(w, flags=args.flags.split(), flush_l2=not args.no_flush)
    if args.raw:
        np.save(args.raw, stamps)
    print(json.dumps({"workload": w.name, "flags": args.flags,
                      "cycles_per_kv_step_median": summarize(stamps[args.row]),
                      "cta_times": summarize_ctas(ctas),
                      "kernel_event_ns": run.last_event_ns, "l2_flushed": not args.no_flush}, indent=1))


if __name__ == "__main__":
    main()
