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
         [--flags=-DNAME=VALUE ...] [--raw stamps.npy] [--persistent]

The plain kernel is traced with the persistent variant switched off
(-DFMHA_PERSISTENT_WAVES=1000000), so every workload runs it.  --persistent
traces the persistent variant instead (fmha_fwd_persistent.cuh): per unit
each CTA ran, the hand-offs around the boundary between consecutive units,
and (from two observer warps) when step commits complete and ring loads land.
--backward traces the backward pass's dQ and dK/dV kernels (CTAs of head 0,
sequence 0): per key block (dQ) or query block (dK/dV) the gradient math, the
waits between blocks and how late the MMA-issuing threads see each hand-off.
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
TR_SOFTMAX, TR_MMA, TR_LOAD = 16, 1040, 1600
TR_OBS_LOAD, TR_OBS_STEP = 272, 784


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
    # the benchmark's L2 flush: write 504 MiB, then read another 504 MiB
    flush = torch.empty(126 * 1024 * 1024, dtype=torch.float32, device=dev)
    reader = torch.zeros(126 * 1024 * 1024, dtype=torch.float32, device=dev) if flush_l2 else None
    sink = torch.empty(1, dtype=torch.float32, device=dev)
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
                sink.copy_(reader.sum().reshape(1))
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


def per_tile(row: np.ndarray, nblk: int) -> dict:
    """Per-tile medians of the hand-off chain, SM cycles.

    notice: P hand-off -> MMA warp acquires it; skew: the last
    of the tile's four softmax warps to hand off P, relative to warp 0 (the
    stamped one); busy: the MMA
    warp was still issuing the other tile when P arrived (cycles from the P
    hand-off to the end of that issue); s_latency: last MMA of the group
    issued -> softmax sees S; v_wait: MMA warp waits for the V block after the
    previous step's last group.
    """
    def sm(t, j, e):
        return int(row[TR_SOFTMAX + t * 512 + j * 8 + e])

    def mma(j, e):
        return int(row[TR_MMA + j * 8 + e])

    res = {}
    for t in (0, 1):
        d = {k: [] for k in ("notice", "skew", "busy", "issue_span", "s_latency", "softmax")}
        for j in range(nblk):
            if not sm(t, j, 0):
                continue
            p_at = sm(t, j, 4)
            d["softmax"].append(p_at - sm(t, j, 0))
            others = [sm(t, j, 4 + w) for w in (1, 2, 3) if sm(t, j, 4 + w)]
            if others:
                d["skew"].append(max(others) - p_at)
            acq, issued = mma(j, 1 + 2 * t), mma(j, 2 + 2 * t)
            # the group the MMA warp issued just before this one
            prev = mma(j, 2) if t == 1 else (mma(j - 1, 4) if j > 0 else 0)
            if prev:
                d["busy"].append(prev - p_at)
            if acq:
                d["notice"].append(acq - p_at)
                if issued:
                    d["issue_span"].append(issued - acq)
                    if j + 1 < nblk and sm(t, j + 1, 0):
                        d["s_latency"].append(sm(t, j + 1, 0) - issued)
        res[f"tile{t}"] = {k: (statistics.median(v) if v else None) for k, v in d.items()}
    vw = [mma(j, 0) - mma(j - 1, 4) for j in range(1, nblk) if mma(j, 0) and mma(j - 1, 4)]
    res["v_wait"] = statistics.median(vw) if vw else None
    return res


def setup_and_ring(row: np.ndarray, nblk: int) -> dict:
    """Set-up phases (cycles from kernel entry), ring-load latency (issue ->
    landed, from the observer warp), and per-step MMA completion."""
    med = lambda v: statistics.median(v) if v else None  # noqa: E731
    s = {i: int(row[i]) for i in range(7)}
    out = {}
    if s[2]:
        out["setup"] = {name: (s[i] - s[2] if s[i] else None) for name, i in
                        (("barriers_init", 3), ("copies_issued", 4), ("tmem_alloc", 5), ("pre_sync", 6),
                         ("sync_done", 0))}
        first = int(row[TR_SOFTMAX])
        out["setup"]["first_S0"] = first - s[2] if first else None
    landed = [int(row[TR_OBS_LOAD + i]) for i in range(2 * nblk)]
    issued = [int(row[TR_LOAD + i]) for i in range(2 * nblk)]
    if s[4] and landed[0]:
        out["early_load_latency"] = [x - s[4] for x in landed[:4] if x]
    out["ring_load_latency"] = med([landed[i] - issued[i] for i in range(4, 2 * nblk) if landed[i] and issued[i]])
    # V_j landed relative to the MMA warp acquiring it (negative: it waited on other things)
    out["v_landed_minus_acquired"] = med([landed[2 * j + 1] - int(row[TR_MMA + j * 8])
                                          for j in range(nblk) if landed[2 * j + 1] and row[TR_MMA + j * 8]])
    # MMA warp: last group issued -> step commit issued -> V_(j+1) acquired
    out["step_commit_issue"] = med([int(row[TR_MMA + j * 8 + 5]) - int(row[TR_MMA + j * 8 + 4])
                                    for j in range(nblk) if row[TR_MMA + j * 8 + 5] and row[TR_MMA + j * 8 + 4]])
    out["after_commit_to_v"] = med([int(row[TR_MMA + (j + 1) * 8]) - int(row[TR_MMA + j * 8 + 5])
                                    for j in range(nblk - 1) if row[TR_MMA + (j + 1) * 8] and row[TR_MMA + j * 8 + 5]])
    # PV issue of tile t (acquired -> about to issue its QK^T)
    for t in (0, 1):
        out[f"pv_issue_t{t}"] = med([int(row[TR_MMA + j * 8 + 6 + t]) - int(row[TR_MMA + j * 8 + 1 + 2 * t])
                                     for j in range(nblk) if row[TR_MMA + j * 8 + 6 + t] and row[TR_MMA + j * 8 + 1 + 2 * t]])
    done = [int(row[TR_OBS_STEP + n]) for n in range(nblk + 1)]
    # step commit n = j + 1 completes after the step's last group was issued
    out["step_complete_after_issue"] = med([done[j + 1] - int(row[TR_MMA + j * 8 + 4])
                                            for j in range(nblk) if done[j + 1] and row[TR_MMA + j * 8 + 4]])
    ep = lambda i: int(row[1560 + i])  # noqa: E731
    # (rows with more blocks than the trace keeps have no valid last step)
    last = done[nblk] if 0 < nblk < 32 and done[nblk] else 0
    if last:
        out["epilogue_after_last_mma"] = {
            "tile0_O_seen": ep(0) - last if ep(0) else None, "tile0_O_stored": ep(1) - last if ep(1) else None,
            "tile1_O_seen": ep(4) - last if ep(4) else None, "tile1_O_staged": ep(6) - last if ep(6) else None,
            "tile1_O_stored": ep(5) - last if ep(5) else None,
            "final_sync": ep(8) - last if ep(8) else None}
        lastP = [int(row[TR_SOFTMAX + t * 512 + (nblk - 1) * 8 + 4]) for t in (0, 1)]
        out["last_P_before_last_mma"] = [last - x if x else None for x in lastP]
    out["step_period_in_pipe"] = med([done[n] - done[n - 1] for n in range(2, nblk + 1) if done[n] and done[n - 1]])
    return out


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
    out["per_tile"] = per_tile(row, nblk)
    out.update(setup_and_ring(row, nblk))
    out["blocks"] = nblk
    out["first_S_ready"] = sm(0, 0, 0) - int(t0) if sm(0, 0, 0) else None
    out["cta_end"] = int(row[1] - t0) if row[1] else None
    return out


PERS_UNITS, PERS_EVENTS = 64, 16  # the persistent kernel's trace slots per CTA


def run_persistent(w: wl.Workload, repeats: int = 3, flags=()):
    """Stamps of the persistent kernel's last launch: per CTA [units, events]
    and the observers' [2, 1024] rows (step commits completed, loads landed)."""
    L = load_trace_lib(flags)
    L.fmha_debug_set_pers_trace.restype = ctypes.c_int
    L.fmha_debug_set_pers_trace.argtypes = [ctypes.c_void_p]
    L.fmha_debug_set_pers_obs_trace.restype = ctypes.c_int
    L.fmha_debug_set_pers_obs_trace.argtypes = [ctypes.c_void_p]
    dev = torch.device("cuda:0")
    inp = wl.make_inputs(w, seed=0)
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    cq = None if inp.cu_seqlens_q is None else inp.cu_seqlens_q.to(dev)
    ck = None if inp.cu_seqlens_k is None else inp.cu_seqlens_k.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.heads, w.total_q), dtype=torch.float32, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    buf = torch.zeros((sms, PERS_UNITS, PERS_EVENTS), dtype=torch.int64, device=dev)
    obs = torch.zeros((sms, 2, 1024), dtype=torch.int64, device=dev)
    for _ in range(repeats):
        buf.zero_()
        obs.zero_()
        L.fmha_debug_set_pers_trace(ctypes.c_void_p(buf.data_ptr()))
        L.fmha_debug_set_pers_obs_trace(ctypes.c_void_p(obs.data_ptr()))
        rc = L.fmha_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                        None if cq is None else cq.data_ptr(), None if ck is None else ck.data_ptr(),
                        w.batch, w.total_q, w.total_k, w.max_seqlen_q, w.max_seqlen_k, w.heads, w.head_dim,
                        w.softmax_scale, int(w.causal), None)
        if rc != 0:
            raise RuntimeError(f"fmha_fwd returned {rc}")
        torch.cuda.synchronize()
    L.fmha_debug_set_pers_trace(None)
    L.fmha_debug_set_pers_obs_trace(None)
    return buf.cpu().numpy(), obs.cpu().numpy()


def summarize_persistent(a: np.ndarray, ob: np.ndarray) -> dict:
    """Per-unit cycles by key blocks, and the boundary between consecutive
    units of a CTA relative to the previous unit's last step commit (issue)."""
    med = lambda v: float(np.median(v)) if len(v) else None  # noqa: E731
    cta = a[:, PERS_UNITS - 1, :]
    live = cta[cta[:, 0] != 0]
    g0 = live[:, 0].min()
    res = {"ctas": int(len(live)),
           "cta_end_ns_min_med_max": [int(x) for x in np.percentile(live[:, 1] - g0, [0, 50, 100])],
           "sm_clock_mhz_median": med((live[:, 3] - live[:, 2]) / (live[:, 1] - live[:, 0]) * 1e3)}
    dur, gaps, per_cta = {}, [], []
    bd = {k: [] for k in ("published", "q0_issued", "k0_issued", "q1_issued", "unit_taken", "k0_seen", "q0_seen",
                          "q1_seen", "qk1_issued", "first_commit")}
    ev = {"published": 8, "q0_issued": 9, "k0_issued": 10, "q1_issued": 11, "unit_taken": 1, "k0_seen": 12,
          "q0_seen": 13, "q1_seen": 14, "qk1_issued": 15, "first_commit": 2}
    bo = {k: [] for k in ("prev_commit_n-1_done", "prev_last_commit_done", "first_commit_done", "k0_landed",
                          "v0_landed")}
    for c in range(a.shape[0]):
        rows = [r for r in a[c][:PERS_UNITS - 1] if r[1] != 0]
        per_cta.append(len(rows))
        cn = ld = 0
        for i, r in enumerate(rows):
            n = int(r[7])
            if r[2] and r[3]:
                dur.setdefault(n, []).append(int(r[3] - r[2]))
            if i + 1 < len(rows) and r[3] and n > 0 and int(rows[i + 1][7]) > 0:
                T, nxt = int(r[3]), rows[i + 1]
                if nxt[2]:
                    gaps.append(int(nxt[2]) - T)
                for k_, e in ev.items():
                    if nxt[e]:
                        bd[k_].append(int(nxt[e]) - T)
                st, lo = ob[c, 0], ob[c, 1]
                if cn + n < 1024 and st[cn + n]:
                    bo["prev_last_commit_done"].append(int(st[cn + n]) - T)
                if cn + n - 1 < 1024 and st[cn + n - 1]:
                    bo["prev_commit_n-1_done"].append(int(st[cn + n - 1]) - T)
                if cn + n + 1 < 1024 and st[cn + n + 1]:
                    bo["first_commit_done"].append(int(st[cn + n + 1]) - T)
                g = ld + 2 * n
                if g + 1 < 1024 and lo[g]:
                    bo["k0_landed"].append(int(lo[g]) - T)
                if g + 1 < 1024 and lo[g + 1]:
                    bo["v0_landed"].append(int(lo[g + 1]) - T)
            cn += n + 1 if n > 0 else 0
            ld += 2 * n
    res["units_per_cta_min_med_max"] = [min(per_cta), med(per_cta), max(per_cta)]
    res["unit_cycles_by_key_blocks"] = {int(k_): {"units": len(v_), "cycles": med(v_), "per_block": round(med(v_) / k_, 1)}
                                        for k_, v_ in sorted(dur.items()) if k_ > 0}
    res["boundary_gap_cycles"] = med(gaps)
    res["boundary_rel_prev_last_commit"] = {k_: med(v_) for k_, v_ in bd.items()}
    res["observers_rel_prev_last_commit"] = {k_: med(v_) for k_, v_ in bo.items()}
    return res


def run_backward(w: wl.Workload, repeats: int = 3, flags=()):
    """Stamps of the backward kernels' last launch: ([query blocks, 1024],
    [key blocks, 1024]) for the dQ and dK/dV kernels."""
    from . import binding

    load_trace_lib(flags)
    L = binding.open_library(TRACE_LIB)  # with the C ABI's argument types
    L.fmha_debug_set_bwd_trace.restype = ctypes.c_int
    L.fmha_debug_set_bwd_trace.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    dev = torch.device("cuda:0")
    inp = wl.make_inputs(w, seed=0)
    dout = wl.make_dout(w, seed=0)
    q, k, v, g = (t.to(dev) for t in (inp.q, inp.k, inp.v, dout))
    cq = None if inp.cu_seqlens_q is None else inp.cu_seqlens_q.to(dev)
    ck = None if inp.cu_seqlens_k is None else inp.cu_seqlens_k.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.heads, w.total_q), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(binding.fmha_bwd_workspace_size(w.heads, w.total_q) // 4, dtype=torch.float32, device=dev)
    tq = torch.zeros(((w.max_seqlen_q + 127) // 128, 1024), dtype=torch.int64, device=dev)
    tk = torch.zeros(((w.max_seqlen_k + 127) // 128, 1024), dtype=torch.int64, device=dev)
    st = torch.cuda.current_stream()
    rc = binding.fmha_fwd_gqa(q, k, v, out, lse, cq, ck, w.batch, w.total_q, w.total_k, w.max_seqlen_q,
                              w.max_seqlen_k, w.heads, w.n_kv_heads, w.head_dim, w.softmax_scale, int(w.causal), st,
                              library=L)
    if rc != 0:
        raise RuntimeError(f"fmha_fwd_gqa returned {rc}")
    for _ in range(repeats):
        L.fmha_debug_set_bwd_trace(ctypes.c_void_p(tq.data_ptr()), ctypes.c_void_p(tk.data_ptr()))
        rc = binding.fmha_bwd(q, k, v, out, g, lse, dq, dk, dv, ws, cq, ck, w.batch, w.total_q, w.total_k,
                              w.max_seqlen_q, w.max_seqlen_k, w.heads, w.n_kv_heads, w.head_dim, w.softmax_scale,
                              int(w.causal), st, library=L)
        if rc != 0:
            raise RuntimeError(f"fmha_bwd returned {rc}")
        torch.cuda.synchronize()
    L.fmha_debug_set_bwd_trace(None, None)
    return tq.cpu().numpy(), tk.cpu().numpy()


def summarize_backward(a: np.ndarray, bk: np.ndarray) -> dict:
    """Medians over steady-state blocks (the 3rd to the 3rd-last of each CTA), SM cycles.

    dQ kernel, per key block j (slots 8 j + e): 0 S and dP ready for the
    gradient warps, 1 dP read and released to the dP issuer, 2 dS stored,
    3 the dP issuer saw that release, 4 the S/dQ issuer saw dS, 5 the S/dQ
    issuer, after issuing dQ(j), saw K of block j + 2, 6 the dP issuer saw V
    of block j + 1.  dK/dV kernel, per query block
    (item) it: 0 stage ready, 1 / 3 half 0 / 1 scores ready, 2 / 4 half 0 / 1
    P stored, 5 / 6 dV issuer saw half 0 / 1, 7 producer passed the stage's
    release; set-up at 1000 (entry) and 1001 (roles start)."""
    med = lambda v: float(np.median(v)) if len(v) else None  # noqa: E731
    d = {k: [] for k in ("period", "math", "wait_between_blocks", "dp_release_seen", "ds_seen", "setup")}
    for row in a:
        if row[1000] == 0:
            continue
        d["setup"].append(row[1001] - row[1000])
        n = 0
        while n < 64 and row[8 * n] != 0:
            n += 1
        for j in range(2, n - 2):
            s0, s1, s2, s3, s4 = (int(row[8 * j + e]) for e in range(5))
            d["period"].append(int(row[8 * (j + 1)]) - s0)
            d["math"].append(s2 - s0)
            d["wait_between_blocks"].append(int(row[8 * (j + 1)]) - s2)
            d["dp_release_seen"].append(s3 - s1)
            d["ds_seen"].append(s4 - s2)
    res = {"dq": {k: med(v) for k, v in d.items()}}
    d = {k: [] for k in ("period", "math_h0", "math_h1", "wait_h0", "wait_h1", "p0_seen", "p1_seen", "setup")}
    for row in bk:
        if row[1000] == 0:
            continue
        d["setup"].append(row[1001] - row[1000])
        n = 0
        while n < 64 and row[8 * n] != 0:
            n += 1
        for it in range(2, n - 2):
            e = [int(row[8 * it + x]) for x in range(8)]
            d["period"].append(int(row[8 * (it + 1) + 1]) - e[1])
            d["math_h0"].append(e[2] - e[1])
            d["math_h1"].append(e[4] - e[3])
            d["wait_h0"].append(int(row[8 * (it + 1) + 1]) - e[4])
            d["wait_h1"].append(e[3] - e[2])
            d["p0_seen"].append(e[5] - e[2])
            d["p1_seen"].append(e[6] - e[4])
    res["dkdv"] = {k: med(v) for k, v in d.items()}
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default=wl.C2.name, choices=sorted({**wl.CONFIGS, **wl.EXTRA}))
    ap.add_argument("--row", type=int, default=0, help="query block (256 rows) of head 0 to show")
    ap.add_argument("--raw", default=None, help="save the raw stamps (.npy)")
    ap.add_argument("--flags", default="", help="extra -D flags for the trace build (tuning variants)")
    ap.add_argument("--no-flush", action="store_true", help="skip the L2 flush before each launch")
    ap.add_argument("--persistent", action="store_true", help="trace the persistent variant")
    ap.add_argument("--backward", action="store_true", help="trace the backward pass's dQ and dK/dV kernels")
    args = ap.parse_args()
    w = {**wl.CONFIGS, **wl.EXTRA}[args.workload]
    if args.backward:
        a, bk = run_backward(w, flags=args.flags.split())
        print(json.dumps({"workload": w.name, "flags": args.flags, "backward": summarize_backward(a, bk)}, indent=1))
        return
    if args.persistent:
        a, ob = run_persistent(w, flags=args.flags.split())
        print(json.dumps({"workload": w.name, "flags": args.flags, "persistent": summarize_persistent(a, ob)}, indent=1))
        return
    stamps, ctas = run(w, flags=["-DFMHA_PERSISTENT_WAVES=1000000", *args.flags.split()], flush_l2=not args.no_flush)
    if args.raw:
        np.save(args.raw, stamps)
        np.save(args.raw.replace(".npy", "") + "_ctas.npy", ctas)
    print(json.dumps({"workload": w.name, "flags": args.flags,
                      "cycles_per_kv_step_median": summarize(stamps[args.row]),
                      "cta_times": summarize_ctas(ctas),
                      "kernel_event_ns": run.last_event_ns, "l2_flushed": not args.no_flush}, indent=1))


if __name__ == "__main__":
    main()
