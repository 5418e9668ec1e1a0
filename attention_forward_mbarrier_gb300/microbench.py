"""Instruction throughput probes on the GPU (see csrc/microbench.cu).

Reports per SM per clock the ex2, bf16x2-conversion and packed-FFMA2 rates
(the quantities "Kernel Bottleneck Tuning", section "1. Measure instruction
throughputs in isolation" lists for GB300), cycles per tcgen05.mma for the
operand arrangements the attention kernel uses, and tensor-memory load
bandwidth.

  python -m attention_forward_mbarrier_gb300.microbench
"""
from __future__ import annotations

import ctypes
import json
import os
import statistics
import subprocess

from . import build as _build

LIB = os.path.join(_build.PKG, "libfmha_microbench.so")
SRC = os.path.join(_build.CSRC, "microbench.cu")


def load():
    deps = [SRC, os.path.join(_build.CSRC, "sm103_ptx.cuh")]
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(d) for d in deps):
        cmd = [_build.nvcc(), *_build.NVCC_FLAGS, "-I", _build.CSRC, "-o", LIB, SRC]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(r.stdout + r.stderr)
    L = ctypes.CDLL(LIB)
    P = ctypes.POINTER(ctypes.c_longlong)
    L.fmha_microbench_alu.restype = ctypes.c_int
    L.fmha_microbench_alu.argtypes = [ctypes.c_int, ctypes.c_int, P, ctypes.c_int]
    L.fmha_microbench_mma.restype = ctypes.c_int
    L.fmha_microbench_mma.argtypes = [ctypes.c_int] * 6 + [P, ctypes.c_int]
    L.fmha_microbench_mma_mix.restype = ctypes.c_int
    L.fmha_microbench_mma_mix.argtypes = [ctypes.c_int, ctypes.c_int, P, ctypes.c_int]
    L.fmha_microbench_boundary.restype = ctypes.c_int
    L.fmha_microbench_boundary.argtypes = [ctypes.c_int, ctypes.c_int, P, ctypes.c_int]
    L.fmha_microbench_exp_loop.restype = ctypes.c_int
    L.fmha_microbench_exp_loop.argtypes = [ctypes.c_int] * 3 + [P, ctypes.c_int]
    F = ctypes.POINTER(ctypes.c_float)
    L.fmha_probe_exp2_poly.restype = ctypes.c_int
    L.fmha_probe_exp2_poly.argtypes = [F, F, F, ctypes.c_int]
    L.fmha_microbench_empty_launch.restype = ctypes.c_int
    L.fmha_microbench_empty_launch.argtypes = [ctypes.c_int] * 3 + [ctypes.c_void_p]
    L.fmha_microbench_pingpong.restype = ctypes.c_int
    L.fmha_microbench_pingpong.argtypes = [ctypes.c_int, ctypes.c_int, P, ctypes.c_int]
    L.fmha_microbench_handoff.restype = ctypes.c_int
    L.fmha_microbench_handoff.argtypes = [ctypes.c_int] * 3 + [P, ctypes.c_int]
    L.fmha_microbench_tmem_ld.restype = ctypes.c_int
    L.fmha_microbench_tmem_ld.argtypes = [ctypes.c_int, P, ctypes.c_int]
    return L


def empty_launch_envelope(L, steps: int = 40) -> dict:
    """Median microseconds between two CUDA events around the launch of an
    empty kernel (144 CTAs of 512 threads, the dense workload's grid), after a
    write-then-read pass over 2 x 504 MiB that flushes L2 and keeps the GPU
    busy while the host enqueues, as the benchmark times its launches."""
    import torch

    dev = torch.device("cuda", 0)
    st = torch.cuda.current_stream(dev)
    scratch = torch.empty(132 << 20, dtype=torch.float32, device=dev)
    reader = torch.zeros(132 << 20, dtype=torch.float32, device=dev)
    sink = torch.empty(1, dtype=torch.float32, device=dev)
    res = {}
    for smem_kb in (0, 200):
        ms = []
        for i in range(steps + 5):
            scratch.zero_()
            sink.copy_(reader.sum().reshape(1))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            rc = L.fmha_microbench_empty_launch(144, 512, smem_kb * 1024, ctypes.c_void_p(st.cuda_stream))
            e1.record(st)
            if rc != 0:
                raise RuntimeError(f"empty launch failed with {rc}")
            torch.cuda.synchronize()
            if i >= 5:
                ms.append(e0.elapsed_time(e1))
        res[f"grid144_block512_smem{smem_kb}k"] = round(statistics.median(ms) * 1000, 2)
    return res


def exp2_poly_values(x):
    """(poly, exp2f) of the probe's FMA-pipe exp2 on a float32 numpy array."""
    import numpy as np

    x = np.ascontiguousarray(x, dtype=np.float32)
    yp, yr = np.empty_like(x), np.empty_like(x)
    F = ctypes.POINTER(ctypes.c_float)
    rc = load().fmha_probe_exp2_poly(x.ctypes.data_as(F), yp.ctypes.data_as(F), yr.ctypes.data_as(F), len(x))
    if rc != 0:
        raise RuntimeError(f"fmha_probe_exp2_poly failed with {rc}")
    return yp, yr


def _median(fn, *args, n_ctas):
    buf = (ctypes.c_longlong * n_ctas)()
    rc = fn(*args, buf, n_ctas)
    if rc != 0:
        raise RuntimeError(f"probe {fn.__name__}{args} failed with {rc}")
    return statistics.median(list(buf))


MMA_CASES = [  # (a_tmem, b_mn, n, issuers, uniform)
    (0, 0, 128, 1, 0), (0, 0, 128, 1, 1), (0, 0, 256, 1, 1), (0, 0, 256, 1, 0), (0, 0, 64, 1, 1),
    (0, 1, 128, 1, 1), (1, 0, 128, 1, 1), (1, 1, 128, 1, 1), (1, 1, 128, 1, 0),
    (0, 0, 128, 2, 1), (1, 1, 128, 2, 1), (1, 1, 128, 2, 0), (1, 1, 128, 3, 1),
]


def main():
    import torch

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    L = load()
    out = {"sms": sms}
    reps = 4096
    for which, name in ((0, "ex2"), (1, "cvt_bf16x2"), (2, "ffma2")):
        _median(L.fmha_microbench_alu, which, 64, n_ctas=sms)
        cyc = _median(L.fmha_microbench_alu, which, reps, n_ctas=sms)
        out[name + "_per_clk_per_sm"] = reps * 8 * 512 / cyc
    _median(L.fmha_microbench_alu, 4, 64, n_ctas=sms)
    cyc = _median(L.fmha_microbench_alu, 4, reps, n_ctas=sms)
    out["ex2_per_clk_per_sm_one_warp_per_subpartition"] = reps * 8 * 128 / cyc
    _median(L.fmha_microbench_alu, 3, 8, n_ctas=sms)
    cyc = _median(L.fmha_microbench_alu, 3, 256, n_ctas=sms)
    out["softmax_exp_loop_cycles_per_128_scores"] = cyc / 256
    # exp-loop variants: cycles per 128-score row (per warp slot)
    loop = {}
    for variant, name in ((0, "fma_ex2_sum_pack"), (1, "fma_ex2_sum"), (2, "ex2_sum"), (3, "fma_sum_pack"),
                          (4, "fma_ex2_sum_alu_pack"), (5, "fma_ex2_f16x2_sum_pack"),
                          (6, "ex2_f16x2_only_64_per_row"), (7, "quarter_pairs_on_fma_pipe"),
                          (8, "eighth_pairs_on_fma_pipe")):
        for threads in (128, 256):
            _median(L.fmha_microbench_exp_loop, variant, threads, 4, n_ctas=sms)
            cyc = _median(L.fmha_microbench_exp_loop, variant, threads, 64, n_ctas=sms)
            loop[f"{name}_{threads // 128}warp_per_subpartition"] = round(cyc / 64, 1)
    out["exp_loop_cycles_per_row"] = loop
    mreps = 512
    rows = []
    for a_tmem, b_mn, n, issuers, uniform in MMA_CASES:
        args = (a_tmem, b_mn, n, issuers, uniform)
        _median(L.fmha_microbench_mma, *args, 16, n_ctas=sms)
        cyc = _median(L.fmha_microbench_mma, *args, mreps, n_ctas=sms)
        per_issuer = cyc / (mreps * 8)
        rows.append({"a": "tmem" if a_tmem else "smem", "b": "mn-major" if b_mn else "k-major", "n": n,
                     "issuers": issuers, "issue": "warp-uniform" if uniform else "lane0",
                     "cycles_per_mma_per_issuer": round(per_issuer, 1),
                     "flop_per_clk_per_sm": round(issuers * 2 * 128 * n * 16 / per_issuer)})
    out["mma"] = rows
    # cycles per MMA from the slope between two run lengths (start-up and
    # drain cancel)
    mix = {}
    for mode, name, per_round in ((0, "pv_then_qk_two_tiles", 32), (1, "qk_only_two_tiles", 16),
                                  (2, "pv_only_two_tiles", 16), (3, "pv_then_qk_with_smem_writes", 32),
                                  (4, "one_tile_with_tmem_ld_st", 16), (5, "one_tile", 16),
                                  (6, "pv_then_qk_commit_every_8", 32), (7, "pv_then_qk_commit_every_mma", 32),
                                  (8, "pv_then_qk_commit_every_32", 32), (9, "qk_one_tile_commit_every_8", 8),
                                  (10, "pv_then_qk_two_tiles_random_operands", 32),
                                  (11, "qk_only_two_tiles_random_operands", 16)):
        _median(L.fmha_microbench_mma_mix, mode, 8, n_ctas=sms)
        c1 = _median(L.fmha_microbench_mma_mix, mode, 64, n_ctas=sms)
        c2 = _median(L.fmha_microbench_mma_mix, mode, 192, n_ctas=sms)
        mix[name] = {"slope": round((c2 - c1) / (128 * per_round), 1), "whole": round(c2 / (192 * per_round), 1)}
    out["mma_stream_cycles_per_mma"] = mix
    # issuing-thread cycles at a step boundary, after 16 MMAs in flight
    bnd = {}
    for mode, name in ((0, "commit_then_try_wait"), (1, "try_wait_only"), (2, "commit_only"),
                       (3, "n256_commit_then_try_wait"), (4, "n256_try_wait_only"), (5, "n256_commit_only"),
                       (6, "commit_then_try_wait_3_warps_polling_elsewhere"),
                       (7, "commit_then_try_wait_3_warps_waiting_on_the_commit"),
                       (8, "commit_then_shared_load")):
        _median(L.fmha_microbench_boundary, mode, 8, n_ctas=sms)
        bnd[name] = round(_median(L.fmha_microbench_boundary, mode, 128, n_ctas=sms) / 128, 1)
    out["step_boundary_cycles"] = bnd
    # an mbarrier hand-off between two warps (half a ping-pong round trip) and
    # a dependent shared-memory load, while the issuing warp runs MMA streams
    hand = {}
    for mode, name in ((0, "no_mma"), (1, "qk_like_ss_n128"), (2, "pv_like_ts_n128"), (3, "attention_stream")):
        _median(L.fmha_microbench_handoff, mode, 0, 16, n_ctas=sms)
        rt = _median(L.fmha_microbench_handoff, mode, 0, 256, n_ctas=sms)
        ld = _median(L.fmha_microbench_handoff, mode, 1, 2048, n_ctas=sms)
        nb = _median(L.fmha_microbench_handoff, mode, 2, 256, n_ctas=sms)
        hand[name] = {"arrive_to_seen": round(rt / 256 / 2, 1), "ld_shared": round(ld / 2048, 1),
                      "named_barrier_arrive_to_sync": round(nb / 256 / 2, 1)}
    out["handoff_cycles_under_mma_stream"] = hand
    # one issuer for both tiles' groups vs one issuer per tile passing a token
    pp = {}
    for variant, name in ((0, "one_issuer_commit_per_group"), (1, "two_issuers_commit_then_token"),
                          (2, "two_issuers_token_then_commit"), (3, "two_issuers_token_no_commit")):
        _median(L.fmha_microbench_pingpong, variant, 8, n_ctas=sms)
        c1 = _median(L.fmha_microbench_pingpong, variant, 64, n_ctas=sms)
        c2 = _median(L.fmha_microbench_pingpong, variant, 192, n_ctas=sms)
        pp[name] = round((c2 - c1) / (128 * 32), 1)
    out["alternating_issuers_cycles_per_mma"] = pp
    out["empty_launch_us"] = empty_launch_envelope(L)
    _median(L.fmha_microbench_tmem_ld, 16, n_ctas=sms)
    cyc = _median(L.fmha_microbench_tmem_ld, reps, n_ctas=sms)
    out["tmem_ld_bytes_per_clk_per_sm"] = reps * 4 * 32 * 32 * 4 / cyc
    print(json.dumps(out, indent=1))


if __name__ == "__main__":
    main()
