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
    L.fmha_microbench_tmem_ld.restype = ctypes.c_int
    L.fmha_microbench_tmem_ld.argtypes = [ctypes.c_int, P, ctypes.c_int]
    return L


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
    _median(L.fmha_microbench_tmem_ld, 16, n_ctas=sms)
    cyc = _median(L.fmha_microbench_tmem_ld, reps, n_ctas=sms)
    out["tmem_ld_bytes_per_clk_per_sm"] = reps * 4 * 32 * 32 * 4 / cyc
    print(json.dumps(out, indent=1))


if __name__ == "__main__":
    main()
