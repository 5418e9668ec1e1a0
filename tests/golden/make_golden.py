"""Write the stored oracle fixtures in this folder.

Calls only ``oracle/`` (and the seeded input generator).  The pages print no
worked numeric example, so the fixtures here are saved inputs with the
oracle's outputs, kept so that a later change of the oracle's arithmetic shows
up as a diff (the "save inputs, compare against saved outputs" discipline of
"Kernel Bottleneck Tuning", section "Validation discipline (every change)").

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from attention_forward_mbarrier_gb300 import workloads as wl  # noqa: E402


def bits_hex(t) -> str:
    b = t.contiguous().view(__import__("torch").int16).numpy().view(np.uint16).ravel()
    return "".join(f"{x:04x}" for x in b)


def main():
    w = wl.varlen("golden_tiny", (5, 3), 1, head_dim=128, causal=True, seqlens_k=(5, 4))
    inp = wl.make_inputs(w, seed=2024)
    out, lse = oracle.oracle_fwd(*inp.oracle_args())
    fixture = {
        "about": "oracle outputs for saved seeded inputs; written by make_golden.py",
        "seqlens_q": list(w.seqlens_q), "seqlens_k": list(w.seqlens_k),
        "heads": w.heads, "head_dim": w.head_dim, "causal": w.causal, "scale": w.softmax_scale,
        "q_bf16_hex": bits_hex(inp.q), "k_bf16_hex": bits_hex(inp.k), "v_bf16_hex": bits_hex(inp.v),
        "out": [repr(float(x)) for x in out.ravel()],
        "lse": [repr(float(x)) for x in lse.ravel()],
    }
    with open(os.path.join(HERE, "oracle_tiny_d128.json"), "w") as f:
        json.dump(fixture, f, indent=0)

    # backward pass: the same kind of case with grouped K/V heads and an upstream gradient
    w = wl.varlen("golden_bwd_tiny", (5, 3), 2, head_dim=32, causal=True, seqlens_k=(5, 4), kv_heads=1)
    inp = wl.make_inputs(w, seed=2025)
    dout = wl.make_dout(w, seed=2025)
    dq, dk, dv = oracle.oracle_bwd(inp.q, inp.k, inp.v, dout, *inp.oracle_args()[3:])
    fixture = {
        "about": "backward-oracle outputs for saved seeded inputs; written by make_golden.py",
        "seqlens_q": list(w.seqlens_q), "seqlens_k": list(w.seqlens_k),
        "heads": w.heads, "kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "causal": w.causal,
        "scale": w.softmax_scale,
        "q_bf16_hex": bits_hex(inp.q), "k_bf16_hex": bits_hex(inp.k), "v_bf16_hex": bits_hex(inp.v),
        "dout_bf16_hex": bits_hex(dout),
        "dq": [repr(float(x)) for x in dq.ravel()],
        "dk": [repr(float(x)) for x in dk.ravel()],
        "dv": [repr(float(x)) for x in dv.ravel()],
    }
    with open(os.path.join(HERE, "oracle_bwd_tiny_d32.json"), "w") as f:
        json.dump(fixture, f, indent=0)


if __name__ == "__main__":
    main()
