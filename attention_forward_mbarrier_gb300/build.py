"""Build libfmha.so in-tree with nvcc for sm_103a (no cmake, one translation unit)."""
from __future__ import annotations

import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libfmha.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
    "-diag-suppress", "1160",
]


def sources() -> list:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False, extra_flags=(), out: str = LIB) -> str:
    """Compile csrc/fmha_api.cu (which includes the kernel) into ``out``."""
    if not force and os.path.exists(out):
        newest = max(os.path.getmtime(f) for f in sources())
        if os.path.getmtime(out) >= newest and not extra_flags:
            return out
    cmd = [nvcc(), *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-I", CSRC,
           "-o", out, os.path.join(CSRC, "fmha_api.cu")]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose:
        print(res.stdout + res.stderr)
    return out


def ptxas_report() -> str:
    """ptxas resource usage (registers, spills) of the kernel, from a fresh build to /tmp."""
    import tempfile

    with tempfile.TemporaryDirectory() as d:
        cmd = [nvcc(), *NVCC_FLAGS, "-Xptxas=-v", "-I", INCLUDE, "-I", CSRC,
               "-o", os.path.join(d, "libfmha_probe.so"), os.path.join(CSRC, "fmha_api.cu")]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
        return res.stdout + res.stderr


if __name__ == "__main__":
    print(build(force=True, verbose=True))
