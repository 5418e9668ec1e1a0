"""CPU oracle for the fused attention forward -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never imports, links or executes anything here, and this package
imports nothing from the product package.

Two independent implementations of the same definition live here:

* ``oracle_fwd`` -- the fp64 C oracle in ``fmha_oracle.c`` (OpenMP over rows),
  called through ctypes on numpy arrays.  It is the reference the GPU parity
  tests compare against.
* ``brute_force_fwd`` -- pure-Python float loops with ``math.exp`` and no max
  shift, for tiny shapes only.  It exists to pin the C oracle.

The definition both follow (sources: "[BUG] Unexpected Slower Performance in
C++ CuTe (77_blackwell_fmha) vs Python CuTe DSL (fmha.py) on Jetson Thor",
section "Implementation Differences in softmax_step"; "[BUG] CuTe DSL 4.7/4.8
regression: FlashAttention-4 SM100 forward kernel spills registers", section
"Steps/Code to reproduce bug"): per sequence, head and query row i,
``s_ij = scale * q_i . k_j`` over the visible keys ``j < Lk`` (and
``j <= i + Lk - Lq`` when causal), ``O_i = softmax_j(s_ij) @ V`` and
``LSE_i = log sum_j exp(s_ij)``.  A row with no visible key has O = 0 and
LSE = -inf.  Readings of points the pages leave open (LSE base, causal
alignment for Lq != Lk, empty rows) are stated in ``fmha_oracle.c``.

A third function covers the backward pass:

* ``oracle_bwd`` -- the fp64 C oracle in ``fmha_bwd_oracle.c``: the gradients
  dQ, dK, dV of L = sum dO . O, written out by the chain rule through the
  softmax (row statistics recomputed from q, k, v; nothing is taken from a
  forward run).  Full outputs, or sampled query rows / key rows.

Parity status: every function here is pinned: the forward ones by
``tests/test_oracle_pins.py`` (closed forms, a library softmax, brute force,
structural invariants and planted mistakes), the backward one by
``tests/test_oracle_bwd_pins.py`` (central finite differences of a float64
forward, closed forms at scale 0, sum rules, grouped heads against repeated
heads, sample modes against full mode, planted mistakes).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fmha_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_BWD_SRC = os.path.join(_HERE, "fmha_bwd_oracle.c")
_BWD_LIB_PATH = os.path.join(_HERE, "liboracle_bwd.so")
_lock = threading.Lock()
_lib = None
_bwd_lib = None


def _compile(src: str, out: str, force: bool) -> str:
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracles (forward, and backward when building the default
    forward library) with gcc + OpenMP into shared libraries."""
    if src == _SRC and out == _LIB_PATH:
        _compile(_BWD_SRC, _BWD_LIB_PATH, force)
    return _compile(src, out, force)


def _load(path: str = _LIB_PATH):
    lib = ctypes.CDLL(path)
    fn = lib.oracle_fmha_fwd
    fn.restype = ctypes.c_int
    fn.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,  # q k v
        ctypes.c_void_p, ctypes.c_void_p,  # out lse
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,  # cu_q cu_k batch
        ctypes.c_int64, ctypes.c_int64,  # total_q total_k
        ctypes.c_int, ctypes.c_int,  # max_seqlen_q max_seqlen_k
        ctypes.c_int, ctypes.c_int, ctypes.c_int,  # heads kv_heads head_dim
        ctypes.c_double, ctypes.c_int,  # scale causal
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,  # rows n_rows n_threads
    ]
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def load_variant(source_text: str, workdir: str):
    """Compile C source text (a variant of ``fmha_oracle.c``) and load it."""
    src = os.path.join(workdir, "variant.c")
    out = os.path.join(workdir, "libvariant.so")
    with open(src, "w") as f:
        f.write(source_text)
    build(force=True, src=src, out=out)
    return _load(out)


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def lib():
    """The loaded oracle library (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _load()
    return _lib


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def _bits(a) -> np.ndarray:
    """bf16 data as a contiguous uint16 numpy array of bit patterns.

    Accepts a numpy uint16 array or a CPU torch bfloat16 tensor.
    """
    if isinstance(a, np.ndarray):
        if a.dtype != np.uint16:
            raise TypeError("expected uint16 bf16 bit patterns")
        return np.ascontiguousarray(a)
    # torch tensor (imported lazily so the oracle does not require torch)
    import torch

    if a.dtype != torch.bfloat16:
        raise TypeError("expected a bfloat16 tensor")
    return a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, batch, max_seqlen_q, max_seqlen_k,
               scale, causal, rows=None, n_threads: int = 0, lib_handle=None):
    """fp64 attention forward from the C oracle.

    q: [total_q, heads, head_dim] bf16 (numpy uint16 bits or torch bf16),
    k, v: [total_k, kv_heads, head_dim] (kv_heads divides heads; query head h
    reads K/V head h // (heads // kv_heads)).  cu_seqlens_q / cu_seqlens_k: int32
    prefix offsets of length batch+1, or None for dense batches.
    rows: optional int64 array of flattened (token * heads + head) indices.
    lib_handle: a library from ``load_variant`` (tests build deliberately
    broken copies of the C source to show the pins catch them).
    Returns (out, lse): full mode out [total_q, heads, head_dim] and lse
    [heads, total_q]; row mode out [n_rows, head_dim] and lse [n_rows].
    """
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    if qb.ndim != 3:
        raise ValueError("q must be [tokens, heads, head_dim]")
    total_q, heads, head_dim = qb.shape
    total_k, kv_heads = kb.shape[0], kb.shape[1]
    if kb.ndim != 3 or kb.shape[2] != head_dim or vb.shape != kb.shape or heads % kv_heads != 0:
        raise ValueError("k and v must be [total_k, kv_heads, head_dim] with kv_heads dividing heads")
    if (cu_seqlens_q is None) != (cu_seqlens_k is None):
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both be given or both be None")
    cu_q = cu_k = None
    if cu_seqlens_q is not None:
        cu_q = np.ascontiguousarray(np.asarray(cu_seqlens_q, dtype=np.int32))
        cu_k = np.ascontiguousarray(np.asarray(cu_seqlens_k, dtype=np.int32))
        if cu_q.shape != (batch + 1,) or cu_k.shape != (batch + 1,):
            raise ValueError("cu_seqlens must have batch + 1 entries")
    if rows is None:
        out = np.zeros((total_q, heads, head_dim), dtype=np.float64)
        lse = np.zeros((heads, total_q), dtype=np.float64)
        rows_arr, n_rows = None, 0
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows = rows_arr.shape[0]
        out = np.zeros((n_rows, head_dim), dtype=np.float64)
        lse = np.zeros((n_rows,), dtype=np.float64)
    handle = lib() if lib_handle is None else lib_handle
    rc = handle.oracle_fmha_fwd(
        qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, out.ctypes.data, lse.ctypes.data,
        cu_q.ctypes.data if cu_q is not None else None,
        cu_k.ctypes.data if cu_k is not None else None,
        int(batch), int(total_q), int(total_k), int(max_seqlen_q), int(max_seqlen_k),
        int(heads), int(kv_heads), int(head_dim), float(scale), int(bool(causal)),
        rows_arr.ctypes.data if rows_arr is not None else None, int(n_rows), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_fmha_fwd rejected its arguments")
    return out, lse


def _bf16_bits_to_float(bits: int) -> float:
    return float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0])


def brute_force_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, batch, max_seqlen_q, max_seqlen_k,
                    scale, causal):
    """Pure-Python float loops, no max shift: exp(s) / sum exp(s) directly.

    Only for tiny shapes with small scores (no overflow).  Same argument
    conventions and return layout as ``oracle_fwd`` in full mode.
    """
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    total_q, heads, head_dim = qb.shape
    group = heads // kb.shape[1]  # query heads per K/V head
    to_f = np.vectorize(_bf16_bits_to_float, otypes=[float])
    Q, K, V = to_f(qb).tolist(), to_f(kb).tolist(), to_f(vb).tolist()
    out = [[[0.0] * head_dim for _ in range(heads)] for _ in range(total_q)]
    lse = [[0.0] * total_q for _ in range(heads)]
    for b in range(batch):
        if cu_seqlens_q is None:
            q0, lq, k0, lk = b * max_seqlen_q, max_seqlen_q, b * max_seqlen_k, max_seqlen_k
        else:
            q0, lq = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1]) - int(cu_seqlens_q[b])
            k0, lk = int(cu_seqlens_k[b]), int(cu_seqlens_k[b + 1]) - int(cu_seqlens_k[b])
        for h in range(heads):
            for i in range(lq):
                weights = []
                for j in range(lk):
                    if causal and j > i + lk - lq:
                        continue
                    dot = 0.0
                    for d in range(head_dim):
                        dot += Q[q0 + i][h][d] * K[k0 + j][h // group][d]
                    weights.append((j, math.exp(scale * dot)))
                if not weights:
                    lse[h][q0 + i] = -math.inf
                    continue
                z = sum(w for _, w in weights)
                for d in range(head_dim):
                    out[q0 + i][h][d] = sum(w * V[k0 + j][h // group][d] for j, w in weights) / z
                lse[h][q0 + i] = math.log(z)
    return np.array(out, dtype=np.float64), np.array(lse, dtype=np.float64)


# ---------------------------------------------------------------- backward pass
def _load_bwd(path: str = _BWD_LIB_PATH):
    lib = ctypes.CDLL(path)
    fn = lib.oracle_fmha_bwd
    fn.restype = ctypes.c_int
    fn.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,  # q k v dout
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,  # dq dk dv
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,  # cu_q cu_k batch
        ctypes.c_int64, ctypes.c_int64,  # total_q total_k
        ctypes.c_int, ctypes.c_int,  # max_seqlen_q max_seqlen_k
        ctypes.c_int, ctypes.c_int, ctypes.c_int,  # heads kv_heads head_dim
        ctypes.c_double, ctypes.c_int,  # scale causal
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,  # rows n_rows keys n_keys
        ctypes.c_int,  # n_threads
    ]
    return lib


def bwd_lib():
    """The loaded backward oracle library (built on first use)."""
    global _bwd_lib
    with _lock:
        if _bwd_lib is None:
            _compile(_BWD_SRC, _BWD_LIB_PATH, False)
            _bwd_lib = _load_bwd()
    return _bwd_lib


def bwd_source_text() -> str:
    with open(_BWD_SRC) as f:
        return f.read()


def load_bwd_variant(source_text: str, workdir: str):
    """Compile C source text (a variant of ``fmha_bwd_oracle.c``) and load it."""
    src = os.path.join(workdir, "bwd_variant.c")
    out = os.path.join(workdir, "libbwd_variant.so")
    with open(src, "w") as f:
        f.write(source_text)
    _compile(src, out, True)
    return _load_bwd(out)


def oracle_bwd(q, k, v, dout, cu_seqlens_q, cu_seqlens_k, batch, max_seqlen_q, max_seqlen_k,
               scale, causal, rows=None, keys=None, want_dq=True, want_dkdv=True,
               n_threads: int = 0, lib_handle=None):
    """fp64 gradients (dq, dk, dv) of L = sum(dout * O) from the C backward oracle.

    q, dout: [total_q, heads, head_dim] bf16 (numpy uint16 bits or torch bf16);
    k, v: [total_k, kv_heads, head_dim].  Other arguments as ``oracle_fwd``.
    rows: optional flattened query indices (token * heads + head) -> dq is
    [n_rows, head_dim]; keys: optional flattened key indices
    (token * kv_heads + kv_head) -> dk, dv are [n_keys, head_dim].  Parts not
    wanted come back as None.
    """
    qb, kb, vb, gb = _bits(q), _bits(k), _bits(v), _bits(dout)
    total_q, heads, head_dim = qb.shape
    total_k, kv_heads = kb.shape[0], kb.shape[1]
    if gb.shape != qb.shape or kb.shape[2] != head_dim or vb.shape != kb.shape or heads % kv_heads:
        raise ValueError("inconsistent shapes")
    if (cu_seqlens_q is None) != (cu_seqlens_k is None):
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both be given or both be None")
    cu_q = cu_k = None
    if cu_seqlens_q is not None:
        cu_q = np.ascontiguousarray(np.asarray(cu_seqlens_q, dtype=np.int32))
        cu_k = np.ascontiguousarray(np.asarray(cu_seqlens_k, dtype=np.int32))
    rows_arr = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    keys_arr = None if keys is None else np.ascontiguousarray(np.asarray(keys, dtype=np.int64))
    dq = dk = dv = None
    if want_dq:
        dq = np.zeros((total_q, heads, head_dim) if rows_arr is None else (len(rows_arr), head_dim))
    if want_dkdv:
        shp = (total_k, kv_heads, head_dim) if keys_arr is None else (len(keys_arr), head_dim)
        dk, dv = np.zeros(shp), np.zeros(shp)
    handle = bwd_lib() if lib_handle is None else lib_handle

    def ptr(a):
        return None if a is None else a.ctypes.data

    rc = handle.oracle_fmha_bwd(
        ptr(qb), ptr(kb), ptr(vb), ptr(gb), ptr(dq), ptr(dk), ptr(dv), ptr(cu_q), ptr(cu_k),
        int(batch), int(total_q), int(total_k), int(max_seqlen_q), int(max_seqlen_k),
        int(heads), int(kv_heads), int(head_dim), float(scale), int(bool(causal)),
        ptr(rows_arr), 0 if rows_arr is None else len(rows_arr),
        ptr(keys_arr), 0 if keys_arr is None else len(keys_arr), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_fmha_bwd rejected its arguments")
    return dq, dk, dv
