"""ctypes binding of libfmha.so: the C ABI of include/fmha.h, same names.

Argument marshalling only: every step of the attention forward runs in the
CUDA library.  If the library is missing this module raises; there is no CPU
fallback.  torch is used for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

FMHA_OK = 0
FMHA_ERR_INVALID_ARG = 1
FMHA_ERR_UNSUPPORTED = 2
FMHA_ERR_CUDA = 3
FMHA_ERR_TIMEOUT = 4

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfmha.so")

# exported symbols, in the order include/fmha.h declares them
SYMBOLS = ("fmha_fwd", "fmha_fwd_gqa", "fmha_fwd_fp8pv", "fmha_fwd_fp8pv_workspace_size", "fmha_bwd", "fmha_bwd_workspace_size", "fmha_bwd_noalloc",
           "fmha_get_device_status", "fmha_status_string", "fmha_version")

_lock = threading.Lock()
_lib = None


class FmhaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})" if what else status_string(status))


def open_library(path: str):
    """Load a build of the library at ``path`` and declare its C signatures."""
    L = ctypes.CDLL(path)
    L.fmha_fwd.restype = ctypes.c_int
    L.fmha_fwd.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_void_p,
    ]
    L.fmha_fwd_gqa.restype = ctypes.c_int
    L.fmha_fwd_gqa.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_void_p,
    ]
    L.fmha_fwd_fp8pv.restype = ctypes.c_int
    L.fmha_fwd_fp8pv.argtypes = [ctypes.c_void_p] * 8 + [ctypes.c_int] * 8 + [ctypes.c_float, ctypes.c_int,
                                                                               ctypes.c_void_p]
    L.fmha_fwd_fp8pv_workspace_size.restype = ctypes.c_size_t
    L.fmha_fwd_fp8pv_workspace_size.argtypes = [ctypes.c_int] * 4
    L.fmha_bwd.restype = ctypes.c_int
    L.fmha_bwd.argtypes = [ctypes.c_void_p] * 12 + [ctypes.c_int] * 8 + [ctypes.c_float, ctypes.c_int,
                                                                         ctypes.c_void_p]
    L.fmha_bwd_noalloc.restype = ctypes.c_int
    L.fmha_bwd_noalloc.argtypes = [ctypes.c_void_p] * 11 + [ctypes.c_int] * 8 + [ctypes.c_float, ctypes.c_int,
                                                                                ctypes.c_void_p]
    L.fmha_bwd_workspace_size.restype = ctypes.c_size_t
    L.fmha_bwd_workspace_size.argtypes = [ctypes.c_int, ctypes.c_int]
    L.fmha_get_device_status.restype = ctypes.c_int
    L.fmha_get_device_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
    L.fmha_status_string.restype = ctypes.c_char_p
    L.fmha_status_string.argtypes = [ctypes.c_int]
    L.fmha_version.restype = ctypes.c_int
    L.fmha_version.argtypes = []
    return L


def lib():
    """Load libfmha.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                                   "or attention_forward_mbarrier_gb300.build.build()")
            _lib = open_library(LIB_PATH)
    return _lib


def _ptr(x) -> Optional[int]:
    """A device pointer from a torch tensor, an int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def fmha_fwd(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
             max_seqlen_q, max_seqlen_k, heads, head_dim, scale, causal, stream=None, library=None) -> int:
    """The C entry point with the same arguments; tensors or raw pointers.

    Returns the status code (FMHA_OK == 0).  See include/fmha.h.  ``library``:
    a handle from ``open_library`` (another build of the library), else the
    in-tree one.
    """
    return int((library or lib()).fmha_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                              _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(batch), int(total_q),
                              int(total_k), int(max_seqlen_q), int(max_seqlen_k), int(heads),
                              int(head_dim), float(scale), int(causal), _stream(stream)))


def fmha_fwd_gqa(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                 max_seqlen_q, max_seqlen_k, heads, kv_heads, head_dim, scale, causal, stream=None,
                 library=None) -> int:
    """The grouped-K/V-head C entry point; tensors or raw pointers.  Returns the status."""
    return int((library or lib()).fmha_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                  _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(batch), int(total_q),
                                  int(total_k), int(max_seqlen_q), int(max_seqlen_k), int(heads),
                                  int(kv_heads), int(head_dim), float(scale), int(causal), _stream(stream)))


def fmha_fwd_fp8pv(q, k, v, out, lse, workspace, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                   max_seqlen_q, max_seqlen_k, heads, kv_heads, head_dim, scale, causal, stream=None,
                   library=None) -> int:
    """The FP8 (e4m3) P V forward entry point; tensors or raw pointers.  Returns the status."""
    return int((library or lib()).fmha_fwd_fp8pv(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(workspace), _ptr(cu_seqlens_q),
        _ptr(cu_seqlens_k), int(batch), int(total_q), int(total_k), int(max_seqlen_q), int(max_seqlen_k),
        int(heads), int(kv_heads), int(head_dim), float(scale), int(causal), _stream(stream)))


def fmha_fwd_fp8pv_workspace_size(batch, total_k, kv_heads, head_dim, library=None) -> int:
    """Bytes of device workspace fmha_fwd_fp8pv needs."""
    return int((library or lib()).fmha_fwd_fp8pv_workspace_size(int(batch), int(total_k), int(kv_heads),
                                                                 int(head_dim)))


def fmha_bwd(q, k, v, out, dout, lse, dq, dk, dv, workspace, cu_seqlens_q, cu_seqlens_k, batch, total_q,
             total_k, max_seqlen_q, max_seqlen_k, heads, kv_heads, head_dim, scale, causal, stream=None,
             library=None) -> int:
    """The backward-pass C entry point; tensors or raw pointers.  Returns the status."""
    return int((library or lib()).fmha_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        _ptr(workspace), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(batch), int(total_q), int(total_k),
        int(max_seqlen_q), int(max_seqlen_k), int(heads), int(kv_heads), int(head_dim), float(scale),
        int(causal), _stream(stream)))


def fmha_bwd_noalloc(q, k, v, out, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, batch, total_q,
                     total_k, max_seqlen_q, max_seqlen_k, heads, kv_heads, head_dim, scale, causal, stream=None,
                     library=None) -> int:
    """fmha_bwd for callers that cannot allocate: its scratch is a fixed array
    inside the library (heads * total_q <= 2**21).  Returns the status."""
    return int((library or lib()).fmha_bwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(batch), int(total_q), int(total_k),
        int(max_seqlen_q), int(max_seqlen_k), int(heads), int(kv_heads), int(head_dim), float(scale),
        int(causal), _stream(stream)))


def fmha_bwd_workspace_size(heads, total_q, library=None) -> int:
    """Bytes of device workspace fmha_bwd needs."""
    return int((library or lib()).fmha_bwd_workspace_size(int(heads), int(total_q)))


def fmha_get_device_status(stream=None, library=None):
    """(status, detail): synchronises the stream and reads/clears the device status word."""
    detail = ctypes.c_int(0)
    st = int((library or lib()).fmha_get_device_status(_stream(stream), ctypes.byref(detail)))
    return st, int(detail.value)


def status_string(status: int) -> str:
    return lib().fmha_status_string(int(status)).decode()


def fmha_status_string(status: int) -> str:
    return status_string(status)


def fmha_version() -> int:
    return int(lib().fmha_version())


def attention_forward(q, k, v, scale, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None,
                      max_seqlen_k=None, causal=False, out=None, lse=None,
                      return_lse=True, stream=None):
    """Convenience wrapper over ``fmha_fwd`` for CUDA torch tensors.

    q: [total_q, heads, 128] bf16 (or [b, s, heads, 128] dense); k/v likewise
    with kv_heads heads (kv_heads dividing heads: grouped K/V heads).
    scale: the softmax scale, always given (e.g. 1/sqrt(head_dim)); no
    default is applied.
    cu_seqlens_*: int32 CUDA tensors [batch + 1] or None (dense).  Allocates
    ``out`` ([total_q, heads, 128] bf16) and ``lse`` ([heads, total_q] fp32)
    with torch when not given.  Raises FmhaError on a non-OK status.
    """
    import torch

    dense4 = q.dim() == 4
    if dense4:
        b, sq, h, d = q.shape
        sk, hk = k.shape[1], k.shape[2]
        qf, kf, vf = q.reshape(b * sq, h, d), k.reshape(b * sk, hk, d), v.reshape(b * sk, hk, d)
        batch, max_seqlen_q, max_seqlen_k = b, sq, sk
        if cu_seqlens_q is not None or cu_seqlens_k is not None:
            raise ValueError("4-D dense inputs take no cu_seqlens")
    else:
        qf, kf, vf = q, k, v
        h, d = q.shape[1], q.shape[2]
        if cu_seqlens_q is None:
            batch = 1
            max_seqlen_q = q.shape[0] if max_seqlen_q is None else max_seqlen_q
            max_seqlen_k = k.shape[0] if max_seqlen_k is None else max_seqlen_k
        else:
            batch = cu_seqlens_q.numel() - 1
            if max_seqlen_q is None or max_seqlen_k is None:
                raise ValueError("varlen calls need max_seqlen_q and max_seqlen_k")
    for name, t in (("q", qf), ("k", kf), ("v", vf)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if out is None:
        out = torch.empty_like(qf)
    if lse is None and return_lse:
        lse = torch.empty((h, qf.shape[0]), dtype=torch.float32, device=qf.device)
    st = fmha_fwd_gqa(qf, kf, vf, out, lse, cu_seqlens_q, cu_seqlens_k, batch, qf.shape[0], kf.shape[0],
                      max_seqlen_q, max_seqlen_k, h, kf.shape[1], d, scale, int(bool(causal)), stream)
    if st != FMHA_OK:
        raise FmhaError(st, "fmha_fwd_gqa")
    if dense4:
        out = out.view(q.shape)
    return (out, lse) if return_lse else out
