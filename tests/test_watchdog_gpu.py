"""Bounded waits on the GPU: a wait that can never complete ends in an error
status the host reads, not in a hang or a trap, and the context stays usable.

A test-only build of the kernel (-DFMHA_TEST_DROP_STEP_COMMIT) never makes the
first step commit, so the softmax of tile 1 and the TMA producer wait on a
barrier phase that nothing completes.  With the per-wait limit lowered to
200 ms the launch must return within seconds, `fmha_get_device_status` must
report FMHA_ERR_TIMEOUT with a decodable (role, barrier) detail, the status
word must be cleared by that read, and the production library must then
compute a correct result in the same process.
"""
import ctypes
import os
import time

import numpy as np
import pytest
import torch

import oracle
from attention_forward_mbarrier_gb300 import binding
from attention_forward_mbarrier_gb300 import build as _build
from attention_forward_mbarrier_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

HOOK_LIB = os.path.join(_build.PKG, "libfmha_testhook.so")
ROLES = {1: "softmax", 2: "correction", 3: "load", 4: "mma", 5: "drain"}


@pytest.fixture(scope="module")
def hook_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build(force=True, extra_flags=["-DFMHA_TEST_DROP_STEP_COMMIT=1", "-DFMHA_WAIT_LIMIT_NS=200000000ull"],
                 out=HOOK_LIB)
    L = ctypes.CDLL(HOOK_LIB)
    L.fmha_fwd.restype = ctypes.c_int
    L.fmha_fwd.argtypes = ([ctypes.c_void_p] * 7 + [ctypes.c_int] * 7 + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p])
    L.fmha_get_device_status.restype = ctypes.c_int
    L.fmha_get_device_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
    return L


def test_expired_wait_reports_timeout_and_context_survives(hook_lib):
    w = wl.dense("watchdog_dense_b1_h2_s512", 1, 512, 2)
    inp = wl.make_inputs(w, seed=7)
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    out = torch.zeros_like(q)
    lse = torch.zeros((w.heads, w.total_q), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream

    t0 = time.perf_counter()
    st = hook_lib.fmha_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), None, None,
                           w.batch, w.total_q, w.total_k, w.max_seqlen_q, w.max_seqlen_k, w.heads, w.head_dim,
                           w.softmax_scale, 0, stream)
    assert st == binding.FMHA_OK
    detail = ctypes.c_int(-1)
    st = hook_lib.fmha_get_device_status(stream, ctypes.byref(detail))
    elapsed = time.perf_counter() - t0
    assert st == binding.FMHA_ERR_TIMEOUT, binding.status_string(st)
    role, barrier = divmod(detail.value, 256)
    assert role in ROLES and 0 <= barrier < 16, detail.value
    assert elapsed < 20.0, elapsed
    # the read cleared the word
    st = hook_lib.fmha_get_device_status(stream, ctypes.byref(detail))
    assert st == binding.FMHA_OK and detail.value == 0

    # the context is still usable: the production library computes correctly
    _build.build()
    out2 = torch.empty_like(q)
    lse2 = torch.empty_like(lse)
    st = binding.fmha_fwd(q, k, v, out2, lse2, None, None, w.batch, w.total_q, w.total_k, w.max_seqlen_q,
                          w.max_seqlen_k, w.heads, w.head_dim, w.softmax_scale, 0, torch.cuda.current_stream())
    assert st == binding.FMHA_OK
    torch.cuda.synchronize()
    st, d = binding.fmha_get_device_status()
    assert st == binding.FMHA_OK, (st, d)
    o_ref, lse_ref = oracle.oracle_fwd(*inp.oracle_args())
    o = out2.float().cpu().numpy().astype(np.float64)
    assert np.abs(o - o_ref).max() <= 2e-2
    assert np.abs(lse2.cpu().numpy() - lse_ref).max() <= 1e-3
