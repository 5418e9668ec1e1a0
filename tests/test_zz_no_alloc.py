"""fmha_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (code running where cudaMalloc is unavailable or not allowed, such as
an allocator's own hooks or a plugin whose host owns all device memory).  Its
scratch is a fixed array inside the library instead of a caller workspace.

Checked through the C ABI against fmha_bwd, the entry point that takes a
workspace, on two calls in a row: a larger problem, then a smaller one that
finds the first call's values still in the shared array.  The tolerance is
the one the backward parity tests use (relative RMS <= 1e-2, max error <=
2e-2 of the largest entry, per gradient).  A problem whose scratch would not
fit the array is refused before any GPU work.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from attention_forward_mbarrier_gb300 import binding
from attention_forward_mbarrier_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

REL_RMS = 1e-2
MAX_REL = 2e-2
MAX_SCRATCH_FLOATS = 1 << 21


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_forward_mbarrier_gb300 import build

    build.build()
    binding.lib()
    torch.cuda.set_device(0)
    yield
    st, detail = binding.fmha_get_device_status()
    assert st == binding.FMHA_OK, (st, detail)


def prepare(w, seed):
    """Device inputs, and the forward's O and LSE, for workload w."""
    dev = torch.device("cuda:0")
    inp = wl.make_inputs(w, seed=seed)
    t = dict(q=inp.q.to(dev), k=inp.k.to(dev), v=inp.v.to(dev), dout=wl.make_dout(w, seed=seed).to(dev))
    t["cq"] = None if inp.cu_seqlens_q is None else inp.cu_seqlens_q.to(dev)
    t["ck"] = None if inp.cu_seqlens_k is None else inp.cu_seqlens_k.to(dev)
    t["out"] = torch.empty_like(t["q"])
    t["lse"] = torch.empty((w.heads, w.total_q), dtype=torch.float32, device=dev)
    st = binding.fmha_fwd_gqa(t["q"], t["k"], t["v"], t["out"], t["lse"], t["cq"], t["ck"], w.batch, w.total_q,
                              w.total_k, w.max_seqlen_q, w.max_seqlen_k, w.heads, w.n_kv_heads, w.head_dim,
                              w.softmax_scale, int(w.causal), torch.cuda.current_stream())
    assert st == binding.FMHA_OK
    return t


def grads(w, t, noalloc):
    dq, dk, dv = (torch.full_like(t[x], float("nan")) for x in ("q", "k", "v"))
    common = (t["cq"], t["ck"], w.batch, w.total_q, w.total_k, w.max_seqlen_q, w.max_seqlen_k, w.heads,
              w.n_kv_heads, w.head_dim, w.softmax_scale, int(w.causal), torch.cuda.current_stream())
    if noalloc:
        st = binding.fmha_bwd_noalloc(t["q"], t["k"], t["v"], t["out"], t["dout"], t["lse"], dq, dk, dv, *common)
    else:
        ws = torch.empty(max(1, binding.fmha_bwd_workspace_size(w.heads, w.total_q) // 4), dtype=torch.float32,
                         device=t["q"].device)
        st = binding.fmha_bwd(t["q"], t["k"], t["v"], t["out"], t["dout"], t["lse"], dq, dk, dv, ws, *common)
    assert st == binding.FMHA_OK, binding.status_string(st)
    torch.cuda.synchronize()
    return dq, dk, dv


def close(got, ref, name):
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), f"{name}: non-finite"
    top = np.abs(r).max()
    rel = np.linalg.norm(g - r) / np.linalg.norm(r)
    assert rel <= REL_RMS, f"{name}: rel-rms {rel:.3e}"
    assert np.abs(g - r).max() <= MAX_REL * top, f"{name}: max error"


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    first = wl.varlen("noalloc_first", (700, 333, 1029), 4, causal=True, kv_heads=2)
    second = wl.varlen("noalloc_second", (300, 129), 2, causal=False, seqlens_k=(257, 400))
    for w, seed in ((first, 61), (second, 62)):
        t = prepare(w, seed)
        want = grads(w, t, noalloc=False)
        got = grads(w, t, noalloc=True)
        for name, a, b in zip(("dq", "dk", "dv"), got, want):
            close(a, b, name)


def test_noalloc_refuses_problem_larger_than_its_scratch():
    # heads * total_q one past the fixed array: refused on the host, no GPU work
    heads, total_q = 2, MAX_SCRATCH_FLOATS // 2 + 1
    st = binding.fmha_bwd_noalloc(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000, 0x9000,
                                  None, None, 1, total_q, total_q, total_q, total_q, heads, heads, 128,
                                  0.088, 1, None)
    assert st == binding.FMHA_ERR_UNSUPPORTED
