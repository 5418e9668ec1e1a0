"""GPU parity of the backward pass (fmha_bwd, through the C ABI) against the
fp64 backward oracle.

The GPU forward (fmha_fwd) produces O and LSE, then fmha_bwd the gradients;
the oracle recomputes everything from q, k, v and dO alone.

Tolerance, per gradient tensor: relative RMS ||d - d_ref|| / ||d_ref|| <=
1e-2 and max |d - d_ref| <= 2e-2 * max |d_ref|.  Derived from the kernel's
arithmetic: P and dS are rounded to bf16 for the tensor-core products (and
D uses the bf16 output O), with fp32 accumulation and bf16 outputs; a float64
emulation of exactly that arithmetic lands at relative RMS 2.4e-3 (4.5e-3
for a sharp softmax) and max error 6e-3 of the largest entry on these
shapes, so the bounds keep a margin of 2-3x.

Small shapes and the dense h16 s2225 and varlen causal 8192-token workloads
are compared in full; the two 32768-token workloads on seeded query rows
(dQ) and keys (dK, dV) plus sum rules checked over every sequence and head
(sum_j dV_j = sum_i dO_i, sum_j dK_j = 0).  Outputs start as NaN canaries:
every row of every sequence must be written.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_mbarrier_gb300 import binding
from attention_forward_mbarrier_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

REL_RMS = 1e-2
MAX_REL = 2e-2


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


def run_fwd_bwd(inp, dO, library=None):
    """GPU forward then backward; returns (dq, dk, dv) on the device."""
    w = inp.workload
    dev = torch.device("cuda:0")
    q, k, v, g = (t.to(dev) for t in (inp.q, inp.k, inp.v, dO))
    cq = None if inp.cu_seqlens_q is None else inp.cu_seqlens_q.to(dev)
    ck = None if inp.cu_seqlens_k is None else inp.cu_seqlens_k.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.heads, w.total_q), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    st = binding.fmha_fwd_gqa(q, k, v, out, lse, cq, ck, w.batch, w.total_q, w.total_k, w.max_seqlen_q,
                              w.max_seqlen_k, w.heads, w.n_kv_heads, w.head_dim, w.softmax_scale,
                              int(w.causal), stream)
    assert st == binding.FMHA_OK, binding.status_string(st)
    nan = float("nan")
    dq = torch.full_like(q, nan)
    dk = torch.full_like(k, nan)
    dv = torch.full_like(v, nan)
    ws = torch.empty(binding.fmha_bwd_workspace_size(w.heads, w.total_q) // 4 or 1, dtype=torch.float32,
                     device=dev)
    st = binding.fmha_bwd(q, k, v, out, g, lse, dq, dk, dv, ws, cq, ck, w.batch, w.total_q, w.total_k,
                          w.max_seqlen_q, w.max_seqlen_k, w.heads, w.n_kv_heads, w.head_dim, w.softmax_scale,
                          int(w.causal), stream, library=library)
    assert st == binding.FMHA_OK, binding.status_string(st)
    torch.cuda.synchronize()
    return dq, dk, dv


def covered(cu, total, dev):
    m = torch.zeros(total, dtype=torch.bool, device=dev)
    for b in range(len(cu) - 1):
        m[int(cu[b]):int(cu[b + 1])] = True
    return m


def assert_all_written(w, dq, dk, dv):
    cq, ck = w.cu_seqlens()
    mq, mk = covered(cq, w.total_q, dq.device), covered(ck, w.total_k, dk.device)
    for name, t, m in (("dq", dq, mq), ("dk", dk, mk), ("dv", dv, mk)):
        n = int(torch.isnan(t[m]).sum())
        assert n == 0, f"{n} {name} elements never written"


def compare_grad(got, ref, name):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{name}: non-finite"
    err = np.abs(got - ref)
    top = float(np.abs(ref).max()) if ref.size else 0.0
    if top == 0.0:
        assert float(np.abs(got).max()) <= 1e-6, f"{name}: expected zeros"
        return 0.0, 0.0
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    mx = float(err.max()) / top
    assert rel <= REL_RMS, f"{name}: rel-rms {rel:.3e}"
    assert mx <= MAX_REL, f"{name}: max-abs / max|ref| {mx:.3e}"
    return rel, mx


def check_full(inp, dO):
    w = inp.workload
    dq, dk, dv = run_fwd_bwd(inp, dO)
    assert_all_written(w, dq, dk, dv)
    rq, rk, rv = oracle.oracle_bwd(inp.q, inp.k, inp.v, dO, *inp.oracle_args()[3:])
    cq, ck = w.cu_seqlens()
    mq = covered(cq, w.total_q, "cpu").numpy()
    mk = covered(ck, w.total_k, "cpu").numpy()
    compare_grad(dq.float().cpu().numpy()[mq], rq[mq], "dq")
    compare_grad(dk.float().cpu().numpy()[mk], rk[mk], "dk")
    compare_grad(dv.float().cpu().numpy()[mk], rv[mk], "dv")


CASES = [
    wl.varlen("bwd_ragged_causal", (1, 127, 128, 129, 255, 256, 257, 383), 2, causal=True),
    wl.varlen("bwd_ragged_noncausal", (1, 127, 128, 129, 255, 256, 257, 383), 2, causal=False),
    wl.varlen("bwd_lq_gt_lk_causal", (300, 200, 5), 2, causal=True, seqlens_k=(100, 450, 1)),
    wl.varlen("bwd_lq_lt_lk_noncausal", (70, 260), 3, causal=False, seqlens_k=(500, 33)),
    wl.varlen("bwd_empty_docs", (0, 130, 0, 40), 1, causal=True, seqlens_k=(0, 130, 7, 40)),
    wl.dense("bwd_dense_b2_causal_s513", 2, 513, 2, causal=True),
    wl.varlen("bwd_gqa_h8_kv2", (1, 129, 300, 513), 8, causal=True, kv_heads=2),
    wl.varlen("bwd_mqa_noncausal", (200, 77), 6, causal=False, seqlens_k=(260, 31), kv_heads=1),
    wl.varlen("bwd_sharp", (700, 300), 2, causal=True, scale=0.5),
    wl.varlen("bwd_scale0", (300, 129), 2, causal=True, scale=0.0),
    wl.varlen("bwd_negative_scale", (300, 129), 2, causal=False, scale=-0.2),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_backward_edge_shapes_full(w):
    check_full(wl.make_inputs(w, seed=51), wl.make_dout(w, seed=51))


@pytest.mark.parametrize("w", [wl.C1, wl.C2, wl.C3], ids=lambda w: w.name)
def test_backward_workloads_full(w):
    check_full(wl.make_inputs(w, seed=0), wl.make_dout(w, seed=0))


def sum_rules(w, dO, dk, dv):
    """Over every sequence and K/V head: sum_j dV_j = sum of dO over the group's
    rows that see a key, and sum_j dK_j = 0 (up to the kernel's rounding)."""
    cq, ck = w.cu_seqlens()
    grp = w.heads // w.n_kv_heads
    g = dO.to(dk.device).float()
    for b in range(w.batch):
        q0, q1, k0, k1 = (int(x) for x in (cq[b], cq[b + 1], ck[b], ck[b + 1]))
        lq, lk = q1 - q0, k1 - k0
        if lk == 0:
            continue
        first = max(0, lq - lk) if w.causal else 0  # rows before it see no key
        gs = g[q0 + first:q1].reshape(lq - first, w.n_kv_heads, grp, -1).sum(dim=(0, 2))
        vs = dv[k0:k1].float().sum(0)
        ks = dk[k0:k1].float().sum(0)
        scale_v = float(dv[k0:k1].float().abs().sum(0).max())
        scale_k = float(dk[k0:k1].float().abs().sum(0).max())
        assert float((vs - gs).abs().max()) <= 2e-2 * scale_v, "sum of dV"
        assert float(ks.abs().max()) <= 2e-2 * scale_k, "sum of dK"


@pytest.mark.parametrize("w,key_heads", [(wl.C4, (0, 31)), (wl.C5, (7,))], ids=lambda x: getattr(x, "name", ""))
def test_backward_large_workloads_sampled(w, key_heads):
    inp = wl.make_inputs(w, seed=0)
    dO = wl.make_dout(w, seed=0)
    dq, dk, dv = run_fwd_bwd(inp, dO)
    assert_all_written(w, dq, dk, dv)
    sum_rules(w, dO, dk, dv)
    rows = wl.sample_rows(w, n_random=384, seed=1)
    keys = wl.sample_keys(w, n_random=384, seed=2)
    keys = keys[np.isin(keys % w.n_kv_heads, key_heads)]  # keys of a few heads: their rows' statistics
    rq, rk, rv = oracle.oracle_bwd(inp.q, inp.k, inp.v, dO, *inp.oracle_args()[3:], rows=rows, keys=keys)
    compare_grad(dq.reshape(-1, w.head_dim)[torch.from_numpy(rows).cuda()].float().cpu().numpy(), rq, "dq")
    kt = torch.from_numpy(keys).cuda()
    compare_grad(dk.reshape(-1, w.head_dim)[kt].float().cpu().numpy(), rk, "dk")
    compare_grad(dv.reshape(-1, w.head_dim)[kt].float().cpu().numpy(), rv, "dv")


def test_backward_deterministic():
    # every output row is written by exactly one CTA (no atomics): repeats agree bitwise
    w = wl.varlen("bwd_repeat", (1000, 555), 4, causal=True, kv_heads=2)
    inp, dO = wl.make_inputs(w, seed=52), wl.make_dout(w, seed=52)
    first = run_fwd_bwd(inp, dO)
    for _ in range(4):
        again = run_fwd_bwd(inp, dO)
        assert all(torch.equal(a, b) for a, b in zip(first, again))


def test_backward_cuda_graph_and_no_fork():
    # The call forks the dK/dV kernel onto a second stream of the library's and
    # joins it back before returning: a CUDA graph captured from the caller's
    # stream replays all three kernels (inputs overwritten in place between
    # replays), and the results equal those of a build that runs every kernel
    # on the caller's stream (-DFMHA_BWD_FORK=0).
    import os

    from attention_forward_mbarrier_gb300 import build as _build

    w = wl.varlen("bwd_graph", (700, 300, 129), 4, causal=True, kv_heads=2)
    first, second = (wl.make_inputs(w, seed=s) for s in (53, 54))
    douts = [wl.make_dout(w, seed=s) for s in (53, 54)]
    dev = torch.device("cuda:0")
    q, k, v, g = (t.to(dev) for t in (first.q, first.k, first.v, douts[0]))
    cu = first.cu_seqlens_q.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.heads, w.total_q), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(binding.fmha_bwd_workspace_size(w.heads, w.total_q) // 4, dtype=torch.float32, device=dev)

    def call(stream, library=None):
        assert binding.fmha_fwd_gqa(q, k, v, out, lse, cu, cu, w.batch, w.total_q, w.total_k, w.max_seqlen_q,
                                    w.max_seqlen_k, w.heads, w.n_kv_heads, w.head_dim, w.softmax_scale, 1,
                                    stream, library=library) == binding.FMHA_OK
        assert binding.fmha_bwd(q, k, v, out, g, lse, dq, dk, dv, ws, cu, cu, w.batch, w.total_q, w.total_k,
                                w.max_seqlen_q, w.max_seqlen_k, w.heads, w.n_kv_heads, w.head_dim,
                                w.softmax_scale, 1, stream, library=library) == binding.FMHA_OK

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # first calls outside the capture (per-process set-up)
        call(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(torch.cuda.current_stream())
    path = os.path.join(_build.PKG, "libfmha_nofork.so")
    _build.build(force=True, extra_flags=["-DFMHA_BWD_FORK=0"], out=path)
    serial = binding.open_library(path)
    for inp, dO in zip((first, second), douts):
        q.copy_(inp.q.to(dev))
        k.copy_(inp.k.to(dev))
        v.copy_(inp.v.to(dev))
        g.copy_(dO.to(dev))
        for t in (dq, dk, dv):
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        got = (dq.clone(), dk.clone(), dv.clone())
        call(torch.cuda.current_stream(), library=serial)
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(got, (dq, dk, dv)))
        rq, rk, rv = oracle.oracle_bwd(inp.q, inp.k, inp.v, dO, *inp.oracle_args()[3:])
        compare_grad(got[0].float().cpu().numpy(), rq, "dq")
        compare_grad(got[1].float().cpu().numpy(), rk, "dk")
        compare_grad(got[2].float().cpu().numpy(), rv, "dv")
    st, detail = binding.fmha_get_device_status(library=serial)
    assert st == binding.FMHA_OK, (st, detail)
