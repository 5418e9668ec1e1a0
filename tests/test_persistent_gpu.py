"""The persistent forward kernel, checked on every row.

The library runs the forward as a persistent kernel (resident CTAs that take
work units from a counter in global memory and overlap consecutive units)
when the plain grid would take more than one wave of CTAs (one CTA per SM).
A test build (-DFMHA_PERSISTENT_WAVES=0 -DFMHA_PERSISTENT_MAX_CTAS=3) takes
that path on every launch with at most 3 CTAs, so that problems small enough
for a full oracle compare run many units per CTA: units whose tiles have no
key blocks, sequences shorter than a tile, empty sequences, Lq != Lk, dense
and varlen, causal and not, head_dim 64 and grouped K/V heads.  Each result
must match the oracle on every row and be bitwise equal to the production
build's (the plain kernel at these sizes): the order in which units run and
which CTA runs them change nothing a unit computes.

The full-size varlen causal 8192 workload, which the production build runs
persistently, is compared on every row in test_parity_gpu.py.
"""
import os

import pytest
import torch

import oracle
from attention_forward_mbarrier_gb300 import binding
from attention_forward_mbarrier_gb300 import build as _build
from attention_forward_mbarrier_gb300 import workloads as wl

from test_parity_gpu import assert_every_row_written, compare, run_gpu

pytestmark = pytest.mark.gpu

PERS_LIB = os.path.join(_build.PKG, "libfmha_perstest.so")


@pytest.fixture(scope="module")
def pers_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    _build.build(force=True, extra_flags=["-DFMHA_PERSISTENT_WAVES=0", "-DFMHA_PERSISTENT_MAX_CTAS=3"],
                 out=PERS_LIB)
    torch.cuda.set_device(0)
    L = binding.open_library(PERS_LIB)
    yield L
    st, detail = binding.fmha_get_device_status(library=L)
    assert st == binding.FMHA_OK, (st, detail)


RAGGED = (1, 127, 128, 129, 255, 256, 257, 383, 700, 1500)

CASES = [
    wl.varlen("pers_ragged_causal", RAGGED, 2, causal=True),
    wl.varlen("pers_ragged_noncausal", RAGGED, 2, causal=False),
    # Lq != Lk: causal tiles whose rows see no key (no blocks), and tails
    wl.varlen("pers_lq_ne_lk", (300, 200, 5, 600), 2, causal=True, seqlens_k=(100, 450, 1, 77)),
    # empty sequences and sequences without keys
    wl.varlen("pers_empty_docs", (0, 130, 0, 40, 300), 2, causal=True, seqlens_k=(0, 130, 7, 0, 300)),
    wl.dense("pers_dense_b3_h4_s300", 3, 300, 4, causal=False),
    wl.dense("pers_dense_b2_h3_s1000_causal", 2, 1000, 3, causal=True),
    wl.varlen("pers_d64_causal", (513, 1, 900), 3, head_dim=64, causal=True),
    wl.varlen("pers_gqa_h8_kv2", (1, 129, 300, 513), 8, causal=True, kv_heads=2),
    wl.varlen("pers_sharp", (700, 300), 2, causal=True, scale=0.5),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_persistent_full(pers_lib, w):
    inp = wl.make_inputs(w, seed=51)
    out, lse = run_gpu(inp, library=pers_lib)
    assert_every_row_written(w, out, lse)
    ref_o, ref_l = oracle.oracle_fwd(*inp.oracle_args())
    compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)
    out_plain, lse_plain = run_gpu(inp)
    assert torch.equal(out, out_plain) and torch.equal(lse, lse_plain)


def test_persistent_without_lse(pers_lib):
    w = wl.varlen("pers_no_lse", (1, 300, 129), 2, causal=True)
    inp = wl.make_inputs(w, seed=52)
    out, _ = run_gpu(inp, with_lse=False, library=pers_lib)
    out_ref, _ = run_gpu(inp, library=pers_lib)
    assert torch.equal(out, out_ref)


def test_persistent_repeats_and_concurrent_streams(pers_lib):
    # the counter slot is reset by each launch's last CTA: repeated launches
    # give the same result, and launches in flight on two streams at once
    # (different slots) do not take each other's units
    wa = wl.varlen("pers_stream_a", (700, 1, 300, 1100), 4, causal=True)
    wb = wl.dense("pers_stream_b", 2, 900, 3, causal=False)
    ia, ib = wl.make_inputs(wa, seed=53), wl.make_inputs(wb, seed=54)
    ref_a, ref_la = run_gpu(ia, library=pers_lib)
    ref_b, ref_lb = run_gpu(ib, library=pers_lib)
    for _ in range(3):
        a, la = run_gpu(ia, library=pers_lib)
        assert torch.equal(a, ref_a) and torch.equal(la, ref_la)

    dev = torch.device("cuda:0")

    def prepare(inp):
        w = inp.workload
        q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
        cq = None if inp.cu_seqlens_q is None else inp.cu_seqlens_q.to(dev)
        ck = None if inp.cu_seqlens_k is None else inp.cu_seqlens_k.to(dev)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.heads, w.total_q), 12345.0, dtype=torch.float32, device=dev)
        return (q, k, v, out, lse, cq, ck, w.batch, w.total_q, w.total_k, w.max_seqlen_q, w.max_seqlen_k,
                w.heads, w.head_dim, w.softmax_scale, int(w.causal))

    args_a, args_b = prepare(ia), prepare(ib)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(4):
        assert binding.fmha_fwd(*args_a, s1, library=pers_lib) == binding.FMHA_OK
        assert binding.fmha_fwd(*args_b, s2, library=pers_lib) == binding.FMHA_OK
    torch.cuda.synchronize()
    assert torch.equal(args_a[3], ref_a) and torch.equal(args_a[4], ref_la)
    assert torch.equal(args_b[3], ref_b) and torch.equal(args_b[4], ref_lb)
