"""The head-grouped launch order, checked on every row.

The library orders its grid in groups of 4 heads when one sequence's K/V
exceeds 96 MiB (the causal 32768-token workload takes this path).  A
test-only build lowers that threshold to 1 MiB (-DFMHA_L2_GROUP_BYTES), so
problems small enough for a full oracle compare take the same code path:
partial last head groups, several sequences, causal and not, head_dim 64 and
grouped K/V heads.  Each result must match the oracle on every row and be
bitwise equal to the production build's (plain grid order): the order in
which CTAs run changes nothing a CTA computes.
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

GROUP_LIB = os.path.join(_build.PKG, "libfmha_grouptest.so")
THRESHOLD = 1 << 20  # bytes of one sequence's K and V above which the grid is head-grouped


@pytest.fixture(scope="module")
def group_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    _build.build(force=True, extra_flags=[f"-DFMHA_L2_GROUP_BYTES={THRESHOLD}"], out=GROUP_LIB)
    torch.cuda.set_device(0)
    L = binding.open_library(GROUP_LIB)
    yield L
    st, detail = binding.fmha_get_device_status(library=L)
    assert st == binding.FMHA_OK, (st, detail)


def test_head_dim_256_keeps_plain_order(group_lib):
    # head_dim 256 runs the plain grid order even above the threshold
    w = wl.varlen("grp_d256_plain", (1500, 300), 6, head_dim=256, causal=True)
    inp = wl.make_inputs(w, seed=42)
    out, lse = run_gpu(inp, library=group_lib)
    ref_o, ref_l = oracle.oracle_fwd(*inp.oracle_args())
    compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)


CASES = [
    # 6 heads: groups of 4 and 2; a one-token sequence
    wl.varlen("grp_causal_h6", (1500, 700, 1), 6, causal=True),
    # 9 heads: groups 4, 4, 1; dense batches
    wl.dense("grp_dense_b2_h9_s1000", 2, 1000, 9, causal=False),
    # Lq != Lk, ragged tails
    wl.varlen("grp_lq_ne_lk_h5", (300, 1333), 5, causal=True, seqlens_k=(2100, 1333)),
    wl.varlen("grp_d64_causal_h5", (2000, 333), 5, head_dim=64, causal=True),
    wl.varlen("grp_gqa_h8_kv2", (1200, 900), 8, causal=True, kv_heads=2),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_grouped_order_full(group_lib, w):
    kv_bytes = w.n_kv_heads * w.max_seqlen_k * w.head_dim * 4
    assert kv_bytes > THRESHOLD and w.heads > 4, "case must take the head-grouped order"
    inp = wl.make_inputs(w, seed=41)
    out, lse = run_gpu(inp, library=group_lib)
    assert_every_row_written(w, out, lse)
    ref_o, ref_l = oracle.oracle_fwd(*inp.oracle_args())
    compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)
    out_plain, lse_plain = run_gpu(inp)
    assert torch.equal(out, out_plain) and torch.equal(lse, lse_plain)


def test_grouped_order_growing_scores(group_lib):
    # The head-grouped kernel through the softmax's redo path: even rows'
    # scores grow by ~17 log2 units per 128-key block (see
    # test_parity_gpu.test_scores_growing_across_key_blocks)
    from dataclasses import replace

    import numpy as np

    n = 1000
    w = wl.dense("grp_growing_h6", 1, n, 6, causal=True)
    inp = wl.make_inputs(w, seed=43)
    q, k = inp.q.float(), inp.k.float()
    q[0::2, :, 0] = 4.0
    q[1::2, :, 0] = 0.0
    k[:, :, 0] = torch.arange(n, dtype=torch.float32)[:, None] * 0.25
    inp = replace(inp, q=q.to(torch.bfloat16), k=k.to(torch.bfloat16))
    assert w.n_kv_heads * w.max_seqlen_k * w.head_dim * 4 > THRESHOLD and w.heads > 4
    out, lse = run_gpu(inp, library=group_lib)
    ref_o, ref_l = oracle.oracle_fwd(*inp.oracle_args())
    compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)
    out_plain, lse_plain = run_gpu(inp)
    assert torch.equal(out, out_plain) and torch.equal(lse, lse_plain)
    assert np.isfinite(out.float().cpu().numpy()).all()
