"""Seeded input recipe: shapes, cu_seqlens and algorithmic FLOP counts."""
import numpy as np
import torch

from attention_forward_mbarrier_gb300 import workloads as wl


def test_cu_seqlens_recipe():
    # cu = round(linspace(0, total, docs + 1)) as int32
    assert wl.C3.seqlens_q == (2048,) * 4
    assert wl.C4.seqlens_q == (4096,) * 8
    assert wl.C5.seqlens_q == (32768,)
    cq, ck = wl.C4.cu_seqlens()
    assert cq.dtype == np.int32 and list(cq) == list(range(0, 32769, 4096))
    assert wl.linspace_docs(10, 3) == (3, 4, 3)


def test_flops_match_closed_form():
    # non-causal: 4 d h L^2 ; causal (Lq == Lk): 4 d h L(L+1)/2 per sequence
    assert wl.C2.flops() == 4 * 128 * 16 * 2225 * 2225
    assert wl.C5.flops() == 4 * 128 * 16 * 32768 * 32769 // 2
    assert wl.C3.flops() == 4 * 4 * 128 * 32 * 2048 * 2049 // 2
    # Lq != Lk causal, bottom-right: row i sees min(lk, i + lk - lq + 1) keys
    w = wl.varlen("x", (5,), 1, head_dim=1, causal=True, seqlens_k=(3,))
    assert w.visible_pairs() == 0 + 0 + 1 + 2 + 3


def test_generator_is_seeded_and_ordered():
    a = wl.make_inputs(wl.C1, seed=0)
    b = wl.make_inputs(wl.C1, seed=0)
    assert torch.equal(a.q, b.q) and torch.equal(a.v, b.v)
    assert a.q.shape == (128, 2, 128) and a.q.dtype == torch.bfloat16
    g = torch.Generator().manual_seed(0)
    q = torch.randn((128, 2, 128), generator=g).to(torch.bfloat16)
    assert torch.equal(q, a.q)
    assert a.cu_seqlens_q is None


def test_sample_rows_cover_sequence_edges():
    rows = wl.sample_rows(wl.C3, n_random=10, seed=0)
    toks = set((rows // wl.C3.heads).tolist())
    for b in (0, 2048, 4096, 6144):
        assert b in toks and b + 2047 in toks
