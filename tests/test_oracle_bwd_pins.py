"""Pins of the backward-pass oracle (oracle/fmha_bwd_oracle.c) to things
other than itself.

* Central finite differences of a float64 forward written here with
  scipy.special.softmax (a library softmax over an explicit mask): the
  gradient of L = sum(dO * O) with respect to every element of q, k and v,
  on tiny varlen shapes (causal and not, Lq != Lk, an empty sequence, a row
  with no visible key, grouped K/V heads).
* Closed forms at scale 0 (every visible key has the same weight): dQ = dK = 0
  and dV_j = sum over the rows i that see key j of dO_i / |visible(i)|.
* Sum rules that hold at any size: per sequence and K/V head, sum_j dK_j = 0
  (each softmax row's dS sums to zero) and sum_j dV_j = sum over the group's
  rows with a visible key of dO_i (each softmax row sums to one); V equal
  across keys gives dQ = dK = 0.
* Grouped K/V heads equal multi-head attention with repeated K/V heads whose
  dK/dV are summed over each group.
* Sampled rows / keys equal the full outputs.
* Planted mistakes in copies of the C source each fail at least one pin.
"""
import re

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from attention_forward_mbarrier_gb300 import workloads as wl


def to_f64(t):
    return t.float().double().numpy()


def forward_f64(Q, K, V, w, scale):
    """O = softmax(scale Q K^T, explicit mask) V in float64 (library softmax)."""
    cq, ck = w.cu_seqlens()
    H, G = w.heads, w.heads // w.n_kv_heads
    O = np.zeros_like(Q)
    for b in range(w.batch):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        lq, lk = q1 - q0, k1 - k0
        if lq == 0 or lk == 0:
            continue
        mask = np.ones((lq, lk), dtype=bool)
        if w.causal:
            mask = np.arange(lk)[None, :] <= np.arange(lq)[:, None] + (lk - lq)
        for h in range(H):
            S = scale * Q[q0:q1, h] @ K[k0:k1, h // G].T
            S = np.where(mask, S, -np.inf)
            rows = mask.any(axis=1)
            P = np.zeros_like(S)
            P[rows] = scipy.special.softmax(S[rows], axis=1)
            O[q0:q1, h] = P @ V[k0:k1, h // G]
    return O


def finite_diff_grads(inp, dO, eps=1e-5):
    w = inp.workload
    scale = w.softmax_scale
    X = [to_f64(inp.q), to_f64(inp.k), to_f64(inp.v)]
    G = to_f64(dO)

    def loss(xs):
        return float((forward_f64(xs[0], xs[1], xs[2], w, scale) * G).sum())

    grads = []
    for a in range(3):
        g = np.zeros_like(X[a])
        it = np.nditer(X[a], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = [x.copy() for x in X]
            xm = [x.copy() for x in X]
            xp[a][idx] += eps
            xm[a][idx] -= eps
            g[idx] = (loss(xp) - loss(xm)) / (2 * eps)
        grads.append(g)
    return grads


def bwd(inp, dO, lib_handle=None, **kw):
    return oracle.oracle_bwd(inp.q, inp.k, inp.v, dO, *inp.oracle_args()[3:], lib_handle=lib_handle, **kw)


TINY = [
    wl.varlen("bwd_tiny_causal", (5, 3, 0, 4), 2, head_dim=8, causal=True, seqlens_k=(5, 6, 2, 2)),
    wl.varlen("bwd_tiny_noncausal", (4, 2), 2, head_dim=8, causal=False, seqlens_k=(3, 5)),
    wl.varlen("bwd_tiny_gqa", (6, 3), 4, head_dim=8, causal=True, kv_heads=2),
    wl.dense("bwd_tiny_dense", 2, 4, 2, head_dim=8, causal=True, scale=0.7),
]


def check_finite_differences(case, lib_handle=None, seed=3):
    inp = wl.make_inputs(case, seed=seed)
    dO = wl.make_dout(case, seed=seed)
    dq, dk, dv = bwd(inp, dO, lib_handle)
    fq, fk, fv = finite_diff_grads(inp, dO)
    for got, ref, name in ((dq, fq, "dq"), (dk, fk, "dk"), (dv, fv, "dv")):
        err = np.abs(got - ref).max()
        assert err <= 1e-6 * max(1.0, np.abs(ref).max()), f"{case.name} {name} err {err:.3e}"


@pytest.mark.parametrize("case", TINY, ids=lambda w: w.name)
def test_matches_finite_differences(case):
    check_finite_differences(case)


def check_scale_zero_closed_form(lib_handle=None):
    w = wl.varlen("bwd_scale0", (7, 4), 2, head_dim=16, causal=True, seqlens_k=(9, 4), scale=0.0)
    inp = wl.make_inputs(w, seed=5)
    dO = wl.make_dout(w, seed=5)
    dq, dk, dv = bwd(inp, dO, lib_handle)
    assert np.abs(dq).max() == 0.0 and np.abs(dk).max() == 0.0
    G = to_f64(dO)
    cq, ck = w.cu_seqlens()
    ref = np.zeros_like(dv)
    for b in range(w.batch):
        lq, lk = int(cq[b + 1] - cq[b]), int(ck[b + 1] - ck[b])
        for i in range(lq):
            vis = [j for j in range(lk) if j <= i + lk - lq]
            for j in vis:
                ref[int(ck[b]) + j] += G[int(cq[b]) + i] / len(vis)
    assert np.abs(dv - ref).max() <= 1e-12


def test_scale_zero_closed_form():
    check_scale_zero_closed_form()


def check_sum_rules(lib_handle=None):
    w = wl.varlen("bwd_sums", (40, 17, 33), 4, head_dim=32, causal=True, kv_heads=2,
                  seqlens_k=(40, 30, 20))
    inp = wl.make_inputs(w, seed=9)
    dO = wl.make_dout(w, seed=9)
    dq, dk, dv = bwd(inp, dO, lib_handle)
    G = to_f64(dO)
    cq, ck = w.cu_seqlens()
    grp = w.heads // w.n_kv_heads
    for b in range(w.batch):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        lq, lk = q1 - q0, k1 - k0
        seen = np.array([min(lk, max(0, i + lk - lq + 1)) > 0 for i in range(lq)])
        for hk in range(w.n_kv_heads):
            assert np.abs(dk[k0:k1, hk].sum(0)).max() <= 1e-10 * max(1.0, np.abs(dk[k0:k1, hk]).max())
            want = sum(G[q0:q1, h][seen].sum(0) for h in range(hk * grp, (hk + 1) * grp))
            assert np.abs(dv[k0:k1, hk].sum(0) - want).max() <= 1e-10 * max(1.0, np.abs(want).max())
    # V equal across the keys of every sequence: O no longer depends on q or k
    inp2 = wl.Inputs(w, inp.q, inp.k, inp.v[:1].expand_as(inp.v).contiguous(), inp.cu_seqlens_q,
                     inp.cu_seqlens_k)
    dq2, dk2, _ = bwd(inp2, dO, lib_handle)
    assert np.abs(dq2).max() <= 1e-12 and np.abs(dk2).max() <= 1e-12


def test_sum_rules():
    check_sum_rules()


def check_grouped_equals_repeated(lib_handle=None):
    w = wl.varlen("bwd_gqa", (9, 13), 6, head_dim=16, causal=True, kv_heads=2)
    inp = wl.make_inputs(w, seed=11)
    dO = wl.make_dout(w, seed=11)
    dq, dk, dv = bwd(inp, dO, lib_handle)
    wm = wl.varlen("bwd_gqa_mha", (9, 13), 6, head_dim=16, causal=True)
    im = wl.Inputs(wm, inp.q, inp.k.repeat_interleave(3, dim=1).contiguous(),
                   inp.v.repeat_interleave(3, dim=1).contiguous(), inp.cu_seqlens_q, inp.cu_seqlens_k)
    dq_m, dk_m, dv_m = bwd(im, dO, lib_handle)
    assert np.abs(dq - dq_m).max() <= 1e-12
    assert np.abs(dk - dk_m.reshape(dk_m.shape[0], 2, 3, -1).sum(2)).max() <= 1e-12
    assert np.abs(dv - dv_m.reshape(dv_m.shape[0], 2, 3, -1).sum(2)).max() <= 1e-12


def test_grouped_equals_repeated():
    check_grouped_equals_repeated()


def test_sample_modes_equal_full():
    w = wl.varlen("bwd_sample", (30, 1, 25), 3, head_dim=16, causal=True, seqlens_k=(30, 4, 50),
                  kv_heads=1)
    inp = wl.make_inputs(w, seed=13)
    dO = wl.make_dout(w, seed=13)
    dq, dk, dv = bwd(inp, dO)
    rows = wl.sample_rows(w, n_random=20, seed=1)
    keys = wl.sample_keys(w, n_random=20, seed=2)
    sq, sk, sv = bwd(inp, dO, rows=rows, keys=keys)
    assert np.array_equal(sq, dq.reshape(-1, 16)[rows])
    assert np.array_equal(sk, dk.reshape(-1, 16)[keys])
    assert np.array_equal(sv, dv.reshape(-1, 16)[keys])
    only_q = bwd(inp, dO, rows=rows, want_dkdv=False)
    assert only_q[1] is None and np.array_equal(only_q[0], sq)


def test_rejects_bad_arguments():
    w = wl.varlen("bwd_bad", (3,), 2, head_dim=8)
    inp = wl.make_inputs(w, seed=1)
    dO = wl.make_dout(w, seed=1)
    with pytest.raises(ValueError):
        bwd(inp, dO, rows=np.array([3 * 2], dtype=np.int64))  # token 3 is outside every sequence
    with pytest.raises(ValueError):
        bwd(inp, dO, keys=np.array([-1], dtype=np.int64))


# ---------------------------------------------------------------- planted mistakes
MISTAKES = {
    "dq without scale": ("out[d] += pr->scale * ds * bf16_to_double(kj[d]);",
                         "out[d] += ds * bf16_to_double(kj[d]);"),
    "D added instead of subtracted": ("const double ds = pij * (dpij - st.d);",
                                      "const double ds = pij * (dpij + st.d);"),
    "D dropped in dK": ("const double ds = pij * (dpij - st->d);", "const double ds = pij * dpij;"),
    "dV from dS": ("dv[d] += pij * bf16_to_double(doi[d]);", "dv[d] += ds * bf16_to_double(doi[d]);"),
    "causal off by one": ("return !pr->causal || j <= i + lk - lq;", "return !pr->causal || j < i + lk - lq;"),
    "top-left causal": ("return !pr->causal || j <= i + lk - lq;", "return !pr->causal || j <= i;"),
    "K/V head by modulo": ("const int hk = h / (pr->heads / pr->kv_heads);\n    rowstat_t st",
                           "const int hk = h % pr->kv_heads;\n    rowstat_t st"),
    "dK from k": ("dk[d] += pr->scale * ds * bf16_to_double(qi[d]);",
                  "dk[d] += pr->scale * ds * bf16_to_double(krow(pr, k0 + j, hk)[d]);"),
    "softmax not normalised": ("const double pij = exp(p[j] - st.m) / st.z;",
                               "const double pij = exp(p[j] - st.m);"),
}


@pytest.mark.parametrize("name", sorted(MISTAKES))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MISTAKES[name]
    src = oracle.bwd_source_text()
    assert src.count(old) >= 1, name
    lib_handle = oracle.load_bwd_variant(src.replace(old, new), str(tmp_path))
    checks = [lambda: [check_finite_differences(c, lib_handle) for c in TINY],
              lambda: check_scale_zero_closed_form(lib_handle),
              lambda: check_sum_rules(lib_handle),
              lambda: check_grouped_equals_repeated(lib_handle)]
    failed = 0
    for chk in checks:
        try:
            chk()
        except AssertionError:
            failed += 1
    assert failed >= 1, f"planted mistake '{name}' passed every pin"
