"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin ties the fp64 C oracle to something the mathematics or an independent
implementation fixes:

* brute force   -- pure-Python loops (no max shift) on tiny varlen shapes,
                   including Lq != Lk and rows with no visible key;
* library       -- scipy.special.softmax / logsumexp on an explicit masked
                   score matrix;
* closed forms  -- scale = 0 gives the mean of the visible V rows and
                   LSE = log(count); identical K rows give the same; causal row
                   0 gives V_0 and LSE = scale q_0.k_0; V = 1 gives O = 1; two
                   keys give the logistic weight and the softplus LSE;
* invariants    -- varlen sequence == the same sequence run alone, key
                   permutation (non-causal), head permutation, K shift;
* planted mistakes -- broken copies of the C source (dropped scale, causal
                   off-by-one, top-left alignment, LSE without the max, no
                   normalisation, q used for k, wrong head, K/V head by modulo
                   instead of by group) must each fail at least one pin;
* grouped K/V heads -- equal to multi-head attention with each K/V head
                   repeated for its group of query heads, and the brute force
                   on a tiny grouped shape.

Definition being pinned: "[BUG] Unexpected Slower Performance in C++ CuTe
(77_blackwell_fmha) vs Python CuTe DSL (fmha.py) on Jetson Thor", section
"Implementation Differences in softmax_step"; "[BUG] CuTe DSL 4.7/4.8
regression: FlashAttention-4 SM100 forward kernel spills registers", section
"Steps/Code to reproduce bug" (varlen causal layout).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_mbarrier_gb300 import workloads as wl

TOL = 1e-12


def to_bits(x) -> np.ndarray:
    """float array -> bf16 bit patterns (exact when x is bf16-representable)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    back = t.to(torch.float32).numpy()
    assert np.array_equal(back, np.asarray(x, dtype=np.float32)), "value not bf16-exact"
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run(fn, q, k, v, seqlens_q, seqlens_k, scale, causal, dense=False, **kw):
    batch = len(seqlens_q)
    if dense:
        cq = ck = None
    else:
        cq = np.concatenate([[0], np.cumsum(seqlens_q)]).astype(np.int32)
        ck = np.concatenate([[0], np.cumsum(seqlens_k)]).astype(np.int32)
    return fn(q, k, v, cq, ck, batch, max(seqlens_q), max(seqlens_k), scale, causal, **kw)


def assert_close(a, b, tol=TOL):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape
    fin = np.isfinite(a) | np.isfinite(b)
    assert np.array_equal(np.isneginf(a), np.isneginf(b))
    if fin.any():
        assert np.max(np.abs(a[fin] - b[fin])) <= tol, np.max(np.abs(a[fin] - b[fin]))


# ----------------------------------------------------------------------------
# pin families, written against an oracle callable so the planted-mistake test
# can run the same checks on broken copies
# ----------------------------------------------------------------------------

def pin_brute_force(fn):
    cases = [
        ((5, 1, 9, 37), (5, 1, 9, 37), 2, 16, True),
        ((5, 1, 9, 37), (5, 1, 9, 37), 2, 16, False),
        ((3, 7, 0, 4), (6, 4, 2, 0), 2, 8, True),   # Lq != Lk, empty rows, empty doc
        ((3, 7), (6, 4), 3, 8, False),
    ]
    for sq, sk, heads, hd, causal in cases:
        w = wl.varlen("bf", sq, heads, head_dim=hd, causal=causal, seqlens_k=sk)
        inp = wl.make_inputs(w, seed=3, dist="uniform")
        a = fn(*inp.oracle_args())
        b = oracle.brute_force_fwd(*inp.oracle_args())
        assert_close(a[0], b[0])
        assert_close(a[1], b[1])


def pin_library(fn):
    from scipy.special import logsumexp, softmax

    w = wl.varlen("lib", (130, 257, 1), 3, head_dim=128, causal=True, seqlens_k=(130, 300, 4))
    inp = wl.make_inputs(w, seed=5)
    out, lse = fn(*inp.oracle_args())
    q, k, v = (x.to(torch.float64).numpy() for x in (inp.q, inp.k, inp.v))
    cq, ck = w.cu_seqlens()
    for b in range(w.batch):
        lq, lk = w.seqlens_q[b], w.seqlens_k[b]
        for h in range(w.heads):
            qs = q[cq[b]:cq[b + 1], h]
            ks = k[ck[b]:ck[b + 1], h]
            vs = v[ck[b]:ck[b + 1], h]
            s = w.softmax_scale * qs @ ks.T
            ii, jj = np.meshgrid(np.arange(lq), np.arange(lk), indexing="ij")
            s = np.where(jj <= ii + lk - lq, s, -np.inf)
            ref_o = softmax(s, axis=1) @ vs
            ref_l = logsumexp(s, axis=1)
            assert np.max(np.abs(out[cq[b]:cq[b + 1], h] - ref_o)) <= 1e-10
            assert np.max(np.abs(lse[h, cq[b]:cq[b + 1]] - ref_l)) <= 1e-10


def pin_scale_zero(fn):
    # scale = 0: every visible key weighs the same -> cumulative mean of V,
    # LSE = log(number of visible keys)
    w = wl.varlen("z", (40, 17), 2, head_dim=32, causal=True)
    inp = wl.make_inputs(w, seed=7)
    args = list(inp.oracle_args())
    args[8] = 0.0
    out, lse = fn(*args)
    v = inp.v.to(torch.float64).numpy()
    cq, _ = w.cu_seqlens()
    for b in range(w.batch):
        seg = v[cq[b]:cq[b + 1]]
        cnt = np.arange(1, seg.shape[0] + 1, dtype=np.float64)
        mean = np.cumsum(seg, axis=0) / cnt[:, None, None]
        assert np.max(np.abs(out[cq[b]:cq[b + 1]] - mean)) <= TOL
        for h in range(w.heads):
            assert np.max(np.abs(lse[h, cq[b]:cq[b + 1]] - np.log(cnt))) <= TOL


def pin_identical_keys(fn):
    # every K row equal: scores are constant along j -> O = mean of visible V,
    # LSE = scale * q_i.k + log(count)   (non-causal: count = Lk)
    rng = np.random.default_rng(11)
    lq, lk, hd = 9, 13, 16
    qf = rng.integers(-4, 5, size=(lq, 1, hd)) / 8.0
    krow = rng.integers(-4, 5, size=(1, 1, hd)) / 8.0
    kf = np.repeat(krow, lk, axis=0)
    vf = rng.integers(-8, 9, size=(lk, 1, hd)) / 8.0
    scale = 0.25
    out, lse = run(fn, to_bits(qf), to_bits(kf), to_bits(vf), (lq,), (lk,), scale, False, dense=True)
    assert np.max(np.abs(out - vf.mean(axis=0)[None])) <= TOL
    s = scale * (qf[:, 0] @ krow[0, 0])
    assert np.max(np.abs(lse[0] - (s + math.log(lk)))) <= TOL


def pin_causal_row0(fn):
    # causal, Lq == Lk: row 0 sees only key 0 -> O_0 = V_0, LSE_0 = scale q_0.k_0
    w = wl.varlen("r0", (6, 11, 3), 2, head_dim=64, causal=True)
    inp = wl.make_inputs(w, seed=13)
    out, lse = fn(*inp.oracle_args())
    q, k, v = (x.to(torch.float64).numpy() for x in (inp.q, inp.k, inp.v))
    cq, _ = w.cu_seqlens()
    for b in range(w.batch):
        t = cq[b]
        assert np.array_equal(out[t], v[t])
        for h in range(w.heads):
            assert abs(lse[h, t] - w.softmax_scale * float(q[t, h] @ k[t, h])) <= TOL


def pin_ones_v(fn):
    # V = 1: softmax weights sum to one, so O = 1 exactly up to rounding
    w = wl.varlen("ones", (33, 70), 2, head_dim=16, causal=True, seqlens_k=(40, 70))
    inp = wl.make_inputs(w, seed=17)
    args = list(inp.oracle_args())
    args[2] = torch.ones_like(inp.v)
    out, _ = fn(*args)
    cq, _ = w.cu_seqlens()
    # doc 0 has Lq < Lk, every row sees >= 8 keys; all rows valid
    assert np.max(np.abs(out - 1.0)) <= 1e-14


def pin_two_keys(fn):
    # two keys, k_1 = 0: weight of key 0 is the logistic function of
    # a = scale q.k_0, and LSE = log(1 + e^a)
    hd = 8
    q = np.zeros((1, 1, hd)); q[0, 0, :3] = [1.0, -0.5, 2.0]
    k = np.zeros((2, 1, hd)); k[0, 0, :3] = [0.5, 1.0, 0.75]
    v = np.zeros((2, 1, hd)); v[0, 0, 0] = 3.0; v[1, 0, 0] = -1.0; v[1, 0, 5] = 2.0
    scale = 0.5
    out, lse = run(fn, to_bits(q), to_bits(k), to_bits(v), (1,), (2,), scale, False, dense=True)
    a = scale * (1.0 * 0.5 - 0.5 * 1.0 + 2.0 * 0.75)
    w0 = 1.0 / (1.0 + math.exp(-a))
    assert abs(out[0, 0, 0] - (3.0 * w0 - 1.0 * (1.0 - w0))) <= TOL
    assert abs(out[0, 0, 5] - 2.0 * (1.0 - w0)) <= TOL
    assert abs(lse[0, 0] - (a + math.log1p(math.exp(-a)))) <= TOL


def pin_varlen_equals_alone(fn):
    w = wl.varlen("va", (50, 129, 7), 2, head_dim=128, causal=True, seqlens_k=(60, 129, 7))
    inp = wl.make_inputs(w, seed=19)
    out, lse = fn(*inp.oracle_args())
    cq, ck = w.cu_seqlens()
    for b in range(w.batch):
        sq, sk = slice(cq[b], cq[b + 1]), slice(ck[b], ck[b + 1])
        o1, l1 = run(fn, inp.q[sq], inp.k[sk], inp.v[sk], (w.seqlens_q[b],), (w.seqlens_k[b],),
                     w.softmax_scale, True, dense=True)
        assert np.array_equal(o1, out[sq])
        assert np.array_equal(l1, lse[:, sq])


def pin_key_permutation(fn):
    w = wl.dense("perm", 1, 31, 2, head_dim=32, seqlen_k=45)
    inp = wl.make_inputs(w, seed=23)
    out, lse = fn(*inp.oracle_args())
    perm = torch.from_numpy(np.random.default_rng(1).permutation(45))
    args = list(inp.oracle_args())
    args[1], args[2] = inp.k[perm], inp.v[perm]
    out2, lse2 = fn(*args)
    assert_close(out, out2, 1e-13)
    assert_close(lse, lse2, 1e-13)


def pin_head_permutation(fn):
    w = wl.varlen("hp", (20, 9), 3, head_dim=16, causal=True)
    inp = wl.make_inputs(w, seed=29)
    out, lse = fn(*inp.oracle_args())
    perm = [2, 0, 1]
    args = list(inp.oracle_args())
    args[0], args[1], args[2] = inp.q[:, perm], inp.k[:, perm], inp.v[:, perm]
    out2, lse2 = fn(*args)
    assert np.array_equal(out2, out[:, perm])
    assert np.array_equal(lse2, lse[perm])


def pin_key_shift(fn):
    # adding c to every key row shifts row i's scores by scale q_i.c (constant
    # in j): O unchanged, LSE shifted by scale q_i.c
    rng = np.random.default_rng(31)
    lq, lk, hd = 12, 12, 16
    qf = rng.integers(-4, 5, size=(lq, 1, hd)) / 8.0
    kf = rng.integers(-4, 5, size=(lk, 1, hd)) / 8.0
    vf = rng.integers(-8, 9, size=(lk, 1, hd)) / 8.0
    c = rng.integers(-2, 3, size=(1, 1, hd)) / 2.0
    scale = 0.3
    o1, l1 = run(fn, to_bits(qf), to_bits(kf), to_bits(vf), (lq,), (lk,), scale, True, dense=True)
    o2, l2 = run(fn, to_bits(qf), to_bits(kf + c), to_bits(vf), (lq,), (lk,), scale, True, dense=True)
    assert np.max(np.abs(o1 - o2)) <= 1e-13
    shift = scale * (qf[:, 0] @ c[0, 0])
    assert np.max(np.abs((l2 - l1)[0] - shift)) <= 1e-13


def pin_grouped_kv_heads(fn):
    # Grouped K/V heads: 6 query heads on 2 K/V heads must equal ordinary
    # multi-head attention with each K/V head repeated for its 3 query heads
    # (query head h reads K/V head h // 3).  Also the pure-Python brute force
    # on a tiny grouped shape.
    w = wl.varlen("gqa", (23, 40), 6, head_dim=16, causal=True, kv_heads=2)
    inp = wl.make_inputs(w, seed=41)
    out, lse = fn(*inp.oracle_args())
    args = list(inp.oracle_args())
    args[1] = inp.k.repeat_interleave(3, dim=1)
    args[2] = inp.v.repeat_interleave(3, dim=1)
    out2, lse2 = fn(*args)
    assert_close(out, out2, 1e-13)
    assert_close(lse, lse2, 1e-13)
    wb = wl.varlen("gqa_bf", (9, 5), 4, head_dim=8, causal=False, seqlens_k=(7, 11), kv_heads=2)
    ib = wl.make_inputs(wb, seed=43, dist="uniform")
    a = fn(*ib.oracle_args())
    b = oracle.brute_force_fwd(*ib.oracle_args())
    assert_close(a[0], b[0])
    assert_close(a[1], b[1])


PINS = [pin_brute_force, pin_library, pin_scale_zero, pin_identical_keys, pin_causal_row0,
        pin_ones_v, pin_two_keys, pin_varlen_equals_alone, pin_key_permutation,
        pin_head_permutation, pin_key_shift, pin_grouped_kv_heads]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(oracle_mod, pin):
    pin(oracle_mod.oracle_fwd)


def test_row_mode_matches_full_mode(oracle_mod):
    w = wl.varlen("rows", (70, 3, 129), 4, head_dim=128, causal=True)
    inp = wl.make_inputs(w, seed=37)
    out, lse = oracle_mod.oracle_fwd(*inp.oracle_args())
    rows = wl.sample_rows(w, n_random=50, seed=2)
    o_r, l_r = oracle_mod.oracle_fwd(*inp.oracle_args(), rows=rows)
    tok, h = rows // w.heads, rows % w.heads
    assert np.array_equal(o_r, out[tok, h])
    assert np.array_equal(l_r, lse[h, tok])


def test_oracle_rejects_bad_arguments(oracle_mod):
    w = wl.varlen("bad", (4,), 1, head_dim=8)
    inp = wl.make_inputs(w)
    args = list(inp.oracle_args())
    args[4] = None  # cu_k missing while cu_q given
    with pytest.raises(ValueError):
        oracle_mod.oracle_fwd(*args)


MUTANTS = {
    "dropped_scale": ("s_buf[j] = scale * dot;", "s_buf[j] = dot;"),
    "causal_off_by_one": ("(j <= i + lk - lq)", "(j < i + lk - lq)"),
    "top_left_alignment": ("(j <= i + lk - lq)", "(j <= i)"),
    "lse_without_max": ("*lse_out = m + log(z);", "*lse_out = log(z);"),
    "no_normalisation": ("o_row[d] /= z;", "o_row[d] /= 1.0;"),
    "q_used_for_k": ("bf16_bits_to_double(qi[d]) * bf16_bits_to_double(kj[d])",
                     "bf16_bits_to_double(qi[d]) * bf16_bits_to_double(qi[d])"),
    "wrong_head_for_v": ("const uint16_t *vj = v + (k0 + j) * kv_stride + (int64_t)hk * head_dim;",
                         "const uint16_t *vj = v + (k0 + j) * kv_stride;"),
    "max_not_subtracted": ("double p = exp(s_buf[j] - m);", "double p = exp(s_buf[j]);"),
    "kv_head_modulo": ("const int hk = h / (heads / kv_heads);", "const int hk = h % kv_heads;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(oracle_mod, tmp_path, name):
    before, after = MUTANTS[name]
    src = oracle_mod.source_text()
    assert src.count(before) == 1, f"mutation anchor for {name} not unique"
    handle = oracle_mod.load_variant(src.replace(before, after), str(tmp_path))

    def broken(*args, **kw):
        return oracle_mod.oracle_fwd(*args, lib_handle=handle, **kw)

    caught = []
    for pin in PINS:
        try:
            pin(broken)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
