"""GPU parity of the FP8 (e4m3) P V forward, fmha_fwd_fp8pv, against the fp64
oracle, and of its quantised V against an independent rounding on the host.

Tolerance (the variant's own): relative RMS of O <= 6e-2 and
max |O - O_ref| <= 2^-3 * max|V|.  Derived from the arithmetic: P and V / s
are each rounded to e4m3 (half an e4m3 unit is 2^-4 relative), so one output
element is off by at most (2^-4 + 2^-4) * max|V| (its weights sum to one);
a float64 emulation of that rounding on causal, dense, sharp-softmax and
grouped shapes gives relative RMS 2.8e-2 .. 3.7e-2 and max error <= 0.16.
The LSE comes from the unrounded P: abs <= 1e-3 as for fmha_fwd.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_mbarrier_gb300 import binding
from attention_forward_mbarrier_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

REL_RMS = 6e-2
MAX_OF_VMAX = 2.0 ** -3
LSE_ABS = 1e-3


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


def run_fp8(inp):
    w = inp.workload
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    cq = None if inp.cu_seqlens_q is None else inp.cu_seqlens_q.to(dev)
    ck = None if inp.cu_seqlens_k is None else inp.cu_seqlens_k.to(dev)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.heads, w.total_q), 12345.0, dtype=torch.float32, device=dev)
    nbytes = binding.fmha_fwd_fp8pv_workspace_size(w.batch, w.total_k, w.n_kv_heads, w.head_dim)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device=dev)  # e4m3 NaN everywhere before the call
    st = binding.fmha_fwd_fp8pv(q, k, v, out, lse, ws, cq, ck, w.batch, w.total_q, w.total_k, w.max_seqlen_q,
                                w.max_seqlen_k, w.heads, w.n_kv_heads, w.head_dim, w.softmax_scale,
                                int(w.causal), torch.cuda.current_stream())
    assert st == binding.FMHA_OK, binding.status_string(st)
    torch.cuda.synchronize()
    return out, lse, ws


def check(inp, rows=None):
    w = inp.workload
    out, lse, _ = run_fp8(inp)
    cq, _ = w.cu_seqlens()
    if rows is None:
        ro, rl = oracle.oracle_fwd(*inp.oracle_args())
        o = out.float().cpu().numpy().astype(np.float64)
        lg = lse.cpu().numpy().astype(np.float64)
    else:
        ro, rl = oracle.oracle_fwd(*inp.oracle_args(), rows=rows)
        tok, h = torch.from_numpy(rows // w.heads).cuda(), torch.from_numpy(rows % w.heads).cuda()
        o = out[tok, h].float().cpu().numpy().astype(np.float64)
        lg = lse[h, tok].cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(o)), "non-finite output"
    vmax = float(inp.v.float().abs().max())
    err = np.abs(o - ro)
    assert err.max() <= MAX_OF_VMAX * vmax, f"O max-abs {err.max():.3e} (max|V| {vmax:.2f})"
    rel = np.linalg.norm(o - ro) / np.linalg.norm(ro)
    assert rel <= REL_RMS, f"O rel-rms {rel:.3e}"
    fin = ~np.isneginf(rl)
    assert np.array_equal(np.isneginf(lg), ~fin)
    assert np.abs(lg[fin] - rl[fin]).max() <= LSE_ABS
    return rel


CASES = [
    wl.varlen("fp8_ragged_causal", (1, 127, 128, 129, 255, 256, 257, 383), 2, causal=True),
    wl.varlen("fp8_ragged_noncausal", (1, 127, 128, 129, 255, 256, 257, 383), 2, causal=False),
    wl.varlen("fp8_lq_ne_lk", (300, 200, 5), 2, causal=True, seqlens_k=(100, 450, 1)),
    wl.varlen("fp8_empty_docs", (0, 130, 0, 40), 1, causal=True, seqlens_k=(0, 130, 7, 40)),
    wl.dense("fp8_dense_b3_s300", 3, 300, 4, causal=False),
    wl.varlen("fp8_gqa_h8_kv2", (1, 129, 300, 513), 8, causal=True, kv_heads=2),
    wl.varlen("fp8_sharp", (700, 300), 2, causal=True, scale=0.5),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fp8_edge_shapes(w):
    check(wl.make_inputs(w, seed=71))


def test_fp8_workloads():
    check(wl.make_inputs(wl.C2, seed=0))
    inp = wl.make_inputs(wl.C5, seed=0)
    check(inp, rows=wl.sample_rows(wl.C5, n_random=256, seed=1))


def test_fp8_scaled_values():
    # V far from 1 in magnitude: the per-head scale keeps e4m3's relative precision
    w = wl.varlen("fp8_big_v", (300, 129), 2, causal=True)
    inp = wl.make_inputs(w, seed=72)
    inp.v = (inp.v.float() * torch.tensor([300.0, 0.01]).view(1, 2, 1)).to(torch.bfloat16)
    out, lse, _ = run_fp8(inp)
    ro, _ = oracle.oracle_fwd(*inp.oracle_args())
    o = out.float().cpu().numpy().astype(np.float64)
    for h in range(2):
        vmax = float(inp.v[:, h].float().abs().max())
        assert np.abs(o[:, h] - ro[:, h]).max() <= MAX_OF_VMAX * vmax


def test_fp8_quantised_v_layout():
    # the workspace's e4m3 V^T equals the host's own rounding of V / s, with
    # sequence b at padded column 16 * (ceil(k0 / 16) + b) and zeros between
    w = wl.varlen("fp8_layout", (37, 0, 200, 129), 3, causal=True, seqlens_k=(37, 5, 200, 129), kv_heads=3)
    inp = wl.make_inputs(w, seed=73)
    _, _, ws = run_fp8(inp)
    ws = ws.cpu()
    H, D = w.n_kv_heads, w.head_dim
    amax = ws[:4 * H].view(torch.int32).view(torch.float32)
    v = inp.v.float()
    want_amax = v.abs().amax(dim=(0, 2))
    assert torch.equal(amax, want_amax)
    kpad = 16 * ((w.total_k + 15) // 16 + w.batch)
    off = (H * 4 + 255) // 256 * 256
    vt = ws[off:off + H * D * kpad].view(H, D, kpad)
    inv = torch.tensor(448.0, dtype=torch.float32) / want_amax
    want = torch.zeros((H, D, kpad), dtype=torch.uint8)
    _, ck = w.cu_seqlens()
    for b in range(w.batch):
        k0, k1 = int(ck[b]), int(ck[b + 1])
        p0 = 16 * ((k0 + 15) // 16 + b)
        q = (v[k0:k1] * inv.view(1, H, 1)).to(torch.float8_e4m3fn).view(torch.uint8)  # [keys, H, D]
        want[:, :, p0:p0 + (k1 - k0)] = q.permute(1, 2, 0)
    assert torch.equal(vt, want)
