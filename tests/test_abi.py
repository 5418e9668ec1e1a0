"""The C ABI library loads, exports every declared symbol, and validates
arguments on the host before touching the GPU (no GPU needed here)."""
import os
import re

import pytest

from attention_forward_mbarrier_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def declared_functions():
    txt = open(os.path.join(ROOT, "include", "fmha.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fmha_\w+)\s*\(", txt, flags=re.M)


def test_header_declares_binding_symbols():
    assert sorted(declared_functions()) == sorted(binding.SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert binding.status_string(0) == "ok"
    assert "timed out" in binding.status_string(binding.FMHA_ERR_TIMEOUT)
    assert binding.status_string(99) == "unknown status"
    assert binding.fmha_version() >= 10100


GOOD = dict(q=0x1000, k=0x2000, v=0x3000, out=0x4000, lse=0x5000, cu_seqlens_q=0x6000,
            cu_seqlens_k=0x7000, batch=2, total_q=300, total_k=300, max_seqlen_q=200,
            max_seqlen_k=200, heads=4, head_dim=128, scale=0.088, causal=1, stream=0)


@pytest.mark.parametrize("change,expected", [
    (dict(q=0), binding.FMHA_ERR_INVALID_ARG),
    (dict(out=0), binding.FMHA_ERR_INVALID_ARG),
    (dict(cu_seqlens_k=0), binding.FMHA_ERR_INVALID_ARG),
    (dict(q=0x1008), binding.FMHA_ERR_INVALID_ARG),  # not 16-byte aligned
    (dict(lse=0x5002), binding.FMHA_ERR_INVALID_ARG),
    (dict(heads=0), binding.FMHA_ERR_INVALID_ARG),
    (dict(batch=-1), binding.FMHA_ERR_INVALID_ARG),
    (dict(causal=2), binding.FMHA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.FMHA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), binding.FMHA_ERR_INVALID_ARG),
    (dict(scale=float("-inf")), binding.FMHA_ERR_INVALID_ARG),
    (dict(head_dim=96), binding.FMHA_ERR_UNSUPPORTED),
    (dict(head_dim=192), binding.FMHA_ERR_UNSUPPORTED),
    (dict(head_dim=512), binding.FMHA_ERR_UNSUPPORTED),
    (dict(batch=70000), binding.FMHA_ERR_UNSUPPORTED),
    # more than 65535 blocks of 256 query rows on the plain grid (this K/V of
    # 4 heads stays under the head-grouped threshold)
    (dict(max_seqlen_q=65535 * 256 + 1, total_q=2 * (65535 * 256 + 1)), binding.FMHA_ERR_UNSUPPORTED),
    # dense mode needs total == batch * max_seqlen
    (dict(cu_seqlens_q=0, cu_seqlens_k=0), binding.FMHA_ERR_INVALID_ARG),
])
def test_invalid_arguments_rejected_on_host(lib, change, expected):
    args = dict(GOOD)
    args.update(change)
    assert binding.fmha_fwd(**args) == expected


@pytest.mark.parametrize("kv_heads,expected", [
    (0, binding.FMHA_ERR_INVALID_ARG),
    (3, binding.FMHA_ERR_INVALID_ARG),   # does not divide heads = 4
    (-2, binding.FMHA_ERR_INVALID_ARG),
    (8, binding.FMHA_ERR_INVALID_ARG),   # more K/V heads than query heads
])
def test_invalid_kv_heads_rejected_on_host(lib, kv_heads, expected):
    args = dict(GOOD)
    args.update(kv_heads=kv_heads)
    assert binding.fmha_fwd_gqa(**args) == expected


def test_grouped_call_with_bad_common_argument_matches_fmha_fwd(lib):
    args = dict(GOOD)
    args.update(kv_heads=2, scale=float("nan"))
    assert binding.fmha_fwd_gqa(**args) == binding.FMHA_ERR_INVALID_ARG


def test_empty_problem_is_ok_without_gpu(lib):
    args = dict(GOOD)
    args.update(batch=0, total_q=0, total_k=0, max_seqlen_q=0, max_seqlen_k=0)
    assert binding.fmha_fwd(**args) == binding.FMHA_OK


def test_no_gpu_gives_cuda_error_not_crash(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert binding.fmha_fwd(**GOOD) == binding.FMHA_ERR_CUDA


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError):
        binding.lib()


def test_kernel_has_no_register_spills():
    rep = build.ptxas_report()
    m = re.findall(r"(\d+) bytes spill stores, (\d+) bytes spill loads", rep)
    assert m, rep
    assert all(a == "0" and b == "0" for a, b in m), rep
    assert "0 bytes stack frame" in rep


BWD_GOOD = dict(q=0x1000, k=0x2000, v=0x3000, out=0x4000, dout=0x5000, lse=0x6000, dq=0x7000, dk=0x8000,
                dv=0x9000, workspace=0xa000, cu_seqlens_q=0xb000, cu_seqlens_k=0xc000, batch=2, total_q=300,
                total_k=300, max_seqlen_q=200, max_seqlen_k=200, heads=4, kv_heads=2, head_dim=128,
                scale=0.088, causal=1, stream=0)


@pytest.mark.parametrize("change,expected", [
    (dict(lse=0), binding.FMHA_ERR_INVALID_ARG),          # the backward pass needs the forward's LSE
    (dict(workspace=0), binding.FMHA_ERR_INVALID_ARG),
    (dict(dout=0), binding.FMHA_ERR_INVALID_ARG),
    (dict(dk=0x8008), binding.FMHA_ERR_INVALID_ARG),      # not 16-byte aligned
    (dict(workspace=0xa002), binding.FMHA_ERR_INVALID_ARG),
    (dict(kv_heads=3), binding.FMHA_ERR_INVALID_ARG),
    (dict(cu_seqlens_q=0), binding.FMHA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.FMHA_ERR_INVALID_ARG),
    (dict(causal=-1), binding.FMHA_ERR_INVALID_ARG),
    (dict(head_dim=64), binding.FMHA_ERR_UNSUPPORTED),
    (dict(max_seqlen_k=65536 * 128, total_k=2 * 65536 * 128), binding.FMHA_ERR_UNSUPPORTED),
])
def test_backward_invalid_arguments_rejected_on_host(lib, change, expected):
    args = dict(BWD_GOOD)
    args.update(change)
    assert binding.fmha_bwd(**args) == expected


def test_backward_workspace_size(lib):
    assert binding.fmha_bwd_workspace_size(16, 32768) == 16 * 32768 * 4
    assert binding.fmha_bwd_workspace_size(-1, 5) == 0
    args = dict(BWD_GOOD)
    args.update(batch=0, total_q=0, total_k=0, max_seqlen_q=0, max_seqlen_k=0)
    assert binding.fmha_bwd(**args) == binding.FMHA_OK


FP8_GOOD = dict(q=0x1000, k=0x2000, v=0x3000, out=0x4000, lse=0x5000, workspace=0x10000, cu_seqlens_q=0x6000,
                cu_seqlens_k=0x7000, batch=2, total_q=300, total_k=300, max_seqlen_q=200, max_seqlen_k=200,
                heads=4, kv_heads=2, head_dim=128, scale=0.088, causal=1, stream=0)


@pytest.mark.parametrize("change,expected", [
    (dict(workspace=0), binding.FMHA_ERR_INVALID_ARG),
    (dict(workspace=0x10010), binding.FMHA_ERR_INVALID_ARG),  # not 256-byte aligned
    (dict(v=0x3008), binding.FMHA_ERR_INVALID_ARG),
    (dict(kv_heads=3), binding.FMHA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), binding.FMHA_ERR_INVALID_ARG),
    (dict(head_dim=64), binding.FMHA_ERR_UNSUPPORTED),
    (dict(head_dim=256), binding.FMHA_ERR_UNSUPPORTED),
])
def test_fp8_invalid_arguments_rejected_on_host(lib, change, expected):
    args = dict(FP8_GOOD)
    args.update(change)
    assert binding.fmha_fwd_fp8pv(**args) == expected


def test_fp8_workspace_size(lib):
    # per-head max words padded to 256 bytes, then kv_heads * head_dim rows of
    # 16 * (ceil(total_k / 16) + batch) bytes
    assert binding.fmha_fwd_fp8pv_workspace_size(4, 8192, 32, 128) == 256 + 32 * 128 * 16 * (512 + 4)
    assert binding.fmha_fwd_fp8pv_workspace_size(1, 1, 80, 128) == 512 + 80 * 128 * 32
    assert binding.fmha_fwd_fp8pv_workspace_size(-1, 5, 1, 128) == 0
    args = dict(FP8_GOOD)
    args.update(batch=0, total_q=0, total_k=0, max_seqlen_q=0, max_seqlen_k=0)
    assert binding.fmha_fwd_fp8pv(**args) == binding.FMHA_OK
