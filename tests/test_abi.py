"""The C-ABI library: it loads, exports what include/fa.h declares, and rejects bad
arguments on the host (these calls return before any CUDA work, so they run without a GPU)."""

from __future__ import annotations

import ctypes
import os
import re

import pytest

from tiled_attention_prefill_gb300 import _build, fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_\w+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    assert declared_functions() == sorted(fa.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_error_strings(lib):
    assert lib.fa_version() == 100
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        s = lib.fa_error_string(code).decode()
        assert s and s != "unknown error code"
    assert lib.fa_error_string(12345).decode() == "unknown error code"


def test_watchdog_setter(lib):
    assert lib.fa_set_watchdog_ns(0) == fa.FA_OK


def _call(lib, q=16, k=32, v=48, o=1 << 40, lse=0, B=1, H=1, N=8, D=64, scale=0.125, causal=0, dtype=0):
    return lib.fa_forward(q or None, k or None, v or None, o or None, lse or None, B, H, N, D, scale, causal, dtype,
                          None)


def test_null_pointers_rejected(lib):
    assert _call(lib, q=0) == fa.FA_ERR_INVALID_ARG
    assert _call(lib, k=0) == fa.FA_ERR_INVALID_ARG
    assert _call(lib, v=0) == fa.FA_ERR_INVALID_ARG
    assert _call(lib, o=0) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("field", ["B", "H", "N"])
@pytest.mark.parametrize("value", [0, -3])
def test_nonpositive_sizes_rejected(lib, field, value):
    assert _call(lib, **{field: value}) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("D", [0, 32, 96, 256])
def test_unsupported_head_dim(lib, D):
    assert _call(lib, D=D) == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("dtype", [-1, 3, 7])
def test_unsupported_dtype(lib, dtype):
    assert _call(lib, dtype=dtype) == fa.FA_ERR_UNSUPPORTED


def test_fp32_dtype_is_validated_like_the_others(lib):
    # FA_DTYPE_FP32 is a fused-forward dtype (tf32 products): it passes validation and would
    # then need a device; bad arguments are still refused first.
    assert _call(lib, dtype=fa.FA_DTYPE_FP32, q=0) == fa.FA_ERR_INVALID_ARG
    assert _call(lib, dtype=fa.FA_DTYPE_FP32, q=24) == fa.FA_ERR_ALIGN
    assert _call(lib, dtype=fa.FA_DTYPE_FP32, D=96) == fa.FA_ERR_UNSUPPORTED


def test_misaligned_pointers(lib):
    assert _call(lib, q=18) == fa.FA_ERR_ALIGN
    assert _call(lib, k=40) == fa.FA_ERR_ALIGN
    assert _call(lib, v=8) == fa.FA_ERR_ALIGN
    assert _call(lib, o=(1 << 40) + 4) == fa.FA_ERR_ALIGN
    assert _call(lib, lse=(1 << 41) + 2) == fa.FA_ERR_ALIGN


def test_too_large(lib):
    assert _call(lib, N=(1 << 30) + 1) == fa.FA_ERR_TOO_LARGE
    assert _call(lib, B=1 << 16, H=1 << 16, N=256) == fa.FA_ERR_TOO_LARGE


def test_output_aliasing_rejected(lib):
    base = 1 << 40
    n_bytes = 1 * 1 * 8 * 64 * 2
    assert _call(lib, q=base, k=base + 4096, v=base + 8192, o=base + 16) == fa.FA_ERR_INVALID_ARG
    o = base + (1 << 20)
    assert _call(lib, q=base, k=base + 4096, v=base + 8192, o=o, lse=o + n_bytes - 4) == fa.FA_ERR_INVALID_ARG


def test_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(1, 1, 8, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        fa.forward(x, x, x)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(ImportError):
        fa.load_library(str(tmp_path / "libmissing.so"))
    assert isinstance(ctypes.CDLL, type)


def test_decomposition_setter(lib):
    assert lib.fa_set_decomposition(1) == fa.FA_OK
    assert lib.fa_set_decomposition(2) == fa.FA_OK
    assert lib.fa_set_decomposition(3) == fa.FA_OK
    assert lib.fa_set_decomposition(4) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_set_decomposition(-1) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_set_decomposition(0) == fa.FA_OK


def _align_up(x, a=256):
    return (x + a - 1) // a * a


def test_splitkv_workspace_bytes(lib):
    for B, H, N, D, S in ((1, 1, 1, 64, 2), (2, 3, 1000, 128, 5), (1, 32, 1024, 64, 256)):
        rows = B * H * N
        want = _align_up(S * rows * D * 4) + _align_up(S * rows * 4)
        assert lib.fa_splitkv_workspace_bytes(B, H, N, D, S) == want
    assert lib.fa_splitkv_workspace_bytes(1, 1, 128, 64, 1) == 0      # one split: no workspace
    assert lib.fa_splitkv_workspace_bytes(1, 1, 128, 96, 2) == 0      # unsupported D
    assert lib.fa_splitkv_workspace_bytes(1, 1, 128, 64, 0) == 0
    assert lib.fa_splitkv_workspace_bytes(1, 1, 128, 64, 257) == 0
    assert lib.fa_splitkv_workspace_bytes(0, 1, 128, 64, 2) == 0


def _splitkv(lib, S=2, ws=1 << 44, ws_bytes=1 << 30, q=16, **kw):
    args = dict(k=32, v=48, o=1 << 40, lse=0, B=1, H=1, N=256, D=64, scale=0.125, causal=0, dtype=0)
    args.update(kw)
    return lib.fa_forward_splitkv(q or None, args["k"] or None, args["v"] or None, args["o"] or None,
                                  args["lse"] or None, args["B"], args["H"], args["N"], args["D"], args["scale"],
                                  args["causal"], args["dtype"], S, ws or None, ws_bytes, None)


def test_splitkv_rejects_bad_arguments_before_any_cuda_call(lib):
    need = lib.fa_splitkv_workspace_bytes(1, 1, 256, 64, 2)
    assert _splitkv(lib, S=-1) == fa.FA_ERR_INVALID_ARG
    assert _splitkv(lib, S=257) == fa.FA_ERR_INVALID_ARG
    assert _splitkv(lib, q=0) == fa.FA_ERR_INVALID_ARG
    assert _splitkv(lib, D=96) == fa.FA_ERR_UNSUPPORTED
    assert _splitkv(lib, ws=0) == fa.FA_ERR_WORKSPACE
    assert _splitkv(lib, ws=(1 << 44) + 16) == fa.FA_ERR_WORKSPACE          # not 256-byte aligned
    assert _splitkv(lib, ws_bytes=need - 1) == fa.FA_ERR_WORKSPACE
    assert _splitkv(lib, ws=1 << 40, ws_bytes=need) == fa.FA_ERR_INVALID_ARG  # overlaps o
    assert _splitkv(lib, ws=0, q=17) == fa.FA_ERR_ALIGN


def _merge(lib, op=1 << 40, lp=1 << 41, P=2, pd=2, o=1 << 42, lse=1 << 43, B=1, H=1, N=8, D=64, dtype=0):
    return lib.fa_merge_partials(op or None, lp or None, P, pd, o or None, lse or None, B, H, N, D, dtype, None)


def test_merge_rejects_bad_arguments_before_any_cuda_call(lib):
    assert _merge(lib, op=0) == fa.FA_ERR_INVALID_ARG
    assert _merge(lib, lp=0) == fa.FA_ERR_INVALID_ARG
    assert _merge(lib, o=0) == fa.FA_ERR_INVALID_ARG
    assert _merge(lib, P=0) == fa.FA_ERR_INVALID_ARG
    assert _merge(lib, N=0) == fa.FA_ERR_INVALID_ARG
    assert _merge(lib, D=96) == fa.FA_ERR_UNSUPPORTED
    assert _merge(lib, pd=3) == fa.FA_ERR_UNSUPPORTED
    assert _merge(lib, dtype=2) == fa.FA_ERR_UNSUPPORTED                   # fp32 output not offered
    assert _merge(lib, op=(1 << 40) + 8) == fa.FA_ERR_ALIGN
    assert _merge(lib, o=(1 << 42) + 8) == fa.FA_ERR_ALIGN
    assert _merge(lib, lp=(1 << 41) + 2) == fa.FA_ERR_ALIGN
    assert _merge(lib, o=(1 << 40) + 256) == fa.FA_ERR_INVALID_ARG         # output inside the parts
    assert _merge(lib, lse=(1 << 41) + 4) == fa.FA_ERR_INVALID_ARG         # lse inside the part lse


def test_naive_workspace_bytes(lib):
    assert lib.fa_naive_workspace_bytes(1, 32, 1024) == 32 * 1024 * 1024 * 2
    assert lib.fa_naive_workspace_bytes(2, 3, 17) == _align_up(2 * 3 * 17 * 17 * 2)
    assert lib.fa_naive_workspace_bytes(0, 1, 8) == 0


def test_naive_rejects_bad_arguments_before_any_cuda_call(lib):
    def call(q=16, dtype=0, D=64, ws=1 << 44, ws_bytes=1 << 30):
        return lib.fa_naive_forward(q or None, 32, 48, 1 << 40, None, 1, 1, 256, D, 0.1, 0, dtype, ws or None,
                                    ws_bytes, None)
    assert call(q=0) == fa.FA_ERR_INVALID_ARG
    assert call(dtype=1) == fa.FA_ERR_UNSUPPORTED        # the naive baseline is fp16 only
    assert call(D=96) == fa.FA_ERR_UNSUPPORTED
    assert call(q=24) == fa.FA_ERR_ALIGN
    assert call(ws=0) == fa.FA_ERR_WORKSPACE
    assert call(ws_bytes=256 * 256 * 2 - 1) == fa.FA_ERR_WORKSPACE
    assert call(ws=1 << 40) == fa.FA_ERR_INVALID_ARG       # workspace overlaps o
    for code in (-8, -9):
        assert lib.fa_error_string(code).decode() != "unknown error code"
