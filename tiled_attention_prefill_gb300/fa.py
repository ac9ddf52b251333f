"""Python binding of the C-ABI library ``libfa_gb300.so`` (ctypes).

Argument marshalling only: every step of the attention forward pass runs in the
library's CUDA kernel. PyTorch supplies device memory and the current stream.
There is no fallback: if the library is missing or the device is unsupported,
the call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa_gb300.so")

FA_DTYPE_FP16 = 0
FA_DTYPE_BF16 = 1
FA_DTYPE_FP32 = 2
FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_ALIGN = -3
FA_ERR_CUDA = -4
FA_ERR_TIMEOUT = -5
FA_ERR_TOO_LARGE = -6
FA_ERR_WORKSPACE = -7
FA_ERR_SCRATCH = -8
FA_ERR_LIBRARY = -9
NOALLOC_SCRATCH_BYTES = 32 << 20
FA_DECOMP_AUTO = 0
FA_DECOMP_TWO_TILES = 1
FA_DECOMP_SPLIT_KV = 2
FA_DECOMP_SPLIT_KV_SERIAL = 3

# Every symbol include/fa.h declares, with its ctypes signature.
SIGNATURES = {
    "fa_forward": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "fa_error_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fa_version": (ctypes.c_int, []),
    "fa_check_device_status": (ctypes.c_int, []),
    "fa_set_watchdog_ns": (ctypes.c_int, [ctypes.c_ulonglong]),
    "fa_last_cuda_error": (ctypes.c_int, []),
    "fa_set_decomposition": (ctypes.c_int, [ctypes.c_int]),
    "fa_debug_force_stall": (ctypes.c_int, [ctypes.c_int]),
    "fa_debug_work_schedule": (ctypes.c_int, [ctypes.c_int] * 7 + [ctypes.c_void_p, ctypes.c_int]),
    "fa_debug_work_plan": (ctypes.c_int, [ctypes.c_int] * 7 + [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]),
    "fa_debug_num_splits": (ctypes.c_int, [ctypes.c_int] * 7),
    "fa_forward_splitkv": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                          ctypes.c_size_t, ctypes.c_void_p]),
    "fa_forward_splitkv_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, ctypes.c_void_p]),
    "fa_naive_forward": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                        ctypes.c_void_p]),
    "fa_naive_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "fa_naive_last_library_error": (ctypes.c_int, []),
    "fa_splitkv_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int]),
    "fa_splitkv_num_splits": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "fa_schedule_pool_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "fa_merge_partials": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
}

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__("fa error %d: %s" % (code, msg))
        self.code = code


def load_library(path: str | None = None):
    """Load (once) and return the ctypes handle of the library; raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError("%s not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
                              "(needs nvcc for sm_103a)" % p)
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        if path is None:
            _lib = lib
        return lib


def error_string(code: int) -> str:
    return load_library().fa_error_string(int(code)).decode()


def _check(code: int):
    if code != FA_OK:
        msg = error_string(code)
        if code == FA_ERR_CUDA:
            msg += " (cudaError %d)" % load_library().fa_last_cuda_error()
        raise FAError(code, msg)


def check_device_status() -> None:
    """Synchronise the current device and raise FAError if a kernel timed out."""
    _check(load_library().fa_check_device_status())


def schedule_pool_status():
    """(used bytes, capacity bytes) of the current device's work-table pool, and the number of
    launches in this process that needed a work table but ran without one."""
    used = ctypes.c_size_t(0)
    cap = ctypes.c_size_t(0)
    fb = ctypes.c_ulonglong(0)
    _check(load_library().fa_schedule_pool_status(ctypes.byref(used), ctypes.byref(cap), ctypes.byref(fb)))
    return int(used.value), int(cap.value), int(fb.value)


def set_watchdog_ns(ns: int) -> None:
    _check(load_library().fa_set_watchdog_ns(int(ns)))


def set_decomposition(mode: int) -> None:
    """Process-wide work decomposition (FA_DECOMP_AUTO / _TWO_TILES / _SPLIT_KV / _SPLIT_KV_SERIAL)."""
    _check(load_library().fa_set_decomposition(int(mode)))


def debug_force_stall(on: bool) -> None:
    """Test hook: following launches stall on purpose so the device-side watchdog fires."""
    _check(load_library().fa_debug_force_stall(1 if on else 0))


def debug_work_schedule(B: int, H: int, N: int, D: int, causal: bool, dtype: int, num_sms: int):
    """The per-CTA work-item lists ``fa_forward`` would use for this shape on ``num_sms`` SMs
    (host only): a list of ``num_sms`` lists of item indices, or None when the shape's items are
    strided over the CTAs instead."""
    lib = load_library()
    args = (int(B), int(H), int(N), int(D), int(bool(causal)), int(dtype), int(num_sms))
    n = lib.fa_debug_work_schedule(*args, None, 0)
    if n < 0:
        _check(n)
    if n == 0:
        return None
    buf = (ctypes.c_int * n)()
    _check(min(0, lib.fa_debug_work_schedule(*args, ctypes.addressof(buf), n)))
    vals = list(buf)
    off, items = vals[:num_sms + 1], vals[num_sms + 1:]
    return [items[off[c]:off[c + 1]] for c in range(num_sms)]


def forward_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, H: int, N: int, D: int,
                scale: float, causal: bool, dtype: int, stream: int) -> int:
    """Direct call of ``fa_forward`` with integer device pointers; returns the status code."""
    return load_library().fa_forward(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr or None, int(B), int(H), int(N), int(D),
                                     float(scale), int(bool(causal)), int(dtype), stream or None)


def _current_stream_handle(torch, index: int) -> int:
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)  # fast path, present in torch 2.x
    if raw is not None:
        return raw(index)
    return torch.cuda.current_stream(index).cuda_stream


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, return_lse: bool = True):
    """Attention forward on CUDA tensors [B, H, N, D] (fp16, bf16, or fp32 computed on tf32
    tensor cores; contiguous).

    Returns (o, lse) with o like q and lse [B, H, N] fp32 (lse is None when
    ``return_lse`` is False and no buffer was given). Runs on the current stream. A batch with
    no query rows (B, H or N is 0) returns empty outputs without a launch.
    """
    import torch

    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if q.dtype not in (torch.float16, torch.bfloat16, torch.float32) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share dtype fp16, bf16 or fp32")
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape [B, H, N, D]")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    dev = q.get_device()
    if k.get_device() != dev or v.get_device() != dev:
        raise ValueError("q, k, v must be on the same device")
    B, H, N, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or out.get_device() != dev:
        raise ValueError("out must be a contiguous tensor like q")
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous()
                            or lse.get_device() != dev):
        raise ValueError("lse must be a contiguous fp32 tensor [B, H, N]")
    if _empty(q):
        return out, lse
    dtype = {torch.float16: FA_DTYPE_FP16, torch.bfloat16: FA_DTYPE_BF16, torch.float32: FA_DTYPE_FP32}[q.dtype]
    sc = -1.0 if scale is None else float(scale)
    lib = _lib if _lib is not None else load_library()
    lse_ptr = lse.data_ptr() if lse is not None else None
    if dev == torch.cuda.current_device():
        rc = lib.fa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr, B, H, N, D, sc,
                            1 if causal else 0, dtype, _current_stream_handle(torch, dev) or None)
    else:
        with torch.cuda.device(dev):
            rc = lib.fa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr, B, H, N, D, sc,
                                1 if causal else 0, dtype, _current_stream_handle(torch, dev) or None)
    if rc != FA_OK:
        _check(rc)
    return out, lse


def _empty(q) -> bool:
    """True for a batch with no query rows (B, H or N is 0), after D is checked: the result is
    empty, and the C entry points, which take sizes >= 1, are not called."""
    if q.numel() != 0:
        return False
    if q.shape[3] not in (64, 128):
        _check(FA_ERR_UNSUPPORTED)
    return True


def _check_qkv(torch, q, k, v):
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if q.dtype not in (torch.float16, torch.bfloat16) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share dtype fp16 or bf16")
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape [B, H, N, D]")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    if k.get_device() != q.get_device() or v.get_device() != q.get_device():
        raise ValueError("q, k, v must be on the same device")


def splitkv_num_splits(B: int, H: int, N: int, D: int, causal: bool) -> int:
    """Split count ``fa_forward_splitkv`` chooses for num_splits = 0 (needs the device)."""
    rc = load_library().fa_splitkv_num_splits(int(B), int(H), int(N), int(D), int(bool(causal)))
    if rc < 0:
        _check(rc)
    return rc


def splitkv_workspace_bytes(B: int, H: int, N: int, D: int, num_splits: int) -> int:
    return int(load_library().fa_splitkv_workspace_bytes(int(B), int(H), int(N), int(D), int(num_splits)))


def forward_splitkv(q, k, v, causal: bool = False, scale: float | None = None, num_splits: int = 0,
                    workspace=None, out=None, lse=None, return_lse: bool = True):
    """Split-KV forward (``fa_forward_splitkv``): same result as :func:`forward`.

    ``num_splits`` 0 lets the library choose. ``workspace`` is a CUDA uint8 tensor of at least
    ``splitkv_workspace_bytes`` bytes (256-byte aligned); allocated here when None. Returns
    (o, lse) like :func:`forward`; the workspace afterwards holds the partial results.
    """
    import torch

    _check_qkv(torch, q, k, v)
    B, H, N, D = q.shape
    dev = q.get_device()
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if _empty(q):
        return out, lse
    with torch.cuda.device(dev):
        splits = num_splits if num_splits > 0 else splitkv_num_splits(B, H, N, D, causal)
        if workspace is None:
            nbytes = splitkv_workspace_bytes(B, H, N, D, splits)
            workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
        dtype = FA_DTYPE_BF16 if q.dtype == torch.bfloat16 else FA_DTYPE_FP16
        sc = -1.0 if scale is None else float(scale)
        rc = load_library().fa_forward_splitkv(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr() if lse is not None else None,
            B, H, N, D, sc, 1 if causal else 0, dtype, int(splits), workspace.data_ptr(), workspace.numel(),
            _current_stream_handle(torch, dev) or None)
    _check(rc)
    return out, lse


def merge_partials(o_parts, lse_parts, out_dtype=None, out=None, lse=None):
    """``fa_merge_partials``: o_parts [P, B, H, N, D] (fp16/bf16/fp32), lse_parts [P, B, H, N] fp32.

    Returns (o [B, H, N, D] in ``out_dtype`` (default: the parts' type, fp16 for fp32 parts),
    lse [B, H, N] fp32).
    """
    import torch

    if o_parts.dim() != 5 or lse_parts.shape != o_parts.shape[:4]:
        raise ValueError("o_parts [P, B, H, N, D] and lse_parts [P, B, H, N] expected")
    if not (o_parts.is_cuda and lse_parts.is_cuda and o_parts.is_contiguous() and lse_parts.is_contiguous()):
        raise ValueError("parts must be contiguous CUDA tensors")
    if lse_parts.dtype != torch.float32:
        raise ValueError("lse_parts must be fp32")
    kinds = {torch.float16: FA_DTYPE_FP16, torch.bfloat16: FA_DTYPE_BF16, torch.float32: FA_DTYPE_FP32}
    if o_parts.dtype not in kinds:
        raise ValueError("o_parts must be fp16, bf16 or fp32")
    P, B, H, N, D = o_parts.shape
    if out_dtype is None:
        out_dtype = torch.float16 if o_parts.dtype == torch.float32 else o_parts.dtype
    if out is None:
        out = torch.empty((B, H, N, D), dtype=out_dtype, device=o_parts.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=o_parts.device)
    dev = o_parts.get_device()
    with torch.cuda.device(dev):
        rc = load_library().fa_merge_partials(
            o_parts.data_ptr(), lse_parts.data_ptr(), P, kinds[o_parts.dtype], out.data_ptr(), lse.data_ptr(),
            B, H, N, D, FA_DTYPE_BF16 if out.dtype == torch.bfloat16 else FA_DTYPE_FP16,
            _current_stream_handle(torch, dev) or None)
    _check(rc)
    return out, lse


def forward_splitkv_noalloc(q, k, v, causal: bool = False, scale: float | None = None, num_splits: int = 0,
                            out=None, lse=None, return_lse: bool = True):
    """``fa_forward_splitkv_noalloc``: split-KV forward whose partials go to the library's built-in
    32 MiB per-device scratch (no workspace argument, no allocation in the library). Calls that
    overlap in time on one device race on that scratch."""
    import torch

    _check_qkv(torch, q, k, v)
    B, H, N, D = q.shape
    dev = q.get_device()
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if _empty(q):
        return out, lse
    dtype = FA_DTYPE_BF16 if q.dtype == torch.bfloat16 else FA_DTYPE_FP16
    sc = -1.0 if scale is None else float(scale)
    with torch.cuda.device(dev):
        rc = load_library().fa_forward_splitkv_noalloc(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr() if lse is not None else None,
            B, H, N, D, sc, 1 if causal else 0, dtype, int(num_splits), _current_stream_handle(torch, dev) or None)
    _check(rc)
    return out, lse


def naive_workspace_bytes(B: int, H: int, N: int) -> int:
    return int(load_library().fa_naive_workspace_bytes(int(B), int(H), int(N)))


def naive_forward(q, k, v, causal: bool = False, scale: float | None = None, workspace=None, out=None, lse=None,
                  return_lse: bool = True):
    """``fa_naive_forward``: the unfused baseline (S = scale QK^T and P written to memory, fp16 only).

    ``workspace``: CUDA uint8 tensor of at least ``naive_workspace_bytes`` bytes (allocated here
    when None). Returns (o, lse) like :func:`forward`.
    """
    import torch

    _check_qkv(torch, q, k, v)
    B, H, N, D = q.shape
    dev = q.get_device()
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(naive_workspace_bytes(B, H, N), dtype=torch.uint8, device=q.device)
    dtype = FA_DTYPE_BF16 if q.dtype == torch.bfloat16 else FA_DTYPE_FP16
    sc = -1.0 if scale is None else float(scale)
    with torch.cuda.device(dev):
        rc = load_library().fa_naive_forward(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr() if lse is not None else None,
            B, H, N, D, sc, 1 if causal else 0, dtype, workspace.data_ptr(), workspace.numel(),
            _current_stream_handle(torch, dev) or None)
    if rc == FA_ERR_LIBRARY:
        raise FAError(rc, error_string(rc) + " (cublasStatus %d)" % load_library().fa_naive_last_library_error())
    _check(rc)
    return out, lse


def debug_num_splits(B: int, H: int, N: int, D: int, causal: bool, num_sms: int, noalloc: bool = False) -> int:
    """The split count ``splitkv_num_splits`` gives for this shape on ``num_sms`` SMs, or with
    ``noalloc`` the one ``forward_splitkv_noalloc`` runs with ``num_splits=0`` (host only)."""
    n = load_library().fa_debug_num_splits(int(B), int(H), int(N), int(D), int(bool(causal)), int(num_sms),
                                           int(bool(noalloc)))
    if n < 0:
        _check(n)
    return n


def debug_work_plan(B: int, H: int, N: int, D: int, causal: bool, dtype: int, num_sms: int):
    """The work decomposition ``fa_forward`` would use for this shape on ``num_sms`` SMs (host
    only): a dict with ``items``, ``single_tile``, ``paired``, ``dispatch`` and ``grid``, and for
    paired launches ``units``, one tuple per CTA (item a, item b or -1, tiles of a, tiles of b,
    tiles of warpgroup 0, tiles of warpgroup 1)."""
    lib = load_library()
    args = (int(B), int(H), int(N), int(D), int(bool(causal)), int(dtype), int(num_sms))
    plan = (ctypes.c_int * 5)()
    n = lib.fa_debug_work_plan(*args, ctypes.addressof(plan), None, 0)
    if n < 0:
        _check(n)
    out = dict(zip(("items", "single_tile", "paired", "dispatch", "grid"), list(plan)))
    out["single_tile"], out["paired"], out["dispatch"] = (bool(out[k]) for k in ("single_tile", "paired", "dispatch"))
    out["units"] = None
    if n > 0:
        buf = (ctypes.c_int * n)()
        _check(min(0, lib.fa_debug_work_plan(*args, ctypes.addressof(plan), ctypes.addressof(buf), n)))
        vals = list(buf)
        out["units"] = [tuple(vals[6 * c:6 * c + 6]) for c in range(n // 6)]
    return out
