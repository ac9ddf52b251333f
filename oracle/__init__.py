"""Attention forward oracle (fp64, CPU).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline of ``bench.py`` may import this package. The CUDA library shares no
code with it and never calls it.

What it computes is the plain definition of the attention forward pass, as
stated in "Android Transformer Optimization: Attention and Mobile GPU
Bottlenecks", section "The Self-Attention Bottleneck Is Memory Traffic, Not
Compute" (S = QK^T, P = softmax(S), O = PV, the score matrix materialised and
swept three times), with the scale 1/sqrt(headDim) applied to the scores as
the SGEMM alpha of "Flash Attention on Android: tiled SGEMM with
RenderScript", section "Architecture: tiled attention with RenderScript BLAS":

    s_ij = scale * q_i . k_j          j in J(i) = {0..N-1} or {0..i} (causal)
    M_i  = max_j s_ij
    L_i  = sum_j exp(s_ij - M_i)
    O_i  = sum_j exp(s_ij - M_i) v_j / L_i
    lse_i = M_i + ln L_i

Entry points:

* ``attention_rows`` / ``attention``: the C implementation
  (``attention_oracle.c``, fp64, OpenMP over rows) for any size, on all rows
  or on a sampled subset of rows.
* ``attention_keys`` and ``attention_rows(..., key_ranges=...)``: the same
  definition restricted to a range of keys, the partial result that split-KV
  work produces (lse = -inf and O = 0 where the range holds no key of J(i)).
* ``merge_partials`` (``merge.py``): partial results over disjoint key sets
  combined by the online-softmax update.
* ``attention_np``: the same definition in numpy, for tiny cases (a second,
  independent writing used to cross-check the C code).
* ``online_softmax_blockwise``: the pages' tiled recurrence (section "The
  Essence of FlashAttention: Reordering the Computation" and "A Complete Tile
  Loop" of the first page: running max m, denominator l and output O, rescaled
  by exp(m_old - m_new) whenever a new tile raises the max, normalised once at
  the end), in fp64 with arbitrary row/column tile sizes. Its agreement with
  the unfused definition is the pages' claim that the reordering does not
  change the result; the tests check that claim.

Every function takes tensors/arrays of shape [B, H, N, D] (any float dtype;
widened exactly to fp64) and returns fp64 numpy arrays: O [B, H, N, D] (or
[R, D] for sampled rows) and lse [B, H, N] (or [R]).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .merge import merge_partials  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_attention.so")
_lock = threading.Lock()
_lib = None


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the C oracle with gcc (OpenMP when available, no fast-math)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math", *extra_flags]
    tmp = out + ".tmp.%d" % os.getpid()
    try:
        subprocess.run(base + ["-fopenmp", src, "-o", tmp, "-lm"], check=True,
                       stdout=subprocess.PIPE, stderr=subprocess.PIPE)
    except subprocess.CalledProcessError:
        subprocess.run(base + [src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build ``_build/liboracle_attention.so`` if missing or older than the source."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_oracle()
    return _LIB_PATH


def load_library(path: str):
    lib = ctypes.CDLL(path)
    f = lib.oracle_attention_rows_f64
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
                  ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    f = lib.oracle_attention_rows_keyrange_f64
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
                  ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    return lib


def _get_lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
        return _lib


def max_threads() -> int:
    return int(_get_lib().oracle_max_threads())


def to_f64(x) -> np.ndarray:
    """Exact widening of a torch tensor or numpy array to a C-contiguous fp64 array."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch  # local: only when given torch tensors
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def attention_rows(q, k, v, scale: float, causal: bool, rows, nthreads: int = 0, lib=None,
                   key_ranges=None):
    """Oracle on sampled rows. ``rows``: int array [R, 2] of (bh, i) with bh = b*H + h.

    ``key_ranges`` (optional, int [R, 2]): request r uses only the keys j of J(i) with
    key_ranges[r, 0] <= j < key_ranges[r, 1] (the partial result of that key range; a range
    with no such key gives o = 0, lse = -inf). Returns (o [R, D], lse [R]) in fp64.
    """
    q64, k64, v64 = to_f64(q), to_f64(k), to_f64(v)
    B, H, N, D = q64.shape
    assert k64.shape == q64.shape and v64.shape == q64.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    R = rows.shape[0]
    o = np.empty((R, D), dtype=np.float64)
    lse = np.empty((R,), dtype=np.float64)
    lib = lib if lib is not None else _get_lib()
    if key_ranges is None:
        rc = lib.oracle_attention_rows_f64(
            q64.ctypes.data, k64.ctypes.data, v64.ctypes.data,
            B * H, N, D, float(scale), int(bool(causal)),
            rows.ctypes.data, R, o.ctypes.data, lse.ctypes.data, int(nthreads))
    else:
        kr = np.ascontiguousarray(np.asarray(key_ranges, dtype=np.int64).reshape(-1, 2))
        assert kr.shape[0] == R
        rc = lib.oracle_attention_rows_keyrange_f64(
            q64.ctypes.data, k64.ctypes.data, v64.ctypes.data,
            B * H, N, D, float(scale), int(bool(causal)),
            rows.ctypes.data, R, kr.ctypes.data, o.ctypes.data, lse.ctypes.data, int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attention_rows_f64 failed with code %d" % rc)
    return o, lse


def attention(q, k, v, scale: float, causal: bool, nthreads: int = 0, lib=None):
    """Oracle on every row. Returns (o [B,H,N,D], lse [B,H,N]) in fp64."""
    B, H, N, D = tuple(q.shape)
    bh, i = np.meshgrid(np.arange(B * H), np.arange(N), indexing="ij")
    rows = np.stack([bh.ravel(), i.ravel()], axis=1)
    o, lse = attention_rows(q, k, v, scale, causal, rows, nthreads=nthreads, lib=lib)
    return o.reshape(B, H, N, D), lse.reshape(B, H, N)


def attention_keys(q, k, v, scale: float, causal: bool, lo: int, hi: int, nthreads: int = 0, lib=None):
    """Partial result of every row over the keys lo <= j < hi (within J(i)).

    Returns (o [B,H,N,D], lse [B,H,N]) in fp64; rows without a key get o = 0, lse = -inf.
    """
    B, H, N, D = tuple(q.shape)
    bh, i = np.meshgrid(np.arange(B * H), np.arange(N), indexing="ij")
    rows = np.stack([bh.ravel(), i.ravel()], axis=1)
    kr = np.tile(np.array([[lo, hi]], dtype=np.int64), (rows.shape[0], 1))
    o, lse = attention_rows(q, k, v, scale, causal, rows, nthreads=nthreads, lib=lib, key_ranges=kr)
    return o.reshape(B, H, N, D), lse.reshape(B, H, N)


def attention_np(q, k, v, scale: float, causal: bool):
    """The same definition in numpy (fp64); materialises S = scale*QK^T per head."""
    q64, k64, v64 = to_f64(q), to_f64(k), to_f64(v)
    B, H, N, D = q64.shape
    o = np.empty_like(q64)
    lse = np.empty((B, H, N), dtype=np.float64)
    allowed = np.tril(np.ones((N, N), dtype=bool)) if causal else np.ones((N, N), dtype=bool)
    for b in range(B):
        for h in range(H):
            s = scale * (q64[b, h] @ k64[b, h].T)          # S, written out in full
            s = np.where(allowed, s, -np.inf)
            m = s.max(axis=1, keepdims=True)                # pass 1
            e = np.exp(s - m)
            l = e.sum(axis=1, keepdims=True)                # pass 2
            o[b, h] = (e @ v64[b, h]) / l                   # pass 3
            lse[b, h] = m[:, 0] + np.log(l[:, 0])
    return o, lse


def online_softmax_blockwise(q, k, v, scale: float, causal: bool, block_m: int, block_n: int):
    """The pages' tiled loop with the online-softmax update, in fp64.

    Outer loop over query row blocks of ``block_m`` rows, inner loop over
    key/value column blocks of ``block_n`` columns (the last block of either
    may be short). Per row: m = -inf, l = 0, O = 0 at the start; for each
    column block, m_new = max(m_old, rowmax(S_blk)), alpha = exp(m_old -
    m_new), l = l*alpha + rowsum(exp(S_blk - m_new)), O = O*alpha +
    exp(S_blk - m_new) @ V_blk; after the last block O /= l. lse = m + ln l.
    Causally masked entries of a block are -inf (exp gives 0).
    """
    q64, k64, v64 = to_f64(q), to_f64(k), to_f64(v)
    B, H, N, D = q64.shape
    o = np.empty_like(q64)
    lse = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            Q, K, V = q64[b, h], k64[b, h], v64[b, h]
            for r0 in range(0, N, block_m):
                r1 = min(r0 + block_m, N)
                Qs = Q[r0:r1]
                m = np.full((r1 - r0, 1), -np.inf)
                l = np.zeros((r1 - r0, 1))
                O = np.zeros((r1 - r0, D))
                for c0 in range(0, N, block_n):
                    c1 = min(c0 + block_n, N)
                    S = scale * (Qs @ K[c0:c1].T)
                    if causal:
                        rows = np.arange(r0, r1)[:, None]
                        cols = np.arange(c0, c1)[None, :]
                        S = np.where(cols <= rows, S, -np.inf)
                    m_new = np.maximum(m, S.max(axis=1, keepdims=True))
                    alpha = np.exp(m - m_new)
                    P = np.exp(S - m_new)
                    l = l * alpha + P.sum(axis=1, keepdims=True)
                    O = O * alpha + P @ V[c0:c1]
                    m = m_new
                o[b, h, r0:r1] = O / l
                lse[b, h, r0:r1] = m[:, 0] + np.log(l[:, 0])
    return o, lse
