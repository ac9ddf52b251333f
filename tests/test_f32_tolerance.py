"""Where the 5e-3 tolerance of the fp32-I/O (tf32) forward comes from (CPU only).

The fp32 variant is the first page's second compile-time build ("Android Transformer
Optimization: Attention and Mobile GPU Bottlenecks", section "Pitfalls I Hit": an fp32
build beside the fp16 one). On GB300 its products run on the tensor cores as tf32:

1. The tensor core reads Q, K and V as tf32: the top 19 bits of each fp32 value, i.e. the
   low 13 mantissa bits dropped (truncation, relative change < 2^-10). Exact attention on
   the truncated inputs differs from exact attention on the fp32 inputs; the oracle computes
   both. The largest difference is at the first rows of causal heads, where O is one or two
   V rows (so up to 2^-10 * max|v|), and the lse moves by the truncation of the scores.
   Pinned below: at most 3.5e-3 in O and lse on every fp32 shape the GPU tests use.
2. The kernel rounds P to tf32 (nearest, ties away from zero, relative change <= 2^-11)
   before the P V product, while l sums the unrounded p. Pinned below with a direct fp64
   computation on truncated inputs: at most 5e-4 in O.
3. Everything else is fp32 arithmetic (scores, exp2, sums over at most a few thousand keys):
   below 1e-5 on these shapes.

So the kernel is within 3.5e-3 + 5e-4 + 1e-5 < 4.1e-3 of the oracle, and the GPU tests use
5e-3 for O and lse.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from tiled_attention_prefill_gb300 import workloads

TRUNC_BOUND = 3.5e-3
P_ROUND_BOUND = 5e-4
GPU_TOL = 5e-3

# the shapes of the GPU tests of the fp32 path (tests/test_f32.py), both masks
SMALL = [(1, 1, 1, 64), (1, 2, 17, 128), (1, 1, 64, 64), (1, 1, 65, 128), (2, 3, 128, 64), (1, 1, 129, 64),
         (1, 2, 200, 128), (1, 1, 257, 64), (1, 2, 640, 128), (1, 1, 1000, 64)]


def tf32_truncate(x: torch.Tensor) -> torch.Tensor:
    """The top 19 bits of each fp32 value (sign, exponent, 10 mantissa bits)."""
    return (x.contiguous().view(torch.int32) & ~0x1FFF).view(torch.float32)


def tf32_round_away(p: np.ndarray) -> np.ndarray:
    """Nearest tf32, ties away from zero, of fp32 values >= 0 (half a tf32 unit added, then truncated)."""
    b = p.astype(np.float32).view(np.int32).astype(np.int64)
    return ((b + 0x1000) & ~0x1FFF).astype(np.int32).view(np.float32).astype(np.float64)


def truncation_effect(w):
    q, k, v = workloads.make_qkv(w)
    ro, rl = oracle.attention(q, k, v, w.scale, w.causal)
    to, tl = oracle.attention(tf32_truncate(q), tf32_truncate(k), tf32_truncate(v), w.scale, w.causal)
    return float(np.abs(ro - to).max()), float(np.abs(rl - tl).max())


def cases():
    out = [workloads.WORKLOADS["c2_f32"], workloads.WORKLOADS["c3_f32"]]
    for (B, H, N, D) in SMALL:
        for causal in (False, True):
            out.append(workloads.Workload("t", B, H, N, D, "fp32", causal, seed=13 * N + D))
    return out


def test_truncation_effect_pinned():
    worst_o = worst_l = 0.0
    for w in cases():
        eo, el = truncation_effect(w)
        assert eo <= TRUNC_BOUND and el <= TRUNC_BOUND, (w, eo, el)
        worst_o, worst_l = max(worst_o, eo), max(worst_l, el)
    # the bound is not loose by an order of magnitude (it is what the tolerance rests on)
    assert max(worst_o, worst_l) > 0.5 * TRUNC_BOUND


def test_truncation_of_a_single_key_is_the_v_truncation():
    # N = 1: O = v_0 exactly, so the effect is exactly |v_0 - trunc(v_0)| < 2^-10 |v_0|.
    w = workloads.Workload("t", 1, 1, 1, 64, "fp32", False, seed=13 + 64)
    q, k, v = workloads.make_qkv(w)
    ro, _ = oracle.attention(q, k, v, w.scale, False)
    to, _ = oracle.attention(tf32_truncate(q), tf32_truncate(k), tf32_truncate(v), w.scale, False)
    v64 = v.double().numpy()
    assert np.array_equal(to, tf32_truncate(v).double().numpy())
    assert np.all(np.abs(ro - to) < 2.0 ** -10 * np.abs(v64) + 1e-30)


def test_p_rounding_effect_pinned():
    """P rounded to tf32 before the product, l from the unrounded p, on truncated inputs."""
    worst = 0.0
    for name, heads in (("c2_f32", range(0, 32, 3)), ("c3_f32", range(0, 32, 8))):
        w = workloads.WORKLOADS[name]
        q, k, v = (tf32_truncate(x).double().numpy() for x in workloads.make_qkv(w))
        for bh in heads:
            s = (q[0, bh] @ k[0, bh].T) * w.scale
            if w.causal:
                s = np.where(np.tril(np.ones(s.shape, dtype=bool)), s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            l = p.sum(axis=1, keepdims=True)
            o_exact = p @ v[0, bh] / l
            o_round = tf32_round_away(p) @ v[0, bh] / l
            worst = max(worst, float(np.abs(o_round - o_exact).max()))
    assert worst <= P_ROUND_BOUND, worst


def test_gpu_tolerance_covers_the_budget():
    assert TRUNC_BOUND + P_ROUND_BOUND + 1e-5 < GPU_TOL
    import tests.test_f32 as t
    assert t.TOL == GPU_TOL
