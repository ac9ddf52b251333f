"""GPU parity of the naive (unfused) baseline against the fp64 oracle.

The baseline stores S = scale QK^T in fp16 before the softmax (the pages' naive form), so its
error budget is larger than the fused kernel's: rounding a score s to fp16 moves it by at
most 2^-11 |s|, about 3e-3 for the |s| < 6 of N(0,1) inputs. That shifts lse by at most that
much (tolerance 4e-3) and O by at most max|ds| * max|v_j - O_i| (tolerance 1e-2, with the
fp16 rounding of P on top, as in the fused kernel).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_prefill_gb300 import fa, workloads

pytestmark = pytest.mark.gpu

TOL_O = 1e-2
TOL_LSE = 4e-3


def run_naive(q, k, v, causal, scale):
    o, lse = fa.naive_forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def check(o, lse, ro, rl, what):
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    assert np.abs(o - ro).max() <= TOL_O, "%s O err %.3e" % (what, np.abs(o - ro).max())
    assert np.abs(lse - rl).max() <= TOL_LSE, "%s lse err %.3e" % (what, np.abs(lse - rl).max())


@pytest.mark.parametrize("shape", [(1, 1, 1, 64), (1, 2, 17, 128), (2, 1, 128, 64), (1, 3, 200, 64),
                                   (1, 1, 256, 128), (1, 2, 1000, 64)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_naive_small_shapes(shape, causal):
    B, H, N, D = shape
    w = workloads.Workload("t", B, H, N, D, "fp16", causal, seed=3 * N + D)
    q, k, v = workloads.make_qkv(w)
    o, lse = run_naive(q, k, v, causal, w.scale)
    ro, rl = oracle.attention(q, k, v, w.scale, causal)
    check(o, lse, ro, rl, str(shape))


@pytest.mark.parametrize("name", ["c2", "c3", "c3c"])
def test_naive_workloads(name):
    w = workloads.WORKLOADS[name]
    q, k, v = workloads.make_qkv(w)
    o, lse = run_naive(q, k, v, w.causal, w.scale)
    ro, rl = oracle.attention(q, k, v, w.scale, w.causal)
    check(o, lse, ro, rl, name)


def test_naive_and_fused_agree():
    """Both paths on the headline workload: within the naive tolerance of each other."""
    w = workloads.WORKLOADS["c2"]
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    o1, l1 = fa.forward(q, k, v, causal=True, scale=w.scale)
    o2, l2 = fa.naive_forward(q, k, v, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= TOL_O
    assert (l1 - l2).abs().max().item() <= TOL_LSE


def test_naive_rejects_bf16():
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.naive_forward(x, x, x)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED
