"""Large sizes on the GPU: a 131072-token sequence, thousands of heads, and sampled rows of
each checked against the fp64 oracle (index arithmetic, scheduling and L2-section ordering at
scale). Tolerances as in test_forward.py."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_prefill_gb300 import fa, workloads

pytestmark = pytest.mark.gpu

TOL_O = {"fp16": 2e-3, "bf16": 1e-2}
TOL_LSE = 1e-3


def sampled_check(w, o, lse, n_heads=3, seed=0):
    rng = np.random.default_rng(seed)
    BH, N = w.B * w.H, w.N
    heads = sorted(set([0, BH - 1] + rng.integers(0, BH, size=n_heads).tolist()))
    rows = []
    for bh in heads:
        idx = set(i for i in (0, 1, 127, 128, N // 2, N - 129, N - 128, N - 1) if 0 <= i < N)
        idx |= set(rng.integers(0, N, size=12).tolist())
        rows += [(bh, i) for i in sorted(idx)]
    rows = np.array(rows, dtype=np.int64)
    q, k, v = workloads.make_qkv(w)
    ro, rl = oracle.attention_rows(q, k, v, w.scale, w.causal, rows)
    go = o.float().cpu().numpy().astype(np.float64).reshape(BH, N, w.D)[rows[:, 0], rows[:, 1]]
    gl = lse.cpu().numpy().astype(np.float64).reshape(BH, N)[rows[:, 0], rows[:, 1]]
    assert np.isfinite(go).all() and np.isfinite(gl).all()
    assert np.abs(go - ro).max() <= TOL_O[w.dtype], np.abs(go - ro).max()
    assert np.abs(gl - rl).max() <= TOL_LSE, np.abs(gl - rl).max()


@pytest.mark.parametrize("D,dtype", [(64, "fp16"), (128, "bf16")])
def test_very_long_causal_sequence(D, dtype):
    w = workloads.Workload("long", 1, 1, 131072, D, dtype, True, seed=77 + D)
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    o, lse = fa.forward(q, k, v, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    fa.check_device_status()
    sampled_check(w, o, lse)
    o2, l2 = fa.forward_splitkv(q, k, v, causal=True, scale=w.scale)  # automatic split count
    torch.cuda.synchronize()
    fa.check_device_status()
    sampled_check(w, o2, l2, seed=1)


def test_many_short_heads():
    w = workloads.Workload("heads", 64, 64, 200, 64, "fp16", True, seed=5)  # B*H = 4096, ragged N
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    o, lse = fa.forward(q, k, v, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    fa.check_device_status()
    sampled_check(w, o, lse, n_heads=8)


def test_many_heads_noncausal_d128():
    w = workloads.Workload("heads128", 8, 256, 384, 128, "bf16", False, seed=6)  # B*H = 2048
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    o, lse = fa.forward(q, k, v, causal=False, scale=w.scale)
    torch.cuda.synchronize()
    fa.check_device_status()
    sampled_check(w, o, lse, n_heads=8)
