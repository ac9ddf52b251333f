"""GPU parity of the paired split-K form (causal launches at D = 64 with between one and two
single-query-tile items per SM: each CTA runs a long and a short query tile at once, the
second warpgroup storing the short one itself before it takes the rest of the long one).
Whole outputs against the fp64 oracle, the same launches with pairing turned off, run-to-run
determinism and a CUDA-graph replay. Tolerances as in test_forward.py."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_prefill_gb300 import fa, workloads

pytestmark = pytest.mark.gpu

TOL_O = {"fp16": 2e-3, "bf16": 1e-2}
TOL_LSE = 1e-3
CODE = {"fp16": fa.FA_DTYPE_FP16, "bf16": fa.FA_DTYPE_BF16}


def num_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def paired_heads(N, D, dtype):
    """A head count whose causal launch at this N is paired on this GPU (one to two items per
    SM, too few two-tile items to fill it)."""
    G, nqt = num_sms(), -(-N // 128)
    for H in range(G // nqt + 1, 2 * G // nqt + 1):
        if fa.debug_work_plan(1, H, N, D, True, CODE[dtype], G)["paired"]:
            return H
    pytest.skip("no paired head count for N=%d on %d SMs" % (N, G))


def check(w, o, lse, ro, rl):
    go = o.double().cpu().numpy()
    gl = lse.double().cpu().numpy()
    assert np.isfinite(go).all() and np.isfinite(gl).all()
    assert np.abs(go - ro).max() <= TOL_O[w.dtype], np.abs(go - ro).max()
    assert np.abs(gl - rl).max() <= TOL_LSE, np.abs(gl - rl).max()


@pytest.mark.parametrize("N,D,dtype", [(1024, 64, "fp16"), (1024, 64, "bf16"), (1000, 64, "fp16"),
                                       (1536, 64, "bf16"), (640, 64, "fp16"), (300, 64, "bf16")])
def test_paired_matches_oracle_and_serial(N, D, dtype):
    H = paired_heads(N, D, dtype)
    w = workloads.Workload("pair", 1, H, N, D, dtype, True, seed=900 + N + D)
    q, k, v = workloads.make_qkv(w)
    ro, rl = oracle.attention(q, k, v, w.scale, True)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.forward(qc, kc, vc, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    fa.check_device_status()
    check(w, o, lse, ro, rl)
    o2, l2 = fa.forward(qc, kc, vc, causal=True, scale=w.scale)  # deterministic
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, l2)
    try:
        fa.set_decomposition(fa.FA_DECOMP_SPLIT_KV_SERIAL)
        os_, ls_ = fa.forward(qc, kc, vc, causal=True, scale=w.scale)
        torch.cuda.synchronize()
        fa.check_device_status()
    finally:
        fa.set_decomposition(fa.FA_DECOMP_AUTO)
    check(w, os_, ls_, ro, rl)


def test_paired_in_a_cuda_graph_matches_eager():
    w = workloads.WORKLOADS["c2"]
    assert fa.debug_work_plan(w.B, w.H, w.N, w.D, True, CODE[w.dtype], num_sms())["paired"]
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.N, device="cuda")
    fa.forward(q, k, v, causal=True, scale=w.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    ref_o, ref_l = o.clone(), lse.clone()
    o.zero_()
    lse.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fa.forward(q, k, v, causal=True, scale=w.scale, out=o, lse=lse)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    fa.check_device_status()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)


def test_paired_batch_with_two_sequences():
    # two sequences of the batch: the pairs mix heads of both
    G = num_sms()
    w = workloads.Workload("pairb", 2, 16, 1024, 64, "fp16", True, seed=31)
    if not fa.debug_work_plan(w.B, w.H, w.N, w.D, True, CODE[w.dtype], G)["paired"]:
        pytest.skip("not paired on %d SMs" % G)
    q, k, v = workloads.make_qkv(w)
    ro, rl = oracle.attention(q, k, v, w.scale, True)
    o, lse = fa.forward(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=w.scale)
    torch.cuda.synchronize()
    fa.check_device_status()
    check(w, o, lse, ro, rl)
