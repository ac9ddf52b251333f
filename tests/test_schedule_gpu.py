"""GPU: causal launches with more than two waves of items run on a persistent grid with
per-CTA item lists (the dispatch-order schedule). Checked against the fp64 oracle on whole
heads, with the schedule in place, when the first call of a shape happens inside CUDA graph
capture (no schedule can be made then: one CTA per item), and with a graph replayed after
the schedule exists. Tolerances as in test_forward.py."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_prefill_gb300 import fa, workloads

pytestmark = pytest.mark.gpu

TOL_O = {"fp16": 2e-3, "bf16": 1e-2, "fp32": 5e-3}
TOL_LSE = {"fp16": 1e-3, "bf16": 1e-3, "fp32": 5e-3}


def check_heads(w, q, k, v, o, lse, heads):
    for bh in heads:
        b, h = divmod(bh, w.H)
        ro, rl = oracle.attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], w.scale, True)
        go = o[b:b + 1, h:h + 1].double().cpu().numpy()
        gl = lse[b:b + 1, h:h + 1].double().cpu().numpy()
        assert np.abs(go - ro).max() <= TOL_O[w.dtype], (bh, np.abs(go - ro).max())
        assert np.abs(gl - rl).max() <= TOL_LSE[w.dtype], (bh, np.abs(gl - rl).max())


@pytest.mark.parametrize("B,H,N,D,dtype", [(1, 64, 1280, 64, "fp16"), (2, 32, 1536, 128, "bf16"),
                                           (1, 40, 1000, 64, "fp32")])
def test_scheduled_causal_matches_oracle(B, H, N, D, dtype):
    w = workloads.Workload("sched", B, H, N, D, dtype, True, seed=300 + H)
    code = {"fp16": fa.FA_DTYPE_FP16, "bf16": fa.FA_DTYPE_BF16, "fp32": fa.FA_DTYPE_FP32}[dtype]
    assert fa.debug_work_schedule(B, H, N, D, True, code, torch.cuda.get_device_properties(0).multi_processor_count) \
        is not None
    q, k, v = workloads.make_qkv(w)
    o, lse = fa.forward(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=w.scale)
    torch.cuda.synchronize()
    fa.check_device_status()
    check_heads(w, q, k, v, o, lse, heads=[0, 1, B * H // 2, B * H - 1])


def test_first_call_inside_graph_capture_then_scheduled_replay():
    # A shape not used by any other test: its first call is captured, so no schedule is made
    # (one CTA per item); a later eager call makes the schedule; a second graph uses it.
    w = workloads.Workload("cap", 1, 48, 1664, 64, "fp16", True, seed=4711)
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    fa.forward(q[:, :1, :256].contiguous(), k[:, :1, :256].contiguous(), v[:, :1, :256].contiguous(), causal=True)
    torch.cuda.synchronize()  # the device is set up (status word) before any capture
    outs = []
    for _ in range(2):
        o = torch.empty_like(q)
        lse = torch.empty(w.B, w.H, w.N, device="cuda")
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                fa.forward(q, k, v, causal=True, scale=w.scale, out=o, lse=lse)
        g.replay()
        torch.cuda.synchronize()
        fa.check_device_status()
        outs.append((o.clone(), lse.clone()))
        o2, l2 = fa.forward(q, k, v, causal=True, scale=w.scale)  # eager: makes the schedule
        torch.cuda.synchronize()
        outs.append((o2, l2))
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    check_heads(w, q.cpu(), k.cpu(), v.cpu(), outs[0][0], outs[0][1], heads=[0, 23, 47])


def test_first_call_on_a_side_stream_then_another_stream():
    # A shape no other test uses: its first call copies the work table asynchronously on a
    # non-blocking side stream; a second call of the same shape, issued right away on another
    # non-blocking stream (no host synchronisation in between), must wait for that copy.
    w = workloads.Workload("async", 1, 56, 1408, 64, "fp16", True, seed=5150)
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    torch.cuda.synchronize()
    used0, cap, fb0 = fa.schedule_pool_status()
    s1 = torch.cuda.Stream()
    s2 = torch.cuda.Stream()
    with torch.cuda.stream(s1):
        o1, l1 = fa.forward(q, k, v, causal=True, scale=w.scale)
    with torch.cuda.stream(s2):
        o2, l2 = fa.forward(q, k, v, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    fa.check_device_status()
    used1, cap1, fb1 = fa.schedule_pool_status()
    assert cap1 == cap == 4 << 20
    assert used1 > used0, "the shape's work table was not made"
    assert fb1 == fb0, "a launch ran without its work table"
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    check_heads(w, q.cpu(), k.cpu(), v.cpu(), o1, l1, heads=[0, 27, 55])
