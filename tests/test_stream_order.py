"""Every entry point back to back on one stream, and the fused forward inside a CUDA graph.

The kernels are launched with programmatic stream serialization (each waits for the previous
kernel's writes with griddepcontrol.wait), so a sequence that mixes them (fused forward, fp32
forward, split-KV partials and merge, the merge on its own, the naive baseline) checks that each
one still sees the results of the one before it. Each output is compared with the oracle.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_prefill_gb300 import fa, workloads

pytestmark = pytest.mark.gpu


def err(a, b):
    return float(np.abs(a.double().cpu().numpy() - b).max())


def test_mixed_sequence_on_one_stream():
    w = workloads.Workload("m", 1, 3, 640, 64, "fp16", True, seed=4242)
    q, k, v = workloads.make_qkv(w)
    ro, rl = oracle.attention(q, k, v, w.scale, True)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    w32 = w.with_(dtype="fp32")
    q32, k32, v32 = workloads.make_qkv(w32)
    ro32, rl32 = oracle.attention(q32, k32, v32, w32.scale, True)
    q32c, k32c, v32c = q32.cuda(), k32.cuda(), v32.cuda()
    # the fused output feeds the next forward as its V: a consumer that must see the producer
    outs = []
    for rep in range(3):
        o1, l1 = fa.forward(qc, kc, vc, causal=True, scale=w.scale)
        o2, l2 = fa.forward_splitkv(qc, kc, vc, causal=True, scale=w.scale, num_splits=3)
        o3, l3 = fa.forward(q32c, k32c, v32c, causal=True, scale=w32.scale)
        o4, l4 = fa.naive_forward(qc, kc, vc, causal=True, scale=w.scale)
        o5, l5 = fa.forward(qc, kc, o1, causal=True, scale=w.scale)  # V = previous output
        parts = torch.stack([o1.float(), o2.float()])
        o6, l6 = fa.merge_partials(parts, torch.stack([l1, l2]), out_dtype=torch.float16)
        outs.append((o1, l1, o2, l2, o3, l3, o4, l4, o5, l5, o6, l6))
    torch.cuda.synchronize()
    fa.check_device_status()
    ro5, rl5 = oracle.attention(q, k, outs[0][0].cpu(), w.scale, True)
    # merging two copies of the same result: the same O, lse + ln 2
    for (o1, l1, o2, l2, o3, l3, o4, l4, o5, l5, o6, l6) in outs:
        assert err(o1, ro) <= 2e-3 and err(l1, rl) <= 1e-3
        assert err(o2, ro) <= 2e-3 and err(l2, rl) <= 1e-3
        assert err(o3, ro32) <= 5e-3 and err(l3, rl32) <= 5e-3
        assert err(o4, ro) <= 1e-2 and err(l4, rl) <= 4e-3
        assert err(o5, ro5) <= 2e-3 and err(l5, rl5) <= 1e-3
        assert err(o6, ro) <= 3e-3 and err(l6, rl + np.log(2.0)) <= 1e-3


def test_fused_forward_in_a_cuda_graph():
    w = workloads.WORKLOADS["c2"]
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.N, device="cuda")
    fa.forward(q, k, v, causal=True, scale=w.scale, out=o, lse=lse)  # one-time setup outside capture
    torch.cuda.synchronize()
    ref_o, ref_l = o.clone(), lse.clone()
    o.zero_()
    lse.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fa.forward(q, k, v, causal=True, scale=w.scale, out=o, lse=lse)
            fa.forward(q, k, v, causal=True, scale=w.scale, out=o, lse=lse)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    fa.check_device_status()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)
