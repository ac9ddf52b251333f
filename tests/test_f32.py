"""GPU parity of the fp32-I/O forward (tf32 tensor-core products) against the fp64 oracle.

Tolerance 5e-3 for O and lse, from the arithmetic (derived and pinned on the CPU in
tests/test_f32_tolerance.py): the tensor core reads the fp32 operands Q, K, V as tf32 (the
low 13 mantissa bits dropped), which moves exact attention by at most 3.5e-3 on these
shapes; the kernel's rounding of P to tf32 adds at most 5e-4; the rest is fp32 arithmetic.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_prefill_gb300 import fa, workloads

pytestmark = pytest.mark.gpu

TOL = 5e-3


def run(q, k, v, causal, scale):
    o, lse = fa.forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    fa.check_device_status()
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def check(o, lse, ro, rl, what):
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    eo, el = np.abs(o - ro).max(), np.abs(lse - rl).max()
    assert eo <= TOL and el <= TOL, "%s: O err %.3e, lse err %.3e" % (what, eo, el)


SHAPES = [(1, 1, 1, 64), (1, 2, 17, 128), (1, 1, 64, 64), (1, 1, 65, 128), (2, 3, 128, 64), (1, 1, 129, 64),
          (1, 2, 200, 128), (1, 1, 257, 64), (1, 2, 640, 128), (1, 1, 1000, 64)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_f32_small_shapes(shape, causal):
    B, H, N, D = shape
    w = workloads.Workload("t", B, H, N, D, "fp32", causal, seed=13 * N + D)
    q, k, v = workloads.make_qkv(w)
    o, lse = run(q, k, v, causal, w.scale)
    ro, rl = oracle.attention(q, k, v, w.scale, causal)
    check(o, lse, ro, rl, str(shape))


@pytest.mark.parametrize("name", ["c2_f32", "c3_f32"])
def test_f32_workloads(name):
    w = workloads.WORKLOADS[name]
    q, k, v = workloads.make_qkv(w)
    o, lse = run(q, k, v, w.causal, w.scale)
    ro, rl = oracle.attention(q, k, v, w.scale, w.causal)
    check(o, lse, ro, rl, name)


def test_f32_no_writes_outside_outputs():
    w = workloads.Workload("g", 1, 3, 333, 128, "fp32", True, seed=77)
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    pad, numel, nl = 4096, q.numel(), w.B * w.H * w.N
    o_big = torch.full((numel + 2 * pad,), 7.0, dtype=torch.float32, device="cuda")
    l_big = torch.full((nl + 2 * pad,), -3.0, dtype=torch.float32, device="cuda")
    o = o_big[pad:pad + numel].view(q.shape)
    lse = l_big[pad:pad + nl].view(w.B, w.H, w.N)
    fa.forward(q, k, v, causal=True, scale=w.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    assert bool((o_big[:pad] == 7.0).all()) and bool((o_big[pad + numel:] == 7.0).all())
    assert bool((l_big[:pad] == -3.0).all()) and bool((l_big[pad + nl:] == -3.0).all())
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, True)
    check(o.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "guard")


def test_f32_bitwise_deterministic():
    w = workloads.WORKLOADS["c2_f32"]
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    o1, l1 = fa.forward(q, k, v, causal=True, scale=w.scale)
    o2, l2 = fa.forward(q, k, v, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_f32_close_to_fp16_path_on_fp16_representable_inputs():
    """Inputs exactly representable in fp16 (and so in tf32): both paths within tolerance."""
    w = workloads.WORKLOADS["c2"]
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    o16, l16 = fa.forward(q, k, v, causal=True, scale=w.scale)
    o32, l32 = fa.forward(q.float(), k.float(), v.float(), causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert (o16.float() - o32).abs().max().item() <= 2e-3 + TOL
    assert (l16 - l32).abs().max().item() <= 1e-3 + TOL


def test_f32_rejected_by_split_and_naive_paths():
    x = torch.zeros(1, 1, 256, 64, dtype=torch.float32, device="cuda")
    lib = fa.load_library()
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    assert lib.fa_forward_splitkv(x.data_ptr(), x.data_ptr(), x.data_ptr(), ws.data_ptr() + 4096 * 0 + (1 << 19),
                                  None, 1, 1, 256, 64, 0.1, 0, fa.FA_DTYPE_FP32, 2, ws.data_ptr(), 1 << 18,
                                  None) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_naive_forward(x.data_ptr(), x.data_ptr(), x.data_ptr(), ws.data_ptr() + (1 << 19), None, 1, 1,
                                256, 64, 0.1, 0, fa.FA_DTYPE_FP32, ws.data_ptr(), 1 << 18, None) == fa.FA_ERR_UNSUPPORTED
