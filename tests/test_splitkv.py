"""GPU parity of the split-KV forward and of the partial-result merge against the fp64 oracle.

The split-KV forward must give the full attention result (same tolerances as the fused
forward: max abs O error 2e-3 fp16 / 1e-2 bf16, LSE 1e-3). Its workspace partials are also
checked one by one against the oracle's key-range partials, and the merge kernel on its own
against the oracle's merge (fp32 parts: O within half an output ulp plus 1e-5, LSE 1e-5
relative).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_prefill_gb300 import fa, workloads

pytestmark = pytest.mark.gpu

TOL_O = {"fp16": 2e-3, "bf16": 1e-2}
TOL_LSE = 1e-3


def assert_close(o, lse, ro, rl, dtype, what=""):
    assert np.isfinite(o).all(), "non-finite O " + what
    err = np.abs(o - ro)
    i = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= TOL_O[dtype], "O %s: max err %.3e at %s" % (what, err.max(), i)
    if lse is not None:
        el = np.abs(lse - rl)
        assert el.max() <= TOL_LSE, "LSE %s: max err %.3e" % (what, el.max())


def run_splitkv(q, k, v, causal, scale, splits, workspace=None):
    o, lse = fa.forward_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, num_splits=splits,
                                workspace=workspace)
    torch.cuda.synchronize()
    fa.check_device_status()
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


SHAPES = [(1, 1, 1, 64), (1, 2, 129, 128), (2, 3, 200, 64), (1, 1, 257, 128), (1, 2, 640, 64), (1, 1, 1000, 128)]


@pytest.mark.parametrize("splits", [2, 3, 8])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_splitkv_small_shapes_against_oracle(shape, dtype, causal, splits):
    B, H, N, D = shape
    w = workloads.Workload("t", B, H, N, D, dtype, causal, seed=11 * N + D + splits)
    q, k, v = workloads.make_qkv(w)
    o, lse = run_splitkv(q, k, v, causal, w.scale, splits)
    ro, rl = oracle.attention(q, k, v, w.scale, causal)
    assert_close(o, lse, ro, rl, dtype, "%s splits=%d" % (shape, splits))


def split_ranges(N, causal, splits):
    """(query tile, split) -> key range [lo, hi) in keys, as the header documents it."""
    nt = (N + 127) // 128
    out = {}
    for qt in range(nt):
        n = qt + 1 if causal else nt
        for s in range(splits):
            out[(qt, s)] = (128 * (s * n // splits), min(N, 128 * ((s + 1) * n // splits)))
    return out


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("D", [64, 128])
def test_workspace_partials_against_oracle_key_ranges(causal, D):
    """Each partial in the workspace equals the oracle's attention over that key range."""
    B, H, N, S = 1, 2, 700, 3
    w = workloads.Workload("t", B, H, N, D, "fp16", causal, seed=501 + D)
    q, k, v = workloads.make_qkv(w)
    nbytes = fa.splitkv_workspace_bytes(B, H, N, D, S)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    run_splitkv(q, k, v, causal, w.scale, S, workspace=ws)
    BH, rows = B * H, B * H * N
    o_bytes = (S * rows * D * 4 + 255) // 256 * 256
    o_part = ws[:S * rows * D * 4].view(torch.float32).view(S, BH, N, D).cpu().numpy().astype(np.float64)
    l_part = ws[o_bytes:o_bytes + S * rows * 4].view(torch.float32).view(S, BH, N).cpu().numpy().astype(np.float64)
    req, kr, idx = [], [], []
    for (qt, s), (lo, hi) in split_ranges(N, causal, S).items():
        for bh in range(BH):
            for i in range(qt * 128, min(N, qt * 128 + 128)):
                req.append((bh, i))
                kr.append((lo, hi))
                idx.append((s, bh, i))
    ro, rl = oracle.attention_rows(q, k, v, w.scale, causal, np.array(req), key_ranges=np.array(kr))
    idx = np.array(idx)
    go = o_part[idx[:, 0], idx[:, 1], idx[:, 2]]
    gl = l_part[idx[:, 0], idx[:, 1], idx[:, 2]]
    empty = ~np.isfinite(rl)
    assert np.all(gl[empty] == -np.inf), "empty ranges must have lse = -inf"
    assert np.isfinite(go[~empty]).all()
    assert np.abs(go[~empty] - ro[~empty]).max() <= TOL_O["fp16"]
    assert np.abs(gl[~empty] - rl[~empty]).max() <= TOL_LSE


@pytest.mark.parametrize("name,splits", [("c1", 2), ("c2", 2), ("c2", 4), ("c3c", 3), ("p2s1024", 2), ("c2", 0)])
def test_splitkv_workloads_full_oracle(name, splits):
    w = workloads.WORKLOADS[name]
    q, k, v = workloads.make_qkv(w)
    o, lse = run_splitkv(q, k, v, w.causal, w.scale, splits)
    ro, rl = oracle.attention(q, k, v, w.scale, w.causal)
    assert_close(o, lse, ro, rl, w.dtype, "%s splits=%d" % (name, splits))


@pytest.mark.parametrize("splits", [0, 4])
def test_splitkv_long_causal_full_oracle(splits):
    """One long causal sequence (the split-KV target case, 16384 tokens): every element against
    the oracle (~34 GFLOP of fp64 on the host cores)."""
    w = workloads.WORKLOADS["lc1"]
    q, k, v = workloads.make_qkv(w)
    o, lse = run_splitkv(q, k, v, w.causal, w.scale, splits)
    ro, rl = oracle.attention(q, k, v, w.scale, w.causal)
    assert_close(o, lse, ro, rl, w.dtype, "lc1 splits=%d" % splits)


def test_one_split_is_the_fused_forward():
    w = workloads.WORKLOADS["c2"]
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    o1, l1 = fa.forward(q, k, v, causal=True, scale=w.scale)
    o2, l2 = fa.forward_splitkv(q, k, v, causal=True, scale=w.scale, num_splits=1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_splitkv_deterministic_and_workspace_reusable():
    w = workloads.WORKLOADS["c3c"]
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    ws = torch.full((fa.splitkv_workspace_bytes(w.B, w.H, w.N, w.D, 4),), 0xFF, dtype=torch.uint8, device="cuda")
    o1, l1 = fa.forward_splitkv(q, k, v, causal=True, scale=w.scale, num_splits=4, workspace=ws)
    o1, l1 = o1.clone(), l1.clone()
    o2, l2 = fa.forward_splitkv(q, k, v, causal=True, scale=w.scale, num_splits=4, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_splitkv_small_workspace_rejected():
    w = workloads.WORKLOADS["c1"]
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    ws = torch.empty(fa.splitkv_workspace_bytes(w.B, w.H, w.N, w.D, 2) - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.forward_splitkv(q, k, v, num_splits=2, workspace=ws)
    assert e.value.code == fa.FA_ERR_WORKSPACE


def test_auto_split_count_is_sane():
    assert fa.splitkv_num_splits(1, 1, 16384, 128, True) > 1     # 128 query tiles on 152 SMs
    assert fa.splitkv_num_splits(4, 16, 4096, 128, True) == 1    # thousands of items already
    assert fa.splitkv_num_splits(1, 1, 100, 64, False) == 1      # a single key tile


@pytest.mark.parametrize("parts_dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("out", ["fp16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
def test_merge_partials_against_oracle(parts_dtype, out, D):
    """Random partial results, some parts empty (lse = -inf, O = NaN), merged on the GPU."""
    P, B, H, N = 4, 2, 3, 77
    g = torch.Generator().manual_seed(7 + D)
    pdt = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}[parts_dtype]
    o_parts = torch.randn((P, B, H, N, D), generator=g).to(pdt)
    lse_parts = (torch.randn((P, B, H, N), generator=g) * 4.0).float()
    empty = torch.rand((P, B, H, N), generator=g) < 0.3
    empty[:, 0, 0, 5] = True                      # a row with no key at all
    lse_parts[empty] = float("-inf")
    o_parts[empty] = float("nan")
    o_dt = torch.float16 if out == "fp16" else torch.bfloat16
    go, gl = fa.merge_partials(o_parts.cuda(), lse_parts.cuda(), out_dtype=o_dt)
    torch.cuda.synchronize()
    ro, rl = oracle.merge_partials(o_parts.double().numpy(), lse_parts.double().numpy())
    go = go.float().cpu().numpy().astype(np.float64)
    gl = gl.cpu().numpy().astype(np.float64)
    assert np.all(go[0, 0, 5] == 0.0) and gl[0, 0, 5] == -np.inf
    assert np.isfinite(go).all()
    half_ulp = np.abs(ro) * (2.0 ** -11 if out == "fp16" else 2.0 ** -8)
    assert np.all(np.abs(go - ro) <= half_ulp + 1e-5)
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(gl), fin)
    assert np.all(np.abs(gl[fin] - rl[fin]) <= 1e-5 * np.maximum(1.0, np.abs(rl[fin])))
