"""The oracle against what the pages and mathematics fix (CPU only)."""

from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest

import oracle
from tests import oracle_pins
from tiled_attention_prefill_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _c_oracle(q, k, v, scale, causal):
    return oracle.attention(q, k, v, scale, causal)


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_c_oracle_pin(pin):
    pin(_c_oracle)


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_numpy_twin_pin(pin):
    pin(oracle.attention_np)


@pytest.mark.parametrize("causal", [False, True])
def test_c_oracle_matches_numpy_twin_on_workload_c1(causal):
    w = workloads.WORKLOADS["c1"]
    q, k, v = workloads.make_qkv(w)
    o1, l1 = oracle.attention(q, k, v, w.scale, causal)
    o2, l2 = oracle.attention_np(q, k, v, w.scale, causal)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("block_m,block_n", [(1, 1), (1, 7), (16, 64), (128, 128), (16, 200), (128, 300)])
@pytest.mark.parametrize("causal", [False, True])
def test_blockwise_recurrence_equals_unfused(block_m, block_n, causal):
    """The pages' claim: reordering into tiles with the online-softmax update does
    not change the result. Tile sizes include ones that do not divide N and one
    larger than N (a single block)."""
    rng = np.random.default_rng(5)
    B, H, N, D = 1, 2, 200, 16
    q, k, v = (rng.standard_normal((B, H, N, D)) for _ in range(3))
    ob, lb = oracle.online_softmax_blockwise(q, k, v, 0.25, causal, block_m, block_n)
    ou, lu = oracle.attention(q, k, v, 0.25, causal)
    np.testing.assert_allclose(ob, ou, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lb, lu, rtol=1e-12, atol=1e-12)


def test_blockwise_recurrence_with_wide_score_range():
    """Scores of the long-sequence stress shape (q, k multiplied by 4) and an
    extreme case where exp(m_old - m_new) underflows to exactly 0 in fp64: the
    recurrence stays finite and equal to the unfused definition."""
    w = workloads.WORKLOADS["c5"].with_(H=1, N=384)
    q, k, v = workloads.make_qkv(w)
    for causal in (False, True):
        ob, lb = oracle.online_softmax_blockwise(q, k, v, w.scale, causal, 128, 128)
        ou, lu = oracle.attention(q, k, v, w.scale, causal)
        np.testing.assert_allclose(ob, ou, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lb, lu, rtol=1e-12, atol=1e-12)
    # key 0 scores -1000 below the keys of the second block: alpha underflows to 0
    N, D = 8, 2
    q = np.zeros((1, 1, N, D)); q[..., 0] = 1.0
    k = np.zeros((1, 1, N, D)); k[0, 0, :4, 0] = -1000.0; k[0, 0, 4:, 0] = 1000.0
    v = np.arange(N * D, dtype=np.float64).reshape(1, 1, N, D)
    ob, lb = oracle.online_softmax_blockwise(q, k, v, 1.0, False, 8, 4)
    assert np.all(np.isfinite(ob)) and np.all(np.isfinite(lb))
    assert math.exp(-2000.0) == 0.0
    np.testing.assert_allclose(ob[0, 0], np.broadcast_to(v[0, 0, 4:].mean(axis=0), (N, D)), rtol=1e-14)
    np.testing.assert_allclose(lb[0, 0], np.full(N, 1000.0 + math.log(4.0)), rtol=1e-14)


def test_sampled_rows_match_full():
    w = workloads.WORKLOADS["c2"].with_(H=3, N=300)
    q, k, v = workloads.make_qkv(w)
    o, lse = oracle.attention(q, k, v, w.scale, True)
    rows = np.array([[0, 0], [2, 299], [1, 17], [0, 128], [2, 127]])
    os_, ls_ = oracle.attention_rows(q, k, v, w.scale, True, rows)
    for r, (bh, i) in enumerate(rows):
        np.testing.assert_array_equal(os_[r], o.reshape(-1, 300, w.D)[bh, i])
        assert ls_[r] == lse.reshape(-1, 300)[bh, i]


def test_thread_count_does_not_change_results():
    w = workloads.WORKLOADS["c1"]
    q, k, v = workloads.make_qkv(w)
    o1, l1 = oracle.attention(q, k, v, w.scale, False, nthreads=1)
    o2, l2 = oracle.attention(q, k, v, w.scale, False, nthreads=4)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_bad_rows_rejected():
    q = np.zeros((1, 1, 4, 8))
    with pytest.raises(RuntimeError):
        oracle.attention_rows(q, q, q, 1.0, False, np.array([[0, 4]]))
    with pytest.raises(RuntimeError):
        oracle.attention_rows(q, q, q, 1.0, False, np.array([[1, 0]]))


def test_page_size_claims():
    g = json.load(open(os.path.join(GOLDEN, "page_size_claims.json")))
    s = g["score_matrix_n2048_fp16"]
    assert s["n"] * s["n"] * s["elem_bytes"] == s["value_bytes"] == 8 * 2**20
    t = g["score_tile_64_fp32"]
    assert t["tile"] * t["tile"] * t["elem_bytes"] == t["value_bytes"] == 16 * 2**10
    # the table's reduction column is its two bandwidth columns, to the printed precision
    for row in g["bandwidth_reduction_table"]["rows"]:
        red = 100.0 * (1.0 - row["tiled_gbs"] / row["naive_gbs"])
        assert abs(red - row["reduction_pct"]) < 1.0, row


def test_workload_byte_and_flop_counts():
    # 4*N^2*D per head, halved when causal; the floor |Q|+|K|+|V|+|O| (+ fp32 lse)
    assert workloads.attention_flops(1, 1, 256, 64, False) == 4 * 256 * 256 * 64
    assert workloads.attention_flops(4, 16, 4096, 128, True) == 2 * 4096 * 4096 * 128 * 64
    assert workloads.min_dram_bytes(1, 32, 1024, 64, with_lse=False) == 16 * 2**20
    assert workloads.min_dram_bytes(4, 16, 4096, 128, with_lse=True) == 256 * 2**20 + 2**20
