"""The work schedule for causal problems with several waves of items (host logic, no GPU):
a persistent grid whose per-CTA item lists follow one-CTA-per-item dispatch. Every item must
appear exactly once, each list in dispatch (item) order, the first wave one item per CTA, and
the estimated loads within the list-scheduling bound."""

from __future__ import annotations

import pytest

from tiled_attention_prefill_gb300 import _build, fa

FP16, BF16, FP32 = 0, 1, 2


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return fa.load_library()


def item_costs(B, H, N, D, dtype, num_items):
    """Estimated cost per item in the kernel's item order (tile steps of the longer warpgroup
    chain + 1), for causal items: two-query-tile items (fp16/bf16) or single 128-row query tiles
    with 64-key tiles split between the two warpgroups (fp32)."""
    BH = B * H
    esz = 4 if dtype == FP32 else 2
    section = max(1, min(BH, (32 << 20) // (2 * N * D * esz)))
    rows = 128 if dtype == FP32 else 256
    num_mb = -(-N // rows)
    assert BH * num_mb == num_items
    costs = []
    for t in range(num_items):
        per_sec = section * num_mb
        sec, r = divmod(t, per_sec)
        hs = min(section, BH - sec * section)
        mb = num_mb - 1 - r // hs
        if dtype == FP32:
            nkt = -(-N // 64)
            nk = min(2 * mb + 2, nkt)
            steps = (nk + 1) // 2
        else:
            nkt = -(-N // 128)
            n0 = min(2 * mb + 1, nkt)
            n1 = min(2 * mb + 2, nkt) if mb * 256 + 128 < N else 0
            steps = max(n0, n1)
        costs.append(steps + 1.0)
    return costs


@pytest.mark.parametrize("shape", [
    (4, 16, 4096, 128, BF16, 152),   # the batched-prefill shape: 1024 items
    (4, 16, 4096, 128, BF16, 148),
    (2, 40, 1000, 64, FP16, 152),    # ragged N
    (1, 64, 2048, 64, FP32, 152),    # fp32 kernel: single query tiles, 64-key tiles
    (1, 8, 16384, 128, FP16, 16),    # few SMs
])
def test_schedule_covers_every_item_once_in_dispatch_order(shape):
    B, H, N, D, dtype, G = shape
    lists = fa.debug_work_schedule(B, H, N, D, True, dtype, G)
    assert lists is not None and len(lists) == G
    flat = [t for lst in lists for t in lst]
    n = len(flat)
    assert sorted(flat) == list(range(n))
    assert n > 2 * G
    for c, lst in enumerate(lists):
        assert lst == sorted(lst)
        assert lst[0] == c                      # the first wave: item c on CTA c
    costs = item_costs(B, H, N, D, dtype, n)
    loads = [sum(costs[t] for t in lst) for lst in lists]
    assert max(loads) <= sum(costs) / G + max(costs) + 1e-9


def test_shapes_without_a_schedule():
    assert fa.debug_work_schedule(1, 32, 1024, 64, True, FP16, 152) is None    # one wave or less
    assert fa.debug_work_schedule(1, 8, 16384, 128, False, FP16, 152) is None  # non-causal: even items
    assert fa.debug_work_schedule(4, 16, 4096, 128, True, BF16, 2000) is None  # under two waves


def test_schedule_argument_checks(lib):
    assert lib.fa_debug_work_schedule(0, 1, 8, 64, 1, 0, 152, None, 0) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_debug_work_schedule(1, 1, 8, 96, 1, 0, 152, None, 0) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_debug_work_schedule(1, 1, 8, 64, 1, 3, 152, None, 0) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_debug_work_schedule(1, 1, 8, 64, 1, 0, 0, None, 0) == fa.FA_ERR_INVALID_ARG
    need = lib.fa_debug_work_schedule(4, 16, 4096, 128, 1, 1, 152, None, 0)
    assert need == 152 + 1 + 1024
    import ctypes
    buf = (ctypes.c_int * need)()
    assert lib.fa_debug_work_schedule(4, 16, 4096, 128, 1, 1, 152, ctypes.addressof(buf), need - 1) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_debug_work_schedule(4, 16, 4096, 128, 1, 1, 152, ctypes.addressof(buf), need) == need
