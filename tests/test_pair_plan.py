"""The paired split-K decomposition (host logic, no GPU). A causal launch at D = 64 with
single-query-tile items, more than one and at most two per SM, runs CTA c of G on items c and
2G - 1 - c at once:
warpgroup 0 takes the first ceil(T/2) K/V tiles of the longer item a, warpgroup 1 all of the
shorter item b and then the rest of a (T = tiles of both). Checked: when pairing applies, that
every item is run once, that each unit's tile counts are the items' causal counts, and that the
two warpgroups' chains differ by at most one tile and never exceed the serial form's."""

from __future__ import annotations

import ctypes

import pytest

from tiled_attention_prefill_gb300 import _build, fa

FP16, BF16, FP32 = 0, 1, 2


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return fa.load_library()


def causal_tiles(B, H, N, D, t):
    """K/V tiles of single-query-tile item t in the kernel's order (heads in L2 sections, each
    section's query tiles longest first)."""
    BH = B * H
    section = max(1, min(BH, (32 << 20) // (2 * N * D * 2)))
    num_mb = -(-N // 128)
    sec, r = divmod(t, section * num_mb)
    hs = min(section, BH - sec * section)
    mb = num_mb - 1 - r // hs
    return min(mb + 1, -(-N // 128))


PAIRED = [
    (1, 32, 1024, 64, FP16, 152),   # the 1B-class prefill shape: 256 items, 104 pairs
    (1, 32, 1024, 64, BF16, 152),
    (2, 16, 1000, 64, BF16, 152),   # ragged N
    (1, 24, 1536, 64, FP16, 152),   # 288 items of 1..12 tiles
    (1, 40, 500, 64, FP16, 152),    # 160 items: only 8 pairs
    (1, 32, 1024, 64, FP16, 132),   # another SM count
    (6, 64, 640, 64, FP16, 1400),   # several L2 sections
]


@pytest.mark.parametrize("shape", PAIRED)
def test_pairs_cover_every_item_once_and_balance_the_warpgroups(shape):
    B, H, N, D, dtype, G = shape
    plan = fa.debug_work_plan(B, H, N, D, True, dtype, G)
    n = plan["items"]
    assert plan["single_tile"] and plan["paired"] and not plan["dispatch"]
    assert G < n <= 2 * G and plan["grid"] == G
    units = plan["units"]
    assert len(units) == G
    seen = []
    for c, (ta, tb, na, nb, n0, n1) in enumerate(units):
        assert {ta, tb} - {-1} == {c, 2 * G - 1 - c} & set(range(n))
        seen += [t for t in (ta, tb) if t >= 0]
        assert na == causal_tiles(B, H, N, D, ta)
        assert nb == (causal_tiles(B, H, N, D, tb) if tb >= 0 else 0)
        assert na >= nb
        assert n0 + n1 == na + nb and n0 - n1 in (0, 1) and n0 <= na
        serial = (na + 1) // 2 + (nb + 1) // 2  # the two items one after another, split-K
        assert max(n0, n1) <= serial
    assert sorted(seen) == list(range(n))


def test_the_prefill_shape_runs_every_cta_in_four_steps():
    # 256 query tiles of 1..8 K/V tiles (32 each) on 152 SMs: serially some CTA needs 5 steps
    # and an item change; paired, every warpgroup runs at most 4 tiles.
    units = fa.debug_work_plan(1, 32, 1024, 64, True, FP16, 152)["units"]
    assert max(max(u[4], u[5]) for u in units) == 4
    serial = max((u[2] + 1) // 2 + (u[3] + 1) // 2 for u in units)
    assert serial == 5


@pytest.mark.parametrize("shape,why", [
    ((1, 32, 512, 128, BF16, 152), "one item per SM or fewer"),
    ((1, 32, 1024, 128, BF16, 152), "D = 128 (measured slower paired)"),
    ((1, 32, 4096, 64, FP16, 152), "two-query-tile items with a dispatch schedule"),
    ((1, 32, 1024, 64, FP16, 152, False), "non-causal"),
    ((1, 40, 1000, 64, FP32, 152), "fp32 kernel"),
    ((1, 64, 1024, 64, FP16, 100), "more than two items per SM"),
])
def test_launches_that_are_not_paired(shape, why):
    B, H, N, D, dtype, G = shape[:6]
    causal = shape[6] if len(shape) > 6 else True
    plan = fa.debug_work_plan(B, H, N, D, causal, dtype, G)
    assert not plan["paired"] and plan["units"] is None, why
    assert plan["grid"] == (G if (plan["dispatch"] or plan["items"] > G) else plan["items"])


def test_serial_mode_turns_pairing_off():
    try:
        fa.set_decomposition(fa.FA_DECOMP_SPLIT_KV_SERIAL)
        plan = fa.debug_work_plan(1, 32, 1024, 64, True, FP16, 152)
        assert plan["single_tile"] and not plan["paired"] and plan["grid"] == 152
        fa.set_decomposition(fa.FA_DECOMP_SPLIT_KV)
        assert fa.debug_work_plan(1, 32, 1024, 64, True, FP16, 152)["paired"]
        fa.set_decomposition(fa.FA_DECOMP_TWO_TILES)
        assert not fa.debug_work_plan(1, 32, 1024, 64, True, FP16, 152)["single_tile"]
    finally:
        fa.set_decomposition(fa.FA_DECOMP_AUTO)


def test_work_plan_argument_checks(lib):
    plan = (ctypes.c_int * 5)()
    p = ctypes.addressof(plan)
    assert lib.fa_debug_work_plan(0, 1, 8, 64, 1, 0, 152, p, None, 0) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_debug_work_plan(1, 1, 8, 64, 1, 0, 152, None, None, 0) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_debug_work_plan(1, 1, 8, 96, 1, 0, 152, p, None, 0) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_debug_work_plan(1, 1, 8, 64, 1, 3, 152, p, None, 0) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_debug_work_plan(1, 1, 8, 64, 1, 0, 0, p, None, 0) == fa.FA_ERR_INVALID_ARG
    need = lib.fa_debug_work_plan(1, 32, 1024, 64, 1, 0, 152, p, None, 0)
    assert need == 6 * 152
    buf = (ctypes.c_int * need)()
    assert lib.fa_debug_work_plan(1, 32, 1024, 64, 1, 0, 152, p, ctypes.addressof(buf), need - 1) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_debug_work_plan(1, 32, 1024, 64, 1, 0, 152, p, ctypes.addressof(buf), need) == need
    assert list(plan) == [256, 1, 1, 0, 152]
