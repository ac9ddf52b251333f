"""The host's choice of work decomposition (no GPU), through fa_debug_work_plan, against the
rules it implements, over random shapes, masks, dtypes and SM counts:

* fp32 storage, or a forced split-K mode: one 128-row query tile per item;
* causal fp16/bf16: two query tiles per item unless that leaves fewer items than SMs;
* non-causal fp16/bf16: single query tiles when twice the items fill whole waves of SMs
  better (by more than the 4% the split costs), else two query tiles;
* a dispatch-order schedule for causal launches with more than two items per SM;
* pairs for causal fp16/bf16 launches at D = 64 with single query tiles, more than one and at
  most two items per SM (not in the serial split-K mode);
* a grid of one CTA per SM, or one per item when there are fewer items than SMs.
"""

from __future__ import annotations

import random

import pytest

from tiled_attention_prefill_gb300 import _build, fa

FP16, BF16, FP32 = 0, 1, 2


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return fa.load_library()


def expected(B, H, N, D, causal, dtype, G, mode):
    BH = B * H
    items_two = BH * -(-N // 256)
    f32 = dtype == FP32
    splitk = mode in (fa.FA_DECOMP_SPLIT_KV, fa.FA_DECOMP_SPLIT_KV_SERIAL) or f32
    if mode == fa.FA_DECOMP_AUTO and not f32:
        if causal:
            splitk = items_two < G
        else:
            def eff(n):
                waves = -(-n // G)
                return n / (waves * G)
            splitk = eff(2 * items_two) * 0.96 > eff(items_two)
    rows = 128 if splitk else 256
    items = BH * -(-N // rows)
    dispatch = causal and items > 2 * G
    paired = (splitk and causal and D == 64 and not f32 and mode != fa.FA_DECOMP_SPLIT_KV_SERIAL
              and G < items <= 2 * G)
    grid = G if (dispatch or items > G) else items
    return {"items": items, "single_tile": splitk, "paired": paired, "dispatch": dispatch, "grid": grid}


@pytest.mark.parametrize("mode", [fa.FA_DECOMP_AUTO, fa.FA_DECOMP_TWO_TILES, fa.FA_DECOMP_SPLIT_KV,
                                  fa.FA_DECOMP_SPLIT_KV_SERIAL])
def test_decomposition_matches_its_rules(mode):
    rnd = random.Random(11 + mode)
    try:
        fa.set_decomposition(mode)
        for _ in range(400):
            B, H = rnd.randint(1, 8), rnd.randint(1, 64)
            N = rnd.choice([rnd.randint(1, 300), rnd.randint(1, 4096), 128 * rnd.randint(1, 64)])
            D = rnd.choice([64, 128])
            causal = rnd.random() < 0.5
            dtype = rnd.choice([FP16, BF16, FP32])
            G = rnd.choice([152, 148, 132, 16, 1, 600])
            got = fa.debug_work_plan(B, H, N, D, causal, dtype, G)
            units = got.pop("units")
            want = expected(B, H, N, D, causal, dtype, G, mode)
            assert got == want, ((B, H, N, D, causal, dtype, G, mode), got, want)
            assert (units is not None) == want["paired"]
            if units is not None:
                assert len(units) == want["grid"]
    finally:
        fa.set_decomposition(fa.FA_DECOMP_AUTO)


def test_the_benchmark_workloads():
    # the decompositions the measured workloads run with on 152 SMs
    from tiled_attention_prefill_gb300 import workloads
    code = {"fp16": FP16, "bf16": BF16, "fp32": FP32}
    want = {"c1": (True, False, False), "c2": (True, True, False), "c3": (False, False, False),
            "c3c": (False, False, False), "c4": (False, False, True), "c5": (True, False, False),
            "p2s512": (True, False, False), "p2s1024": (False, False, False), "lc1": (True, False, False),
            "c2_f32": (True, False, False), "c3_f32": (True, False, False)}
    for name, w in workloads.WORKLOADS.items():
        got = fa.debug_work_plan(w.B, w.H, w.N, w.D, w.causal, code[w.dtype], 152)
        assert (got["single_tile"], got["paired"], got["dispatch"]) == want[name], (name, got)
