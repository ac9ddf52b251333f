"""The oracle's key-range partials and merge against their pins, and planted mistakes in both."""

from __future__ import annotations

import os

import numpy as np
import pytest

import oracle
from oracle import merge as merge_mod
from tests import merge_pins, oracle_pins

SRC_C = os.path.join(os.path.dirname(oracle.__file__), "attention_oracle.c")
SRC_MERGE = merge_mod.__file__


def _partial(lib=None):
    def fn(q, k, v, scale, causal, lo, hi):
        return oracle.attention_keys(q, k, v, scale, causal, lo, hi, lib=lib)
    return fn


@pytest.mark.parametrize("pin", merge_pins.PARTIAL_PINS, ids=lambda p: p.__name__)
def test_partial_pin(pin):
    pin(_partial())


@pytest.mark.parametrize("pin", merge_pins.MERGE_PINS, ids=lambda p: p.__name__)
def test_merge_pin(pin):
    pin(oracle.merge_partials)


@pytest.mark.parametrize("causal", [False, True])
def test_split_then_merge_equals_full(causal):
    """Key tiles of 16 split into ranges as a split-KV forward would; merged, they give the full result."""
    N = 70
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((1, 2, N, 8)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, 0.4, causal)
    for cuts in ([0, 16, 48, N], [0, 64, N], [0, 0, 32, N, N]):
        parts = [oracle.attention_keys(q, k, v, 0.4, causal, a, b) for a, b in zip(cuts[:-1], cuts[1:])]
        mo, ml = oracle.merge_partials(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        np.testing.assert_allclose(mo, o, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(ml, lse, rtol=1e-12, atol=1e-12)


def test_full_range_partial_is_the_full_result():
    rng = np.random.default_rng(6)
    q, k, v = (rng.standard_normal((1, 1, 33, 8)) for _ in range(3))
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, 0.4, causal)
        po, pl = oracle.attention_keys(q, k, v, 0.4, causal, 0, 33)
        assert np.array_equal(po, o) and np.array_equal(pl, lse)


def test_bad_key_range_rejected():
    q = np.zeros((1, 1, 4, 4))
    with pytest.raises(RuntimeError):
        oracle.attention_rows(q, q, q, 1.0, False, [[0, 0]], key_ranges=[[2, 5]])
    with pytest.raises(RuntimeError):
        oracle.attention_rows(q, q, q, 1.0, False, [[0, 0]], key_ranges=[[3, 2]])


C_MUTATIONS = {
    "range_end_ignored": ("    if (nj > hi)\n        nj = hi;\n", ""),
    "empty_range_lse_zero": ("        *lse_out = -INFINITY;\n        return;", "        *lse_out = 0.0;\n        return;"),
    "empty_range_not_detected": ("if (lo >= nj) {", "if (lo > nj) {"),
    "pass_3_skips_first_key": ("for (int64_t j = lo; j < nj; ++j) {\n        const double p",
                               "for (int64_t j = lo + 1; j < nj; ++j) {\n        const double p"),
}


@pytest.mark.parametrize("name", sorted(C_MUTATIONS))
def test_planted_range_mistake_is_caught(name, tmp_path):
    old, new = C_MUTATIONS[name]
    text = open(SRC_C).read()
    assert text.count(old) == 1, "mutation anchor not found: " + old
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib = oracle.load_library(oracle.compile_oracle(str(src), str(tmp_path / "libmutant.so")))
    failed = []
    for pin in merge_pins.PARTIAL_PINS:
        try:
            pin(_partial(lib))
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, "mutation %s passed every pin" % name


def test_range_extension_keeps_full_pins(tmp_path):
    """The full-range path of the extended C oracle still passes every full-attention pin."""
    for pin in oracle_pins.ALL_PINS:
        pin(lambda q, k, v, s, c: oracle.attention(q, k, v, s, c))


MERGE_MUTATIONS = {
    "new_part_weight_sign": ("np.exp(m_s - m_new)", "np.exp(m_new - m_s)"),
    "accumulator_not_rescaled": ("acc = acc * alpha[..., None]", "acc = acc"),
    "empty_part_output_not_masked": ("o_s = np.where(has[..., None], o_parts[s], 0.0)", "o_s = o_parts[s]"),
    "lse_without_running_max": ("lse = np.where(any_key, m + np.log(", "lse = np.where(any_key, np.log("),
    "running_max_not_updated": ("        m = m_new\n", "        m = np.where(np.isfinite(m), m, 0.0)\n"),
    "denominator_not_rescaled": ("l = l * alpha + l_s * beta", "l = l + l_s * beta"),
}


@pytest.mark.parametrize("name", sorted(MERGE_MUTATIONS))
def test_planted_merge_mistake_is_caught(name):
    old, new = MERGE_MUTATIONS[name]
    text = open(SRC_MERGE).read()
    assert text.count(old) == 1, "mutation anchor not found: " + old
    ns = {"__name__": "merge_mutant"}
    exec(compile(text.replace(old, new), "merge_mutant", "exec"), ns)
    failed = []
    for pin in merge_pins.MERGE_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(ns["merge_partials"])
        except (AssertionError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, "mutation %s passed every pin" % name
