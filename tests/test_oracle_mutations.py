"""Planted mistakes in the C oracle must each fail at least one pin.

Each mutation is a textual edit of ``oracle/attention_oracle.c`` compiled into
a throw-away library on the CPU; the real oracle is untouched.
"""

from __future__ import annotations

import os

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attention_oracle.c")

MUTATIONS = {
    "scale_dropped": ("s_row[j] = scale * acc;", "s_row[j] = acc;"),
    "causal_window_one_wider": ("causal ? (i + 1) : N", "causal ? (i + 2 < N ? i + 2 : N) : N"),
    "keys_used_as_values": ("const double *vj = vh + j * D;", "const double *vj = kh + j * D;"),
    "lse_in_base_two": ("*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    "divide_by_count": ("o_row[d] /= l;", "o_row[d] /= (double)nj;"),
    "max_not_subtracted_in_pass_3": ("const double p = exp(s_row[j] - m);", "const double p = exp(s_row[j]);"),
    "query_row_shifted": ("q + (bh * N + i) * D;", "q + (bh * N + (i + 1) % N) * D;"),
    "q_dot_k_off_by_one_feature": ("acc += qi[d] * kj[d];", "acc += qi[d] * kj[(d + 1) % D];"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, "mutation anchor not found: " + old
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib = oracle.load_library(oracle.compile_oracle(str(src), str(tmp_path / "libmutant.so")))

    def mutant(q, k, v, scale, causal):
        return oracle.attention(q, k, v, scale, causal, lib=lib)

    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, "mutation %s passed every pin" % name
