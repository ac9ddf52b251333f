"""Merge of partial attention results (fp64, numpy). TEST INFRASTRUCTURE, like the rest of
this package.

A partial result of query row i over a set of keys K_s is (O_s, lse_s): O_s is the softmax-
weighted mean of V over K_s and lse_s = ln sum_{j in K_s} exp(s_ij). When the key sets
partition J(i), the full result follows from the online-softmax update of "Android
Transformer Optimization: Attention and Mobile GPU Bottlenecks", section "The Essence of
FlashAttention: Reordering the Computation", applied with whole key sets as the blocks. A
part, summarised by its lse, is a block whose running max is m_s = lse_s and whose
denominator relative to that max is l_s = exp(lse_s - m_s) = 1, with normalised output O_s.
The update per part, in the order the parts are given:

    m_new = max(m, m_s)
    alpha = exp(m - m_new)                    (rescales what was accumulated so far)
    beta  = exp(m_s - m_new)                  (weight of the new part)
    l     = l * alpha + l_s * beta
    acc   = acc * alpha + (l_s * O_s) * beta
    m     = m_new

with m = -inf, l = 0, acc = 0 at the start, then O = acc / l and lse = m + ln l. A part with
lse_s = -inf holds no key and is skipped (whatever its O holds). A row with no key in any
part gets O = 0, lse = -inf.
"""

from __future__ import annotations

import numpy as np


def merge_partials(o_parts, lse_parts):
    """Combine P partial results. o_parts [P, ..., D], lse_parts [P, ...] -> (o [..., D], lse [...]) fp64."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    assert o_parts.shape[:-1] == lse_parts.shape, (o_parts.shape, lse_parts.shape)
    shape = lse_parts.shape[1:]
    m = np.full(shape, -np.inf)
    l = np.zeros(shape)
    acc = np.zeros(o_parts.shape[1:])
    for s in range(lse_parts.shape[0]):
        m_s = lse_parts[s]
        has = m_s > -np.inf                        # a part at -inf holds no key: skipped
        m_new = np.where(has, np.maximum(m, m_s), m)
        with np.errstate(invalid="ignore"):        # (-inf) - (-inf) only where masked out
            alpha = np.where(has, np.exp(m - m_new), 1.0)
            beta = np.where(has, np.exp(m_s - m_new), 0.0)
        l_s = 1.0
        o_s = np.where(has[..., None], o_parts[s], 0.0)
        l = l * alpha + l_s * beta
        acc = acc * alpha[..., None] + (l_s * o_s) * beta[..., None]
        m = m_new
    any_key = l > 0
    o = np.where(any_key[..., None], acc / np.where(any_key, l, 1.0)[..., None], 0.0)
    lse = np.where(any_key, m + np.log(np.where(any_key, l, 1.0)), -np.inf)
    return o, lse
