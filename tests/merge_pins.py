"""Pins for partial results over key ranges and for their merge.

``pin_partial_*`` take ``fn(q, k, v, scale, causal, lo, hi) -> (o, lse)``: the attention of
every row restricted to the keys lo <= j < hi of J(i) (fp64 numpy, shapes [B,H,N,D] and
[B,H,N]; a row without such a key gives o = 0, lse = -inf). ``pin_merge_*`` take
``fn(o_parts, lse_parts) -> (o, lse)``. Each raises AssertionError on disagreement.

No expected value comes from the oracle: the references are closed forms and library routines
(torch's fp64 CPU scaled_dot_product_attention and logsumexp on sliced keys).
"""

from __future__ import annotations

import math

import numpy as np
import torch

RTOL = 1e-11
ATOL = 1e-11


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _sdpa_masked(q, k, v, scale, allowed):
    """Library reference: softmax attention of q over the keys where ``allowed`` [N_q, N_k] holds,
    with lse from torch.logsumexp; rows with no allowed key get o = 0, lse = -inf."""
    qt, kt, vt = (torch.from_numpy(np.ascontiguousarray(x)) for x in (q, k, v))
    s = scale * torch.einsum("bhid,bhjd->bhij", qt, kt)
    mask = torch.from_numpy(allowed)
    s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    any_key = mask.any(dim=-1)
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=mask | ~any_key[:, None], scale=scale)
    o = torch.where(any_key[None, None, :, None], o, torch.zeros_like(o))
    return o.numpy(), lse.numpy()


def _allowed(N, causal, lo, hi):
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    a = (j >= lo) & (j < hi) & np.ones((N, 1), dtype=bool)
    if causal:
        a &= j <= i
    return a


def pin_partial_single_key(fn):
    """Range [j, j+1): O_i = v_j and lse_i = s_ij where key j is visible, else O = 0, lse = -inf."""
    q, k, v = _rand((1, 2, 9, 8), 21), _rand((1, 2, 9, 8), 22), _rand((1, 2, 9, 8), 23)
    scale = 0.41
    for causal in (False, True):
        for j in (0, 4, 8):
            o, lse = fn(q, k, v, scale, causal, j, j + 1)
            for h in range(2):
                for i in range(9):
                    if causal and j > i:
                        assert np.all(o[0, h, i] == 0.0) and lse[0, h, i] == -np.inf
                    else:
                        np.testing.assert_allclose(o[0, h, i], v[0, h, j], rtol=RTOL, atol=ATOL)
                        np.testing.assert_allclose(lse[0, h, i], scale * float(q[0, h, i] @ k[0, h, j]),
                                                   rtol=RTOL, atol=ATOL)


def pin_partial_empty_range(fn):
    """An empty range holds no key: O = 0 and lse = -inf on every row."""
    q, k, v = _rand((1, 1, 7, 4), 31), _rand((1, 1, 7, 4), 32), _rand((1, 1, 7, 4), 33)
    for causal in (False, True):
        for lo in (0, 3, 7):
            o, lse = fn(q, k, v, 0.5, causal, lo, lo)
            assert np.all(o == 0.0) and np.all(lse == -np.inf)


def pin_partial_ranges_against_library(fn):
    """Several ranges, both masks: torch SDPA / logsumexp over the sliced, masked keys."""
    N = 37
    q, k, v = _rand((2, 2, N, 8), 41), _rand((2, 2, N, 8), 42), _rand((2, 2, N, 8), 43, 2.0)
    scale = 0.3
    for causal in (False, True):
        for lo, hi in ((0, N), (0, 5), (5, 20), (20, N), (13, 14), (30, 37)):
            o, lse = fn(q, k, v, scale, causal, lo, hi)
            ro, rl = _sdpa_masked(q, k, v, scale, _allowed(N, causal, lo, hi))
            np.testing.assert_allclose(o, ro, rtol=1e-10, atol=1e-10)
            np.testing.assert_allclose(lse, rl, rtol=1e-10, atol=1e-10)


PARTIAL_PINS = [pin_partial_single_key, pin_partial_empty_range, pin_partial_ranges_against_library]


def pin_merge_two_parts_closed_form(fn):
    """Two parts: lse = logaddexp(a, b); O = sig(a - b) O_1 + (1 - sig(a - b)) O_2."""
    o1, o2 = _rand((5, 3), 51), _rand((5, 3), 52)
    a, b = _rand((5,), 53, 3.0), _rand((5,), 54, 3.0)
    o, lse = fn(np.stack([o1, o2]), np.stack([a, b]))
    for r in range(5):
        sig = 1.0 / (1.0 + math.exp(-(a[r] - b[r])))
        np.testing.assert_allclose(o[r], sig * o1[r] + (1.0 - sig) * o2[r], rtol=RTOL, atol=ATOL)
        np.testing.assert_allclose(lse[r], max(a[r], b[r]) + math.log1p(math.exp(-abs(a[r] - b[r]))),
                                   rtol=RTOL, atol=ATOL)


def pin_merge_single_part_is_identity(fn):
    o1, a = _rand((4, 6), 61), _rand((4,), 62)
    o, lse = fn(o1[None], a[None])
    np.testing.assert_allclose(o, o1, rtol=RTOL, atol=ATOL)
    np.testing.assert_allclose(lse, a, rtol=RTOL, atol=ATOL)


def pin_merge_skips_empty_parts(fn):
    """A part at lse = -inf contributes nothing whatever its O holds (NaN included); a row with
    no key in any part gets O = 0 and lse = -inf."""
    o1, o2 = _rand((3, 4), 71), np.full((3, 4), np.nan)
    a = _rand((3,), 72)
    b = np.full((3,), -np.inf)
    o, lse = fn(np.stack([o2, o1, o2]), np.stack([b, a, b]))
    np.testing.assert_allclose(o, o1, rtol=RTOL, atol=ATOL)
    np.testing.assert_allclose(lse, a, rtol=RTOL, atol=ATOL)
    o, lse = fn(np.stack([o2, o2]), np.stack([b, b]))
    assert np.all(o == 0.0) and np.all(lse == -np.inf)


def pin_merge_order_independent(fn):
    o_parts, lse_parts = _rand((5, 6, 3), 81), _rand((5, 6), 82, 4.0)
    o, lse = fn(o_parts, lse_parts)
    perm = [3, 0, 4, 2, 1]
    o2, lse2 = fn(o_parts[perm], lse_parts[perm])
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=1e-12, atol=1e-12)


def pin_merge_large_lse(fn):
    """Weights depend on lse differences only: lse 1e4 and 1e4 + ln 3 weigh 1/4 and 3/4."""
    o1, o2 = _rand((2, 3), 91), _rand((2, 3), 92)
    a = np.full((2,), 1e4)
    o, lse = fn(np.stack([o1, o2]), np.stack([a, a + math.log(3.0)]))
    np.testing.assert_allclose(o, 0.25 * o1 + 0.75 * o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, 1e4 + math.log(4.0), rtol=1e-14, atol=1e-10)


def pin_merge_partition_against_library(fn):
    """Partials of a partition of the keys, each from torch SDPA / logsumexp on its slice, merge
    to torch SDPA / logsumexp over all keys (both masks; empty parts included)."""
    N = 41
    q, k, v = _rand((1, 3, N, 8), 101), _rand((1, 3, N, 8), 102), _rand((1, 3, N, 8), 103)
    scale = 0.35
    for causal in (False, True):
        cuts = [(0, 0), (0, 7), (7, 7), (7, 30), (30, N)]
        parts = [_sdpa_masked(q, k, v, scale, _allowed(N, causal, lo, hi)) for lo, hi in cuts]
        o, lse = fn(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        ro, rl = _sdpa_masked(q, k, v, scale, _allowed(N, causal, 0, N))
        np.testing.assert_allclose(o, ro, rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(lse, rl, rtol=1e-10, atol=1e-10)


MERGE_PINS = [pin_merge_two_parts_closed_form, pin_merge_single_part_is_identity, pin_merge_skips_empty_parts,
              pin_merge_order_independent, pin_merge_large_lse, pin_merge_partition_against_library]
