"""Pins for the attention oracle: facts fixed by the pages and by mathematics.

Each ``pin_*`` takes an oracle callable ``fn(q, k, v, scale, causal) -> (o,
lse)`` (fp64 numpy, shapes [B,H,N,D] and [B,H,N]) and raises AssertionError
when the callable disagrees with the fact. The same pins run on the C oracle,
on its numpy twin and, in ``test_oracle_mutations.py``, on deliberately broken
copies of the C oracle, each of which must fail at least one pin.

None of the expected values below comes from the oracle itself: they are
closed forms, invariants, or a library routine (torch's fp64 CPU
scaled_dot_product_attention and logsumexp).
"""

from __future__ import annotations

import math

import numpy as np
import torch

RTOL = 1e-11
ATOL = 1e-11


def _rand(shape, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * scale


def pin_single_key(fn):
    """N=1: softmax over one key is 1, so O_0 = v_0 and lse_0 = s_00 (both masks)."""
    for causal in (False, True):
        q, k, v = _rand((2, 3, 1, 8), 1), _rand((2, 3, 1, 8), 2), _rand((2, 3, 1, 8), 3)
        scale = 0.37
        o, lse = fn(q, k, v, scale, causal)
        np.testing.assert_allclose(o, v, rtol=RTOL, atol=ATOL)
        s = scale * np.einsum("bhnd,bhnd->bhn", q, k)
        np.testing.assert_allclose(lse, s, rtol=RTOL, atol=ATOL)


def pin_two_keys_closed_form(fn):
    """N=2: O_i = sig(d) v_0 + (1 - sig(d)) v_1 with d = s_i0 - s_i1; lse = logaddexp.

    Causal: row 0 sees key 0 only (O_0 = v_0, lse_0 = s_00); row 1 as non-causal.
    """
    q, k, v = _rand((1, 2, 2, 4), 11), _rand((1, 2, 2, 4), 12), _rand((1, 2, 2, 4), 13)
    scale = 0.5
    for causal in (False, True):
        o, lse = fn(q, k, v, scale, causal)
        for h in range(2):
            for i in range(2):
                s0 = scale * float(q[0, h, i] @ k[0, h, 0])
                s1 = scale * float(q[0, h, i] @ k[0, h, 1])
                if causal and i == 0:
                    exp_o, exp_lse = v[0, h, 0], s0
                else:
                    sig = 1.0 / (1.0 + math.exp(-(s0 - s1)))
                    exp_o = sig * v[0, h, 0] + (1.0 - sig) * v[0, h, 1]
                    exp_lse = max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1)))
                np.testing.assert_allclose(o[0, h, i], exp_o, rtol=RTOL, atol=ATOL)
                assert abs(lse[0, h, i] - exp_lse) <= 1e-12 * max(1.0, abs(exp_lse))


def pin_hand_worked_example(fn):
    """D=1, N=2, scale=1, q=(1,2), k=(1,0), v=(10,20), worked by hand.

    Non-causal: row 0 weights (e/(e+1), 1/(e+1)) so O_0 = 10 + 10/(e+1), lse_0 = ln(e+1);
    row 1 weights (e^2/(e^2+1), 1/(e^2+1)) so O_1 = 10 + 10/(e^2+1), lse_1 = ln(e^2+1).
    Causal: row 0 sees key 0 only: O_0 = 10, lse_0 = 1.
    """
    q = np.array([[[[1.0], [2.0]]]])
    k = np.array([[[[1.0], [0.0]]]])
    v = np.array([[[[10.0], [20.0]]]])
    e = math.e
    o, lse = fn(q, k, v, 1.0, False)
    np.testing.assert_allclose(o[0, 0, :, 0], [10 + 10 / (e + 1), 10 + 10 / (e * e + 1)], rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0], [math.log(e + 1), math.log(e * e + 1)], rtol=1e-14)
    o, lse = fn(q, k, v, 1.0, True)
    np.testing.assert_allclose(o[0, 0, :, 0], [10.0, 10 + 10 / (e * e + 1)], rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0], [1.0, math.log(e * e + 1)], rtol=1e-14)


def _sdpa_reference(q, k, v, scale, causal):
    """torch's fp64 CPU scaled_dot_product_attention and logsumexp (library routines)."""
    tq, tk, tv = (torch.from_numpy(np.asarray(x, dtype=np.float64)) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    s = torch.matmul(tq, tk.transpose(-1, -2)) * scale
    if causal:
        n = s.shape[-1]
        s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.numpy(), lse.numpy()


def pin_library_sdpa(fn):
    """Brute force against torch's fp64 SDPA on small shapes, both masks, N up to 64."""
    for (B, H, N, D), seed in (((1, 1, 1, 8), 21), ((2, 3, 5, 16), 22), ((1, 2, 33, 8), 23),
                               ((1, 1, 64, 64), 24), ((2, 1, 17, 128), 25)):
        q, k, v = _rand((B, H, N, D), seed), _rand((B, H, N, D), seed + 100), _rand((B, H, N, D), seed + 200)
        scale = 1.0 / math.sqrt(D)
        for causal in (False, True):
            o, lse = fn(q, k, v, scale, causal)
            ro, rlse = _sdpa_reference(q, k, v, scale, causal)
            np.testing.assert_allclose(o, ro, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(lse, rlse, rtol=1e-12, atol=1e-12)


def pin_constant_value_rows(fn):
    """Every V row equal to c gives O_i = c for every row (weights sum to one)."""
    B, H, N, D = 1, 2, 40, 16
    q, k = _rand((B, H, N, D), 31, 3.0), _rand((B, H, N, D), 32, 3.0)
    c = _rand((D,), 33)
    v = np.broadcast_to(c, (B, H, N, D)).copy()
    for causal in (False, True):
        o, _ = fn(q, k, v, 0.25, causal)
        np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=1e-12, atol=1e-12)


def pin_zero_query(fn):
    """Q = 0: all scores are 0, so O_i = mean of v_j over J(i) and lse_i = ln|J(i)|."""
    B, H, N, D = 1, 2, 23, 8
    q = np.zeros((B, H, N, D))
    k, v = _rand((B, H, N, D), 41), _rand((B, H, N, D), 42)
    o, lse = fn(q, k, v, 0.3, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, np.full((B, H, N), math.log(N)), rtol=1e-13)
    o, lse = fn(q, k, v, 0.3, True)
    cnt = np.arange(1, N + 1, dtype=np.float64)
    expect = np.cumsum(v, axis=2) / cnt[None, None, :, None]
    np.testing.assert_allclose(o, expect, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(cnt), lse.shape), rtol=1e-13, atol=1e-15)


def pin_key_value_permutation(fn):
    """Non-causal: permuting key and value rows together changes neither O nor lse."""
    B, H, N, D = 2, 2, 37, 16
    q, k, v = _rand((B, H, N, D), 51), _rand((B, H, N, D), 52), _rand((B, H, N, D), 53)
    perm = np.random.default_rng(54).permutation(N)
    o1, l1 = fn(q, k, v, 0.25, False)
    o2, l2 = fn(q, k[:, :, perm], v[:, :, perm], 0.25, False)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-13, atol=1e-13)


def pin_one_hot_dominant(fn):
    """A score that beats every other by far more than 40 selects its V row exactly.

    Keys are one-hot basis vectors; query i points at key t(i) with weight 1e3,
    so s_i,t(i) - s_ij >= 1e3*scale = 250 for every other j: the other weights
    are below e^-250 relative, far under fp64 resolution.
    """
    B, H, N, D = 1, 1, 16, 16
    k = np.eye(N, D)[None, None]
    v = _rand((B, H, N, D), 61)
    rng = np.random.default_rng(62)
    for causal in (False, True):
        targets = np.array([rng.integers(0, i + 1) if causal else rng.integers(0, N) for i in range(N)])
        q = np.zeros((B, H, N, D))
        q[0, 0, np.arange(N), targets] = 1e3
        o, lse = fn(q, k, v, 0.25, causal)
        np.testing.assert_allclose(o[0, 0], v[0, 0, targets], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(lse[0, 0], np.full(N, 250.0), rtol=1e-13)


def pin_row_shift(fn):
    """Adding c_i to every score of row i leaves O unchanged and adds c_i to lse.

    Realised with one extra feature: q'_i = (q_i, c_i/scale), k'_j = (k_j, 1).
    """
    B, H, N, D = 1, 2, 29, 8
    q, k, v = _rand((B, H, N, D), 71), _rand((B, H, N, D), 72), _rand((B, H, N, D), 73)
    c = _rand((B, H, N), 74, 5.0)
    scale = 0.5
    q2 = np.concatenate([q, (c / scale)[..., None]], axis=-1)
    k2 = np.concatenate([k, np.ones((B, H, N, 1))], axis=-1)
    v2 = v
    for causal in (False, True):
        o1, l1 = fn(q, k, v, scale, causal)
        # pad v to the same head dim is not needed: only q/k gain a feature
        o2, l2 = fn(q2, k2, np.concatenate([v2, np.zeros((B, H, N, 1))], axis=-1), scale, causal)
        np.testing.assert_allclose(o2[..., :D], o1, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(l2, l1 + c, rtol=1e-12, atol=1e-12)


ALL_PINS = [
    pin_single_key,
    pin_two_keys_closed_form,
    pin_hand_worked_example,
    pin_library_sdpa,
    pin_constant_value_rows,
    pin_zero_query,
    pin_key_value_permutation,
    pin_one_hot_dominant,
    pin_row_shift,
]
