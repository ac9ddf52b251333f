"""GPU parity: the CUDA path (through the C-ABI binding) against the fp64 oracle.

Tolerances (max abs error over all compared elements): O within 2e-3 for fp16 I/O
and 1e-2 for bf16 I/O, LSE within 1e-3.
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


def run_cuda(q, k, v, causal, scale, lse=True):
    o, l = fa.forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, return_lse=lse)
    torch.cuda.synchronize()
    fa.check_device_status()
    o64 = o.float().cpu().numpy().astype(np.float64)
    l64 = l.cpu().numpy().astype(np.float64) if l is not None else None
    return o64, l64


def ulp(x, dtype):
    """Unit in the last place of the I/O type at |x| (fp16: 10 fraction bits, bf16: 7)."""
    frac_bits, min_exp = {"fp16": (10, -14), "bf16": (7, -126)}[dtype]
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** min_exp)))
    return 2.0 ** (e - frac_bits)


def worst_element(o, lse, ro, rl, dtype):
    """Where the largest O error is, its size in output ulps, and the largest lse error."""
    err_o = np.abs(o - ro)
    i = np.unravel_index(np.argmax(err_o), err_o.shape)
    rep = {"o_max_abs": float(err_o[i]), "o_at": tuple(int(x) for x in i), "o_want": float(ro[i]),
           "o_got": float(o[i]), "o_err_ulps": float(err_o[i] / ulp(ro[i], dtype))}
    if lse is not None:
        err_l = np.abs(lse - rl)
        j = np.unravel_index(np.argmax(err_l), err_l.shape)
        rep.update(lse_max_abs=float(err_l[j]), lse_at=tuple(int(x) for x in j))
    return rep


def assert_close(o, lse, ro, rl, dtype, what=""):
    assert np.isfinite(o).all(), "non-finite O " + what
    err_o = np.abs(o - ro)
    i = np.unravel_index(np.argmax(err_o), err_o.shape)
    assert err_o.max() <= TOL_O[dtype], "O %s: max err %.3e at %s (got %r want %r)" % (
        what, err_o.max(), i, o[i], ro[i])
    if lse is not None:
        assert np.isfinite(lse).all(), "non-finite LSE " + what
        err_l = np.abs(lse - rl)
        j = np.unravel_index(np.argmax(err_l), err_l.shape)
        assert err_l.max() <= TOL_LSE, "LSE %s: max err %.3e at %s" % (what, err_l.max(), j)


SMALL_SHAPES = [
    (1, 1, 1, 64), (1, 1, 2, 128), (1, 2, 17, 64), (1, 1, 127, 128), (1, 1, 128, 64), (1, 1, 129, 128),
    (2, 3, 200, 64), (1, 2, 256, 128), (1, 1, 257, 64), (1, 2, 384, 128), (1, 1, 513, 64), (1, 1, 1000, 128),
]


DECOMPS = {"two_tiles": fa.FA_DECOMP_TWO_TILES, "split_kv": fa.FA_DECOMP_SPLIT_KV}


@pytest.fixture
def decomposition(request):
    fa.set_decomposition(DECOMPS[request.param])
    yield request.param
    fa.set_decomposition(fa.FA_DECOMP_AUTO)


@pytest.mark.parametrize("decomposition", list(DECOMPS), indirect=True)
@pytest.mark.parametrize("shape", SMALL_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_small_shapes_against_oracle(shape, dtype, causal, decomposition):
    B, H, N, D = shape
    w = workloads.Workload("t", B, H, N, D, dtype, causal, seed=7 * N + D + B)
    q, k, v = workloads.make_qkv(w)
    o, lse = run_cuda(q, k, v, causal, w.scale)
    ro, rl = oracle.attention(q, k, v, w.scale, causal)
    assert_close(o, lse, ro, rl, dtype, "%s %s" % (shape, decomposition))


@pytest.mark.parametrize("decomposition", list(DECOMPS), indirect=True)
@pytest.mark.parametrize("name", ["c1", "c2", "c3c"])
def test_workload_both_decompositions(name, decomposition):
    """The same workloads forced through each decomposition."""
    w = workloads.WORKLOADS[name]
    q, k, v = workloads.make_qkv(w)
    o, lse = run_cuda(q, k, v, w.causal, w.scale)
    ro, rl = oracle.attention(q, k, v, w.scale, w.causal)
    assert_close(o, lse, ro, rl, w.dtype, name + " " + decomposition)


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c3c", "c4", "c5", "p2s512", "p2s1024", "lc1"])
def test_workload_full_oracle(name):
    """Every output element of each workload against the oracle, the full-size ones included.

    c5 (Q, K scaled by 4) is the long-sequence case where exp(m_old - m_new) underflows and
    the kernel's deferred rescale acts; c4 is the batched bf16 causal prefill. The oracle
    takes a few seconds (c4) to about twenty (c5) on 16 host cores. The worst element, its
    error in output ulps and the worst lse error are printed (pytest -rP shows them)."""
    w = workloads.WORKLOADS[name]
    q, k, v = workloads.make_qkv(w)
    o, lse = run_cuda(q, k, v, w.causal, w.scale)
    ro, rl = oracle.attention(q, k, v, w.scale, w.causal)
    print("parity %s: %r" % (name, worst_element(o, lse, ro, rl, w.dtype)))
    assert_close(o, lse, ro, rl, w.dtype, name)


def test_lse_optional():
    w = workloads.WORKLOADS["c1"]
    q, k, v = workloads.make_qkv(w)
    o, lse = run_cuda(q, k, v, False, w.scale, lse=False)
    assert lse is None
    ro, _ = oracle.attention(q, k, v, w.scale, False)
    assert_close(o, None, ro, None, "fp16", "no-lse")


def test_default_scale():
    w = workloads.WORKLOADS["c1"].with_(D=128)
    q, k, v = workloads.make_qkv(w)
    o, lse = run_cuda(q, k, v, True, None)
    ro, rl = oracle.attention(q, k, v, 1.0 / np.sqrt(128.0), True)
    assert_close(o, lse, ro, rl, "fp16", "default scale")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_no_writes_outside_outputs(dtype):
    """Guard regions around O and LSE keep their sentinel values (out-of-bounds write check)."""
    w = workloads.Workload("g", 1, 3, 333, 128, dtype, True, seed=99)
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    pad = 4096
    numel = q.numel()
    o_big = torch.full((numel + 2 * pad,), 7.0, dtype=q.dtype, device="cuda")
    l_big = torch.full((w.B * w.H * w.N + 2 * pad,), -3.0, dtype=torch.float32, device="cuda")
    o = o_big[pad:pad + numel].view(q.shape)
    lse = l_big[pad:pad + w.B * w.H * w.N].view(w.B, w.H, w.N)
    fa.forward(q, k, v, causal=True, scale=w.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    fa.check_device_status()
    assert bool((o_big[:pad] == 7.0).all()) and bool((o_big[pad + numel:] == 7.0).all())
    assert bool((l_big[:pad] == -3.0).all()) and bool((l_big[pad + w.B * w.H * w.N:] == -3.0).all())
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, True)
    assert_close(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ro, rl, dtype)


def test_bitwise_deterministic():
    w = workloads.WORKLOADS["c3c"]
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    o1, l1 = fa.forward(q, k, v, causal=True, scale=w.scale)
    o2, l2 = fa.forward(q, k, v, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_errors_surface_as_exceptions():
    x = torch.zeros(1, 1, 8, 96, dtype=torch.float16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.forward(x, x, x)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED


def test_runs_on_a_side_stream():
    w = workloads.WORKLOADS["c1"].with_(H=4, N=700)
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = fa.forward(q, k, v, causal=False, scale=w.scale)
    s.synchronize()
    ro, rl = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, False)
    assert_close(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ro, rl, "fp16")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_extreme_score_range(dtype, D, causal):
    """Q and K scaled by 16 (scores of a few hundred): the row max jumps by far more than the
    deferred-rescale threshold between tiles, and almost every P underflows to zero, so most
    rows attend to one or a few keys. Ragged N, several tiles, single-query-tile items.

    Tolerance from the arithmetic (these are not the five configurations the stated
    tolerances are for): P is rounded to the 16-bit type with relative error <= u (2^-8 for
    bf16, 2^-11 for fp16). The running max can trail the row max by up to 2^8, so even the
    dominant key's p is rounded, while l sums the unrounded p: O_i is off by at most
    u * max_j |v_j| from that, plus u * |O_i| from rounding the output; fp32 scores and sums
    add less than 1e-5 here (the scaled scores' fp32 error is ~2e-4, and they enter O only
    through the exponentials of the few largest). lse: 1e-3 as for the configurations (its
    fp32 error is ~4e-4 at these magnitudes)."""
    w = workloads.Workload("x16", 1, 4, 700, D, dtype, causal, seed=91 + D, qk_mult=16.0)
    q, k, v = workloads.make_qkv(w)
    o, lse = run_cuda(q, k, v, causal, w.scale)
    ro, rl = oracle.attention(q, k, v, w.scale, causal)
    u = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8}[dtype]
    vmax = np.abs(v.double().numpy()).max(axis=2, keepdims=True)  # per head and feature
    bound = u * (vmax + np.abs(ro)) + 1e-5
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    ratio = np.abs(o - ro) / bound
    i = np.unravel_index(np.argmax(ratio), ratio.shape)
    assert ratio.max() <= 1.0, "O x16: error %.3e at %s, bound %.3e" % (abs(o[i] - ro[i]), i, bound[i])
    assert np.abs(lse - rl).max() <= TOL_LSE


@pytest.mark.parametrize("D", [64, 128])
def test_explicit_scale(D):
    """A scale other than 1/sqrt(D) reaches the kernel (it is folded with log2 e there)."""
    w = workloads.Workload("scl", 2, 3, 333, D, "fp16", True, seed=17 + D)
    q, k, v = workloads.make_qkv(w)
    for scale in (0.05, 0.3):
        o, lse = run_cuda(q, k, v, True, scale)
        ro, rl = oracle.attention(q, k, v, scale, True)
        assert_close(o, lse, ro, rl, "fp16", "scale %g" % scale)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_zero_queries_give_the_mean_of_v(D, causal):
    """Q = 0: every score is 0, so O_i is the mean of V over J(i) and lse_i = ln |J(i)|."""
    w = workloads.Workload("q0", 1, 2, 520, D, "fp16", causal, seed=5 + D)
    q, k, v = workloads.make_qkv(w)
    q = torch.zeros_like(q)
    o, lse = run_cuda(q, k, v, causal, w.scale)
    v64 = v.double().numpy()
    n = np.arange(1, w.N + 1, dtype=np.float64)
    if causal:
        ro = np.cumsum(v64, axis=2) / n[None, None, :, None]
        rl = np.broadcast_to(np.log(n), lse.shape)
    else:
        ro = np.broadcast_to(v64.mean(axis=2, keepdims=True), v64.shape)
        rl = np.full(lse.shape, np.log(w.N))
    assert_close(o, lse, ro, rl, "fp16", "Q = 0")


@pytest.mark.parametrize("shape", [(0, 2, 128, 64), (1, 0, 256, 128), (2, 3, 0, 64)])
def test_empty_batch_gives_empty_outputs(shape):
    """No query rows (B, H or N is 0): empty O and lse of the right shapes, from every forward."""
    for dt in (torch.float16, torch.bfloat16, torch.float32):
        x = torch.empty(shape, dtype=dt, device="cuda")
        o, lse = fa.forward(x, x, x, causal=True)
        assert o.shape == shape and o.dtype == dt and lse.shape == shape[:3] and lse.dtype == torch.float32
    x = torch.empty(shape, dtype=torch.float16, device="cuda")
    for f in (fa.forward_splitkv, fa.forward_splitkv_noalloc):
        o, lse = f(x, x, x, causal=False)
        assert o.shape == shape and lse.shape == shape[:3]
    bad = torch.empty(shape[:3] + (96,), dtype=torch.float16, device="cuda")
    with pytest.raises(fa.FAError):
        fa.forward(bad, bad, bad)  # the head size is still checked
