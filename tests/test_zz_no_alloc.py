"""fa_forward_splitkv_noalloc: the split-KV forward on the library's built-in scratch.

Collected last (file name) so that it also runs after every other test in the same process;
it must pass on its own as well. Two calls in a row on different inputs are each compared
with fa_forward_splitkv on a caller workspace (same split count): the second call must not
see anything the first left in the scratch.
"""

from __future__ import annotations

import pytest
import torch

from tiled_attention_prefill_gb300 import fa, workloads


def test_oversize_split_count_rejected_before_any_cuda_call():
    lib = fa.load_library()
    # lc1 (1 x 1 x 16384 x 128) with 8 splits needs 8 * 16384 * (128 + 1) * 4 bytes > 32 MiB.
    assert fa.splitkv_workspace_bytes(1, 1, 16384, 128, 8) > fa.NOALLOC_SCRATCH_BYTES
    rc = lib.fa_forward_splitkv_noalloc(16, 32, 48, 1 << 40, None, 1, 1, 16384, 128, 0.1, 1, 0, 8, None)
    assert rc == fa.FA_ERR_SCRATCH
    assert "32 MiB" in fa.error_string(fa.FA_ERR_SCRATCH)


@pytest.mark.gpu
@pytest.mark.parametrize("name,splits", [("lc1", 2), ("c2", 3), ("c1", 0)])
def test_two_calls_in_a_row_match_the_workspace_entry_point(name, splits):
    w = workloads.WORKLOADS[name]
    q1, k1, v1 = (x.cuda() for x in workloads.make_qkv(w))
    q2, k2, v2 = (x.cuda() for x in workloads.make_qkv(w.with_(seed=w.seed + 500)))
    S = splits if splits > 0 else fa.splitkv_num_splits(w.B, w.H, w.N, w.D, w.causal)
    assert fa.splitkv_workspace_bytes(w.B, w.H, w.N, w.D, S) <= fa.NOALLOC_SCRATCH_BYTES
    a1, la1 = fa.forward_splitkv_noalloc(q1, k1, v1, causal=w.causal, scale=w.scale, num_splits=splits)
    a2, la2 = fa.forward_splitkv_noalloc(q2, k2, v2, causal=w.causal, scale=w.scale, num_splits=splits)
    r1, lr1 = fa.forward_splitkv(q1, k1, v1, causal=w.causal, scale=w.scale, num_splits=S)
    r2, lr2 = fa.forward_splitkv(q2, k2, v2, causal=w.causal, scale=w.scale, num_splits=S)
    torch.cuda.synchronize()
    fa.check_device_status()
    assert torch.equal(a1, r1) and torch.equal(la1, lr1)
    assert torch.equal(a2, r2) and torch.equal(la2, lr2)
    assert not torch.equal(a1, a2)


@pytest.mark.gpu
def test_one_split_causal_multiwave_matches_fa_forward():
    # One split runs the fused forward; this causal shape has more than two waves of work
    # items, so it also exercises the per-shape work table that lives in module memory.
    w = workloads.WORKLOADS["c4"]
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    a, la = fa.forward_splitkv_noalloc(q, k, v, causal=True, scale=w.scale, num_splits=1)
    r, lr = fa.forward(q, k, v, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    fa.check_device_status()
    assert torch.equal(a, r) and torch.equal(la, lr)


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,D,causal", [(1, 1, 16384, 128, True), (1, 1, 65536, 64, True),
                                            (1, 1, 16384, 128, False)])
def test_automatic_split_count_fits_the_scratch(B, H, N, D, causal):
    # num_splits = 0: the cost model's choice, lowered to the largest count whose partials fit
    # the 32 MiB scratch; never FA_ERR_SCRATCH. Same result as the workspace entry point with
    # that count.
    w = workloads.Workload("auto", B, H, N, D, "fp16", causal, seed=77 + N)
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    S = fa.splitkv_num_splits(B, H, N, D, causal)
    while S > 1 and fa.splitkv_workspace_bytes(B, H, N, D, S) > fa.NOALLOC_SCRATCH_BYTES:
        S -= 1
    a, la = fa.forward_splitkv_noalloc(q, k, v, causal=causal, scale=w.scale, num_splits=0)
    r, lr = fa.forward_splitkv(q, k, v, causal=causal, scale=w.scale, num_splits=S)
    torch.cuda.synchronize()
    fa.check_device_status()
    assert torch.equal(a, r) and torch.equal(la, lr)
