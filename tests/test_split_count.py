"""The split-KV split count (host logic, no GPU): the cost model's choices on a 152-SM GB300 and
the lowering that keeps fa_forward_splitkv_noalloc's automatic count inside its 32 MiB scratch.
"""
import pytest

from tiled_attention_prefill_gb300 import fa

SCRATCH = fa.NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return fa.load_library()  # built by __graft_entry__.build(); a missing library fails the test


# (B, H, N, D, causal) -> the count chosen on 152 SMs. Each was timed on a GB300 against every
# count from 1 to 8 (CUDA events, inputs cycled beyond L2): the chosen count was the fastest,
# or, for 1 x 1 x 32768 x 64 causal, within 3% of it.
CHOICES_152 = [
    ((1, 1, 16384, 128, True), 2),   # 101.1 us at 1 split, 60.1 at 2
    ((1, 4, 8192, 64, True), 1),     # 47.7 us at 1, 62.3 at 2
    ((1, 2, 32768, 128, True), 1),   # 377.0 us at 1, 380.2 at 2
    ((1, 2, 16384, 128, False), 1),  # 190.6 us at 1, 205.7 at 4
    ((1, 1, 32768, 64, True), 2),    # 175.1 us at 2, 170.2 at 1
    ((4, 16, 4096, 128, True), 1),   # thousands of query tiles: whole waves already
    ((1, 1, 100, 64, False), 1),     # one key tile
]


@pytest.mark.parametrize("shape,want", CHOICES_152)
def test_cost_model_choices_on_152_sms(shape, want):
    assert fa.debug_num_splits(*shape, num_sms=152) == want


def test_one_split_is_estimated_across_heads():
    # With one split the fused forward balances the items of all heads together; estimated head
    # by head, 1 x 4 x 8192 x 64 causal once chose 2 splits, which measured 31% slower.
    assert fa.debug_num_splits(1, 4, 8192, 64, True, num_sms=152) == 1
    assert fa.debug_num_splits(1, 1, 16384, 128, True, num_sms=152) > 1


SHAPES = [(B, H, N, D, c) for B, H in ((1, 1), (1, 2), (2, 3), (1, 8)) for N in (128, 1000, 4096, 16384, 65536, 131072)
          for D in (64, 128) for c in (False, True)]


@pytest.mark.parametrize("num_sms", [148, 152, 160])
def test_noalloc_auto_count_fits_the_scratch(num_sms):
    for B, H, N, D, c in SHAPES:
        s = fa.debug_num_splits(B, H, N, D, c, num_sms=num_sms)
        s_na = fa.debug_num_splits(B, H, N, D, c, num_sms=num_sms, noalloc=True)
        assert 1 <= s_na <= s
        if s_na > 1:
            assert fa.splitkv_workspace_bytes(B, H, N, D, s_na) <= SCRATCH
        if fa.splitkv_workspace_bytes(B, H, N, D, s) <= SCRATCH:
            assert s_na == s  # lowered only when the model's count does not fit
        elif s_na < s:
            assert s_na == 1 or fa.splitkv_workspace_bytes(B, H, N, D, s_na + 1) > SCRATCH  # the largest that fits


def test_noalloc_auto_on_the_long_single_head_shapes():
    # Shapes the model splits whose partials at that count exceed 32 MiB: the automatic no-alloc
    # count is lowered, never an FA_ERR_SCRATCH.
    lowered = 0
    for shape in ((1, 1, 65536, 64, True), (1, 1, 16384, 128, False), (1, 1, 131072, 64, True)):
        for num_sms in (148, 152, 160):
            s = fa.debug_num_splits(*shape, num_sms=num_sms)
            s_na = fa.debug_num_splits(*shape, num_sms=num_sms, noalloc=True)
            assert s_na == 1 or fa.splitkv_workspace_bytes(*shape[:4], s_na) <= SCRATCH
            lowered += s_na < s
    # 1 x 1 x 65536 x 64 causal: 2 splits (32.5 MiB) on 148-160 SMs; 1 x 1 x 16384 x 128
    # non-causal: 5 splits (40 MiB) on 160 SMs, lowered to 3.
    assert lowered == 4
    assert fa.debug_num_splits(1, 1, 16384, 128, False, num_sms=160, noalloc=True) == 3


def test_bad_arguments():
    with pytest.raises(fa.FAError):
        fa.debug_num_splits(1, 1, 1024, 96, False, num_sms=152)
    with pytest.raises(fa.FAError):
        fa.debug_num_splits(1, 1, 1024, 64, False, num_sms=0)
    with pytest.raises(fa.FAError):
        fa.debug_num_splits(0, 1, 1024, 64, False, num_sms=152)
