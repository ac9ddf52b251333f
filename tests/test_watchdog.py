"""Failure detection on the GPU without faulting it.

Every device-side wait in the kernel is bounded; when one gives up, the kernel records a
status bit, all roles leave their loops, outstanding copies and MMAs are drained, tensor
memory is freed and the kernel returns. The test hook fa_debug_force_stall makes the MMA warp
wait on a barrier that nothing arrives on, with a 1 ms limit: the host must see
FA_ERR_TIMEOUT, and the next call without the hook must still produce correct results (the
context stays usable).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_prefill_gb300 import fa, workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,decomp", [("c3", fa.FA_DECOMP_TWO_TILES), ("c2", fa.FA_DECOMP_SPLIT_KV),
                                         ("c2", fa.FA_DECOMP_SPLIT_KV_SERIAL), ("c4", fa.FA_DECOMP_AUTO)])
def test_watchdog_timeout_reported_and_context_survives(name, decomp):
    w = workloads.WORKLOADS[name]
    q, k, v = (x.cuda() for x in workloads.make_qkv(w))
    fa.check_device_status()  # clear anything left over
    fa.set_decomposition(decomp)
    try:
        fa.set_watchdog_ns(1_000_000)
        fa.debug_force_stall(True)
        fa.forward(q, k, v, causal=w.causal, scale=w.scale)
        with pytest.raises(fa.FAError) as err:
            fa.check_device_status()
        assert err.value.code == fa.FA_ERR_TIMEOUT
    finally:
        fa.debug_force_stall(False)
        fa.set_watchdog_ns(0)
        fa.set_decomposition(fa.FA_DECOMP_AUTO)
    fa.check_device_status()  # the status word was cleared by the check above
    o, lse = fa.forward(q, k, v, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    fa.check_device_status()
    rows = np.array([[0, 0], [0, 1], [3, 129], [w.B * w.H - 1, w.N - 1], [7, w.N // 2]])
    ro, rl = oracle.attention_rows(q.cpu(), k.cpu(), v.cpu(), w.scale, w.causal, rows)
    o_s = o.float().cpu().numpy().reshape(-1, w.N, w.D)[rows[:, 0], rows[:, 1]]
    l_s = lse.cpu().numpy().reshape(-1, w.N)[rows[:, 0], rows[:, 1]]
    tol = 1e-2 if w.dtype == "bf16" else 2e-3
    assert np.abs(o_s - ro).max() <= tol
    assert np.abs(l_s - rl).max() <= 1e-3
