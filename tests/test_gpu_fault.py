"""Failure detection on the GPU without a GPU fault.

Every pipeline wait inside the attention kernel is bounded in time.  A test
hook makes the kernel's TMA warp skip the query-tile load, so the first wait
for it can never be satisfied ("a flag that nothing sets"): the wait runs out
after the short limit set here, the kernel records GBATTN_DEV_WAIT_TIMEOUT in
the device status word, drains what it issued, frees tensor memory and
returns.  The host reads the status, and the very next normal call on the same
context must produce correct results.
"""

import numpy as np
import pytest
import torch

from attention_fp16_flashattention_gb300 import inputs
from oracle import attention as OA

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_stays_usable(gb):
    q, k, v = inputs.dense_inputs(1, 1, 256, 128, seed=61)
    tq, tk, tv = (torch.from_numpy(x).cuda() for x in (q, k, v))
    assert gb.device_status() == 0
    gb.set_wait_limit_ns(50_000_000)          # 50 ms
    gb.test_inject_fault(1)
    try:
        gb.attn_dense_fwd(tq, tk, tv)
        flags = gb.device_status()            # synchronises the stream
    finally:
        gb.test_inject_fault(0)
        gb.set_wait_limit_ns(1_000_000_000)
    assert flags & gb.DEV_WAIT_TIMEOUT
    o = gb.attn_dense_fwd(tq, tk, tv)
    ro, _ = OA.dense_attention(q, k, v, inputs.softmax_scale(128))
    err = np.abs(o.float().cpu().numpy() - ro) - (2e-3 + 1e-2 * np.abs(ro))
    assert np.all(err <= 0)
    assert gb.device_status() == 0
