"""Failure detection on the GPU without a GPU fault.

Every pipeline wait inside the attention kernel is bounded in time.  A test
hook makes the kernel's TMA warp skip the query-tile load (mode 1), or stop
after two rounds of its K/V ring with MMAs of both issuing warps in flight
(mode 2), so a wait can never be satisfied ("a flag that nothing sets"): it
runs out after the short limit set here, the kernel records
GBATTN_DEV_WAIT_TIMEOUT in the device status word, lets what it issued finish,
frees tensor memory and returns.  The host reads the status, and the very next
normal call on the same context must produce correct results.
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


def _close(o, ro):
    err = np.abs(o.float().cpu().numpy() - ro) - (2e-3 + 1e-2 * np.abs(ro))
    return bool(np.all(err <= 0))


def _mid_stream_abort(gb, call):
    """Run `call` with the loads stopping mid-stream; return the status flags."""
    assert gb.device_status() == 0
    gb.set_wait_limit_ns(50_000_000)          # 50 ms
    gb.test_inject_fault(2)
    try:
        call()
        flags = gb.device_status()
    finally:
        gb.test_inject_fault(0)
        gb.set_wait_limit_ns(1_000_000_000)
    return flags


def test_mid_stream_timeout_dense_two_issuers(gb):
    q, k, v = inputs.dense_inputs(1, 2, 256, 128, seed=62, skv=2048)      # 16 key tiles
    tq, tk, tv = (torch.from_numpy(x).cuda() for x in (q, k, v))
    assert _mid_stream_abort(gb, lambda: gb.attn_dense_fwd(tq, tk, tv)) & gb.DEV_WAIT_TIMEOUT
    ro, _ = OA.dense_attention(q, k, v, inputs.softmax_scale(128))
    assert _close(gb.attn_dense_fwd(tq, tk, tv), ro)
    assert gb.device_status() == 0


def test_mid_stream_timeout_masked_three_slot_ring(gb):
    q, k, v = inputs.dense_inputs(1, 2, 200, 128, seed=63, skv=1024)      # 8 key tiles
    mask = inputs.additive_mask(200, 1024, 63)
    tq, tk, tv = (torch.from_numpy(x).cuda() for x in (q, k, v))
    tm = torch.from_numpy(mask).cuda()
    flags = _mid_stream_abort(gb, lambda: gb.attn_dense_mask_fwd(tq, tk, tv, tm))
    assert flags & gb.DEV_WAIT_TIMEOUT
    ro, _ = OA.dense_masked_attention(q, k, v, mask[None, None], inputs.softmax_scale(128))
    assert _close(gb.attn_dense_mask_fwd(tq, tk, tv, tm), ro)
    assert gb.device_status() == 0


def test_mid_stream_timeout_causal_one_issuer(gb):
    q, k, v = inputs.causal_inputs(1, 6, 1, 256, 2048, 256, seed=64)      # about 5 key tiles per chunk
    tq, tk, tv = (torch.from_numpy(x).cuda() for x in (q, k, v))
    assert _mid_stream_abort(gb, lambda: gb.attn_causal_prefill_fwd(tq, tk, tv)) & gb.DEV_WAIT_TIMEOUT
    ro, _ = OA.causal_prefill_attention(q, k, v, inputs.softmax_scale(256), 256)
    assert _close(gb.attn_causal_prefill_fwd(tq, tk, tv), ro)
    assert gb.device_status() == 0
