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


def test_mid_stream_timeout_sparse_and_full_layout(gb):
    from oracle import vsa as OV
    q, k, v = inputs.vsa_inputs(1, 2, 128, seed=65, grid=(4, 32, 32))
    tq, tk, tv = (torch.from_numpy(x).cuda() for x in (q, k, v))
    idx = gb.vsa_select_blocks(tq, tk, topk=8)
    for mode in (1, 2):
        assert gb.device_status() == 0
        gb.set_wait_limit_ns(50_000_000)
        gb.test_inject_fault(mode)
        try:
            gb.vsa_sparse_fwd(tq, tk, tv, idx)
            flags = gb.device_status()
        finally:
            gb.test_inject_fault(0)
            gb.set_wait_limit_ns(1_000_000_000)
        assert flags & gb.DEV_WAIT_TIMEOUT, mode
    ro, _ = OA.vsa_sparse_attention(q, k, v, OV.vsa_select(q, k, 64, 8), 64, inputs.softmax_scale(128))
    assert _close(gb.vsa_sparse_fwd(tq, tk, tv, idx), ro)
    # the full layout (prefix query tiles walk every prefix key tile)
    q, k, v, valid = inputs.vsa_full_inputs(1, 2, 128, seed=66, grid=(5, 10, 9), prefix=256)
    tq, tk, tv, tval = (torch.from_numpy(x).cuda() for x in (q, k, v, valid))
    idx = gb.vsa_select_blocks(tq, tk, 5, prefix=256, cube_valid=tval)
    call = lambda: gb.vsa_sparse_fwd(tq, tk, tv, idx, prefix=256, cube_valid=tval)
    assert _mid_stream_abort(gb, call) & gb.DEV_WAIT_TIMEOUT
    ro, _ = OA.vsa_sparse_attention(q, k, v, idx.cpu().numpy(), 64, inputs.softmax_scale(128),
                                    valid=valid, prefix=256)
    assert _close(call(), ro)
    assert gb.device_status() == 0


def test_mid_stream_timeout_paged_converter_warps(gb):
    """The fused paged prefill: the load warp stops after two ring rounds, so the
    E4M3 converter warps' waits for page bytes run out as well as the MMA and
    softmax warps' waits."""
    q = inputs.causal_inputs(1, 6, 1, 256, 32, 256, 67)[0]
    kp, vp, table = inputs.paged_e4m3_inputs(1, 2048, 256, 67, page_size=32)
    tq, tk, tv, tt = (torch.from_numpy(x).cuda() for x in (q, kp, vp, table))
    for split in (False, True):
        call = lambda: gb.attn_causal_prefill_paged_fwd(tq, tk, tv, tt, 2048, 0.0625, 0.125,
                                                        prob_split=split)
        assert _mid_stream_abort(gb, call) & gb.DEV_WAIT_TIMEOUT, split
        kf, vf = gb.e4m3_paged_to_fp16(tk, tv, tt, 2048, 0.0625, 0.125)
        ref = gb.attn_causal_prefill_fwd(tq, kf[None], vf[None], prob_split=split)
        assert torch.equal(call(), ref)
    assert gb.device_status() == 0


def test_timeout_paged_decode(gb):
    """The decode warps run their own rings: with nothing loaded (mode 1) or the
    loads stopping after two ring rounds (mode 2) their waits run out, each warp
    waits for the stages it issued and returns; the merge still completes."""
    from oracle import decode as OD
    # the tiles are split evenly over every warp of the GPU (8 per SM): about 7000
    # tiles leave each warp more than two rounds of its ring for mode 2 to cut
    q, kp, vp, table, lens = inputs.paged_decode_inputs(2, 6, 1, 1, (65536, 49152), 256, seed=68)
    args = [torch.from_numpy(x).cuda() for x in (q, kp, vp, table, lens)]
    for mode in (1, 2):
        assert gb.device_status() == 0
        gb.set_wait_limit_ns(50_000_000)
        gb.test_inject_fault(mode)
        try:
            gb.attn_paged_decode_fwd(*args, 0.0625, 0.125)
            flags = gb.device_status()
        finally:
            gb.test_inject_fault(0)
            gb.set_wait_limit_ns(1_000_000_000)
        assert flags & gb.DEV_WAIT_TIMEOUT, mode
    o = gb.attn_paged_decode_fwd(*args, 0.0625, 0.125)
    ro, _ = OD.paged_decode_attention(q, kp, vp, table, lens, 0.0625, 0.125,
                                      inputs.softmax_scale(256))
    assert _close(o, ro)
    assert gb.device_status() == 0
