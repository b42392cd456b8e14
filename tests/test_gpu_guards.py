"""Guard bands around every output (in place of the memcheck runs the pages
report: "Integrate H3 SM70 execution, metrics and VSA diagnostics", Test
Result).  Each entry point writes into a view at the middle of a larger
buffer filled with a sentinel; after the call on ragged sizes (tails that are
not whole tiles, pages, cubes or sequences) the guard bands must still hold
the sentinel, the rows the definition fixes (padded causal queries, padding
slots of boundary cubes) must hold their defined values, and the output must
match the oracle.  Sentinels are bit patterns no correct result here can
produce (-7776 in FP16, FP32 and int32)."""

import numpy as np
import pytest
import torch

from attention_fp16_flashattention_gb300 import inputs
from oracle import attention as OA
from oracle import decode as OD
from oracle import e4m3 as OE
from oracle import vsa as OV

pytestmark = pytest.mark.gpu

GUARD = 4096            # elements on each side (a multiple of 16 bytes for every dtype)
SENT = -7776         # exact in FP16, FP32 and int32


def t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


class Guarded:
    """A tensor of `shape` inside a buffer with GUARD sentinel elements on both sides."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape))
        self.buf = torch.full((GUARD + n + GUARD,), SENT, dtype=dtype, device="cuda")
        self.view = self.buf[GUARD:GUARD + n].view(*shape)

    def intact(self):
        b = self.buf.cpu()
        return bool(torch.all(b[:GUARD] == SENT)) and bool(torch.all(b[-GUARD:] == SENT))


def close(got, ref):
    got = np.asarray(got, dtype=np.float64)
    return bool(np.all(np.abs(got - ref) <= 2e-3 + 1e-2 * np.abs(ref)))


def test_guards_dense_and_masked(gb):
    q, k, v = inputs.dense_inputs(1, 3, 300, 128, seed=81, skv=200)
    o, lse = Guarded((1, 3, 300, 128), torch.float16), Guarded((1, 3, 300), torch.float32)
    gb.attn_dense_fwd(t(q), t(k), t(v), o=o.view, lse=lse.view)
    torch.cuda.synchronize()
    ro, rl = OA.dense_attention(q, k, v, inputs.softmax_scale(128))
    assert o.intact() and lse.intact()
    assert close(o.view.float().cpu().numpy(), ro) and np.allclose(lse.view.cpu().numpy(), rl, atol=1e-3)
    q, k, v = inputs.dense_inputs(1, 2, 200, 128, seed=82, skv=264)
    mask = inputs.additive_mask(200, 264, 82)
    o, lse = Guarded((1, 2, 200, 128), torch.float16), Guarded((1, 2, 200), torch.float32)
    gb.attn_dense_mask_fwd(t(q), t(k), t(v), t(mask), o=o.view, lse=lse.view)
    torch.cuda.synchronize()
    ro, _ = OA.dense_masked_attention(q, k, v, mask[None, None], inputs.softmax_scale(128))
    assert o.intact() and lse.intact() and close(o.view.float().cpu().numpy(), ro)
    assert gb.device_status() == 0


@pytest.mark.parametrize("split", [False, True])
def test_guards_causal_padded_queries(gb, split):
    Qp, q_real, KV = 192, 150, 1056
    q, k, v = inputs.causal_inputs(1, 6, 1, Qp, KV, 256, seed=83)
    o, lse = Guarded((1, 6, Qp, 256), torch.float16), Guarded((1, 6, Qp), torch.float32)
    gb.attn_causal_prefill_fwd(t(q), t(k), t(v), q_real=q_real, o=o.view, lse=lse.view,
                               prob_split=split)
    torch.cuda.synchronize()
    ro, _ = OA.causal_prefill_attention(q, k, v, inputs.softmax_scale(256), q_real)
    got = o.view.float().cpu().numpy()
    assert o.intact() and lse.intact() and close(got, ro)
    assert np.all(got[:, :, q_real:] == 0)
    assert np.all(np.isneginf(lse.view.cpu().numpy()[:, :, q_real:]))
    assert gb.device_status() == 0


def test_guards_bridge_and_fused_paged(gb):
    kv_len = 1000                                   # not a multiple of the 32-token page
    kp, vp, table = inputs.paged_e4m3_inputs(1, 1024, 256, seed=84, page_size=32)
    ko, vo = Guarded((1, kv_len, 256), torch.float16), Guarded((1, kv_len, 256), torch.float16)
    gb.e4m3_paged_to_fp16(t(kp), t(vp), t(table), kv_len, 0.0625, 0.125, k_out=ko.view,
                          v_out=vo.view)
    torch.cuda.synchronize()
    rk, rv = OE.paged_e4m3_to_fp16(kp, vp, table, kv_len, 0.0625, 0.125)
    assert ko.intact() and vo.intact()
    assert np.array_equal(ko.view.cpu().numpy().view(np.uint16), rk)
    assert np.array_equal(vo.view.cpu().numpy().view(np.uint16), rv)
    KV = 2080
    q = inputs.causal_inputs(1, 6, 1, 128, 32, 256, 85)[0]
    kp, vp, table = inputs.paged_e4m3_inputs(1, 2112, 256, seed=85, page_size=32)
    o, lse = Guarded((1, 6, 128, 256), torch.float16), Guarded((1, 6, 128), torch.float32)
    gb.attn_causal_prefill_paged_fwd(t(q), t(kp), t(vp), t(table), KV, 0.0625, 0.125, q_real=100,
                                     o=o.view, lse=lse.view)
    torch.cuda.synchronize()
    assert o.intact() and lse.intact()
    assert np.all(o.view.float().cpu().numpy()[:, :, 100:] == 0)
    assert gb.device_status() == 0


def test_guards_paged_decode(gb):
    q, kp, vp, table, lens = inputs.paged_decode_inputs(3, 6, 1, 2, (70, 1111, 2049), 256, seed=86)
    o, lse = Guarded((3, 6, 2, 256), torch.float16), Guarded((3, 6, 2), torch.float32)
    gb.attn_paged_decode_fwd(*(t(x) for x in (q, kp, vp, table, lens)), 0.0625, 0.125, o=o.view,
                             lse=lse.view)
    torch.cuda.synchronize()
    ro, _ = OD.paged_decode_attention(q, kp, vp, table, lens, 0.0625, 0.125,
                                      inputs.softmax_scale(256))
    assert o.intact() and lse.intact() and close(o.view.float().cpu().numpy(), ro)
    assert gb.device_status() == 0


def test_guards_vsa_selection_pairs_sparse_coarse(gb):
    prefix = 128
    q, k, v, valid = inputs.vsa_full_inputs(1, 2, 128, seed=87, grid=(3, 9, 10), prefix=prefix)
    nc = valid.size                                 # odd cube counts leave one cube unpaired
    tq, tk, tv, tval = t(q), t(k), t(v), t(valid)
    idx = Guarded((1, 2, nc, 5), torch.int32)
    gb.vsa_select_blocks(tq, tk, 5, prefix=prefix, cube_valid=tval, idx=idx.view)
    idx2, oc = Guarded((1, 2, nc, 5), torch.int32), Guarded((1, 2, nc, 128), torch.float32)
    gb.vsa_select_blocks_coarse(tq, tk, tv, 5, prefix=prefix, cube_valid=tval, idx=idx2.view,
                                coarse=oc.view)
    pairs = Guarded((1, 2, (nc + 1) // 2, 2), torch.int32)
    gb.vsa_pair_query_cubes(idx.view, pairs=pairs.view)
    o, lse = Guarded(q.shape, torch.float16), Guarded(q.shape[:3], torch.float32)
    gb.vsa_sparse_fwd(tq, tk, tv, idx.view, prefix=prefix, cube_valid=tval, pairs=pairs.view,
                      o=o.view, lse=lse.view)
    torch.cuda.synchronize()
    for g in (idx, idx2, oc, pairs, o, lse):
        assert g.intact()
    ridx = OV.vsa_select(q, k, 64, 5, valid, prefix=prefix)
    assert np.array_equal(idx.view.cpu().numpy(), ridx)
    assert np.array_equal(idx2.view.cpu().numpy(), ridx)
    p = pairs.view.cpu().numpy()
    for h in range(2):
        cubes = sorted(x for x in p[0, h].ravel() if x >= 0)
        assert cubes == list(range(nc))             # every cube exactly once
    got = o.view.float().cpu().numpy()
    ro, _ = OA.vsa_sparse_attention(q, k, v, ridx, 64, inputs.softmax_scale(128), valid=valid,
                                    prefix=prefix)
    assert close(got, ro)
    for c in range(nc):                             # padding slots of boundary cubes
        pad = slice(prefix + c * 64 + valid[c], prefix + (c + 1) * 64)
        assert np.all(got[:, :, pad] == 0)
    assert gb.device_status() == 0
