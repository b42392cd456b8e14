"""The fused paged-E4M3 causal prefill against the bridge followed by the FP16
prefill (bit for bit: the same FP16 keys and values, the same arithmetic), and
against the oracle on the paged workload's small shapes."""

import numpy as np
import pytest
import torch

from attention_fp16_flashattention_gb300 import inputs
from oracle import attention as OA
from oracle import e4m3 as OE
from oracle.fp16 import fp16_bits_to_f64

pytestmark = pytest.mark.gpu


def t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def two_ways(gb, Hq, Hkv, Q, KV, ps, ks, vs, seed, q_real=None, codes="finite", split=False):
    q = inputs.causal_inputs(1, Hq, Hkv, Q, 32, 256, seed)[0]
    if codes == "finite":
        kp, vp, table = inputs.paged_e4m3_inputs(Hkv, KV, 256, seed, page_size=ps)
    else:
        _, kp, vp, tb, _ = inputs.paged_decode_inputs(1, 1, Hkv, 1, (KV,), 256, seed, page_size=ps,
                                                      codes=codes)
        table = tb[0]
    tq, tk, tv, tt = t(q), t(kp), t(vp), t(table)
    lse_f = torch.empty((1, Hq, Q), dtype=torch.float32, device="cuda")
    of = gb.attn_causal_prefill_paged_fwd(tq, tk, tv, tt, KV, ks, vs, q_real=q_real, lse=lse_f,
                                          prob_split=split)
    kf, vf = gb.e4m3_paged_to_fp16(tk, tv, tt, KV, ks, vs)
    lse_b = torch.empty((1, Hq, Q), dtype=torch.float32, device="cuda")
    ob = gb.attn_causal_prefill_fwd(tq, kf[None], vf[None], q_real=q_real, lse=lse_b,
                                    prob_split=split)
    torch.cuda.synchronize()
    assert gb.device_status() == 0
    return q, kp, vp, table, of, lse_f, ob, lse_b


@pytest.mark.parametrize("Hq,Hkv,Q,KV,ps,ks,vs", [
    (6, 1, 256, 1024, 32, 0.0625, 0.125),          # the workload's layout, folded scales
    (6, 1, 320, 4096, 16, 0.0625, 0.125),          # small pages, several key chunks
    (4, 2, 128, 2048, 64, float(np.float16(0.3)), float(np.float16(0.7))),   # FP16-valued scales
    (6, 1, 192, 1536, 128, 1 / 3, 0.3),            # general scales (round-to-odd)
    (6, 1, 64, 2080, 32, 0.0625, 0.125),           # KV not a multiple of 128 (ragged last tile)
    (6, 1, 128, 1536, 256, 0.0625, 0.125)])        # pages of 256 tokens (two 128-key tiles each)
def test_fused_equals_bridge_then_prefill(gb, Hq, Hkv, Q, KV, ps, ks, vs):
    for split in (False, True):
        _, _, _, _, of, lf, ob, lb = two_ways(gb, Hq, Hkv, Q, KV, ps, ks, vs, seed=90 + ps,
                                              split=split)
        assert torch.equal(of, ob), split
        assert torch.equal(lf, lb), split


def test_fused_padded_queries_and_nan_codes_past_the_end(gb):
    # 64-token pages: the last page holds keys 2048..2111, of which 2080.. are past the end
    q, kp, vp, table, of, lf, ob, lb = two_ways(gb, 6, 1, 256, 2080, 64, 0.0625, 0.125, seed=97,
                                                q_real=200)
    assert torch.equal(of, ob) and torch.equal(lf, lb)
    # NaN codes in the unused slots of the last page change nothing
    kp2, vp2 = kp.copy(), vp.copy()
    last = table[(2080 - 1) // 64]
    kp2[last, 2080 % 64:] = 0x7F
    vp2[last, 2080 % 64:] = 0xFF
    o2 = gb.attn_causal_prefill_paged_fwd(t(q), t(kp2), t(vp2), t(table), 2080, 0.0625, 0.125,
                                          q_real=200)
    torch.cuda.synchronize()
    assert torch.equal(o2, of)


def test_fused_matches_oracle(gb):
    q, kp, vp, table, of, lf, _, _ = two_ways(gb, 6, 1, 256, 1024, 32, 0.0625, 0.125, seed=98,
                                              codes="moderate")
    kb, vb = OE.paged_e4m3_to_fp16(kp, vp, table, 1024, 0.0625, 0.125)
    k = fp16_bits_to_f64(kb).astype(np.float16)[None]
    v = fp16_bits_to_f64(vb).astype(np.float16)[None]
    ro, rl = OA.causal_prefill_attention(q, k, v, inputs.softmax_scale(256), 256)
    got = of.float().cpu().numpy()
    assert np.all(np.abs(got - ro) <= 2e-3 + 1e-2 * np.abs(ro))
    assert np.all(np.abs(lf.cpu().numpy() - rl) <= 2e-3 + 1e-2 * np.abs(rl))


def test_fused_prob_split_matches_oracle_on_uniform_codes(gb):
    """The workload's code distribution (uniform over the finite E4M3 codes, |v| up
    to 56) with hi + lo probabilities, at the stated tolerance on every row."""
    q, kp, vp, table, of, lf, _, _ = two_ways(gb, 6, 1, 512, 4096, 32, 0.0625, 0.125, seed=96,
                                              split=True)
    kb, vb = OE.paged_e4m3_to_fp16(kp, vp, table, 4096, 0.0625, 0.125)
    k = fp16_bits_to_f64(kb).astype(np.float16)[None]
    v = fp16_bits_to_f64(vb).astype(np.float16)[None]
    ro, rl = OA.causal_prefill_attention(q, k, v, inputs.softmax_scale(256), 512)
    got = of.float().cpu().numpy()
    assert np.all(np.abs(got - ro) <= 2e-3 + 1e-2 * np.abs(ro))
    assert np.all(np.abs(lf.cpu().numpy() - rl) <= 2e-3 + 1e-2 * np.abs(rl))


def test_fused_bad_page_flagged(gb):
    q = inputs.causal_inputs(1, 6, 1, 64, 32, 256, 99)[0]
    kp, vp, table = inputs.paged_e4m3_inputs(1, 512, 256, 99)
    bad = table.copy()
    bad[3] = 1_000_000
    gb.attn_causal_prefill_paged_fwd(t(q), t(kp), t(vp), t(bad), 512, 0.0625, 0.125)
    torch.cuda.synchronize()
    assert gb.device_status() & gb.DEV_BAD_PAGE


def test_fused_full_workload_equals_bridge_then_prefill(gb):
    """The paged_e4m3 workload (Q=8192 at the tail of KV=131072)."""
    w = inputs.WORKLOADS["paged_e4m3"]
    q = inputs.causal_inputs(w["B"], w["Hq"], w["Hkv"], w["Q"], 32, w["D"], w["seed"])[0]
    kp, vp, table = inputs.paged_e4m3_inputs(w["Hkv"], w["KV"], w["D"], w["seed"], w["page_size"])
    tq, tk, tv, tt = t(q), t(kp), t(vp), t(table)
    kf, vf = gb.e4m3_paged_to_fp16(tk, tv, tt, w["KV"], w["k_scale"], w["v_scale"])
    for split in (False, True):
        of = gb.attn_causal_prefill_paged_fwd(tq, tk, tv, tt, w["KV"], w["k_scale"], w["v_scale"],
                                              prob_split=split)
        ob = gb.attn_causal_prefill_fwd(tq, kf[None], vf[None], prob_split=split)
        torch.cuda.synchronize()
        assert gb.device_status() == 0
        assert torch.equal(of, ob), split
