"""GPU parity: the CUDA library against the CPU oracle on the same seeded inputs.

Bars: the E4M3 bridge and the VSA selection are bit-exact; attention outputs
satisfy |o - ref| <= 2e-3 + 1e-2 |ref| element by element against the float64
oracle.  Small workloads are checked on every row; the full-size workloads
(32768-token video heads, 131072-key prefill) on 4096 seeded (head, row)
samples in the same launch configuration the benchmark times.
"""

import numpy as np
import pytest
import torch

from attention_fp16_flashattention_gb300 import inputs
from oracle import attention as OA
from oracle import e4m3 as OE
from oracle import vsa as OV

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2
DEV = "cuda"


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    excess = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
    bad = int((excess > 0).sum())
    assert bad == 0, f"{what}: {bad} of {excess.size} outside tolerance, max excess {excess.max():.3e}"


_CACHE = {}


def workload(name):
    """Seeded full-size inputs, generated once per test session."""
    if name not in _CACHE:
        w = inputs.WORKLOADS[name]
        if name == "dense_video":
            _CACHE[name] = inputs.dense_inputs(w["B"], w["H"], w["S"], w["D"], w["seed"], video=True)
        elif name == "vsa_video":
            _CACHE[name] = inputs.vsa_inputs(w["B"], w["H"], w["D"], w["seed"], w["grid"], w["cube"])
        elif name == "paged_e4m3":
            _CACHE[name] = inputs.paged_e4m3_inputs(w["Hkv"], w["KV"], w["D"], w["seed"],
                                                    w["page_size"])
    return _CACHE[name]


def t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def rows_of(o, rows):
    """Pick (head, row) samples from a [B, H, S, D] tensor."""
    flat = o.reshape(-1, o.shape[2], o.shape[3])
    hi = torch.from_numpy(rows[:, 0]).to(o.device)
    ri = torch.from_numpy(rows[:, 1]).to(o.device)
    return flat[hi, ri].float().cpu().numpy()


# ------------------------------------------------------------------ bridge
@pytest.mark.parametrize("k_scale,v_scale", [
    (1.0, 1.0), (0.0625, 0.125),                                   # the workload's scales
    (float(np.float16(0.3)), float(np.float16(1 / 3))),            # FP16 scales that round
    (2.0 ** -14, 2.0 ** -20),                                      # subnormal FP16 results
    (1 / 3, 0.3), (1.7e-3, 300.0), (7.123e-5, 2.0 ** -14)])         # FP32-only scales
def test_bridge_all_codes_bit_exact(gb, k_scale, v_scale):
    codes = np.arange(256, dtype=np.uint8)
    P, ps, Hkv, D = 8, 32, 1, 256
    kp = np.resize(codes, P * ps * Hkv * D).reshape(P, ps, Hkv, D)
    vp = np.ascontiguousarray(kp[::-1])
    table = np.random.default_rng(0).permutation(P).astype(np.int32)
    ko, vo = gb.e4m3_paged_to_fp16(t(kp), t(vp), t(table), P * ps, k_scale, v_scale)
    rk, rv = OE.paged_e4m3_to_fp16(kp, vp, table, P * ps, k_scale, v_scale)
    tok = np.arange(P * ps)
    for got, ref, pages in ((ko, rk, kp), (vo, rv, vp)):
        g = got.cpu().numpy().view(np.uint16)
        nan = np.isnan(OE.e4m3fn_decode(pages[table[tok // ps], tok % ps])).transpose(1, 0, 2)
        assert np.array_equal(g[~nan], ref[~nan])
        # NaN codes decode to a NaN (payload not fixed by the pages)
        assert np.all((g[nan] & 0x7C00) == 0x7C00) and np.all((g[nan] & 0x3FF) != 0)
    assert gb.device_status() == 0


def test_bridge_live_length_multi_head_and_bad_page(gb):
    kp, vp, table = inputs.paged_e4m3_inputs(3, 700, 64, seed=5, page_size=16, num_phys_pages=60)
    kv_len = 677
    ko, vo = gb.e4m3_paged_to_fp16(t(kp), t(vp), t(table), kv_len, 0.0625, 0.125)
    rk, rv = OE.paged_e4m3_to_fp16(kp, vp, table, kv_len, 0.0625, 0.125)
    assert np.array_equal(ko.cpu().numpy().view(np.uint16), rk)
    assert np.array_equal(vo.cpu().numpy().view(np.uint16), rv)
    assert gb.device_status() == 0
    bad = table.copy()
    bad[3] = 60                                     # out of range physical page
    ko, vo = gb.e4m3_paged_to_fp16(t(kp), t(vp), t(bad), kv_len, 0.0625, 0.125)
    assert gb.device_status() & gb.DEV_BAD_PAGE
    k = ko.cpu().numpy().view(np.uint16)
    assert np.all(k[:, 3 * 16:4 * 16] == 0)
    assert np.array_equal(k[:, :48], rk[:, :48]) and np.array_equal(k[:, 64:], rk[:, 64:])


@pytest.mark.parametrize("Hkv,D,kv_len,k_scale,v_scale", [
    (1, 16, 333, 0.0625, 0.125),       # two 8-byte chunks per token row
    (5, 48, 301, 1 / 3, 0.3),          # rows of 6 chunks, round-to-odd scaling
    (2, 208, 259, float(np.float16(0.3)), 2.0 ** -14)])
def test_bridge_head_widths_bit_exact(gb, Hkv, D, kv_len, k_scale, v_scale):
    """Head widths whose rows are not a multiple of a warp's 32 chunks, several KV heads and
    a live length that ends inside a page."""
    kp, vp, table = inputs.paged_e4m3_inputs(Hkv, kv_len + 20, D, seed=D + Hkv, page_size=16)
    ko, vo = gb.e4m3_paged_to_fp16(t(kp), t(vp), t(table), kv_len, k_scale, v_scale)
    rk, rv = OE.paged_e4m3_to_fp16(kp, vp, table, kv_len, k_scale, v_scale)
    assert np.array_equal(ko.cpu().numpy().view(np.uint16), rk)   # finite codes only
    assert np.array_equal(vo.cpu().numpy().view(np.uint16), rv)
    assert gb.device_status() == 0


def test_bridge_full_size_bit_exact(gb):
    w = inputs.WORKLOADS["paged_e4m3"]
    kp, vp, table = workload("paged_e4m3")
    ko, vo = gb.e4m3_paged_to_fp16(t(kp), t(vp), t(table), w["KV"], w["k_scale"], w["v_scale"])
    rk, rv = OE.paged_e4m3_to_fp16(kp, vp, table, w["KV"], w["k_scale"], w["v_scale"])
    assert np.array_equal(ko.cpu().numpy().view(np.uint16), rk)
    assert np.array_equal(vo.cpu().numpy().view(np.uint16), rv)


# ------------------------------------------------------------------ dense
def test_dense_small_all_rows(gb):
    w = inputs.WORKLOADS["dense_small"]
    q, k, v = inputs.dense_inputs(w["B"], w["H"], w["S"], w["D"], w["seed"])
    lse = torch.empty((w["B"], w["H"], w["S"]), dtype=torch.float32, device=DEV)
    o = gb.attn_dense_fwd(t(q), t(k), t(v), lse=lse)
    ro, rl = OA.dense_attention(q, k, v, inputs.softmax_scale(128))
    assert_close(o.float().cpu().numpy(), ro, "dense_small")
    assert np.allclose(lse.cpu().numpy(), rl, atol=1e-3, rtol=1e-4)
    assert gb.device_status() == 0


@pytest.mark.parametrize("Sq,Skv", [(1, 1), (200, 333), (128, 4096), (517, 129), (64, 1000),
                                     (256, 384), (128, 512), (130, 640), (300, 897)])
def test_dense_ragged(gb, Sq, Skv):
    q, k, v = inputs.dense_inputs(2, 3, Sq, 128, seed=Sq * 7 + Skv, skv=Skv)
    o = gb.attn_dense_fwd(t(q), t(k), t(v))
    ro, _ = OA.dense_attention(q, k, v, inputs.softmax_scale(128))
    assert_close(o.float().cpu().numpy(), ro, f"dense {Sq}x{Skv}")
    assert gb.device_status() == 0


def test_dense_large_scores_and_rescaling(gb):
    # big logits make the running max jump often (exercises the O rescale path)
    q, k, v = inputs.dense_inputs(1, 2, 256, 128, seed=77, skv=2048)
    ramp = np.linspace(0.2, 4.0, 2048, dtype=np.float32)[None, None, :, None]
    k = (k.astype(np.float32) * ramp).astype(np.float16)
    o = gb.attn_dense_fwd(t(q), t(k), t(v))
    ro, _ = OA.dense_attention(q, k, v, inputs.softmax_scale(128))
    assert_close(o.float().cpu().numpy(), ro, "dense rescale")


def test_dense_video_sampled(gb):
    w = inputs.WORKLOADS["dense_video"]
    q, k, v = workload("dense_video")
    o = gb.attn_dense_fwd(t(q), t(k), t(v))
    rows = inputs.sample_rows(w["B"] * w["H"], w["S"], 4096, seed=7003)
    ro, _ = OA.dense_attention(q, k, v, inputs.softmax_scale(128), rows=rows)
    assert_close(rows_of(o, rows), ro, "dense_video")
    assert gb.device_status() == 0


# ------------------------------------------------------------------ causal
def _causal_check(gb, B, Hq, Hkv, Qp, q_real, KV, seed, workspace=None, rows=None):
    q, k, v = inputs.causal_inputs(B, Hq, Hkv, Qp, KV, 256, seed)
    lse = torch.empty((B, Hq, Qp), dtype=torch.float32, device=DEV)
    o = gb.attn_causal_prefill_fwd(t(q), t(k), t(v), q_real=q_real, lse=lse, workspace=workspace)
    ro, rl = OA.causal_prefill_attention(q, k, v, inputs.softmax_scale(256), q_real, rows=rows)
    if rows is None:
        assert_close(o.float().cpu().numpy(), ro, "causal")
        real = np.isfinite(rl)
        assert np.allclose(lse.cpu().numpy()[real], rl[real], atol=1e-3, rtol=1e-4)
        assert np.all(o.float().cpu().numpy()[:, :, q_real:] == 0)
    else:
        assert_close(rows_of(o, rows), ro, "causal sampled")
    assert gb.device_status() == 0
    return o


def test_causal_small_all_rows(gb):
    w = inputs.WORKLOADS["causal_small"]
    _causal_check(gb, w["B"], w["Hq"], w["Hkv"], w["Q"], w["Q"], w["KV"], w["seed"])


@pytest.mark.parametrize("Qp,q_real,KV", [(64, 64, 64), (64, 1, 32), (192, 150, 1024),
                                          (256, 256, 256), (128, 100, 4000)])
def test_causal_edges(gb, Qp, q_real, KV):
    _causal_check(gb, 1, 6, 1, Qp, q_real, KV, seed=Qp + q_real + KV)


def test_causal_gqa_two_kv_heads_batch2(gb):
    _causal_check(gb, 2, 4, 2, 256, 200, 1056, seed=9)


def test_causal_split_counts_agree(gb):
    w = inputs.WORKLOADS["causal_small"]
    q, k, v = (t(x) for x in inputs.causal_inputs(1, 6, 1, 1024, 4096, 256, w["seed"]))
    o_one = gb.attn_causal_prefill_fwd(q, k, v, workspace=torch.empty(16, dtype=torch.uint8,
                                                                      device=DEV))
    o_split = gb.attn_causal_prefill_fwd(q, k, v)
    ro, _ = OA.causal_prefill_attention(*inputs.causal_inputs(1, 6, 1, 1024, 4096, 256, w["seed"]),
                                        inputs.softmax_scale(256), 1024)
    assert_close(o_one.float().cpu().numpy(), ro, "one chunk")
    assert_close(o_split.float().cpu().numpy(), ro, "split")


def test_paged_e4m3_prefill_sampled(gb):
    """The paged_e4m3 workload (bridge, then causal prefill with the probabilities
    carried as FP16 hi + lo) at the stated tolerance on 4096 sampled rows.

    With the pages' single FP16 P the output moves by up to 2^-11 sum_j w_j |v_j|,
    which for these E4M3 values (|v| up to 56) exceeds the stated bound in rows
    whose output cancels; hi + lo carries about 22 bits of every probability."""
    w = inputs.WORKLOADS["paged_e4m3"]
    kp, vp, table = workload("paged_e4m3")
    q = inputs.causal_inputs(w["B"], w["Hq"], w["Hkv"], w["Q"], 32, w["D"], w["seed"])[0]
    ko, vo = gb.e4m3_paged_to_fp16(t(kp), t(vp), t(table), w["KV"], w["k_scale"], w["v_scale"])
    o = gb.attn_causal_prefill_fwd(t(q), ko[None], vo[None], q_real=w["Q"], prob_split=True)
    rk, rv = OE.paged_e4m3_to_fp16(kp, vp, table, w["KV"], w["k_scale"], w["v_scale"])
    k16 = rk.view(np.float16)[None]
    v16 = rv.view(np.float16)[None]
    rows = inputs.sample_rows(w["B"] * w["Hq"], w["Q"], 4096, seed=7005)
    ro, _ = OA.causal_prefill_attention(q, k16, v16, inputs.softmax_scale(w["D"]), w["Q"], rows=rows)
    assert_close(rows_of(o, rows), ro, "paged_e4m3 prefill")
    assert gb.device_status() == 0


def test_prob_split_small_all_rows(gb):
    w = inputs.WORKLOADS["causal_small"]
    q, k, v = inputs.causal_inputs(1, 6, 1, 1024, 4096, 256, w["seed"])
    lse = torch.empty((1, 6, 1024), dtype=torch.float32, device=DEV)
    o = gb.attn_causal_prefill_fwd(t(q), t(k), t(v), lse=lse, prob_split=True)
    ro, rl = OA.causal_prefill_attention(q, k, v, inputs.softmax_scale(256), 1024)
    assert_close(o.float().cpu().numpy(), ro, "prob split")
    assert np.allclose(lse.cpu().numpy(), rl, atol=1e-3, rtol=1e-4)
    assert gb.device_status() == 0


# ------------------------------------------------------------------ VSA
def test_vsa_select_small_and_ties(gb):
    q, k, v = inputs.vsa_inputs(1, 3, 128, seed=3, grid=(4, 32, 32))
    idx = gb.vsa_select_blocks(t(q), t(k), topk=16)
    assert np.array_equal(idx.cpu().numpy(), OV.vsa_select(q, k, 64, 16))
    k2 = k.copy()
    k2[:, :, 5 * 64:6 * 64] = k2[:, :, 2 * 64:3 * 64]    # duplicate cubes -> exact score ties
    k2[:, :, 7 * 64:9 * 64] = 0                          # two all-zero cubes tie too
    for topk in (1, 7, 64):
        idx = gb.vsa_select_blocks(t(q), t(k2), topk=topk)
        assert np.array_equal(idx.cpu().numpy(), OV.vsa_select(q, k2, 64, topk)), topk
    nc = q.shape[2] // 64
    idx = gb.vsa_select_blocks(t(q), t(k), topk=nc)
    assert np.array_equal(idx.cpu().numpy(), np.broadcast_to(np.arange(nc), idx.shape))
    # every key cube equal (all 64 scores tie: more undecided keys than a warp ranks in
    # place, so the fallback kernel decides), and half of them equal
    k3 = np.broadcast_to(k[:, :, None, :64], (1, 3, nc, 64, 128)).reshape(k.shape).copy()
    k4 = k.reshape(1, 3, nc, 64, 128).copy()
    k4[:, :, ::2] = k3.reshape(1, 3, nc, 64, 128)[:, :, ::2]
    k4 = k4.reshape(k.shape)
    for kk in (k3, k4):
        for topk in (5, 40):
            idx = gb.vsa_select_blocks(t(q), t(kk), topk=topk)
            assert np.array_equal(idx.cpu().numpy(), OV.vsa_select(q, kk, 64, topk)), topk
    assert gb.device_status() == 0


def test_vsa_select_full_size_bit_exact(gb):
    w = inputs.WORKLOADS["vsa_video"]
    q, k, _ = workload("vsa_video")
    idx = gb.vsa_select_blocks(t(q), t(k), topk=w["topk"])
    ref = OV.vsa_select(q, k, 64, w["topk"])
    assert np.array_equal(idx.cpu().numpy(), ref)


def test_vsa_sparse_small_all_rows(gb):
    q, k, v = inputs.vsa_inputs(1, 2, 128, seed=4, grid=(4, 32, 32))
    ridx = OV.vsa_select(q, k, 64, 8)
    o = gb.vsa_sparse_fwd(t(q), t(k), t(v), t(ridx))
    ro, _ = OA.vsa_sparse_attention(q, k, v, ridx, 64, inputs.softmax_scale(128))
    assert_close(o.float().cpu().numpy(), ro, "vsa small")
    assert gb.device_status() == 0


def test_vsa_sparse_all_cubes_equals_dense_and_odd_cube_count(gb):
    q, k, v = inputs.dense_inputs(1, 2, 64 * 7, 128, seed=21)      # 7 cubes: odd pair count
    nc = 7
    idx = np.broadcast_to(np.arange(nc, dtype=np.int32), (1, 2, nc, nc)).copy()
    o = gb.vsa_sparse_fwd(t(q), t(k), t(v), t(idx))
    ro, _ = OA.dense_attention(q, k, v, inputs.softmax_scale(128))
    assert_close(o.float().cpu().numpy(), ro, "vsa all cubes")
    idx3 = np.stack([np.sort(np.random.default_rng(c).choice(nc, 3, replace=False))
                     for c in range(nc)]).astype(np.int32)
    idx3 = np.broadcast_to(idx3, (1, 2, nc, 3)).copy()
    o = gb.vsa_sparse_fwd(t(q), t(k), t(v), t(idx3))
    ro, _ = OA.vsa_sparse_attention(q, k, v, idx3, 64, inputs.softmax_scale(128))
    assert_close(o.float().cpu().numpy(), ro, "vsa 3 of 7")


def test_vsa_bad_index_flagged(gb):
    q, k, v = inputs.dense_inputs(1, 1, 64 * 4, 128, seed=22)
    idx = np.array([[[[0, 2], [1, 1], [3, 9], [0, 1]]]], dtype=np.int32)   # repeat, out of range
    gb.vsa_sparse_fwd(t(q), t(k), t(v), t(idx))
    assert gb.device_status() & gb.DEV_BAD_INDEX


def test_vsa_full_size_sampled(gb):
    w = inputs.WORKLOADS["vsa_video"]
    q, k, v = workload("vsa_video")
    tq, tk, tv = t(q), t(k), t(v)
    idx = gb.vsa_select_blocks(tq, tk, topk=w["topk"])
    o = gb.vsa_sparse_fwd(tq, tk, tv, idx)
    ridx = OV.vsa_select(q, k, 64, w["topk"])
    assert np.array_equal(idx.cpu().numpy(), ridx)
    rows = inputs.sample_rows(w["B"] * w["H"], q.shape[2], 4096, seed=7004)
    ro, _ = OA.vsa_sparse_attention(q, k, v, ridx, 64, inputs.softmax_scale(128), rows=rows)
    assert_close(rows_of(o, rows), ro, "vsa_video")
    assert gb.device_status() == 0


# ------------------------------------------------------------------ determinism
def test_repeat_runs_are_bitwise_identical(gb):
    q, k, v = (t(x) for x in inputs.causal_inputs(1, 6, 1, 512, 8192, 256, seed=31))
    a = gb.attn_causal_prefill_fwd(q, k, v)
    b = gb.attn_causal_prefill_fwd(q, k, v)
    qd, kd, vd = (t(x) for x in inputs.dense_inputs(1, 4, 1024, 128, seed=32))
    c = gb.attn_dense_fwd(qd, kd, vd)
    d = gb.attn_dense_fwd(qd, kd, vd)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(c, d)
