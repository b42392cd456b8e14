"""The VSA coarse ("compression") branch through the C ABI: pooled Q/K/V,
cube-level attention over all key cubes, and the gated sum with the fine
(selected-cube) output, against the oracle on every row of small layouts
(plain, and prefix + boundary cubes) and on sampled rows of the full-size
workload."""

import numpy as np
import pytest
import torch

from attention_fp16_flashattention_gb300 import inputs
from oracle import attention as OA
from oracle import vsa as OV

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


def t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def assert_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    bad = np.abs(got - ref) > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance"


def _gate(shape, seed):
    return np.random.default_rng(seed).uniform(-1.0, 1.0, shape).astype(np.float16)


@pytest.mark.parametrize("layout", ["plain", "full"])
def test_coarse_branch_all_rows(gb, layout):
    scale = inputs.softmax_scale(128)
    if layout == "plain":
        q, k, v = inputs.vsa_inputs(1, 2, 128, seed=71, grid=(4, 32, 32))
        prefix, valid, topk = 0, None, 8
    else:
        q, k, v, valid = inputs.vsa_full_inputs(1, 2, 128, seed=72, grid=(5, 10, 9), prefix=128)
        prefix, topk = 128, 5
    g = _gate(q.shape, 73)
    tv_ = None if valid is None else t(valid)
    idx, oc = gb.vsa_select_blocks_coarse(t(q), t(k), t(v), topk, prefix=prefix, cube_valid=tv_)
    o = gb.vsa_sparse_fwd(t(q), t(k), t(v), idx, prefix=prefix, cube_valid=tv_,
                          pairs=gb.vsa_pair_query_cubes(idx), coarse=oc, gate=t(g))
    torch.cuda.synchronize()
    ridx = OV.vsa_select(q, k, 64, topk, valid, prefix=prefix)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    roc = OV.coarse_attention(q, k, v, 64, scale, valid, prefix=prefix)
    assert_close(oc.cpu().numpy(), roc, "coarse output")
    rfine, _ = OA.vsa_sparse_attention(q, k, v, ridx, 64, scale, valid=valid, prefix=prefix)
    ro = OV.gated_output(rfine, roc, g, 64, valid, prefix)
    assert_close(o.float().cpu().numpy(), ro, "gated output")
    assert gb.device_status() == 0


def test_coarse_zero_gate_equals_fine_bit_for_bit(gb):
    q, k, v = inputs.vsa_inputs(1, 2, 128, seed=74, grid=(4, 32, 32))
    idx, oc = gb.vsa_select_blocks_coarse(t(q), t(k), t(v), 8)
    fine = gb.vsa_sparse_fwd(t(q), t(k), t(v), idx)
    gated = gb.vsa_sparse_fwd(t(q), t(k), t(v), idx, coarse=oc,
                              gate=torch.zeros(q.shape, dtype=torch.float16, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(fine, gated)
    assert torch.equal(idx, gb.vsa_select_blocks(t(q), t(k), 8))


def test_coarse_full_size_sampled(gb):
    w = inputs.WORKLOADS["vsa_video"]
    q, k, v = inputs.vsa_inputs(w["B"], w["H"], w["D"], w["seed"], w["grid"], w["cube"])
    scale = inputs.softmax_scale(128)
    g = _gate(q.shape, 75)
    tq, tk, tv = t(q), t(k), t(v)
    idx, oc = gb.vsa_select_blocks_coarse(tq, tk, tv, w["topk"])
    o = gb.vsa_sparse_fwd(tq, tk, tv, idx, pairs=gb.vsa_pair_query_cubes(idx), coarse=oc,
                          gate=t(g))
    torch.cuda.synchronize()
    ridx = OV.vsa_select(q, k, 64, w["topk"])
    assert np.array_equal(idx.cpu().numpy(), ridx)
    roc = OV.coarse_attention(q, k, v, 64, scale)
    assert_close(oc.cpu().numpy(), roc, "coarse output")
    rows = inputs.sample_rows(w["B"] * w["H"], q.shape[2], 4096, seed=7006)
    rfine, _ = OA.vsa_sparse_attention(q, k, v, ridx, 64, scale, rows=rows)
    hi, ri = rows[:, 0], rows[:, 1]
    ref = rfine + g.reshape(-1, q.shape[2], 128)[hi, ri] * roc.reshape(-1, 512, 128)[hi, ri // 64]
    got = o.reshape(-1, q.shape[2], 128)[torch.from_numpy(hi).cuda(), torch.from_numpy(ri).cuda()]
    assert_close(got.float().cpu().numpy(), ref, "gated sampled")
    assert gb.device_status() == 0
