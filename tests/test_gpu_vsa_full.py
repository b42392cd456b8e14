"""GPU parity of the full VSA layout: prefix tokens, boundary cubes, padding slots.

Selection must equal the oracle bit for bit; attention outputs satisfy
|o - ref| <= 2e-3 + 1e-2 |ref| (and the same for lse) on every row of small
layouts and on 4096 seeded rows of the B1 H24 workload the benchmark times
(1024 prefix tokens + an 8x62x62 grid in 512 cubes, 30752 real tokens).
"""

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


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        excess = np.where(both_inf, -1.0, np.abs(got - ref) - (ATOL + RTOL * np.abs(ref)))
    bad = int((excess > 0).sum())
    assert bad == 0, f"{what}: {bad} of {excess.size} outside tolerance, max excess {excess.max():.3e}"


def run(gb, q, k, v, valid, prefix, topk):
    tq, tk, tv = t(q), t(k), t(v)
    tval = t(valid)
    idx = gb.vsa_select_blocks(tq, tk, topk, prefix=prefix, cube_valid=tval)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    o = gb.vsa_sparse_fwd(tq, tk, tv, idx, prefix=prefix, cube_valid=tval, lse=lse)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), o.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("grid,prefix,topk", [
    ((5, 10, 9), 128, 5),        # 18 cubes, boundary cubes of 2..64 real tokens
    ((8, 13, 12), 0, 7),         # no prefix, boundary cubes
    ((4, 16, 16), 256, 6),       # full cubes with a prefix
    ((3, 6, 7), 128, 2)])        # odd cube count, tiny cubes
def test_full_vsa_small(gb, grid, prefix, topk):
    q, k, v, valid = inputs.vsa_full_inputs(1, 2, 128, seed=60 + prefix, grid=grid, prefix=prefix)
    scale = inputs.softmax_scale(128)
    idx, o, lse = run(gb, q, k, v, valid, prefix, topk)
    ridx = OV.vsa_select(q, k, 64, topk, valid, prefix=prefix)
    assert np.array_equal(idx, ridx)
    ro, rl = OA.vsa_sparse_attention(q, k, v, ridx, 64, scale, valid=valid, prefix=prefix)
    assert gb.device_status() == 0
    assert_close(o, ro, "o")
    assert_close(lse, rl, "lse")


def test_full_vsa_padding_contents_do_not_matter(gb):
    q, k, v, valid = inputs.vsa_full_inputs(1, 2, 128, seed=70, grid=(5, 10, 9), prefix=128)
    idx0, o0, l0 = run(gb, q, k, v, valid, 128, 5)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for c, n in enumerate(valid):
        pad = slice(128 + 64 * c + n, 128 + 64 * (c + 1))
        q2[..., pad, :] = 3.0
        k2[..., pad, :] = -7.0
        v2[..., pad, :] = 50.0          # finite (the padding weight is exactly zero)
    idx1, o1, l1 = run(gb, q2, k2, v2, valid, 128, 5)
    assert np.array_equal(idx0, idx1)
    real = np.ones(q.shape[2], bool)
    for c, n in enumerate(valid):
        real[128 + 64 * c + n:128 + 64 * (c + 1)] = False
    assert np.array_equal(o0[..., real, :], o1[..., real, :])
    assert np.all(o1[..., ~real, :] == 0) and np.all(np.isneginf(l1[..., ~real]))


def test_full_vsa_bad_counts_flagged(gb):
    q, k, v, valid = inputs.vsa_full_inputs(1, 1, 128, seed=71, grid=(4, 8, 8), prefix=0)
    bad = valid.copy()
    bad[1] = 0
    run(gb, q, k, v, bad, 0, 2)
    assert gb.device_status() & gb.DEV_BAD_INDEX


def test_full_vsa_workload_sampled_rows(gb):
    w = inputs.WORKLOADS["vsa_full"]
    q, k, v, valid = inputs.vsa_full_inputs(w["B"], w["H"], w["D"], w["seed"], w["grid"],
                                            w["cube"], w["prefix"])
    idx, o, lse = run(gb, q, k, v, valid, w["prefix"], w["topk"])
    assert gb.device_status() == 0
    ridx = OV.vsa_select(q, k, 64, w["topk"], valid, prefix=w["prefix"])
    assert np.array_equal(idx, ridx)
    S = q.shape[2]
    rows = inputs.sample_rows(w["B"] * w["H"], S, 4096, w["seed"])
    ro, rl = OA.vsa_sparse_attention(q, k, v, ridx, 64, inputs.softmax_scale(w["D"]), rows=rows,
                                     valid=valid, prefix=w["prefix"])
    fo = o.reshape(-1, S, w["D"])[rows[:, 0], rows[:, 1]]
    fl = lse.reshape(-1, S)[rows[:, 0], rows[:, 1]]
    assert_close(fo, ro, "o")
    assert_close(fl, rl, "lse")
