"""GPU parity of dense attention with an additive mask against the CPU oracle.

|o - ref| <= 2e-3 + 1e-2 |ref| and the same for lse, element by element, on
all rows for small shapes (ragged query and key tails, fully hidden rows,
shared, per-head and per-batch masks) and on 4096 seeded rows of the
B1 H24 S8192 workload the benchmark times.
"""

import numpy as np
import pytest
import torch

from attention_fp16_flashattention_gb300 import inputs
from oracle import attention as OA

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


def random_mask(shape, seed, hide=0.15, scale=2.0):
    rng = np.random.default_rng(seed)
    m = (rng.standard_normal(shape) * scale).astype(np.float16)
    m[rng.random(shape) < hide] = -np.inf
    return m


def run(gb, q, k, v, mask, scale):
    B, H, Sq, _ = q.shape
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
    o = gb.attn_dense_mask_fwd(t(q), t(k), t(v), t(mask), lse=lse, scale=scale)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("B,H,Sq,Skv,mshape", [
    (1, 2, 256, 256, "shared"),
    (1, 2, 128, 512, "shared"),
    (2, 3, 300, 904, "per_head"),
    (2, 2, 130, 136, "per_batch_head"),
    (1, 1, 64, 8, "shared"),
    (1, 2, 1000, 1000, "shared"),
    (1, 2, 200, 384, "shared"),           # 3 key tiles: all S buffers used once
    (2, 1, 128, 640, "per_batch_head"),   # 5 key tiles: the 3-slot ring wraps
    (1, 2, 256, 2056, "shared")])         # 17 key tiles with a ragged last one
def test_masked_parity(gb, B, H, Sq, Skv, mshape):
    q, k, v = inputs.dense_inputs(B, H, Sq, 128, seed=80 + Sq, skv=Skv)
    shape = {"shared": (Sq, Skv), "per_head": (1, H, Sq, Skv),
             "per_batch_head": (B, H, Sq, Skv)}[mshape]
    mask = random_mask(shape, 81 + Skv)
    if mshape == "shared":
        mask[Sq // 3] = -np.inf                    # a fully hidden query row
    scale = inputs.softmax_scale(128)
    o, lse = run(gb, q, k, v, mask, scale)
    ro, rl = OA.dense_masked_attention(q, k, v, mask, scale)
    assert gb.device_status() == 0
    assert_close(o, ro, "o")
    assert_close(lse, rl, "lse")


def test_zero_mask_matches_dense(gb):
    q, k, v = inputs.dense_inputs(1, 2, 384, 128, seed=90, skv=640)
    zero = np.zeros((384, 640), np.float16)
    om, lm = run(gb, q, k, v, zero, inputs.softmax_scale(128))
    lse = torch.empty((1, 2, 384), dtype=torch.float32, device="cuda")
    od = gb.attn_dense_fwd(t(q), t(k), t(v), lse=lse).float().cpu().numpy()
    torch.cuda.synchronize()
    assert np.abs(om - od).max() < 2e-3
    assert np.abs(lm - lse.cpu().numpy()).max() < 1e-4


def test_masked_rejects_unaligned_rows(gb):
    q, k, v = inputs.dense_inputs(1, 1, 64, 128, seed=91, skv=100)
    with pytest.raises(gb.GbattnError):
        run(gb, q, k, v, np.zeros((64, 100), np.float16), 0.1)


def test_masked_full_workload_sampled_rows(gb):
    """The benchmark's launch (B1 H24 S8192, shared ALiBi-style mask), 4096 rows."""
    w = inputs.WORKLOADS["dense_masked"]
    q, k, v = inputs.dense_inputs(w["B"], w["H"], w["S"], w["D"], w["seed"])
    mask = inputs.additive_mask(w["S"], w["S"], w["seed"])
    scale = inputs.softmax_scale(w["D"])
    o, lse = run(gb, q, k, v, mask, scale)
    assert gb.device_status() == 0
    rows = inputs.sample_rows(w["B"] * w["H"], w["S"], 4096, w["seed"])
    ro, rl = OA.dense_masked_attention(q, k, v, mask, scale, rows=rows)
    flat_o = o.reshape(-1, w["S"], w["D"])
    flat_l = lse.reshape(-1, w["S"])
    assert_close(flat_o[rows[:, 0], rows[:, 1]], ro, "o")
    assert_close(flat_l[rows[:, 0], rows[:, 1]], rl, "lse")
