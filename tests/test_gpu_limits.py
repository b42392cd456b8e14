"""GPU parity at the implementation limits of the hot path.

* VSA with 1024 key cubes per head (the most the selection's 32-key chunks and
  the pairing's bitsets take) and top-k = 512 (the most a list may hold): the
  union of a query-cube pair's two lists runs to about 780 cubes (390 of the
  512 tiles a list may hold).  Selection bit-exact against the oracle, pairing
  a perfect matching, sparse attention on 256 seeded rows within |o - ref| <=
  2e-3 + 1e-2 |ref|.
* Paged decode with 4096 sequences (the most one launch takes), ragged short
  caches, within the same tolerance on every row.
"""

import numpy as np
import pytest
import torch

from attention_fp16_flashattention_gb300 import inputs
from oracle import attention as OA
from oracle import decode as OD
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


def test_vsa_at_the_cube_and_topk_limits(gb):
    grid = (16, 64, 64)                                   # 4 x 16 x 16 = 1024 cubes
    q, k, v = inputs.vsa_inputs(1, 1, 128, seed=71, grid=grid)
    tq, tk, tv = t(q), t(k), t(v)
    idx = gb.vsa_select_blocks(tq, tk, 512)
    pairs = gb.vsa_pair_query_cubes(idx)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    o = gb.vsa_sparse_fwd(tq, tk, tv, idx, pairs=pairs, lse=lse)
    torch.cuda.synchronize()
    assert gb.device_status() == 0
    ridx = OV.vsa_select(q, k, 64, 512)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    p = pairs.cpu().numpy().reshape(-1, 2)
    seen = p.reshape(-1)
    assert np.array_equal(np.sort(seen[seen >= 0]), np.arange(1024))
    rows = inputs.sample_rows(1, q.shape[2], 256, seed=7071)
    ro, rl = OA.vsa_sparse_attention(q, k, v, ridx, 64, inputs.softmax_scale(128), rows=rows)
    got = o.float().cpu().numpy().reshape(-1, q.shape[2], 128)[rows[:, 0], rows[:, 1]]
    assert_close(got, ro, "o")
    assert_close(lse.cpu().numpy().reshape(-1, q.shape[2])[rows[:, 0], rows[:, 1]], rl, "lse")


def test_decode_at_the_sequence_limit(gb):
    B = 4096
    lens = np.random.default_rng(72).integers(1, 41, size=B)
    q, kp, vp, table, lens = inputs.paged_decode_inputs(B, 6, 1, 1, lens, 128, 72, page_size=16,
                                                        codes="moderate")
    scale = inputs.softmax_scale(128)
    lse = torch.empty((B, 6, 1), dtype=torch.float32, device="cuda")
    o = gb.attn_paged_decode_fwd(t(q), t(kp), t(vp), t(table), t(lens), 0.0625, 0.125,
                                 lse=lse, scale=scale)
    torch.cuda.synchronize()
    assert gb.device_status() == 0
    ro, rl = OD.paged_decode_attention(q, kp, vp, table, lens, 0.0625, 0.125, scale)
    assert_close(o.float().cpu().numpy(), ro, "o")
    assert_close(lse.cpu().numpy(), rl, "lse")
