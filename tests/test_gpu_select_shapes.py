"""The selection's workspace contract and its small and ragged shapes.

* The workspace may hold anything before a call: a workspace filled with 0xFF
  bytes gives the oracle's selection, twice in a row.
* One or two cubes per head over several heads, a ragged second 128-cube score
  tile (NC = 160), and boundary cubes with a prefix over two batches.
"""

import numpy as np
import pytest
import torch

from attention_fp16_flashattention_gb300 import inputs
from oracle import vsa as OV

pytestmark = pytest.mark.gpu


def t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def test_garbage_workspace_gives_the_oracle_selection(gb):
    q, k, _ = inputs.vsa_inputs(1, 3, 128, seed=101, grid=(4, 32, 32))
    B, H, S, D = q.shape
    ws = torch.full((gb.vsa_select_workspace_size(B, H, S, D, 64),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    ref = OV.vsa_select(q, k, 64, 12)
    for _ in range(2):
        idx = gb.vsa_select_blocks(t(q), t(k), topk=12, workspace=ws)
        assert np.array_equal(idx.cpu().numpy(), ref)
    assert gb.device_status() == 0


@pytest.mark.parametrize("grid,H,topk", [((4, 4, 4), 5, 1),      # one cube per head
                                         ((4, 4, 8), 3, 1),      # two cubes per head
                                         ((4, 4, 8), 3, 2),
                                         ((8, 32, 40), 2, 24)])  # NC = 160: a ragged second tile
def test_small_and_ragged_cube_counts(gb, grid, H, topk):
    q, k, _ = inputs.vsa_inputs(1, H, 128, seed=102 + grid[2], grid=grid)
    idx = gb.vsa_select_blocks(t(q), t(k), topk=topk)
    assert np.array_equal(idx.cpu().numpy(), OV.vsa_select(q, k, 64, topk))
    assert gb.device_status() == 0


def test_boundary_cubes_with_prefix_and_two_batches(gb):
    q, k, _, valid = inputs.vsa_full_inputs(2, 2, 128, seed=107, grid=(5, 10, 9), prefix=128)
    idx = gb.vsa_select_blocks(t(q), t(k), 7, prefix=128, cube_valid=t(valid))
    assert np.array_equal(idx.cpu().numpy(), OV.vsa_select(q, k, 64, 7, valid, prefix=128))
    assert gb.device_status() == 0
