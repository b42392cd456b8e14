"""The item counter of vsa_sparse_fwd (persistent CTAs; items handed out by a
counter in a caller workspace, or split statically without one).

* a zeroed workspace: the output matches the oracle and the counter is zero
  again after the call (and after a call that the fault hook aborts);
* no workspace (static split) and the workspace give bit-identical outputs,
  with and without the full VSA layout (prefix tiles and boundary cubes);
* a counter that did not start at zero is flagged (DEV_BAD_INDEX) instead of
  being used as an item number;
* the workspace argument is checked (size, alignment) before anything runs.
"""

import numpy as np
import pytest
import torch

from attention_fp16_flashattention_gb300 import inputs
from oracle import attention as OA
from oracle import vsa as OV

pytestmark = pytest.mark.gpu


def t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def close(got, ref):
    got = np.asarray(got, dtype=np.float64)
    return bool(np.all(np.abs(got - ref) <= 2e-3 + 1e-2 * np.abs(ref)))


def counter(gb):
    return torch.zeros(int(gb.load().vsa_sparse_workspace_size()), dtype=torch.uint8, device="cuda")


def test_counter_output_and_reset(gb):
    q, k, v = inputs.vsa_inputs(1, 3, 128, seed=91, grid=(4, 16, 32))
    tq, tk, tv = t(q), t(k), t(v)
    idx = gb.vsa_select_blocks(tq, tk, topk=12)
    pairs = gb.vsa_pair_query_cubes(idx)
    ws = counter(gb)
    for _ in range(3):                         # the counter is reused call after call
        o = gb.vsa_sparse_fwd(tq, tk, tv, idx, pairs=pairs, workspace=ws)
        torch.cuda.synchronize()
        assert int(ws.sum()) == 0
    assert gb.device_status() == 0
    ro, _ = OA.vsa_sparse_attention(q, k, v, OV.vsa_select(q, k, 64, 12), 64, inputs.softmax_scale(128))
    assert close(o.float().cpu().numpy(), ro)
    o_static = gb.vsa_sparse_fwd(tq, tk, tv, idx, pairs=pairs, workspace=False)
    assert torch.equal(o, o_static)


def test_counter_full_layout_matches_static_split(gb):
    q, k, v, valid = inputs.vsa_full_inputs(1, 2, 128, seed=92, grid=(3, 9, 10), prefix=256)
    tq, tk, tv, tval = t(q), t(k), t(v), t(valid)
    idx = gb.vsa_select_blocks(tq, tk, 6, prefix=256, cube_valid=tval)
    ws = counter(gb)
    a = gb.vsa_sparse_fwd(tq, tk, tv, idx, prefix=256, cube_valid=tval, workspace=ws)
    b = gb.vsa_sparse_fwd(tq, tk, tv, idx, prefix=256, cube_valid=tval, workspace=False)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and int(ws.sum()) == 0
    assert gb.device_status() == 0


def test_counter_reset_after_an_aborted_call(gb):
    q, k, v = inputs.vsa_inputs(1, 2, 128, seed=93, grid=(4, 16, 16))
    tq, tk, tv = t(q), t(k), t(v)
    idx = gb.vsa_select_blocks(tq, tk, topk=8)
    ws = counter(gb)
    assert gb.device_status() == 0
    gb.set_wait_limit_ns(50_000_000)
    gb.test_inject_fault(1)                    # the query tiles never load: every CTA times out
    try:
        gb.vsa_sparse_fwd(tq, tk, tv, idx, workspace=ws)
        flags = gb.device_status()
    finally:
        gb.test_inject_fault(0)
        gb.set_wait_limit_ns(1_000_000_000)
    assert flags & gb.DEV_WAIT_TIMEOUT
    assert int(ws.sum()) == 0                  # the aborted CTAs drew on to their last draw
    o = gb.vsa_sparse_fwd(tq, tk, tv, idx, workspace=ws)
    assert torch.equal(o, gb.vsa_sparse_fwd(tq, tk, tv, idx, workspace=False))
    assert gb.device_status() == 0


def test_counter_not_at_zero_is_flagged(gb):
    q, k, v = inputs.vsa_inputs(1, 2, 128, seed=94, grid=(4, 16, 16))
    tq, tk, tv = t(q), t(k), t(v)
    idx = gb.vsa_select_blocks(tq, tk, topk=8)
    ws = counter(gb)
    ws.view(torch.int32)[0] = 1 << 30          # far past any item number of this launch
    assert gb.device_status() == 0
    gb.vsa_sparse_fwd(tq, tk, tv, idx, workspace=ws)
    assert gb.device_status() & gb.DEV_BAD_INDEX
    ws.zero_()
    o = gb.vsa_sparse_fwd(tq, tk, tv, idx, workspace=ws)
    assert torch.equal(o, gb.vsa_sparse_fwd(tq, tk, tv, idx, workspace=False))
    assert gb.device_status() == 0


def test_counter_argument_checks(gb):
    q, k, v = inputs.vsa_inputs(1, 1, 128, seed=95, grid=(4, 16, 16))
    tq, tk, tv = t(q), t(k), t(v)
    idx = gb.vsa_select_blocks(tq, tk, topk=4)
    small = torch.zeros(8, dtype=torch.uint8, device="cuda")
    before = gb.launch_count()
    with pytest.raises(gb.GbattnError) as e:
        gb.vsa_sparse_fwd(tq, tk, tv, idx, workspace=small)
    assert e.value.status == 6                 # GBATTN_ERR_WORKSPACE
    odd = torch.zeros(64, dtype=torch.uint8, device="cuda")[4:20]
    with pytest.raises(gb.GbattnError) as e:
        gb.vsa_sparse_fwd(tq, tk, tv, idx, workspace=odd)
    assert e.value.status == 4                 # GBATTN_ERR_ALIGN
    assert gb.launch_count() == before
