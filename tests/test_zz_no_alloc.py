"""vsa_select_blocks_noalloc: the selection for callers that cannot allocate.

Some callers cannot allocate device memory at the point where they select
key cubes (a plugin whose host program fixed its memory at start-up, or code
whose device memory belongs to a pool it cannot reach).  The no-allocation
entry point takes only inputs and outputs and keeps its scratch in a fixed
array inside the library.  These tests call it through the C ABI:

* twice in a row on two different inputs, each result against the ordinary
  entry point and against the CPU oracle (selection indices compared exactly,
  the tolerance used for selection everywhere in these tests);
* with prefix tokens and padded boundary cubes;
* at the largest size the fixed scratch holds (B*H*S = 1,048,576 tokens x
  heads), and one cube row past it, which must be rejected before anything
  runs.

The file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

from attention_fp16_flashattention_gb300 import inputs
from oracle import vsa as OV

pytestmark = pytest.mark.gpu

WORKSPACE_ERR = 6


def _noalloc(lib):
    fn = lib.vsa_select_blocks_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 7 + \
        [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return fn


def _call(fn, tq, tk, topk, prefix=0, valid=None):
    B, H, S, D = tq.shape
    idx = torch.full((B, H, (S - prefix) // 64, topk), -1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    vp = None if valid is None else ctypes.c_void_p(valid.data_ptr())
    rc = fn(ctypes.c_void_p(tq.data_ptr()), ctypes.c_void_p(tk.data_ptr()), B, H, S, D, 64,
            topk, prefix, vp, ctypes.c_void_p(idx.data_ptr()), stream)
    return rc, idx


def test_noalloc_select_matches_workspace_entry_point_and_oracle_twice(gb):
    fn = _noalloc(gb.load())
    topk = 16
    for seed in (41, 42):                       # two calls in a row, different inputs
        q, k, _ = inputs.vsa_inputs(1, 4, 128, seed=seed, grid=(8, 32, 32))
        tq = torch.from_numpy(q).cuda()
        tk = torch.from_numpy(k).cuda()
        ref = gb.vsa_select_blocks(tq, tk, topk=topk)
        rc, idx = _call(fn, tq, tk, topk)
        assert rc == 0, gb.status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref)
        assert np.array_equal(idx.cpu().numpy(), OV.vsa_select(q, k, 64, topk))
    assert gb.device_status() == 0


def test_noalloc_prefix_and_boundary_cubes(gb):
    fn = _noalloc(gb.load())
    q, k, _, valid = inputs.vsa_full_inputs(1, 2, 128, seed=43, grid=(5, 10, 9), prefix=128)
    tq, tk, tval = (torch.from_numpy(x).cuda() for x in (q, k, valid))
    rc, idx = _call(fn, tq, tk, 5, prefix=128, valid=tval)
    assert rc == 0, gb.status_string(rc)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), OV.vsa_select(q, k, 64, 5, valid, prefix=128))
    assert gb.device_status() == 0


def test_noalloc_at_the_scratch_limit_and_one_row_past_it(gb):
    fn = _noalloc(gb.load())
    # B=1, H=32, S=32768: 16,384 query cubes, exactly the fixed scratch
    B, H, S, D = 1, 32, 32768, 128
    assert gb.load().vsa_select_workspace_size(B, H, S, D, 64) == \
        (48 << 20) + (192 << 10)
    q, k, _ = inputs.dense_inputs(B, H, S, D, seed=44)
    tq, tk = torch.from_numpy(q).cuda(), torch.from_numpy(k).cuda()
    rc, idx = _call(fn, tq, tk, 64)
    assert rc == 0, gb.status_string(rc)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), OV.vsa_select(q, k, 64, 64))
    del tq, tk
    # one more cube per head (S = 32832) needs 32 more rows and a wider score
    # row: rejected, nothing launched
    big = torch.empty(16, dtype=torch.float16, device="cuda")
    before = gb.launch_count()
    rc = fn(ctypes.c_void_p(big.data_ptr()), ctypes.c_void_p(big.data_ptr()), 1, 32, 32832, 128,
            64, 64, 0, None, ctypes.c_void_p(big.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == WORKSPACE_ERR
    assert gb.launch_count() == before
    assert gb.device_status() == 0
