"""vsa_select_blocks_noalloc: the selection for callers that cannot allocate.

Some callers cannot allocate device memory at the point where they select
key cubes (a plugin whose host program fixed its memory at start-up, or code
whose device memory belongs to a pool it cannot reach).  The no-allocation
entry point takes only inputs and outputs and keeps its scratch in a fixed
array inside the library.  This test calls it through the C ABI twice in a
row, on two different inputs, and checks each result against the ordinary
entry point (selection indices are compared exactly, the tolerance used for
selection everywhere in these tests), then checks that oversized calls are
rejected before anything runs.  The file is named so that pytest collects it
last.
"""

import ctypes

import numpy as np
import pytest
import torch

from attention_fp16_flashattention_gb300 import inputs

pytestmark = pytest.mark.gpu

WORKSPACE_ERR = 6


def _noalloc(lib):
    fn = lib.vsa_select_blocks_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 7 + \
        [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return fn


def test_noalloc_select_matches_workspace_entry_point_twice(gb):
    fn = _noalloc(gb.load())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    topk = 16
    for seed in (41, 42):                       # two calls in a row, different inputs
        q, k, _ = inputs.vsa_inputs(1, 4, 128, seed=seed, grid=(8, 32, 32))
        tq = torch.from_numpy(q).cuda()
        tk = torch.from_numpy(k).cuda()
        B, H, S, D = tq.shape
        ref = gb.vsa_select_blocks(tq, tk, topk=topk)
        idx = torch.full((B, H, S // 64, topk), -1, dtype=torch.int32, device="cuda")
        rc = fn(ctypes.c_void_p(tq.data_ptr()), ctypes.c_void_p(tk.data_ptr()), B, H, S, D, 64,
                topk, 0, None, ctypes.c_void_p(idx.data_ptr()), stream)
        assert rc == 0, gb.status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref)
    assert gb.device_status() == 0


def test_noalloc_rejects_sizes_beyond_fixed_scratch(gb):
    fn = _noalloc(gb.load())
    q = torch.empty(16, dtype=torch.float16, device="cuda")
    idx = torch.empty(16, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    before = gb.launch_count()
    # 1 x 24 heads x 32768 tokens needs 12.6 MB of scratch (fits); 48 heads need 25 MB.
    rc = fn(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()), 1, 48, 32768, 128, 64,
            64, 0, None, ctypes.c_void_p(idx.data_ptr()), stream)
    assert rc == WORKSPACE_ERR
    assert gb.launch_count() == before
