"""Host logic of bench.py (CPU only): the work model and the max-over-ranks timing.

The useful-FLOP counts are checked against the closed forms of the workloads
(4 * D per visible query/key pair), and the cross-rank reduction that turns
per-rank times into the reported time is run on two gloo ranks.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def test_work_model_closed_forms():
    assert bench.dense_flops(1, 24, 32768, 32768, 128) == 13_194_139_533_312
    assert bench.causal_pairs(8192, 131072) == 8192 * 122880 + 8192 * 8193 // 2
    assert bench.causal_flops(1, 6, 8192, 131072, 256) == 6_390_936_502_272
    assert bench.causal_flops(1, 6, 1024, 4096, 256) == 22_551_724_032
    assert bench.vsa_flops(1, 24, 32768, 128, 64) == 1_649_267_441_664
    assert bench.bridge_bytes(131072, 1, 256, 32) == 201_342_976


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(10.0 + rank * 5.0, world)
    bench.barrier(world)
    q.put((rank, t))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert out == {0: 15.0, 1: 15.0}
