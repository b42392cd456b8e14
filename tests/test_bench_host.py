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
    # decode: 417,843 cached tokens of K and V bytes, 13,060 page-table entries, Q and O in FP16
    lens = (131072, 122887, 98313, 65571)
    assert bench.decode_bytes(lens, 4, 6, 1, 1, 256, 32) == \
        2 * 417_843 * 256 + 4 * 13_060 + 2 * 2 * 24 * 256 == 214_012_432


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


def test_clock_samples_are_cut_to_the_timed_window():
    """Only samples stamped inside the timed window count; idle samples (low power) drop."""
    import datetime

    rows = [  # timestamp, index, sm, max, power, active, hw, hwt, swt, swp
        "2026/12/02 10:00:00.000, 0, 900, 2070, 150.0, Idle, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:00.050, 0, 1950, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:00:00.100, 0, 1960, 2070, 1310.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:00:00.150, 0, 2010, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:00.200, 0, 1100, 2070, 900.0, 0x8, Active, Not Active, Not Active, Not Active",
    ]
    t0 = datetime.datetime(2026, 12, 2, 10, 0, 0, 40000)
    t1 = datetime.datetime(2026, 12, 2, 10, 0, 0, 160000)
    assert bench.summarize_clocks(rows, (t0, t1)) == {
        "sm_mhz": 1960.0, "sm_max_mhz": 2070.0, "samples": 3, "reasons": ["sw_power_cap"]}
    # the hardware slowdown outside the window is not reported; inside it is
    wide = bench.summarize_clocks(rows, (t0, datetime.datetime(2026, 12, 2, 10, 0, 1)))
    assert "hw_slowdown" in wide["reasons"] and wide["samples"] == 4
    # a window that holds no sample falls back to every sample; an unknown stamp is kept
    late = datetime.datetime(2026, 12, 2, 11, 0, 0)
    assert bench.summarize_clocks(rows, (late, late))["samples"] == 4
    odd = ["12:00:00, 0, 1500, 2070, 800.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    assert bench.summarize_clocks(odd, (t0, t1))["sm_mhz"] == 1500.0
