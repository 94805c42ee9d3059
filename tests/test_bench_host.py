"""Host-side logic of bench.py: work accounting and the multi-rank aggregation
(world size 2 over gloo on the CPU; no GPU involved)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_work_accounting_matches_hand_counts():
    # prefill rotation: 2048 rows x (4096*2 in + 2048 codes + 4 scale) bytes
    assert bench.fwht_bytes(2048, 4096) == 16_777_216 + 4_202_496
    assert bench.kv_bytes(8192, 32, 128) == 134_217_728 + 35_651_584
    assert bench.gemm_ops(2048, 14336, 4096) == 2 * 2048 * 14336 * 4096
    assert bench.gemm_bytes(16, 4096, 4096) == 16 * 2048 + 4096 * 2048 + 64 + 16384 + 2 * 16 * 4096


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        units, secs = bench.aggregate(float(rank + 1) * 1e12, 0.5 + rank)
        q.put((rank, units, secs))
    finally:
        dist.destroy_process_group()


def test_aggregate_two_ranks_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for _, units, secs in res:
        assert units == pytest.approx(3e12)   # sum of the ranks' work
        assert secs == pytest.approx(1.5)     # slowest rank


def test_aggregate_single_process_is_identity():
    assert bench.aggregate(5.0, 2.0) == (5.0, 2.0)


def test_peaks_file_or_fallback():
    p = bench.load_peaks()
    assert p["hbm_gbs"] > 1000 and p["bf16_tflops"] > 100
    assert p["source"] in ("measured", "fallback")
