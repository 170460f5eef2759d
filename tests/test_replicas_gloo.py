"""Multi-GPU runs of bench.py are independent replicas (the decode step has no
exchange between GPUs): the only cross-rank logic is the timing aggregate --
the slowest rank's timed region, and every rank's bytes over it.  Checked
here with two gloo ranks on the CPU."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 * (rank + 1))       # rank 1 is the slowest
        gbs = bench.replica_throughput_gbs(4_000_000_000, world, ms)
        dist.barrier()
        out[rank] = (ms, gbs)
    finally:
        dist.destroy_process_group()


def test_two_replicas_aggregate_with_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1]
    ms, gbs = out[0]
    assert ms == 20.0
    assert gbs == pytest.approx(2 * 4.0 / 0.020)  # 8 GB over the slowest 20 ms


def test_single_process_aggregate_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.replica_throughput_gbs(1_000_000_000, 1, 1.0) == pytest.approx(1000.0)
