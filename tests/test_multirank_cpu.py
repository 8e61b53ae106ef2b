"""The multi-GPU path is replicas (sequences are independent: no collective on
the data path). Its host side runs here as two gloo ranks on the CPU: the job
time is the slowest rank's, throughput counts every rank's work, and each rank
draws its own seeded inputs."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [10.0, 25.0][rank]                      # rank 1 is the slow one
        tmax = bench.reduce_over_ranks(ms, "max", world, "cpu")
        tps = bench.reduce_over_ranks(100.0 * (rank + 1), "sum", world, "cpu")
        wl = bench.AttnWorkload("attn-batched", rank, host_only=True)
        out[rank] = (tmax, tps, bench.job_gbs(1_000_000, world, tmax),
                     [int(x) for x in wl.lengths[:8]])
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replica_aggregation():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        tmax, tps, gbs, _ = res[r]
        assert tmax == 25.0                          # every rank sees the slowest time
        assert tps == 300.0                          # throughput sums over ranks
        assert abs(gbs - 2 * 1_000_000 / 25e-3 / 1e9) < 1e-12
    assert res[0][3] != res[1][3]                    # each replica has its own inputs


def test_single_rank_is_identity():
    assert bench.reduce_over_ranks(3.5, "max", 1, "cpu") == 3.5
    assert np.isclose(bench.job_gbs(2_000_000_000, 1, 1000.0), 2.0)
