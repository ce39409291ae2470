"""The benchmark's multi-rank arithmetic on CPU: two gloo ranks, max-over-ranks timing,
whole-job throughput of independent replicas, and distinct per-rank inputs."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from kv_cache_vector_19_b300 import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        times = [1.0 + rank, 10.0 - rank, 3.0]
        got = bench.max_over_ranks(times, world, "cpu")
        w = workloads.preset("tiny", tokens=256, seed=0 + rank)   # the bench draws rank r with seed + r
        k0 = workloads.generate(w)["k"][0, 0, 0, :8].float()
        gathered = [torch.zeros(8) for _ in range(world)]
        dist.all_gather(gathered, k0)
        q.put((rank, got, [g.tolist() for g in gathered]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_draw_distinct_inputs():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, gathered in results:
        assert got == [2.0, 10.0, 3.0]
        assert gathered[0] != gathered[1]          # replicas work on different sequences


def test_job_throughput_counts_every_replica():
    assert bench.job_gbs(1, 2e9, 1000.0) == 2.0
    assert bench.job_gbs(4, 2e9, 1000.0) == 8.0       # weak scaling: 4 replicas, same time
    assert bench.max_over_ranks([5.0, 6.0], 1, "cpu") == [5.0, 6.0]
