"""Multi-process path of the benchmark on CPU: two gloo ranks stand in for
two GPUs running independent replicas (the block does not shard, so the only
cross-rank steps are the barrier and the max-over-ranks timing)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_info()
        dist.barrier()
        # each replica times its own steps; the job is as slow as the slowest
        ms = bench.max_over_ranks(100.0 + 25.0 * rank, dist)
        value = bench.replica_value(ws, 4096, 5, ms)
        # the reference arm runs on rank 0 only; other ranks leave at once
        ref = bench.run_reference(bench.parse_args(["--impl", "reference"]), ws, r) if r else None
        q.put((r, ws, local, ms, value, ref))
    finally:
        dist.destroy_process_group()


def test_two_replicas_max_time_and_aggregate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, ws, local, ms, value, ref) in enumerate(res):
        assert (rank, ws, local) == (r, 2, r)
        assert ms == pytest.approx(125.0)                  # the slower rank's time
        assert value == pytest.approx(2 * 4096 * 5 / 0.125)  # tokens of both replicas
        assert ref is None


def test_single_process_value():
    assert bench.max_over_ranks(7.0, None) == 7.0
    assert bench.replica_value(1, 4096, 5, 100.0) == pytest.approx(204800.0)
