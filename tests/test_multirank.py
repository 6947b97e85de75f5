"""Host side of the multi-GPU path, as gloo ranks on the CPU (world size 2).

Rows are independent, so ranks split them with no exchange; the benchmark
only needs the barrier and the max of the per-rank step time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

from reduce_residual_rmsnorm_gb300.workloads import row_split


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        start, count = row_split(4099, world, rank)
        local_ms = 1.0 + rank * 0.25  # a slower rank 1
        bench.barrier(world)
        worst = bench.max_over_ranks(local_ms, world)
        # --gpus must match the torchrun world
        ok = bench.check_world(world) == "run"
        try:
            bench.check_world(world + 1)
            ok = False
        except SystemExit:
            pass
        q.put((rank, start, count, worst, ok))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_rows_and_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    (r0, s0, c0, w0, ok0), (r1, s1, c1, w1, ok1) = res
    assert (s0, c0) == (0, 2050) and (s1, c1) == (2050, 2049)
    assert w0 == w1 == 1.25
    assert ok0 and ok1


@pytest.mark.parametrize("T,W", [(0, 3), (1, 4), (4096, 8), (32768, 3), (7, 7), (5, 2)])
def test_row_split_partitions_all_rows(T, W):
    spans = [row_split(T, W, r) for r in range(W)]
    pos = 0
    for start, count in spans:
        assert start == pos and count >= 0
        pos += count
    assert pos == T
    assert max(c for _, c in spans) - min(c for _, c in spans) <= 1
