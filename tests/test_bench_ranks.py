"""The multi-rank bench path without a GPU: two gloo ranks on the CPU take
the slowest rank's time, and the whole-job value counts every rank's bytes."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 * (rank + 1))
        out.put((rank, got, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [20.0, 20.0]
    assert [r[2] for r in res] == [(0, 2, 0), (1, 2, 1)]


def test_single_process_is_identity_and_value_scales_with_ranks():
    assert bench.max_over_ranks(3.5) == 3.5
    one = bench.step_value(2_359_296_000, 10, 1, 15.0)
    assert one == pytest.approx(4 * 2_359_296_000 * 10 / 0.015 / 1e9)
    assert bench.step_value(2_359_296_000, 10, 4, 15.0) == pytest.approx(4 * one)
