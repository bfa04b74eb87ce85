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


def test_stage_roofline_bytes_and_fractions():
    """The per-stage roofline of the bench line: algorithmic bytes from the
    table's counts, the rate over the stage time, its fraction of the peak."""
    S, R, G, D, L, N = 576000, 576, 2, 72, 576, 576000 * 4096
    ms = [0.020, 0.020, 0.010, 0.700, 0.700]
    r = bench.stage_roofline(ms, S, R, G, D, L, N, 7000.0)
    assert r["encode"]["algorithmic_bytes"] == 8 * S + 20 * R + 4 * L
    assert r["rebuild"]["algorithmic_bytes"] == 8 * S + 24 * R + 48 * G + 4 * (L + 1)
    assert r["pack"]["algorithmic_bytes"] == r["unpack"]["algorithmic_bytes"] == 2 * N
    assert r["pack"]["gbs"] == pytest.approx(2 * N / 0.7e-3 / 1e9)
    assert r["pack"]["frac"] == pytest.approx(r["pack"]["gbs"] / 7000.0)
    assert r["pack"]["bound"] == "hbm" and r["plan"]["bound"] == "latency"


def test_per_workload_figures_reproduce_from_stage_times():
    """path_figures: the value is the fastest launch mode's 4 N per step, and
    pack / unpack rates and their roofline fraction come from the stages'
    mean times (what a reader recomputes from the line)."""
    import numpy as np
    from paged_kv_cache_kvx_gb300 import workloads as W
    wl = W.tiny()
    N, K = wl.payload_bytes, 4
    stage = np.array([[0.01, 0.02, 0.005, 0.5, 0.4]] * K)
    m = dict(total_ms=4.0, stage=stage, launches=40, graph_ms=3.0, graph_launches=40, over_ms=3.5,
             over_launches=44, nruns=8, ngroups=2, ndescs=2)
    f = bench.path_figures(wl, m, K, 1, 7000.0, "measured")
    assert f["launch_mode"] == "cuda_graph" and f["gpu_launches"] == 40
    assert f["value"] == pytest.approx(4 * N * K / 3.0e-3 / 1e9)
    assert f["ms_per_step"] == pytest.approx(0.75)
    assert f["pack_gbs"] == pytest.approx(2 * N / 0.5e-3 / 1e9)
    assert f["unpack_gbs"] == pytest.approx(2 * N / 0.4e-3 / 1e9)
    assert f["roofline"]["kernel"] == "kvx_pack"
    assert f["roofline"]["frac"] == pytest.approx(f["pack_gbs"] / 7000.0)
    assert f["frac_of_measured_peak"] == pytest.approx(4 * N / 0.9e-3 / 1e9 / 7000.0)
    assert f["encode_msegs_per_s"] == pytest.approx(wl.segments / 0.01e-3 / 1e6)
    assert f["rebuild_msegs_per_s"] == pytest.approx(wl.segments / 0.005e-3 / 1e6)
    assert f["pack_payload_gbs"] == pytest.approx(f["pack_gbs"] / 2)
    assert f["unpack_payload_gbs"] == pytest.approx(N / 0.4e-3 / 1e9)
    assert f["stage_ms_mean"]["rebuild"] == pytest.approx(0.005)
