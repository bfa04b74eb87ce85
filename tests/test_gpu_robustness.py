"""Bounded waits, graph capture of the whole path, and byte-exact slabs at
full size where the plan maps remote offsets 1:1 onto slab offsets."""
import time

import numpy as np
import pytest
import torch

from paged_kv_cache_kvx_gb300 import kvx, workloads as W

pytestmark = pytest.mark.gpu


def test_bounded_waits_report_a_timeout():
    """A grid barrier, an mbarrier and the planner's cross-block flag wait that
    nothing will release each give up within seconds and say so in their own
    status word; the context stays usable afterwards."""
    status = torch.zeros(3, dtype=torch.int32, device="cuda")
    t0 = time.time()
    kvx.kvx_selftest_timeouts(status)
    torch.cuda.synchronize()
    assert time.time() - t0 < 30
    assert status.cpu().tolist() == [kvx.S_TIMEOUT] * 3
    x = torch.arange(10, device="cuda")
    assert int(x.sum().item()) == 45


def test_captured_step_replays_bit_exact():
    """One step captured as a CUDA graph (counts stay on the device) replays
    to the same plan and the same bytes as the step launched call by call;
    rebuild on a side stream joins before the step ends."""
    wl = W.worst(blocks=61, slots=18, npos=128, seed=3)
    tr = kvx.Transfer(wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    tr.set_addr(wl.addr)
    pool = torch.empty(wl.pool_bytes, dtype=torch.uint8, device="cuda")
    W.fill_pool_torch(pool, wl.seed)
    slab = torch.empty(tr.slab_bytes, dtype=torch.uint8, device="cuda")
    dst = torch.full((wl.pool_bytes,), W.CANARY, dtype=torch.uint8, device="cuda")
    tr.step(pool, slab, dst)
    torch.cuda.synchronize()
    assert tr.read_status() == 0
    want_plan = tr.read_plan()
    want_local = tr.read_local()
    want_slab = slab.clone()
    want_dst = dst.clone()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    slab.zero_()
    dst.fill_(W.CANARY)
    tr.local.zero_()
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        tr.step(pool, slab, dst, side=side)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert tr.read_status() == 0
    got = tr.read_plan()
    for k in ("groups", "descs"):
        assert got[k].tobytes() == want_plan[k].tobytes()
    assert np.array_equal(tr.read_local(), want_local)
    assert torch.equal(slab, want_slab) and torch.equal(dst, want_dst)


@pytest.mark.parametrize("name", ["default", "wide64k"])
def test_identity_plans_copy_every_byte(name):
    """Bump-allocated holders: every dense group's slab offset equals its
    remote base, so the whole slab must equal the pool byte for byte."""
    wl = W.CONFIGS[name]()
    tr = kvx.Transfer(wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    tr.set_addr(wl.addr)
    pool = torch.empty(wl.pool_bytes, dtype=torch.uint8, device="cuda")
    W.fill_pool_torch(pool, wl.seed)
    slab = torch.zeros(tr.slab_bytes, dtype=torch.uint8, device="cuda")
    tr.encode()
    tr.plan()
    tr.pack(pool, slab)
    torch.cuda.synchronize()
    plan = tr.read_plan()
    assert tr.read_status() == 0
    assert np.array_equal(plan["groups"]["local"], plan["groups"]["base"])
    assert tr.slab_bytes == wl.pool_bytes
    assert torch.equal(slab, pool)


def test_overlapped_transfers_bit_exact():
    """Independent passes over two metadata sets, each pass's encode and plan
    overlapping the previous pass's copies (stream launches, then the same
    passes captured once as a graph and replayed): every output equals the
    oracle's."""
    import oracle
    from paged_kv_cache_kvx_gb300 import kvx, workloads as W
    wl = {v.name: v for v in W.small_variants()}["worst"]
    trs = [kvx.Transfer(wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes) for _ in range(2)]
    for tr in trs:
        tr.set_addr(wl.addr)
    host_pool = W.holder_pool_np(wl)
    pool = torch.from_numpy(host_pool).cuda()
    slab = torch.zeros(trs[0].slab_bytes, dtype=torch.uint8, device="cuda")
    dst = torch.full((wl.pool_bytes,), W.CANARY, dtype=torch.uint8, device="cuda")
    main, ctl, side = (torch.cuda.Stream() for _ in range(3))
    t = oracle.encode_runs(wl.addr)
    p = oracle.plan(t, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    st, local = oracle.rebuild(t, p, wl.blocks, wl.lanes, wl.seg_len)
    want_slab = np.zeros(p.slab_bytes, np.uint8)
    assert oracle.pack(host_pool, p.descs, want_slab) == 0
    want_dst = np.full(wl.pool_bytes, W.CANARY, np.uint8)
    assert oracle.unpack(want_slab, p.descs, want_dst) == 0

    def check():
        for tr in trs:
            assert tr.read_status() == 0
            g = tr.read_plan()
            assert g["descs"].tobytes() == p.descs.tobytes()
            assert np.array_equal(tr.read_local(), local)
        assert np.array_equal(slab.cpu().numpy(), want_slab)
        assert np.array_equal(dst.cpu().numpy(), want_dst)

    kvx.overlapped_steps(trs, pool, slab, dst, 5, main, ctl, side)
    torch.cuda.synchronize()
    check()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=main):
        kvx.overlapped_steps(trs, pool, slab, dst, 4, main, ctl, side)
    slab.zero_()
    dst.fill_(W.CANARY)
    for tr in trs:
        tr.status.zero_()
        tr.local.fill_(0)
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    check()
