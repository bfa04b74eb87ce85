"""Shared GPU-test plumbing: run the CUDA path and the oracle on one table."""
import numpy as np
import torch

import oracle
from paged_kv_cache_kvx_gb300 import kvx, workloads as W


def oracle_all(addr, B, seg_len, numa, pool):
    t = oracle.encode_runs(addr)
    p = oracle.plan(t, B, seg_len, numa, pool)
    st, local = (oracle.rebuild(t, p, B, addr.shape[1], seg_len) if p.status == 0 else (None, None))
    return t, p, st, local


def gpu_plan(addr, B, seg_len, numa, pool):
    tr = kvx.Transfer(B, seg_len, numa, pool)
    tr.set_addr(addr)
    tr.encode()
    tr.plan()
    tr.rebuild()
    torch.cuda.synchronize()
    return tr


def assert_table_equal(tr, t):
    rpl, base, stride, count = tr.read_table()
    assert np.array_equal(rpl, t.runs_per_lane)
    assert np.array_equal(base, t.run_base)
    assert np.array_equal(stride, t.run_stride)
    assert np.array_equal(count, t.run_count)


def assert_plan_equal(tr, p):
    g = tr.read_plan()
    assert tr.read_counts() == (p.groups.size, p.descs.size, p.slab_bytes)
    assert g["groups"].tobytes() == p.groups.tobytes(), "groups differ"
    assert g["descs"].tobytes() == p.descs.tobytes(), "descs differ"
    assert np.array_equal(g["lane_first"], p.lane_first)
    assert np.array_equal(g["run_block"], p.run_block)
    assert np.array_equal(g["run_group"], p.run_group)
    assert np.array_equal(g["run_off"], p.run_off)


def check_all(addr, B, seg_len, numa, pool, data=True):
    """Element-by-element parity of every output; with data=True also the
    slab and the unpacked pool bytes."""
    t, p, st, local = oracle_all(addr, B, seg_len, numa, pool)
    tr = gpu_plan(addr, B, seg_len, numa, pool)
    assert_table_equal(tr, t)
    assert p.status == 0
    assert_plan_equal(tr, p)
    assert np.array_equal(tr.read_local(), local)
    assert tr.read_status() == 0
    if data:
        seed = 99
        host_pool = W.pool_bytes_np(seed, 0, pool)
        dpool = torch.from_numpy(host_pool).cuda()
        slab = torch.zeros(max(1, tr.slab_bytes), dtype=torch.uint8, device="cuda")
        dst = torch.full((pool,), W.CANARY, dtype=torch.uint8, device="cuda")
        tr.pack(dpool, slab[: tr.slab_bytes] if tr.slab_bytes else slab[:0])
        tr.unpack(slab[: tr.slab_bytes] if tr.slab_bytes else slab[:0], dst)
        torch.cuda.synchronize()
        assert tr.read_status() == 0
        want_slab = np.zeros(p.slab_bytes, dtype=np.uint8)
        assert oracle.pack(host_pool, p.descs, want_slab) == 0
        assert np.array_equal(slab[: tr.slab_bytes].cpu().numpy(), want_slab)
        want_dst = np.full(pool, W.CANARY, dtype=np.uint8)
        assert oracle.unpack(want_slab, p.descs, want_dst) == 0
        assert np.array_equal(dst.cpu().numpy(), want_dst)
    return tr, t, p, local


def assert_equal_chunked(dev: torch.Tensor, want: np.ndarray, chunk: int = 1 << 30):
    """Every byte of a device buffer equals the host array (compared a chunk
    at a time, so the host holds one extra chunk, not a second copy)."""
    assert dev.numel() == want.size, (dev.numel(), want.size)
    for a in range(0, want.size, chunk):
        b = min(want.size, a + chunk)
        got = dev[a:b].cpu().numpy()
        if not np.array_equal(got, want[a:b]):
            k = int(np.flatnonzero(got != want[a:b])[0])
            raise AssertionError("first difference at byte %d: %d != %d" % (a + k, got[k], want[a + k]))


def host_generator_bytes(dev_pool: torch.Tensor, seed: int, probes: int = 8) -> np.ndarray:
    """The holder pool's bytes on the host, copied from the device buffer that
    workloads.fill_pool_torch filled, with a few 64 KiB windows checked
    against the numpy generator (so they are the generator's bytes, not
    anything the CUDA path wrote)."""
    host = dev_pool.cpu().numpy()
    rng = np.random.default_rng(seed)
    n = host.size
    for a in rng.integers(0, max(1, n - 65536), size=probes):
        a = int(a) & ~7
        m = min(65536, n - a)
        assert np.array_equal(host[a:a + m], W.pool_bytes_np(seed, a, m)), a
    return host
