"""CUDA path vs the CPU oracle, element by element (bit-exact: every output
is integer or byte data).

Small inputs: every output array and every slab / pool byte.  Full sizes of
the five configurations (and the 64 KiB shape): every run-table, plan and
rebuild array in full, and every byte of the packed slab and of the unpacked
pool against the oracle's pack and unpack of the same holder bytes.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_kvx_gb300 import kvx, workloads as W
from tables import random_holder, random_holder_large, random_lanes
from gpu_helpers import (assert_equal_chunked, assert_plan_equal, assert_table_equal, check_all,
                         gpu_plan, host_generator_bytes,
                         oracle_all)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl", W.small_variants(), ids=lambda w: w.name)
def test_small_variants_bit_exact(wl):
    check_all(wl.addr, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)


def test_random_holders_bit_exact():
    rng = np.random.default_rng(2024)
    for trial in range(60):
        B = int(rng.integers(1, 40))
        addr, seg_len, numa, pool = random_holder(rng, B, int(rng.integers(1, 9)), int(rng.integers(1, 4)))
        check_all(addr, B, seg_len, numa, pool)


@pytest.mark.parametrize("seed", range(40))
def test_random_large_holders_bit_exact(seed):
    """Seeded holders of up to ~90 MB with every feature mixed: 1-3 NUMA
    regions, bump or permuted placement with spill moves, 512 B to 8 KiB
    segments, K-only caches; most take the cooperative planner and several
    copy paths.  Every output of the five calls equals the oracle's, and the
    two-stage copies give the oracle's slab and destination too."""
    addr, seg_len, numa, pool = random_holder_large(np.random.default_rng(2025 + seed))
    B = addr.shape[0]
    tr, t, p, local = check_all(addr, B, seg_len, numa, pool)
    host_pool = W.pool_bytes_np(99, 0, pool)
    want_slab = np.zeros(p.slab_bytes, dtype=np.uint8)
    assert oracle.pack(host_pool, p.descs, want_slab) == 0
    want_dst = np.full(pool, W.CANARY, dtype=np.uint8)
    assert oracle.unpack(want_slab, p.descs, want_dst) == 0
    dpool = torch.from_numpy(host_pool).cuda()
    slab = torch.zeros(max(1, tr.slab_bytes), dtype=torch.uint8, device="cuda")[: tr.slab_bytes]
    dst = torch.full((pool,), W.CANARY, dtype=torch.uint8, device="cuda")
    tr.prepare_pack(dpool, slab)
    tr.prepare_unpack(slab, dst)
    tr.pack_prepared(dpool, slab)
    tr.unpack_prepared(slab, dst)
    torch.cuda.synchronize()
    assert tr.read_status() == 0
    assert np.array_equal(slab.cpu().numpy(), want_slab)
    assert np.array_equal(dst.cpu().numpy(), want_dst)


def test_chunk_outgrows_stride_long_stretch():
    """A long base-adjacent stretch whose blocks overlap: the fits cut runs
    many times inside one stretch (the sequential walker)."""
    B, L, seg = 3, 300, 16
    addr = np.zeros((B, L), dtype=np.uint64)
    for b in range(B):
        addr[b] = b * 7 * seg + np.arange(L) * seg  # stride 112 < chunk
    check_all(addr, B, np.full(L, seg, np.uint32), np.zeros(L, np.uint32), int(addr.max()) + seg)


def test_random_lanes_many_tiles_all_radix_digits():
    """Unstructured addresses over 40 bits, node ids in several bytes: R spans
    several 2048-run tiles and every radix digit is active."""
    rng = np.random.default_rng(77)
    for B, L in ((777, 40), (1500, 9), (5, 1100)):
        addr, seg_len, numa, pool = random_lanes(rng, B, L)
        t, p, st, local = oracle_all(addr, B, seg_len, numa, pool)
        tr = gpu_plan(addr, B, seg_len, numa, pool)
        assert_table_equal(tr, t)
        assert p.status == 0 and tr.read_status() == 0
        assert_plan_equal(tr, p)
        assert np.array_equal(tr.read_local(), local)


@pytest.mark.parametrize("per_sm,extra", [(512, -2), (512, 0), (512, 2), (1024, 0), (1024, 2)])
def test_planner_tile_size_boundary(per_sm, extra):
    """Around 512 and 1024 runs per SM: the cooperative planner cuts the runs
    into the smallest tiles (512, 1024 or 2048 runs) of which there are no
    more than blocks (extra 0 uses every block).  Both sides of each boundary
    equal the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    L = 64
    B = per_sm * sms // 32 + extra  # pair runs: R = 32 * B
    addr, seg_len, numa, pool = random_lanes(np.random.default_rng(4242 + per_sm + extra), B, L)
    t, p, st, local = oracle_all(addr, B, seg_len, numa, pool)
    assert t.num_runs == L * ((B + 1) // 2)
    tr = gpu_plan(addr, B, seg_len, numa, pool)
    assert_table_equal(tr, t)
    assert p.status == 0 and tr.read_status() == 0
    assert_plan_equal(tr, p)
    assert np.array_equal(tr.read_local(), local)


def test_planner_more_tiles_than_one_sweep():
    """2,560,000 pair runs (10,000 x 512 random lanes): 1250 tiles of 2048
    runs, more than eight per planner block, so every radix pass sweeps its
    offsets for a block's tiles in two chunks and the histogram phase counts
    more than eight tiles per block.  Plan and rebuilt pointers equal the
    oracle's."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, L = 10000, 512
    assert (L * B // 2 + 2047) // 2048 > 8 * sms
    addr, seg_len, numa, pool = random_lanes(np.random.default_rng(10512), B, L)
    t, p, st, local = oracle_all(addr, B, seg_len, numa, pool)
    assert t.num_runs == L * B // 2 and p.status == 0
    tr = gpu_plan(addr, B, seg_len, numa, pool)
    assert tr.read_status() == 0
    assert_table_equal(tr, t)
    assert_plan_equal(tr, p)
    assert np.array_equal(tr.read_local(), local)
    del tr
    torch.cuda.empty_cache()


@pytest.mark.parametrize("case", ["one_per_sm", "two_per_sm", "sweep_chunks"])
def test_planner_two_blocks_per_sm(case):
    """kvx_plan_set_sm_share(2): a table of at most one 2048-run tile per SM is
    planned by one block per distinct SM (the first to start on each), a
    larger one by up to two blocks per SM, and the plan equals the oracle's
    either way (and the one-block-per-SM plan)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    L = 512
    B = {"one_per_sm": 2 * 2048 * (sms - 10) // L,       # ~sms - 10 tiles
         "two_per_sm": 2 * 2048 * (2 * sms - 10) // L,   # ~2 sms - 10 tiles
         "sweep_chunks": 10000}[case]                   # 1250 tiles
    addr, seg_len, numa, pool = random_lanes(np.random.default_rng(7000 + B), B, L)
    t, p, st, local = oracle_all(addr, B, seg_len, numa, pool)
    assert p.status == 0
    try:
        kvx.kvx_plan_set_sm_share(2)
        tr = gpu_plan(addr, B, seg_len, numa, pool)
    finally:
        kvx.kvx_plan_set_sm_share(1)
    assert tr.read_status() == 0
    assert_table_equal(tr, t)
    assert_plan_equal(tr, p)
    assert np.array_equal(tr.read_local(), local)
    del tr
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,L,kind", [(20011, 6, "random"), (30013, 9, "random"), (40960, 4, "bump"),
                                      (9001, 2, "bump"), (30011, 40, "random"), (25000, 70, "bump")])
def test_tall_tables_block_per_lane_scan(B, L, kind):
    """Tables with far more row tiles than lanes: the encoder's lane scan is
    spread over the grid, one warp per lane and chunk of 32 row tiles, each
    chunk folding in the totals of the lane's earlier chunks (pair runs, and
    long runs broken by relocated blocks).  The last two also have a ragged
    last lane tile (40 lanes: 32 + 8; 70: 32 + 32 + 6)."""
    rng = np.random.default_rng(B + L)
    if kind == "random":
        addr, seg_len, numa, pool = random_lanes(rng, B, L)
    else:
        seg = 64
        pos = np.arange(B, dtype=np.int64)
        rel = np.sort(rng.choice(B, size=B // 40, replace=False))
        pos[rel] = B + np.arange(rel.size)
        addr = (pos[:, None] * (L * seg) + np.arange(L)[None, :] * seg).astype(np.uint64)
        seg_len, numa = np.full(L, seg, np.uint32), np.zeros(L, np.uint32)
        pool = int(addr.max()) + seg
    t = oracle.encode_runs(addr)
    tr = kvx.Transfer(B, seg_len, numa, pool)
    tr.set_addr(addr)
    tr.encode()
    torch.cuda.synchronize()
    assert tr.read_status() == 0
    assert_table_equal(tr, t)


@pytest.mark.parametrize("kind", ["bump", "random"])
def test_encoder_blocks_with_several_tiles(kind):
    """A table of more tiles than the encoder's grid has blocks: 40,000 x 512
    is 16 lane tiles x 79 row tiles of 8 slices x 64 blocks, 1264 tiles,
    against at most six blocks per SM.  Blocks then loop over tiles, and the
    emit walks each slice again instead of writing from the start masks.
    Bit-exact against the oracle (relocated bump layout: long runs broken;
    random: pair runs)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, L = 40000, 512
    assert 16 * ((B + 511) // 512) > 6 * sms  # more tiles than resident blocks
    rng = np.random.default_rng(40512 + len(kind))
    if kind == "random":
        addr, seg_len, numa, pool = random_lanes(rng, B, L)
    else:
        seg = 64
        pos = np.arange(B, dtype=np.int64)
        rel = np.sort(rng.choice(B, size=B // 50, replace=False))
        pos[rel] = B + np.arange(rel.size)
        addr = (pos[:, None] * (L * seg) + np.arange(L)[None, :] * seg).astype(np.uint64)
        seg_len, numa = np.full(L, seg, np.uint32), np.zeros(L, np.uint32)
        pool = int(addr.max()) + seg
    t = oracle.encode_runs(addr)
    tr = kvx.Transfer(B, seg_len, numa, pool)
    tr.set_addr(addr)
    tr.encode()
    torch.cuda.synchronize()
    assert tr.read_status() == 0
    assert_table_equal(tr, t)
    del tr
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,L", [(0, 4), (1, 2), (1, 7 * 2), (2, 2), (3, 50), (65, 34), (513, 2)])
def test_edge_shapes(B, L):
    rng = np.random.default_rng(B * 1000 + L)
    slots = L // 2
    if B == 0:
        addr = np.zeros((0, L), dtype=np.uint64)
        seg_len = np.full(L, 64, np.uint32)
        tr = gpu_plan(addr, 0, seg_len, np.zeros(L, np.uint32), 4096)
        assert tr.read_status() == 0 and tr.read_counts() == (0, 0, 0)
        rpl, base, _, _ = tr.read_table()
        assert np.all(rpl == 0) and base.size == 0
        return
    addr, seg_len, numa, pool = random_holder(rng, B, slots, 2)
    check_all(addr, B, seg_len, numa, pool)


def test_unaligned_segments_use_the_byte_path():
    """Segment lengths that are not multiples of 16 bytes."""
    rng = np.random.default_rng(5)
    B, L = 9, 6
    seg_len = np.array([3, 5, 7, 11, 13, 17], np.uint32)
    addr = np.zeros((B, L), dtype=np.uint64)
    pos = rng.permutation(B)
    chunk = int(seg_len.sum()) + 1
    for b in range(B):
        off = 0
        for l in range(L):
            addr[b, l] = pos[b] * chunk + off
            off += int(seg_len[l])
    check_all(addr, B, seg_len, np.zeros(L, np.uint32), int(addr.max()) + 17)


# --------------------------------------------------------- negative tables

def _gpu_plan_table(B, seg_len, numa, pool, rpl, base, stride, count, num_runs=None,
                    table_lanes=None, group_cap=None, desc_cap=None):
    L = seg_len.size
    tr = kvx.Transfer(B, seg_len, numa, pool)
    R = base.size
    assert R <= tr.run_cap
    tr.runs_per_lane[: rpl.size].copy_(torch.from_numpy(rpl.astype(np.uint32).view(np.int32)))
    if R:
        tr.run_base[:R].copy_(torch.from_numpy(base.astype(np.uint64).view(np.int64)))
        tr.run_stride[:R].copy_(torch.from_numpy(stride.astype(np.int64)))
        tr.run_count[:R].copy_(torch.from_numpy(count.astype(np.uint32).view(np.int32)))
    tr.num_runs.fill_(R if num_runs is None else num_runs)
    tr.plan(table_lanes=table_lanes, group_cap=group_cap, desc_cap=desc_cap)
    torch.cuda.synchronize()
    return tr


@pytest.mark.parametrize("name", ["worst", "many_small"])
def test_plan_into_arrays_off_16_byte_boundaries(name):
    """Group and descriptor arrays that start 8 bytes past a 16-byte boundary
    (the planner then writes its records field by field instead of in
    16-byte pieces): the same plan as the oracle's, from the single-block
    planner (worst: 1116 runs) and the cooperative one (many_small: 4368)."""
    wl = {v.name: v for v in W.small_variants()}[name]
    B, L = wl.addr.shape
    t = oracle.encode_runs(wl.addr)
    p = oracle.plan(t, B, wl.seg_len, wl.numa, wl.pool_bytes)
    tr = kvx.Transfer(B, wl.seg_len, wl.numa, wl.pool_bytes)
    tr.set_addr(wl.addr)
    tr.encode()
    gbuf = torch.zeros(tr.groups.numel() + 16, dtype=torch.uint8, device="cuda")
    dbuf = torch.zeros(tr.descs.numel() + 16, dtype=torch.uint8, device="cuda")
    g_ptr, d_ptr = gbuf.data_ptr() + 8, dbuf.data_ptr() + 8
    assert g_ptr % 16 == 8 and d_ptr % 16 == 8
    kvx.kvx_plan_groups(tr.runs_per_lane, tr.L, tr.run_base, tr.run_stride, tr.run_count, tr.num_runs,
                        tr.run_cap, tr.B, tr.seg_len, tr.numa, tr.L, tr.pool_bytes, g_ptr, tr.group_cap,
                        d_ptr, tr.desc_cap, tr.lane_first, tr.run_block, tr.run_group, tr.run_off,
                        tr.counts, tr.status, tr.plan_ws)
    torch.cuda.synchronize()
    assert tr.read_status() == 0
    ng, nd, slab = tr.read_counts()
    assert (ng, nd, slab) == (len(p.groups), len(p.descs), p.slab_bytes)
    got_g = gbuf.cpu().numpy()[8: 8 + ng * oracle.GROUP_DTYPE.itemsize]
    got_d = dbuf.cpu().numpy()[8: 8 + nd * oracle.DESC_DTYPE.itemsize]
    assert got_g.tobytes() == p.groups.tobytes()
    assert got_d.tobytes() == p.descs.tobytes()


def _validation_cases_match(B, seg_len0, numa, pool0, t):
    """Corrupt the table one class at a time; the CUDA planner must report
    exactly the oracle's status bits and plan nothing."""
    cases = [("ok", dict()), ("arrays", dict(num_runs=t.num_runs - 1))]
    c = t.run_count.copy(); c[2] = 7
    cases.append(("coverage", dict(count=c)))
    c = t.run_count.copy(); c[1] = 0
    cases.append(("zero_count", dict(count=c)))
    sl = seg_len0.copy(); sl[2] = 0
    cases.append(("zero_len", dict(seg_len=sl)))
    cases.append(("span_pool", dict(pool=pool0 - 1)))
    st = t.run_stride.copy(); st[0] = 2**62
    cases.append(("span_wrap", dict(stride=st)))
    st = t.run_stride.copy(); st[3] = -(2**50)
    cases.append(("span_negative", dict(stride=st)))
    c = t.run_count.copy(); c[0] = 0
    cases.append(("several", dict(count=c, seg_len=sl, pool=10)))
    for name, kw in cases:
        seg_len = kw.get("seg_len", seg_len0)
        pool = kw.get("pool", pool0)
        table = oracle.RunTable(t.runs_per_lane, t.run_base, kw.get("stride", t.run_stride),
                                kw.get("count", t.run_count))
        p = oracle.plan(table, B, seg_len, numa, pool, num_runs=kw.get("num_runs"))
        tr = _gpu_plan_table(B, seg_len, numa, pool, table.runs_per_lane, table.run_base,
                             table.run_stride, table.run_count, num_runs=kw.get("num_runs"))
        assert tr.read_status() == p.status, name
        assert tr.read_counts() == (p.groups.size, p.descs.size, p.slab_bytes), name
        if p.status == 0:
            assert_plan_equal(tr, p)
    tr = _gpu_plan_table(B, seg_len0, numa, pool0, t.runs_per_lane, t.run_base, t.run_stride,
                         t.run_count, table_lanes=seg_len0.size - 1)
    assert tr.read_status() == kvx.S_LANES and tr.read_counts() == (0, 0, 0)
    tr = _gpu_plan_table(B, seg_len0, numa, pool0, t.runs_per_lane, t.run_base, t.run_stride,
                         t.run_count, group_cap=1)
    assert tr.read_status() == kvx.S_CAPACITY and tr.read_counts() == (0, 0, 0)
    tr = _gpu_plan_table(B, seg_len0, numa, pool0, t.runs_per_lane, t.run_base, t.run_stride,
                         t.run_count, desc_cap=1)
    assert tr.read_status() == kvx.S_CAPACITY and tr.read_counts() == (0, 0, 0)


def test_validation_status_matches_oracle_multi_tile():
    """The same corruptions on a 3000-run table (the multi-block planner)."""
    rng = np.random.default_rng(31)
    addr, seg_len, numa, pool = random_lanes(rng, 300, 20)
    t = oracle.encode_runs(addr)
    assert t.num_runs > 2048
    _validation_cases_match(300, seg_len, numa, pool, t)


def test_validation_status_matches_oracle():
    wl = W.tiny()
    t = oracle.encode_runs(wl.addr)
    _validation_cases_match(wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes, t)
    cases = []
    cases.append(("ok", dict()))
    cases.append(("arrays", dict(num_runs=t.num_runs - 1)))
    c = t.run_count.copy(); c[2] = 7
    cases.append(("coverage", dict(count=c)))
    c = t.run_count.copy(); c[1] = 0
    cases.append(("zero_count", dict(count=c)))
    sl = wl.seg_len.copy(); sl[2] = 0
    cases.append(("zero_len", dict(seg_len=sl)))
    cases.append(("span_pool", dict(pool=wl.pool_bytes - 1)))
    s = t.run_stride.copy(); s[0] = 2**62
    cases.append(("span_wrap", dict(stride=s)))
    s = t.run_stride.copy(); s[3] = -(2**20)
    cases.append(("span_negative", dict(stride=s)))
    c = t.run_count.copy(); c[0] = 0
    cases.append(("several", dict(count=c, seg_len=sl, pool=10)))
    for name, kw in cases:
        seg_len = kw.get("seg_len", wl.seg_len)
        pool = kw.get("pool", wl.pool_bytes)
        table = oracle.RunTable(t.runs_per_lane, t.run_base, kw.get("stride", t.run_stride),
                                kw.get("count", t.run_count))
        p = oracle.plan(table, wl.blocks, seg_len, wl.numa, pool, num_runs=kw.get("num_runs"))
        tr = _gpu_plan_table(wl.blocks, seg_len, wl.numa, pool, table.runs_per_lane,
                             table.run_base, table.run_stride, table.run_count,
                             num_runs=kw.get("num_runs"))
        assert tr.read_status() == p.status, name
        assert tr.read_counts() == (p.groups.size, p.descs.size, p.slab_bytes), name
    # wrong lane count
    tr = _gpu_plan_table(wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes, t.runs_per_lane,
                         t.run_base, t.run_stride, t.run_count, table_lanes=wl.lanes - 1)
    assert tr.read_status() == kvx.S_LANES and tr.read_counts() == (0, 0, 0)
    # one-block run with a stride
    rpl = np.full(8, 2, np.uint32)
    base = np.repeat(t.run_base, 2)
    base[1::2] = t.run_base + 7 * t.run_stride.astype(np.uint64)
    stride = np.repeat(t.run_stride, 2)
    stride[1::2] = 0
    count = np.tile(np.array([7, 1], np.uint32), 8)
    tr = _gpu_plan_table(wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes, rpl, base, stride, count)
    p = oracle.plan(oracle.RunTable(rpl, base, stride, count), wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    assert tr.read_status() == p.status == 0
    assert_plan_equal(tr, p)
    stride[1] = 5
    tr = _gpu_plan_table(wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes, rpl, base, stride, count)
    assert tr.read_status() == kvx.S_STRIDE1
    # capacities
    tr = _gpu_plan_table(wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes, t.runs_per_lane,
                         t.run_base, t.run_stride, t.run_count, group_cap=1)
    assert tr.read_status() == kvx.S_CAPACITY and tr.read_counts() == (0, 0, 0)
    tr = _gpu_plan_table(wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes, t.runs_per_lane,
                         t.run_base, t.run_stride, t.run_count, desc_cap=1)
    assert tr.read_status() == kvx.S_CAPACITY and tr.read_counts() == (0, 0, 0)


def test_rebuild_bounds_match_oracle():
    wl = W.tiny()
    t, p, st, local = oracle_all(wl.addr, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    tr = gpu_plan(wl.addr, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    g = p.groups.copy()
    g["chunk"][0] -= 4096
    tr.groups[: g.nbytes].copy_(torch.from_numpy(g.view(np.uint8)))
    tr.status.zero_()
    tr.rebuild()
    torch.cuda.synchronize()
    st, want = oracle.rebuild(t, p, wl.blocks, wl.lanes, wl.seg_len, groups=g)
    assert tr.read_status() == st == oracle.S_BOUNDS
    assert np.array_equal(tr.read_local(), want)
    # slab one byte short: group 1's carve no longer fits
    tr.groups[: p.groups.nbytes].copy_(torch.from_numpy(p.groups.view(np.uint8)))
    tr.status.zero_()
    tr.rebuild(slab_bytes=p.slab_bytes - 1)
    torch.cuda.synchronize()
    st, want = oracle.rebuild(t, p, wl.blocks, wl.lanes, wl.seg_len, slab_bytes=p.slab_bytes - 1)
    assert tr.read_status() == st == oracle.S_BOUNDS
    assert np.array_equal(tr.read_local(), want)


# mutation -> (small variant, status the oracle's rebuild gives)
CORRUPT_GROUPS = {
    "block": ("default_s", oracle.S_BOUNDS),
    "count": ("default_s", oracle.S_BOUNDS),
    "dense": ("many_small", oracle.S_BOUNDS),
    "off": ("default_s", oracle.S_BOUNDS),
    "chunk_small": ("default_s", oracle.S_BOUNDS),
    "local": ("default_s", oracle.S_BOUNDS),
    # the page's dense formula reads remote(b) - group_remote from the runs,
    # so a dense group's stride field takes no part: same pointers, no error
    "stride_dense": ("default_s", 0),
    # a non-dense group's mirror subtracts G.base + i*G.stride: blocks after
    # the first move out of their slices
    "stride_nondense": ("worst", oracle.S_BOUNDS),
}


@pytest.mark.parametrize("mutate", sorted(CORRUPT_GROUPS))
def test_rebuild_corrupt_groups_match_oracle(mutate):
    """Group records that break one check each, on groups of many blocks: the
    first block moved (its runs no longer start there), the block count cut,
    a non-dense group marked dense (its stride then differs from its chunk
    and every block is checked on its own), the chunk one byte short of its
    last run's end, a chunk shorter than the segments, a carve past the slab,
    and the stride field alone altered on a dense and on a non-dense group.
    Every pointer and the status word match the oracle's rebuild of the same
    records, which works from the runs' own addresses."""
    name, want_status = CORRUPT_GROUPS[mutate]
    wl = {v.name: v for v in W.small_variants()}[name]
    B, L = wl.addr.shape
    t, p, st, local = oracle_all(wl.addr, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    tr = gpu_plan(wl.addr, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    g = p.groups.copy()
    k = int(np.flatnonzero(g["count"] > 1)[0])
    if mutate == "block":
        g["block"][k] += 1
    elif mutate == "count":
        g["count"][k] -= 1
    elif mutate == "dense":
        nd = np.flatnonzero((g["dense"] == 0) & (g["count"] > 1))
        g["dense"][int(nd[0])] = 1
    elif mutate == "off":
        g["chunk"][k] -= 1
    elif mutate == "chunk_small":
        g["chunk"][k] = max(1, int(g["chunk"][k]) // 3)
    elif mutate == "local":
        g["local"][k] += np.uint64(p.slab_bytes)
    elif mutate == "stride_dense":
        assert g["dense"][k] == 1
        g["stride"][k] += 4096
    else:
        nd = np.flatnonzero((g["dense"] == 0) & (g["count"] > 1) & (g["stride"] > 0))
        k = int(nd[0])
        g["stride"][k] += 4096
    tr.groups[: g.nbytes].copy_(torch.from_numpy(g.view(np.uint8)))
    tr.status.zero_()
    tr.rebuild()
    torch.cuda.synchronize()
    stw, want = oracle.rebuild(t, p, B, L, wl.seg_len, groups=g)
    assert stw == want_status
    assert tr.read_status() == stw
    assert np.array_equal(tr.read_local(), want)
    if want_status:
        # only the altered group's pointers are rejected
        bad = want == np.uint64(2**64 - 1)
        assert bad.any() and not bad.all()


def test_pack_descriptor_checks_match_oracle():
    wl = W.tiny()
    t, p, st, local = oracle_all(wl.addr, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    tr = gpu_plan(wl.addr, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    host_pool = W.holder_pool_np(wl)
    pool = torch.from_numpy(host_pool).cuda()
    for mutate in ("tiling", "bounds"):
        d = p.descs.copy()
        if mutate == "tiling":
            d["local"][1] += 16
        else:
            d["remote"][1] = wl.pool_bytes - 8
        tr.descs[: d.nbytes].copy_(torch.from_numpy(d.view(np.uint8)))
        slab = torch.zeros(p.slab_bytes, dtype=torch.uint8, device="cuda")
        tr.status.zero_()
        tr.pack(pool, slab)
        torch.cuda.synchronize()
        want = np.zeros(p.slab_bytes, dtype=np.uint8)
        stw = oracle.pack(host_pool, d, want)
        assert tr.read_status() == stw, mutate
        assert np.array_equal(slab.cpu().numpy(), want), mutate


def _desc_list(rng, lengths, bad=()):
    """Descriptors tiling [0, sum(lengths)) of the slab in order, read from
    disjoint pool ranges placed in a shuffled order with small gaps (16-byte
    aligned unless the length is not a multiple of 16); indices in bad point
    past the end of the pool.  Returns (descs, slab bytes, pool bytes)."""
    n = len(lengths)
    d = np.zeros(n, dtype=oracle.DESC_DTYPE)
    remote = np.zeros(n, dtype=np.int64)
    cur = 0
    for k in rng.permutation(n):
        ln = int(lengths[k])
        cur += int(rng.integers(0, 4)) * 16 + (int(rng.integers(1, 16)) if ln % 16 else 0)
        remote[k] = cur
        cur += ln
    pool_bytes = cur + 4096
    local = 0
    for k in range(n):
        ln = int(lengths[k])
        r = pool_bytes - ln // 2 if k in bad else int(remote[k])
        d[k] = (r, local, ln, 0, 0)
        local += ln
    return d, local, pool_bytes


@pytest.mark.parametrize("mix", ["ring_4k", "ring_2k_6k", "register_32k", "short_mixed",
                                 "unaligned", "with_bad"])
def test_copy_paths_descriptor_mix(mix):
    """Tiles of one descriptor (bulk ring), tiles shared by aligned 2-16 KiB
    descriptors (per-descriptor pieces on the 16 KiB-stage rings), and the
    rest (register path): pack and unpack bit-exact against the oracle,
    skipped out-of-range descriptors included."""
    rng = np.random.default_rng(sum(map(ord, mix)))
    if mix == "ring_4k":
        lens = [4096] * 700 + [1 << 20] * 3 + [4096] * 33
    elif mix == "ring_2k_6k":
        lens = list(rng.choice([2048, 6144, 10240], size=900))
    elif mix == "register_32k":
        lens = [32768] * 200
    elif mix == "short_mixed":
        lens = list(rng.choice([1024, 4096, 512, 8192], size=900))
    elif mix == "unaligned":
        lens = list(rng.choice([4096, 4100, 2056], size=700))
    else:
        lens = [4096] * 600
    bad = {5, 77, 301} if mix == "with_bad" else set()
    d, slab_bytes, pool_bytes = _desc_list(rng, [int(x) for x in lens], bad)
    host_pool = rng.integers(0, 256, pool_bytes, dtype=np.uint8)
    want_slab = np.zeros(slab_bytes, np.uint8)
    st_p = oracle.pack(host_pool, d, want_slab)
    want_pool = np.full(pool_bytes, 0xA5, np.uint8)
    st_u = oracle.unpack(want_slab, d, want_pool)
    dd = torch.from_numpy(d.view(np.uint8).copy()).cuda()
    nd = torch.tensor([len(d), 0, 0], dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(kvx.kvx_copy_workspace_size(slab_bytes), dtype=torch.uint8, device="cuda")
    pool = torch.from_numpy(host_pool).cuda()
    slab = torch.zeros(slab_bytes, dtype=torch.uint8, device="cuda")
    kvx.kvx_pack(pool, pool_bytes, dd, nd, len(d), slab, slab_bytes, status, ws)
    torch.cuda.synchronize()
    assert int(status.item()) == st_p
    assert np.array_equal(slab.cpu().numpy(), want_slab)
    dst = torch.full((pool_bytes,), 0xA5, dtype=torch.uint8, device="cuda")
    status.zero_()
    kvx.kvx_unpack(slab, slab_bytes, dd, nd, len(d), dst, pool_bytes, status, ws)
    torch.cuda.synchronize()
    assert int(status.item()) == st_u
    assert np.array_equal(dst.cpu().numpy(), want_pool)


@pytest.mark.parametrize("mix", ["ring_4k", "ring_2k_6k", "short_mixed", "unaligned", "with_bad"])
def test_prepared_copies_match_oracle(mix):
    """The two-stage copies: kvx_copy_prepare, then kvx_pack_prepared and
    kvx_unpack_prepared (each along its own preparation), bit-exact against
    the oracle on every copy path; status bits as kvx_pack / kvx_unpack."""
    rng = np.random.default_rng(sum(map(ord, mix)) + 1)
    lens = {"ring_4k": [4096] * 700 + [1 << 20] * 3 + [4096] * 33,
            "ring_2k_6k": list(rng.choice([2048, 6144, 10240], size=900)),
            "short_mixed": list(rng.choice([1024, 4096, 512, 8192], size=900)),
            "unaligned": list(rng.choice([4096, 4100, 2056], size=700)),
            "with_bad": [4096] * 600}[mix]
    bad = {5, 77, 301} if mix == "with_bad" else set()
    d, slab_bytes, pool_bytes = _desc_list(rng, [int(x) for x in lens], bad)
    host_pool = rng.integers(0, 256, pool_bytes, dtype=np.uint8)
    want_slab = np.zeros(slab_bytes, np.uint8)
    st_p = oracle.pack(host_pool, d, want_slab)
    want_pool = np.full(pool_bytes, 0xA5, np.uint8)
    st_u = oracle.unpack(want_slab, d, want_pool)
    dd = torch.from_numpy(d.view(np.uint8).copy()).cuda()
    nd = torch.tensor([len(d), 0, 0], dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsb = kvx.kvx_copy_workspace_size(slab_bytes)
    ws_p = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    ws_u = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    pool = torch.from_numpy(host_pool).cuda()
    slab = torch.zeros(slab_bytes, dtype=torch.uint8, device="cuda")
    dst = torch.full((pool_bytes,), 0xA5, dtype=torch.uint8, device="cuda")
    # both preparations first, then both copies
    kvx.kvx_copy_prepare(pool, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws_p)
    kvx.kvx_copy_prepare(dst, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws_u)
    torch.cuda.synchronize()
    assert int(st.item()) == st_p == st_u  # the checks are the same in both directions
    kvx.kvx_pack_prepared(pool, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws_p)
    kvx.kvx_unpack_prepared(slab, slab_bytes, dd, nd, len(d), dst, pool_bytes, st, ws_u)
    torch.cuda.synchronize()
    assert int(st.item()) == st_p
    assert np.array_equal(slab.cpu().numpy(), want_slab)
    assert np.array_equal(dst.cpu().numpy(), want_pool)


@pytest.mark.parametrize("prepared", [False, True])
def test_copies_with_descriptors_off_16_byte_boundaries(prepared):
    """A descriptor array that starts 8 bytes past a 16-byte boundary (the ABI
    asks only for the struct's own alignment): every copy path, one-call and
    two-stage, bit-exact against the oracle."""
    rng = np.random.default_rng(23)
    lens = [4096] * 400 + [1 << 20] * 2 + list(rng.choice([512, 2048, 6144, 32768], size=300))
    d, slab_bytes, pool_bytes = _desc_list(rng, [int(x) for x in lens])
    host_pool = rng.integers(0, 256, pool_bytes, dtype=np.uint8)
    want_slab = np.zeros(slab_bytes, np.uint8)
    assert oracle.pack(host_pool, d, want_slab) == 0
    want_pool = np.full(pool_bytes, 0xA5, np.uint8)
    assert oracle.unpack(want_slab, d, want_pool) == 0
    raw = torch.zeros(d.nbytes + 16, dtype=torch.uint8, device="cuda")
    off = 8 if raw.data_ptr() % 16 == 0 else 0
    raw[off: off + d.nbytes].copy_(torch.from_numpy(d.view(np.uint8).copy()))
    dd = raw.data_ptr() + off
    assert dd % 16 == 8
    nd = torch.tensor([len(d), 0, 0], dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(kvx.kvx_copy_workspace_size(slab_bytes), dtype=torch.uint8, device="cuda")
    pool = torch.from_numpy(host_pool).cuda()
    slab = torch.zeros(slab_bytes, dtype=torch.uint8, device="cuda")
    dst = torch.full((pool_bytes,), 0xA5, dtype=torch.uint8, device="cuda")
    if prepared:
        kvx.kvx_copy_prepare(pool, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws)
        kvx.kvx_pack_prepared(pool, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws)
        kvx.kvx_copy_prepare(dst, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws)
        kvx.kvx_unpack_prepared(slab, slab_bytes, dd, nd, len(d), dst, pool_bytes, st, ws)
    else:
        kvx.kvx_pack(pool, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws)
        kvx.kvx_unpack(slab, slab_bytes, dd, nd, len(d), dst, pool_bytes, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(slab.cpu().numpy(), want_slab)
    assert np.array_equal(dst.cpu().numpy(), want_pool)


@pytest.mark.parametrize("prepared", [False, True])
def test_copies_with_pool_and_slab_off_16_byte_boundaries(prepared):
    """Pool and slab buffers that start one byte past a 16-byte boundary: no
    bulk copy may run (every tile takes the register path's byte copies), and
    the bytes still match the oracle's."""
    rng = np.random.default_rng(29)
    lens = [4096] * 64 + [65536] * 4 + [512] * 32
    d, slab_bytes, pool_bytes = _desc_list(rng, lens)
    host_pool = rng.integers(0, 256, pool_bytes, dtype=np.uint8)
    want_slab = np.zeros(slab_bytes, np.uint8)
    assert oracle.pack(host_pool, d, want_slab) == 0
    want_pool = np.full(pool_bytes, 0xA5, np.uint8)
    assert oracle.unpack(want_slab, d, want_pool) == 0
    dd = torch.from_numpy(d.view(np.uint8).copy()).cuda()
    nd = torch.tensor([len(d), 0, 0], dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(kvx.kvx_copy_workspace_size(slab_bytes), dtype=torch.uint8, device="cuda")
    pool_raw = torch.zeros(pool_bytes + 1, dtype=torch.uint8, device="cuda")
    pool_raw[1:].copy_(torch.from_numpy(host_pool))
    slab_raw = torch.zeros(slab_bytes + 1, dtype=torch.uint8, device="cuda")
    dst_raw = torch.full((pool_bytes + 1,), 0xA5, dtype=torch.uint8, device="cuda")
    pool, slab, dst = pool_raw.data_ptr() + 1, slab_raw.data_ptr() + 1, dst_raw.data_ptr() + 1
    assert pool % 16 and slab % 16 and dst % 16
    if prepared:
        kvx.kvx_copy_prepare(pool, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws)
        kvx.kvx_pack_prepared(pool, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws)
        kvx.kvx_copy_prepare(dst, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws)
        kvx.kvx_unpack_prepared(slab, slab_bytes, dd, nd, len(d), dst, pool_bytes, st, ws)
    else:
        kvx.kvx_pack(pool, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws)
        kvx.kvx_unpack(slab, slab_bytes, dd, nd, len(d), dst, pool_bytes, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(slab_raw.cpu().numpy()[1:], want_slab)
    assert np.array_equal(dst_raw.cpu().numpy()[1:], want_pool)


def test_prepared_copy_misuse_moves_nothing():
    """Lists serve the one copy they were made for: a second copy along the
    same preparation, a copy along a workspace prepared for other
    descriptors, and one along a workspace never prepared (cleared) each
    move no byte and raise KVX_S_DESC; kvx_pack after all that is intact."""
    rng = np.random.default_rng(11)
    d, slab_bytes, pool_bytes = _desc_list(rng, [4096] * 300 + [65536] * 20 + [2048] * 100)
    host_pool = rng.integers(0, 256, pool_bytes, dtype=np.uint8)
    want = np.zeros(slab_bytes, np.uint8)
    assert oracle.pack(host_pool, d, want) == 0
    dd = torch.from_numpy(d.view(np.uint8).copy()).cuda()
    dd2 = dd.clone()
    nd = torch.tensor([len(d), 0, 0], dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(kvx.kvx_copy_workspace_size(slab_bytes), dtype=torch.uint8, device="cuda")
    pool = torch.from_numpy(host_pool).cuda()
    slab = torch.zeros(slab_bytes, dtype=torch.uint8, device="cuda")

    kvx.kvx_copy_prepare(pool, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws)
    kvx.kvx_pack_prepared(pool, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and np.array_equal(slab.cpu().numpy(), want)
    # second use of the same lists
    slab.zero_()
    kvx.kvx_pack_prepared(pool, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.S_DESC and not slab.any().item()
    # lists made for another descriptor array
    st.zero_()
    kvx.kvx_copy_prepare(pool, pool_bytes, dd2, nd, len(d), slab, slab_bytes, st, ws)
    kvx.kvx_pack_prepared(pool, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.S_DESC and not slab.any().item()
    # a workspace that was never prepared
    st.zero_()
    ws.zero_()
    kvx.kvx_unpack_prepared(slab, slab_bytes, dd, nd, len(d), pool, pool_bytes, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == kvx.S_DESC
    assert np.array_equal(pool.cpu().numpy(), host_pool)
    # the fused call is unaffected
    st.zero_()
    kvx.kvx_pack(pool, pool_bytes, dd, nd, len(d), slab, slab_bytes, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and np.array_equal(slab.cpu().numpy(), want)


# ------------------------------------------------------------ full sizes

FULL = ["tiny", "default", "worst", "mixed", "many_small", "wide64k"]


def _used_positions(wl):
    """Per region: (byte base, chunk, used-position mask) -- from the generator."""
    out = []
    for (first, nslots, base, npos), pos in zip(wl.regions, wl.pos):
        used = np.zeros(npos, dtype=bool)
        used[pos] = True
        out.append((base, 2 * nslots * wl.seg, used))
    return out


@pytest.mark.parametrize("name", ["worst", "many_small", "mixed"])
def test_full_size_plan_two_blocks_per_sm(name):
    """The full worst (141 tiles: one block per distinct SM), many_small (284
    tiles: up to two blocks per SM) and mixed (66 short tiles) tables planned
    at kvx_plan_set_sm_share(2): run table, plan and rebuilt pointers equal to
    the oracle's, as at the default share."""
    wl = W.CONFIGS[name]()
    t, p, st, local = oracle_all(wl.addr, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    assert p.status == 0 and st == 0
    try:
        kvx.kvx_plan_set_sm_share(2)
        tr = gpu_plan(wl.addr, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    finally:
        kvx.kvx_plan_set_sm_share(1)
    assert tr.read_status() == 0
    assert_table_equal(tr, t)
    assert_plan_equal(tr, p)
    assert np.array_equal(tr.read_local(), local)
    del tr
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["worst", "many_small", "mixed"])
def test_full_size_prepared_copies(name):
    """At full size, the two-stage copies (both preparations first, as the
    overlapped passes do) give the same slab and destination bytes as the
    one-call copies, and both equal the holder's bytes where segments lie."""
    wl = W.CONFIGS[name]()
    tr = gpu_plan(wl.addr, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    assert tr.read_status() == 0
    pool = torch.empty(wl.pool_bytes, dtype=torch.uint8, device="cuda")
    W.fill_pool_torch(pool, wl.seed)
    slab = torch.empty(tr.slab_bytes, dtype=torch.uint8, device="cuda")
    tr.pack(pool, slab)
    slab2 = torch.zeros_like(slab)
    dst2 = torch.full((wl.pool_bytes,), W.CANARY, dtype=torch.uint8, device="cuda")
    tr.prepare_pack(pool, slab2)
    tr.prepare_unpack(slab2, dst2)
    tr.pack_prepared(pool, slab2)
    tr.unpack_prepared(slab2, dst2)
    torch.cuda.synchronize()
    assert tr.read_status() == 0
    assert torch.equal(slab, slab2)
    del slab, slab2
    for base, chunk, used in _used_positions(wl):
        n = used.size * chunk
        a = pool[base:base + n].view(used.size, chunk)
        d = dst2[base:base + n].view(used.size, chunk)
        u = torch.from_numpy(used).cuda()
        assert torch.equal(a[u], d[u])
        if (~used).any():
            assert bool((d[~u] == W.CANARY).all())


@pytest.mark.parametrize("name", FULL)
def test_full_size_config(name):
    """Every configuration at its full size: the run table, the plan and the
    rebuilt pointers element by element, then every byte of the packed slab
    against the oracle's pack of the same holder bytes, and every byte of the
    unpacked destination pool (canary-filled) against the oracle's unpack."""
    wl = W.CONFIGS[name]()
    t, p, st, local = oracle_all(wl.addr, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    assert p.status == 0 and st == 0
    tr = gpu_plan(wl.addr, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    assert tr.read_status() == 0
    assert_table_equal(tr, t)
    assert_plan_equal(tr, p)
    assert np.array_equal(tr.read_local(), local)

    pool = torch.empty(wl.pool_bytes, dtype=torch.uint8, device="cuda")
    W.fill_pool_torch(pool, wl.seed)
    slab = torch.empty(tr.slab_bytes, dtype=torch.uint8, device="cuda")
    dst = torch.full((wl.pool_bytes,), W.CANARY, dtype=torch.uint8, device="cuda")
    tr.pack(pool, slab)
    tr.unpack(slab, dst)
    torch.cuda.synchronize()
    assert tr.read_status() == 0
    host_pool = host_generator_bytes(pool, wl.seed)
    del pool
    want_slab = np.empty(p.slab_bytes, dtype=np.uint8)
    assert oracle.pack(host_pool, p.descs, want_slab) == 0
    del host_pool
    assert_equal_chunked(slab, want_slab)
    del slab
    want_dst = np.full(wl.pool_bytes, W.CANARY, dtype=np.uint8)
    assert oracle.unpack(want_slab, p.descs, want_dst) == 0
    del want_slab
    assert_equal_chunked(dst, want_dst)
    del dst, want_dst
    torch.cuda.empty_cache()
    assert wl.pool_bytes == sum(r[3] * 2 * r[1] * wl.seg for r in wl.regions)
