"""Pins the CPU oracle to facts that do not come from the oracle itself.

Sources (pegaflow PR #350, "run-encode QueryBlocksForTransfer addresses and
coalesce RDMA READs"):
  * Problem section: 576k segments, one fixed64 each (~4.6 MB); per lane the
    bump-allocated addresses are arithmetic.
  * Wire format paragraph: a fully bump-allocated holder collapses every lane
    to one run (~13 KB response).
  * Requester step 4: the degenerate worst case is per-segment reads.
  * READ splitting: 32 MiB pieces; the unsplit 1125 MiB READ of one region.
  * Results table: descriptors 576,000 -> 72 and 115,200 -> 226.
  * Testing section: assert_plan_replays -- every (block, lane) address is
    re-derived through both the descriptor copy and the run arithmetic.
Plus brute-force enumeration on tiny tables, hand-worked fixtures under
tests/golden/, and closed-form / invariant checks.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from oracle import GROUP_DTYPE, DESC_DTYPE
from paged_kv_cache_kvx_gb300 import workloads as W
from conftest import GOLDEN


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _u64(x):
    return int(x) & (2**64 - 1)


def _i64(x):
    x = _u64(x)
    return x - 2**64 if x >= 2**63 else x


# ------------------------------------------------------------------ helpers

def replay(wl_addr, seg_len, table, p, local):
    """assert_plan_replays: every (b, l) address through the run arithmetic
    and through the descriptor that covers its local pointer."""
    B, L = wl_addr.shape
    # run arithmetic
    r = 0
    for l in range(L):
        blk = 0
        for _ in range(int(table.runs_per_lane[l])):
            base, stride, cnt = int(table.run_base[r]), int(table.run_stride[r]), int(table.run_count[r])
            for i in range(cnt):
                assert _u64(base + i * stride) == int(wl_addr[blk + i, l])
            blk += cnt
            r += 1
        assert blk == B
    # descriptor copy
    starts = p.descs["local"].astype(np.uint64)
    idx = np.searchsorted(starts, local.reshape(-1), side="right") - 1
    d = p.descs[idx]
    lens = np.tile(seg_len.astype(np.uint64), B)
    flat_local = local.reshape(-1)
    assert np.all(flat_local >= d["local"])
    assert np.all(flat_local + lens <= d["local"] + d["len"])
    back = d["remote"] + (flat_local - d["local"])
    assert np.array_equal(back, wl_addr.reshape(-1))


def check_tiling(p):
    """Descriptors tile [0, slab) in order with no gap or overlap (Trust
    boundary: no overlapping local writes)."""
    if p.descs.size == 0:
        assert p.slab_bytes == 0
        return
    ends = p.descs["local"] + p.descs["len"]
    assert p.descs["local"][0] == 0
    assert np.array_equal(p.descs["local"][1:], ends[:-1])
    assert int(ends[-1]) == p.slab_bytes
    assert np.all(p.descs["len"] > 0)
    assert np.all(p.descs["len"] <= oracle.MAX_READ_BYTES)


def full_pipeline(wl):
    t = oracle.encode_runs(wl.addr)
    p = oracle.plan(t, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    assert p.status == 0
    st, local = oracle.rebuild(t, p, wl.blocks, wl.lanes, wl.seg_len)
    assert st == 0
    return t, p, local


# ------------------------------------------------------------------- encode

def test_encode_golden_lanes():
    g = _load("encode_lanes.json")
    for case in g["cases"]:
        lane = np.array([_u64(v) for v in case["lane"]], dtype=np.uint64).reshape(-1, 1)
        t = oracle.encode_runs(lane)
        got = [[int(t.run_base[i]), int(t.run_stride[i]), int(t.run_count[i])] for i in range(t.num_runs)]
        want = [[_u64(b), _i64(s), c] for b, s, c in case["runs"]]
        assert got == want, case["why"]
        assert int(t.runs_per_lane[0]) == len(want)


def _greedy_by_enumeration(lane):
    """All 2^(B-1) cut sets of one lane; keep the decompositions where every
    piece is arithmetic, only the last piece may be a single element, and every
    non-last piece is maximal (its progression does not continue into the next
    element).  Exactly one survives; it is the greedy encoding."""
    B = len(lane)
    survivors = []
    for mask in range(1 << (B - 1)):
        cuts = [0] + [i + 1 for i in range(B - 1) if mask >> i & 1] + [B]
        pieces = [lane[cuts[k]:cuts[k + 1]] for k in range(len(cuts) - 1)]
        ok = True
        for k, pc in enumerate(pieces):
            last = k == len(pieces) - 1
            if len(pc) == 1 and not last:
                ok = False
                break
            if len(pc) >= 2:
                st = _u64(pc[1] - pc[0])
                if any(_u64(pc[i + 1] - pc[i]) != st for i in range(len(pc) - 1)):
                    ok = False
                    break
                if not last and _u64(pieces[k + 1][0] - pc[-1]) == st:
                    ok = False
                    break
        if ok:
            runs = []
            for pc in pieces:
                st = _u64(pc[1] - pc[0]) if len(pc) >= 2 else 0
                runs.append((_u64(pc[0]), _i64(st), len(pc)))
            survivors.append(runs)
    assert len(survivors) == 1
    return survivors[0]


def test_encode_matches_brute_force_enumeration():
    rng = np.random.default_rng(11)
    for B in range(1, 11):
        for _ in range(30):
            # small step alphabet so equal consecutive differences are common
            steps = rng.choice([-3, 0, 2, 2, 2, 5], size=B - 1)
            lane = np.concatenate([[1000], 1000 + np.cumsum(steps)]).astype(np.int64)
            lane_u = [_u64(v) for v in lane]
            t = oracle.encode_runs(np.array(lane_u, dtype=np.uint64).reshape(-1, 1))
            got = [(int(t.run_base[i]), int(t.run_stride[i]), int(t.run_count[i]))
                   for i in range(t.num_runs)]
            assert got == _greedy_by_enumeration(lane_u)


def test_encode_bump_allocated_one_run_per_lane():
    """Wire format paragraph: a fully bump-allocated holder collapses every
    lane to a single run, ~13 KB instead of ~4.6 MB for the default shape."""
    fig = _load("page5_figures.json")
    wl = W.default()
    assert wl.segments == fig["default_shape"]["segments"]
    assert wl.payload_bytes == fig["default_shape"]["set_bytes"]
    t = oracle.encode_runs(wl.addr)
    assert t.num_runs == wl.lanes == 576
    assert np.all(t.runs_per_lane == 1)
    assert np.all(t.run_count == wl.blocks)
    chunk = 2 * (wl.slots // 2) * wl.seg
    assert np.all(t.run_stride == chunk) and chunk == 1179648
    old = wl.segments * 8
    new = t.runs_per_lane.nbytes + t.run_base.nbytes + t.run_stride.nbytes + t.run_count.nbytes
    assert old == fig["response_bytes_before"]
    assert new == 13824 and new <= fig["response_bytes_after_max"]
    tt = oracle.encode_runs(W.tiny().addr)
    assert tt.num_runs == 8 and np.all(tt.run_count == 8)


def test_encode_random_lane_gives_pairs_and_bound():
    """Random addresses have no equal consecutive differences: every run is a
    pair (one-element tail when B is odd); runs per lane <= ceil(B/2)."""
    rng = np.random.default_rng(3)
    for B in (1, 2, 7, 64, 101):
        addr = rng.integers(0, 2**62, size=(B, 5), dtype=np.uint64)
        t = oracle.encode_runs(addr)
        assert np.all(t.runs_per_lane == (B + 1) // 2)
        want = [2] * (B // 2) + ([1] if B % 2 else [])
        r = 0
        for l in range(5):
            assert t.run_count[r:r + len(want)].tolist() == want
            r += len(want)


# --------------------------------------------------------------------- plan

def test_plan_golden_hand_cases():
    g = _load("plan_hand.json")
    for case in g["cases"]:
        addr = np.array(case["addr"], dtype=np.uint64)
        B, L = addr.shape
        seg_len = np.full(L, case["seg"], dtype=np.uint32)
        numa = np.array(case["numa"], dtype=np.uint32)
        t = oracle.encode_runs(addr)
        assert t.runs_per_lane.tolist() == case["runs_per_lane"], case["name"]
        got_runs = [[int(t.run_base[i]), int(t.run_stride[i]), int(t.run_count[i])] for i in range(t.num_runs)]
        assert got_runs == case["runs"], case["name"]
        p = oracle.plan(t, B, seg_len, numa, case["pool_bytes"])
        assert p.status == 0, case["name"]
        assert [list(map(int, x)) for x in p.groups.tolist()] == case["groups"], case["name"]
        assert [[int(d["remote"]), int(d["local"]), int(d["len"]), int(d["group"])] for d in p.descs] \
            == case["descs"], case["name"]
        assert p.slab_bytes == case["slab_bytes"]
        st, local = oracle.rebuild(t, p, B, L, seg_len)
        assert st == 0
        assert local.tolist() == case["local"], case["name"]


def test_plan_default_two_dense_regions_72_descs():
    """Results table: 576,000 -> 72 descriptors; READ splitting: each NUMA
    region is one 1125 MiB dense group split at 32 MiB."""
    fig = _load("page5_figures.json")
    wl = W.default()
    t, p, local = full_pipeline(wl)
    assert p.groups.size == 2
    assert np.all(p.groups["dense"] == 1)
    sizes = p.groups["count"].astype(np.uint64) * p.groups["chunk"]
    assert sizes.tolist() == [fig["dense_region_read_bytes"]] * 2
    assert p.descs.size == fig["descs_default"]["after"]
    assert p.slab_bytes == wl.payload_bytes
    check_tiling(p)
    assert int(p.descs["len"].max()) == fig["max_read_bytes"]


def test_plan_wide64k_226_descs():
    fig = _load("page5_figures.json")
    wl = W.wide64k()
    assert wl.segments == fig["descs_wide64k"]["before"]
    t, p, local = full_pipeline(wl)
    assert p.descs.size == fig["descs_wide64k"]["after"]
    assert p.groups.size == 2 and np.all(p.groups["dense"] == 1)
    check_tiling(p)


def test_plan_tiny_two_groups_two_descs():
    wl = W.tiny()
    t, p, local = full_pipeline(wl)
    assert p.groups.size == 2 and p.descs.size == 2
    assert p.slab_bytes == 256 * 1024
    replay(wl.addr, wl.seg_len, t, p, local)


def test_plan_degenerate_is_per_segment_reads():
    """Requester step 4: the degenerate worst case is per-segment reads."""
    wl = W.scattered(blocks=9, slots=4, seg=64)
    t, p, local = full_pipeline(wl)
    assert p.descs.size == wl.segments
    assert np.all(p.descs["len"] == 64)
    replay(wl.addr, wl.seg_len, t, p, local)


@pytest.mark.parametrize("wl", W.small_variants(), ids=lambda w: w.name)
def test_plan_replays_and_tiles(wl):
    t, p, local = full_pipeline(wl)
    check_tiling(p)
    replay(wl.addr, wl.seg_len, t, p, local)
    assert p.slab_bytes == wl.payload_bytes


def _group_members(p, t, numa, seg_len):
    """Per group, its runs in sorted order (recomputed from run_group)."""
    L = t.runs_per_lane.size
    lane = np.repeat(np.arange(L), t.runs_per_lane)
    members = {}
    for r in range(t.num_runs):
        members.setdefault(int(p.run_group[r]), []).append(r)
    out = []
    for gi in range(p.groups.size):
        rs = sorted(members[gi], key=lambda r: int(t.run_base[r]))
        out.append(rs)
    return out, lane


def _random_table(rng, B, slots, nodes):
    """Holder with random block placement per region and random per-lane
    gaps: exercises non-dense groups, fits cuts and negative strides."""
    L = 2 * slots
    seg = int(rng.choice([16, 32, 48]))
    numa = rng.integers(0, nodes, size=L).astype(np.uint32)
    # per block, lay lanes back to back in a random lane order, with the
    # block start drawn from a small set of positions (repeats allowed ->
    # arithmetic runs and adjacency both occur)
    step = int(rng.choice([L * seg // 2, L * seg, L * seg + seg]))
    pos = rng.permutation(B + 3)[:B] if rng.random() < 0.5 else np.arange(B)
    gap = rng.random() < 0.3
    addr = np.zeros((B, L), dtype=np.uint64)
    for b in range(B):
        off = 0
        for l in range(L):
            addr[b, l] = pos[b] * step + off
            off += seg + (seg if gap and l % 3 == 2 else 0)
    pool = int(addr.max()) + seg if B else seg
    return addr, np.full(L, seg, np.uint32), numa, pool


def test_plan_grouping_is_the_greedy_partition():
    """Characterisation of step 3 without re-running it: sorted by (node,
    base, lane, block), every group is a contiguous block of that order whose
    members share node, block range and stride, are base-adjacent and fit the
    stride; and every group boundary is forced (the next group's first run
    would not be accepted).  That partition is unique, so it is the greedy
    one."""
    rng = np.random.default_rng(5)
    for trial in range(150):
        B = int(rng.integers(1, 9))
        addr, seg_len, numa, pool = _random_table(rng, B, int(rng.integers(1, 5)), int(rng.integers(1, 3)))
        t = oracle.encode_runs(addr)
        p = oracle.plan(t, B, seg_len, numa, pool)
        assert p.status == 0
        L = addr.shape[1]
        lane = np.repeat(np.arange(L), t.runs_per_lane)
        key = sorted(range(t.num_runs), key=lambda r: (int(numa[lane[r]]), int(t.run_base[r]),
                                                       int(lane[r]), int(p.run_block[r])))
        gseq = [int(p.run_group[r]) for r in key]
        # contiguous and numbered in order
        assert gseq == sorted(gseq) and gseq[0] == 0 and set(gseq) == set(range(p.groups.size))
        for gi, g in enumerate(p.groups):
            rs = [r for r in key if int(p.run_group[r]) == gi]
            first = rs[0]
            chunk = 0
            for r in rs:
                assert numa[lane[r]] == g["node"] and p.run_block[r] == g["block"]
                assert t.run_count[r] == g["count"] and t.run_stride[r] == g["stride"]
                assert int(t.run_base[r]) == int(g["base"]) + chunk
                assert int(p.run_off[r]) == chunk
                chunk += int(seg_len[lane[r]])
            assert chunk == int(g["chunk"]) and int(t.run_base[first]) == int(g["base"])
            if len(rs) > 1 and g["count"] > 1:
                assert int(g["stride"]) > 0 and chunk <= int(g["stride"])
            dense = g["count"] == 1 or int(g["stride"]) == chunk
            assert int(g["dense"]) == int(dense)
            # boundary forced
            if gi + 1 < p.groups.size:
                nxt = [r for r in key if int(p.run_group[r]) == gi + 1][0]
                same = (numa[lane[nxt]] == g["node"] and p.run_block[nxt] == g["block"]
                        and t.run_count[nxt] == g["count"] and t.run_stride[nxt] == g["stride"]
                        and int(t.run_base[nxt]) == int(g["base"]) + chunk)
                grown = chunk + int(seg_len[lane[nxt]])
                fits = g["count"] == 1 or (int(g["stride"]) > 0 and grown <= int(g["stride"]))
                assert not (same and fits)
        check_tiling(p)
        st, local = oracle.rebuild(t, p, B, L, seg_len)
        assert st == 0
        replay(addr, seg_len, t, p, local)


def test_plan_carve_and_desc_closed_forms():
    """Carve: groups back to back in planner order, local = prefix of
    count*chunk; descriptors: dense -> ceil(count*chunk/32Mi), non-dense ->
    count*ceil(chunk/32Mi); every piece is 32 MiB except the last of a span."""
    for wl in W.small_variants() + [W.worst(), W.mixed(blocks=700)]:
        t, p, _ = full_pipeline(wl)
        sizes = p.groups["count"].astype(np.uint64) * p.groups["chunk"]
        assert np.array_equal(p.groups["local"], np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.uint64))
        M = oracle.MAX_READ_BYTES
        per = np.where(p.groups["dense"] == 1, -(-sizes.astype(np.int64) // M),
                       p.groups["count"].astype(np.int64) * -(-p.groups["chunk"].astype(np.int64) // M))
        assert int(per.sum()) == p.descs.size
        # nodes are carved in ascending order (one partition per node)
        assert np.all(np.diff(p.groups["node"].astype(np.int64)) >= 0)


def test_plan_worst_case_closed_form():
    """Worst case: a permuted block order.  Every greedy run spans blocks
    whose positions step by a constant; each run of a region shares its block
    range with the same run of every lane of the region.  With a positive step
    the region's 288 lanes tile one chunk <= stride (one group, dense iff the
    step is one chunk); a negative step never fits (288 one-run groups)."""
    wl = W.worst(blocks=200, npos=512)
    t, p, local = full_pipeline(wl)
    pos = wl.pos[0]
    # greedy runs over the positions of one lane equal those of every lane
    lane_t = oracle.encode_runs(pos.astype(np.uint64).reshape(-1, 1))
    chunk_r = (wl.slots // 2) * 2 * wl.seg
    n_groups = n_descs = 0
    for i in range(lane_t.num_runs):
        step, cnt = int(lane_t.run_stride[i]), int(lane_t.run_count[i])
        if cnt == 1 or step > 0:
            n_groups += 1
            dense = cnt == 1 or step == 1
            M = oracle.MAX_READ_BYTES
            n_descs += -(-cnt * chunk_r // M) if dense else cnt
        else:
            n_groups += wl.slots // 2 * 2
            n_descs += (wl.slots // 2 * 2) * cnt
    assert p.groups.size == 2 * n_groups
    assert p.descs.size == 2 * n_descs
    assert np.all(p.groups["chunk"][p.groups["stride"] > 0] == chunk_r)


# ---------------------------------------------------------- negative tables

def _base_table():
    wl = W.tiny()
    t = oracle.encode_runs(wl.addr)
    return wl, t


def _plan_status(t, wl, **kw):
    seg_len = kw.pop("seg_len", wl.seg_len)
    numa = kw.pop("numa", wl.numa)
    B = kw.pop("B", wl.blocks)
    pool = kw.pop("pool", wl.pool_bytes)
    return oracle.plan(t, B, seg_len, numa, pool, **kw).status


def test_validate_rejects_each_class():
    """Requester step 1 and the Trust boundary: wrong lane count, parallel
    arrays out of sync, bad coverage, zero-count runs, zero-size slots, span
    overflow -- each rejected with its own status bit, and nothing planned."""
    wl, t = _base_table()
    assert _plan_status(t, wl) == 0
    # lane count
    t2 = oracle.RunTable(t.runs_per_lane[:-1].copy(), t.run_base, t.run_stride, t.run_count)
    assert _plan_status(t2, wl) == oracle.S_LANES
    # arrays out of sync: per-lane counts sum != array length
    assert _plan_status(t, wl, num_runs=t.num_runs - 1) == oracle.S_ARRAYS
    # coverage: a lane's counts do not add to B
    t3 = oracle.RunTable(t.runs_per_lane, t.run_base, t.run_stride, t.run_count.copy())
    t3.run_count[2] = 7
    assert _plan_status(t3, wl) == oracle.S_COVERAGE
    # zero-count run (also breaks coverage)
    t4 = oracle.RunTable(t.runs_per_lane, t.run_base, t.run_stride, t.run_count.copy())
    t4.run_count[1] = 0
    assert _plan_status(t4, wl) == oracle.S_ZERO_COUNT | oracle.S_COVERAGE
    # zero-size K slot
    sl = wl.seg_len.copy()
    sl[2] = 0
    assert _plan_status(t, wl, seg_len=sl) == oracle.S_ZERO_LEN
    # span overflow: the pool is one byte short
    assert _plan_status(t, wl, pool=wl.pool_bytes - 1) == oracle.S_SPAN
    # span overflow through 64-bit wrap of base + i*stride
    t5 = oracle.RunTable(t.runs_per_lane, t.run_base.copy(), t.run_stride.copy(), t.run_count)
    t5.run_stride[0] = 2**62
    assert _plan_status(t5, wl) == oracle.S_SPAN
    # negative stride below address 0
    t6 = oracle.RunTable(t.runs_per_lane, t.run_base.copy(), t.run_stride.copy(), t.run_count)
    t6.run_stride[3] = -(2**20)
    assert _plan_status(t6, wl) == oracle.S_SPAN
    # one-block run with a stride
    t7 = oracle.RunTable(np.full(8, 2, np.uint32),
                         np.repeat(t.run_base, 2), np.repeat(t.run_stride, 2),
                         np.tile(np.array([7, 1], np.uint32), 8))
    t7.run_base[1::2] = t.run_base + 7 * t.run_stride.astype(np.uint64)
    t7.run_stride[1::2] = 0
    assert _plan_status(t7, wl) == 0
    t7.run_stride[1] = 5
    assert _plan_status(t7, wl) == oracle.S_STRIDE1
    # lanes with no runs at all
    t8 = oracle.RunTable(np.zeros(8, np.uint32), t.run_base[:0], t.run_stride[:0], t.run_count[:0])
    assert _plan_status(t8, wl) == oracle.S_COVERAGE
    # several classes at once are all reported
    t9 = oracle.RunTable(t.runs_per_lane, t.run_base.copy(), t.run_stride, t.run_count.copy())
    t9.run_count[0] = 0
    assert _plan_status(t9, wl, seg_len=sl, pool=10) == (oracle.S_ZERO_COUNT | oracle.S_COVERAGE
                                                         | oracle.S_ZERO_LEN | oracle.S_SPAN)
    # output capacity
    p = oracle.plan(t, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes, group_cap=1)
    assert p.status == oracle.S_CAPACITY and p.groups.size == 0
    p = oracle.plan(t, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes, desc_cap=1)
    assert p.status == oracle.S_CAPACITY and p.descs.size == 0


def test_empty_prefix():
    """B = 0: no runs, no groups, an empty slab."""
    addr = np.zeros((0, 6), dtype=np.uint64)
    t = oracle.encode_runs(addr)
    assert t.num_runs == 0 and np.all(t.runs_per_lane == 0)
    p = oracle.plan(t, 0, np.full(6, 64, np.uint32), np.zeros(6, np.uint32), 1024)
    assert p.status == 0 and p.groups.size == 0 and p.descs.size == 0 and p.slab_bytes == 0


# ------------------------------------------------------------------ rebuild

@pytest.mark.parametrize("wl", W.small_variants(), ids=lambda w: w.name)
def test_rebuild_page_formula_equals_block_mirror_formula(wl):
    """Step 5's formula (dense) and the dense-local-mirror formula (non-dense)
    against a second expression: local = G.local + (b - G.block)*G.chunk +
    run_off, evaluated here in numpy."""
    t, p, local = full_pipeline(wl)
    B, L = wl.addr.shape
    lane = np.repeat(np.arange(L), t.runs_per_lane)
    want = np.zeros((B, L), dtype=np.uint64)
    for r in range(t.num_runs):
        g = p.groups[p.run_group[r]]
        b0 = int(p.run_block[r])
        for i in range(int(t.run_count[r])):
            want[b0 + i, lane[r]] = int(g["local"]) + (b0 + i - int(g["block"])) * int(g["chunk"]) + int(p.run_off[r])
    assert np.array_equal(local, want)
    # one slab byte range per segment, none overlapping, covering the slab
    order = np.argsort(local.reshape(-1), kind="stable")
    lens = np.tile(wl.seg_len.astype(np.uint64), B)[order]
    loc = local.reshape(-1)[order]
    if loc.size:
        assert loc[0] == 0 and np.array_equal(loc[1:], loc[:-1] + lens[:-1])
        assert int(loc[-1] + lens[-1]) == p.slab_bytes


def test_rebuild_bounds_checks():
    wl = W.tiny()
    t, p, local = full_pipeline(wl)
    g = p.groups.copy()
    g["local"][1] += 1           # group 1 carve now ends past the slab
    st, loc = oracle.rebuild(t, p, wl.blocks, wl.lanes, wl.seg_len, groups=g)
    assert st == oracle.S_BOUNDS
    bad = np.isin(np.arange(wl.lanes), np.nonzero(wl.numa == 1)[0])
    assert np.all(loc[:, bad] == np.uint64(2**64 - 1)) and np.array_equal(loc[:, ~bad], local[:, ~bad])
    rg = p.run_group.copy()
    rg[0] = 99                   # group index out of range
    st, loc = oracle.rebuild(t, p, wl.blocks, wl.lanes, wl.seg_len, run_group=rg)
    assert st == oracle.S_BOUNDS and np.all(loc[:, 0] == np.uint64(2**64 - 1))
    g = p.groups.copy()
    g["chunk"][0] -= 4096        # segments no longer inside their block slice
    st, loc = oracle.rebuild(t, p, wl.blocks, wl.lanes, wl.seg_len, groups=g)
    assert st == oracle.S_BOUNDS
    # group 0 (dense, lanes 0-3): local = 16384*b + 4096*l sits in the shrunk
    # slice [12288*b, 12288*(b+1)) with its 4096 bytes only while b + l <= 2
    b, l = np.meshgrid(np.arange(wl.blocks), np.arange(4), indexing="ij")
    flagged = loc[:, :4] == np.uint64(2**64 - 1)
    assert np.array_equal(flagged, b + l > 2)
    assert np.array_equal(loc[:, :4][~flagged], local[:, :4][~flagged])


# -------------------------------------------------------------- pack/unpack

@pytest.mark.parametrize("wl", [w for w in W.small_variants() if w.pool_bytes < 2**27],
                         ids=lambda w: w.name)
def test_pack_unpack_identity_and_canary(wl):
    """pack then unpack restores every segment byte; bytes outside segments
    keep the canary; the slab holds each segment at its rebuilt pointer."""
    t, p, local = full_pipeline(wl)
    pool = W.holder_pool_np(wl)
    slab = np.zeros(p.slab_bytes, dtype=np.uint8)
    assert oracle.pack(pool, p.descs, slab) == 0
    B, L = wl.addr.shape
    for b in range(B):
        for l in range(L):
            a, lo, n = int(wl.addr[b, l]), int(local[b, l]), int(wl.seg_len[l])
            assert np.array_equal(slab[lo:lo + n], pool[a:a + n])
    dst = np.full(wl.pool_bytes, W.CANARY, dtype=np.uint8)
    assert oracle.unpack(slab, p.descs, dst) == 0
    mask = np.zeros(wl.pool_bytes, dtype=bool)
    for b in range(B):
        for l in range(L):
            a = int(wl.addr[b, l])
            mask[a:a + int(wl.seg_len[l])] = True
    assert np.array_equal(dst[mask], pool[mask])
    assert np.all(dst[~mask] == W.CANARY)


def test_pack_rejects_bad_descriptors():
    wl = W.tiny()
    t, p, local = full_pipeline(wl)
    pool = W.holder_pool_np(wl)
    slab = np.zeros(p.slab_bytes, dtype=np.uint8)
    d = p.descs.copy()
    d["local"][1] += 16          # no longer tiles the slab
    assert oracle.pack(pool, d, slab) == oracle.S_DESC
    assert np.all(slab == 0)
    d = p.descs.copy()
    d["remote"][1] = wl.pool_bytes - 8   # reads past the pool
    assert oracle.pack(pool, d, slab) == oracle.S_BOUNDS
    assert np.array_equal(slab[:131072], pool[:131072]) and np.all(slab[131072:] == 0)
    small = np.zeros(p.slab_bytes - 1, dtype=np.uint8)
    assert oracle.pack(pool, p.descs, small) == oracle.S_BOUNDS
    dst = np.zeros(wl.pool_bytes - 1, dtype=np.uint8)
    assert oracle.unpack(slab, p.descs, dst) == oracle.S_BOUNDS


def test_payload_generator_is_splitmix64():
    """The payload words are splitmix64 of (seed ^ index); first outputs of
    the published generator seeded with 0 (state advanced by the golden
    gamma before mixing) pin the constants."""
    # splitmix64 stream seeded with 0: next() mixes 1*gamma, 2*gamma, ...
    gamma = 0x9E3779B97F4A7C15
    xs = np.array([(k * gamma - gamma) & (2**64 - 1) for k in (1, 2, 3)], dtype=np.uint64)
    got = W.splitmix64_np(xs)
    assert [hex(int(v)) for v in got] == ["0xe220a8397b1dcdaf", "0x6e789e6aa1b965f4",
                                         "0x6c45d188009454f"]
