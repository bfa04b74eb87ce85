"""Pins for the oracle's widening functions, each against facts that do not
come from the oracle itself.

  * verify_encode -- pegaflow PR #350, Holder paragraph: each block is checked
    against the slot template before its addresses join the run
    accumulators, so a mid-block mismatch leaks nothing and the prefix ends
    at the first failing block.  Pinned by closed forms on bump-allocated
    holders (one run per lane of the prefix length) and by special cases.
  * seal_blocks -- the PR's named follow-up, seal from template metadata:
    every segment is installed from the slab at its rebuilt offset.  Pinned
    by brute force: after pack + seal, each destination segment holds the
    holder bytes of the same (block, lane), whatever the receiver's layout.
  * paged_writes -- "RDMA point-to-point communication for LLM systems",
    TransferEngine API listing (page sets {indices, stride, offset}).
    Pinned by hand-worked fixtures, numpy fancy indexing as the special case
    stride == page_len, and permutation round trips.
"""
import json
import os

import numpy as np
import pytest

import oracle
from paged_kv_cache_kvx_gb300 import workloads as W
from conftest import GOLDEN
from tables import random_holder

S_SPAN, S_BOUNDS = 32, 128


def _bump(B, slots, seg):
    """Fully bump-allocated holder: addr(b, l) = b * L * seg + l * seg."""
    L = 2 * slots
    b = np.arange(B, dtype=np.uint64)[:, None]
    l = np.arange(L, dtype=np.uint64)[None, :]
    return b * np.uint64(L * seg) + l * np.uint64(seg)


# ------------------------------------------------------------ verify_encode

@pytest.mark.parametrize("k", [0, 1, 2, 5, 11])
@pytest.mark.parametrize("lane", [0, 3, 7])
def test_verify_stops_at_first_mismatch_closed_form(k, lane):
    B, slots, seg = 12, 4, 64
    L = 2 * slots
    addr = _bump(B, slots, seg)
    tmpl = np.full(L, seg, np.uint32)
    size = np.tile(tmpl, (B, 1))
    size[k, lane] = seg + 16           # one segment of block k has another size
    size[k + 1:, :] = seg              # later blocks match again: the scan has stopped
    prefix, t = oracle.verify_encode(addr, size, tmpl)
    assert prefix == k
    if k == 0:
        assert t.num_runs == 0 and not t.runs_per_lane.any()
        return
    # a bump-allocated prefix of k blocks: one run per lane, count k
    assert (t.runs_per_lane == 1).all()
    assert (t.run_count == k).all()
    assert (t.run_base == addr[0]).all()
    want_stride = L * seg if k >= 2 else 0
    assert (t.run_stride == want_stride).all()


def test_verify_all_blocks_pass():
    rng = np.random.default_rng(7)
    addr, seg_len, _, _ = random_holder(rng, 9, 3, 2)
    size = np.tile(seg_len, (9, 1))
    prefix, t = oracle.verify_encode(addr, size, seg_len)
    assert prefix == 9
    assert int(t.run_count.sum()) == 9 * addr.shape[1]
    # every lane's runs cover exactly the 9 blocks
    r = 0
    for l in range(addr.shape[1]):
        n = int(t.runs_per_lane[l])
        assert int(t.run_count[r:r + n].sum()) == 9
        r += n


def test_verify_mid_block_mismatch_leaks_nothing():
    """A mismatch in the last lane of block 4: lanes before it in the same
    block must not receive block 4 either."""
    B, slots, seg = 8, 3, 32
    L = 2 * slots
    addr = _bump(B, slots, seg)
    tmpl = np.full(L, seg, np.uint32)
    size = np.tile(tmpl, (B, 1))
    size[4, L - 1] = 0
    prefix, t = oracle.verify_encode(addr, size, tmpl)
    assert prefix == 4
    r = 0
    for l in range(L):
        n = int(t.runs_per_lane[l])
        assert int(t.run_count[r:r + n].sum()) == 4
        r += n


def test_verify_template_differs_per_lane():
    """The template is per lane: a K lane of 64 B and a V lane of 32 B."""
    B, L = 6, 4
    tmpl = np.array([64, 32, 64, 32], np.uint32)
    addr = np.zeros((B, L), np.uint64)
    for b in range(B):
        addr[b] = b * 192 + np.array([0, 64, 96, 160])
    size = np.tile(tmpl, (B, 1))
    prefix, _ = oracle.verify_encode(addr, size, tmpl)
    assert prefix == B
    size[3] = size[3][::-1]            # a block with K and V sizes swapped
    prefix, _ = oracle.verify_encode(addr, size, tmpl)
    assert prefix == 3


# ---------------------------------------------------------------- seal

def _plan_and_pack(addr, seg_len, numa, pool_bytes, pool):
    B, L = addr.shape
    t = oracle.encode_runs(addr)
    p = oracle.plan(t, B, seg_len, numa, pool_bytes)
    assert p.status == 0
    slab = np.zeros(p.slab_bytes, np.uint8)
    assert oracle.pack(pool, p.descs, slab) == 0
    return t, p, slab


def _segments_match(dst, dst_addr, pool, addr, seg_len):
    B, L = addr.shape
    for b in range(B):
        for l in range(L):
            n = int(seg_len[l])
            d, a = int(dst_addr[b, l]), int(addr[b, l])
            assert (dst[d:d + n] == pool[a:a + n]).all(), (b, l)


def _receiver_layout(B, seg_len, lane_major=True, rng=None):
    """The receiver's own placement of every segment (block-major [B][L])."""
    L = seg_len.size
    order = [(b, l) for l in range(L) for b in range(B)] if lane_major else \
        [(b, l) for b in range(B) for l in range(L)]
    if rng is not None:
        order = [order[i] for i in rng.permutation(len(order))]
    dst_addr = np.zeros((B, L), np.uint64)
    off = 0
    for b, l in order:
        dst_addr[b, l] = off
        off += int(seg_len[l])
    return dst_addr, off


@pytest.mark.parametrize("wl", W.small_variants()[:3], ids=lambda w: w.name)
def test_seal_to_holder_layout_is_unpack(wl):
    pool = W.holder_pool_np(wl)
    t, p, slab = _plan_and_pack(wl.addr, wl.seg_len, wl.numa, wl.pool_bytes, pool)
    B, L = wl.addr.shape
    dst = np.full(wl.pool_bytes, 0xA5, np.uint8)
    assert oracle.seal_blocks(t, p, B, L, wl.seg_len, slab, wl.addr, dst) == 0
    # segment bytes restored, holes keep the canary
    covered = np.zeros(wl.pool_bytes, bool)
    for b in range(B):
        for l in range(L):
            a, n = int(wl.addr[b, l]), int(wl.seg_len[l])
            covered[a:a + n] = True
    assert (dst[covered] == pool[covered]).all()
    assert (dst[~covered] == 0xA5).all()


@pytest.mark.parametrize("seed", [1, 2, 3, 4])
def test_seal_to_receiver_layout_brute_force(seed):
    rng = np.random.default_rng(seed)
    addr, seg_len, numa, pool_bytes = random_holder(rng, 7, 3, 2)
    pool = rng.integers(0, 256, pool_bytes, dtype=np.uint8)
    t, p, slab = _plan_and_pack(addr, seg_len, numa, pool_bytes, pool)
    B, L = addr.shape
    dst_addr, size = _receiver_layout(B, seg_len, lane_major=seed % 2 == 0,
                                      rng=rng if seed > 2 else None)
    dst = np.zeros(size, np.uint8)
    assert oracle.seal_blocks(t, p, B, L, seg_len, slab, dst_addr, dst) == 0
    _segments_match(dst, dst_addr, pool, addr, seg_len)


def test_seal_destination_out_of_range_is_skipped():
    wl = W.CONFIGS["tiny"]()
    pool = W.holder_pool_np(wl)
    t, p, slab = _plan_and_pack(wl.addr, wl.seg_len, wl.numa, wl.pool_bytes, pool)
    B, L = wl.addr.shape
    dst_addr, size = _receiver_layout(B, wl.seg_len)
    dst_addr[2, 5] = size - int(wl.seg_len[5]) + 1      # one byte past the end
    dst = np.zeros(size, np.uint8)
    assert oracle.seal_blocks(t, p, B, L, wl.seg_len, slab, dst_addr, dst) == S_BOUNDS
    for b in range(B):
        for l in range(L):
            if (b, l) == (2, 5):
                continue
            n, d, a = int(wl.seg_len[l]), int(dst_addr[b, l]), int(wl.addr[b, l])
            assert (dst[d:d + n] == pool[a:a + n]).all(), (b, l)


def test_seal_corrupt_group_is_skipped():
    """A group carve moved past the slab: its segments fail the rebuild
    check and are not written; the other group's segments are."""
    wl = W.CONFIGS["tiny"]()
    pool = W.holder_pool_np(wl)
    t, p, slab = _plan_and_pack(wl.addr, wl.seg_len, wl.numa, wl.pool_bytes, pool)
    B, L = wl.addr.shape
    groups = p.groups.copy()
    groups["local"][1] += np.uint64(p.slab_bytes)
    dst_addr, size = _receiver_layout(B, wl.seg_len)
    dst = np.full(size, 0x5A, np.uint8)
    st = oracle.seal_blocks(t, p, B, L, wl.seg_len, slab, dst_addr, dst, groups=groups)
    assert st == S_BOUNDS
    for b in range(B):
        for l in range(L):
            n, d, a = int(wl.seg_len[l]), int(dst_addr[b, l]), int(wl.addr[b, l])
            g = int(p.run_group[int(p.lane_first[l])])
            if g == 1:
                assert (dst[d:d + n] == 0x5A).all()
            else:
                assert (dst[d:d + n] == pool[a:a + n]).all()


# --------------------------------------------------------------- paged writes

def _paged(case, dst=None):
    src = np.arange(case["src_bytes"], dtype=np.uint64).astype(np.uint8)
    if dst is None:
        dst = np.zeros(case["dst_bytes"], np.uint8)
    st = oracle.paged_writes(case["page_len"], src, case["src_idx"], case["src_stride"],
                             case["src_offset"], dst, case["dst_idx"], case["dst_stride"],
                             case["dst_offset"])
    return st, dst


def _golden():
    with open(os.path.join(GOLDEN, "paged_hand.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden(), ids=lambda c: c["name"])
def test_paged_hand_fixtures(case):
    st, dst = _paged(case)
    assert st == case["status"]
    assert dst.tolist() == case["dst"]


@pytest.mark.parametrize("page_len", [1, 16, 4096])
def test_paged_identity_is_memcpy(page_len):
    rng = np.random.default_rng(page_len)
    n = 9
    src = rng.integers(0, 256, n * page_len + 5, dtype=np.uint8)
    dst = np.zeros(n * page_len, np.uint8)
    idx = np.arange(n, dtype=np.uint32)
    assert oracle.paged_writes(page_len, src, idx, page_len, 0, dst, idx, page_len, 0) == 0
    assert (dst == src[:n * page_len]).all()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_paged_matches_fancy_indexing(seed):
    """stride == page_len and offset == 0: page sets are rows of a 2-D view,
    so the paged write is numpy's row gather/scatter."""
    rng = np.random.default_rng(seed)
    page, ns, nd, n = 48, 40, 30, 25
    src = rng.integers(0, 256, ns * page, dtype=np.uint8)
    dst = rng.integers(0, 256, nd * page, dtype=np.uint8)
    s_idx = rng.integers(0, ns, n).astype(np.uint32)
    d_idx = rng.permutation(nd)[:n].astype(np.uint32)
    want = dst.copy().reshape(nd, page)
    want[d_idx] = src.reshape(ns, page)[s_idx]
    assert oracle.paged_writes(page, src, s_idx, page, 0, dst, d_idx, page, 0) == 0
    assert (dst.reshape(nd, page) == want).all()


def test_paged_permutation_round_trip():
    rng = np.random.default_rng(5)
    page, n, stride, off = 24, 50, 40, 8
    src = rng.integers(0, 256, off + n * stride, dtype=np.uint8)
    perm = rng.permutation(n).astype(np.uint32)
    ident = np.arange(n, dtype=np.uint32)
    mid = np.zeros(n * page + 3, np.uint8)
    assert oracle.paged_writes(page, src, ident, stride, off, mid, perm, page, 3) == 0
    out = np.zeros(off + n * stride, np.uint8)
    assert oracle.paged_writes(page, mid, perm, page, 3, out, ident, stride, off) == 0
    for i in range(n):
        a = off + i * stride
        assert (out[a:a + page] == src[a:a + page]).all()


def test_paged_empty():
    src = np.arange(16, dtype=np.uint8)
    dst = np.full(8, 7, np.uint8)
    assert oracle.paged_writes(4, src, [], 4, 0, dst, [], 4, 0) == 0
    assert oracle.paged_writes(0, src, [3, 1], 4, 0, dst, [0, 1], 4, 0) == 0
    assert (dst == 7).all()


# ------------------------------------------------------- zero-size V lanes

def _compressed(wl):
    """The same holder with the V lanes dropped: the bytes a K-only cache
    really has."""
    return (np.ascontiguousarray(wl.addr[:, ::2]), np.ascontiguousarray(wl.seg_len[::2]),
            np.ascontiguousarray(wl.numa[::2]))


def _plan_of(addr, seg_len, numa, pool):
    t = oracle.encode_runs(addr)
    return t, oracle.plan(t, addr.shape[0], seg_len, numa, pool)


K_ONLY = [dict(layout="bump", name="tiny", blocks=8, slots=4, seg=4096, seed=1),
          dict(layout="bump", name="bump_s", blocks=37, slots=24, seg=4096, seed=2),
          dict(layout="worst", blocks=61, slots=18, npos=128, seed=3)]


def _check_k_only_plan(wl, p, t, p2, t2):
    """The plan of a K-only table against the plan of the same table without
    its V lanes: identical reads and slab; the byte-carrying groups equal the
    K-only groups field by field; every empty V run sits in a group of chunk
    0 placed after its node's other groups (so at the end of the node's
    partition); rebuilt K pointers are unchanged and V pointers are empty
    ranges at the end of their node's partition."""
    assert p.status == 0 and p2.status == 0
    for k in ["remote", "local", "len"]:
        assert (p.descs[k] == p2.descs[k]).all(), k
    assert p.slab_bytes == p2.slab_bytes == wl.blocks * int(wl.seg_len.sum())
    full = p.groups[p.groups["chunk"] > 0]
    for k in ["base", "stride", "chunk", "local", "block", "count", "node", "dense"]:
        assert (full[k] == p2.groups[k]).all(), k
    # group order: node ascending, and inside a node the empty groups last
    nodes = p.groups["node"]
    assert (np.diff(nodes.astype(np.int64)) >= 0).all()
    for n in np.unique(nodes):
        sel = p.groups[nodes == n]
        ch = sel["chunk"] == 0
        assert not (ch[:-1] & ~ch[1:]).any()       # no byte-carrying group after an empty one
        part_end = int((sel["local"] + sel["count"].astype(np.uint64) * sel["chunk"]).max())
        assert (sel["local"][ch] == part_end).all()
    # every V run is in an empty group, every K run in a byte-carrying one
    L = wl.lanes
    for l in range(L):
        r0, r1 = int(p.lane_first[l]), int(p.lane_first[l + 1])
        ch = p.groups["chunk"][p.run_group[r0:r1]]
        assert ((ch == 0) == (l % 2 == 1)).all()
    st, local = oracle.rebuild(t, p, wl.blocks, L, wl.seg_len)
    assert st == 0
    _, local2 = oracle.rebuild(t2, p2, wl.blocks, L // 2, wl.seg_len[::2].copy())
    assert (local[:, ::2] == local2).all()
    for l in range(1, L, 2):
        g = p.groups[p.run_group[int(p.lane_first[l])]]
        assert (local[:, l] == g["local"]).all()


@pytest.mark.parametrize("null_v", [False, True])
@pytest.mark.parametrize("kw", K_ONLY, ids=lambda k: k.get("name", k["layout"]))
def test_k_only_plan_is_the_k_lanes_plan(kw, null_v):
    """Empty V segments where the next segment starts (allocation order) or
    at address 0: either way they move no byte and change no read."""
    kw = dict(kw)
    wl = W.k_only(kw.pop("layout"), null_v=null_v, **kw)
    assert (wl.seg_len[1::2] == 0).all()
    t, p = _plan_of(wl.addr, wl.seg_len, wl.numa, wl.pool_bytes)
    a2, s2, n2 = _compressed(wl)
    t2, p2 = _plan_of(a2, s2, n2, wl.pool_bytes)
    _check_k_only_plan(wl, p, t, p2, t2)


def test_k_only_empty_groups_closed_form():
    """Bump-allocated K-only tiny table, V at the next segment: each V lane
    is one run (stride = the block chunk); runs of V lanes are adjacent only
    through zero lengths (V(j) + 0 != V(j+1)), so every V lane is its own
    empty group: 2 + 4 groups, 2 reads."""
    wl = W.k_only("bump", name="tiny", blocks=8, slots=4, seg=4096, seed=1)
    t, p = _plan_of(wl.addr, wl.seg_len, wl.numa, wl.pool_bytes)
    assert p.status == 0
    assert p.groups.size == 6 and p.descs.size == 2
    assert list(p.groups["chunk"]) == [8192, 0, 0, 8192, 0, 0]
    assert list(p.groups["local"]) == [0, 65536, 65536, 65536, 131072, 131072]


def test_zero_size_k_still_rejected():
    wl = W.k_only("bump", name="tiny", blocks=8, slots=4, seg=4096, seed=1)
    t = oracle.encode_runs(wl.addr)
    sl = wl.seg_len.copy()
    sl[4] = 0                                      # K of slot 2
    assert oracle.plan(t, wl.blocks, sl, wl.numa, wl.pool_bytes).status == 16


def test_k_only_pack_moves_only_k_bytes():
    wl = W.k_only("worst", blocks=23, slots=6, npos=64, seed=9)
    t, p = _plan_of(wl.addr, wl.seg_len, wl.numa, wl.pool_bytes)
    pool = W.holder_pool_np(wl)
    slab = np.zeros(p.slab_bytes, np.uint8)
    assert oracle.pack(pool, p.descs, slab) == 0
    dst = np.full(wl.pool_bytes, 0xA5, np.uint8)
    assert oracle.unpack(slab, p.descs, dst) == 0
    covered = np.zeros(wl.pool_bytes, bool)
    for b in range(wl.blocks):
        for l in range(0, wl.lanes, 2):
            covered[int(wl.addr[b, l]):int(wl.addr[b, l]) + int(wl.seg_len[l])] = True
    assert (dst[covered] == pool[covered]).all() and (dst[~covered] == 0xA5).all()
