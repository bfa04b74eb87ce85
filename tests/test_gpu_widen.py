"""CUDA path vs the CPU oracle for the widening calls: kvx_paged_writes
(paged writes by page indices) and kvx_seal_blocks (seal from template
metadata).  Byte data and status words: bit-exact."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_kvx_gb300 import kvx, workloads as W
from conftest import GOLDEN
from gpu_helpers import assert_equal_chunked, gpu_plan, host_generator_bytes
from tables import random_holder, random_holder_large

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _u32_dev(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.uint32))
    return _dev(a.view(np.int32) if a.size else np.zeros(1, np.int32))


# --------------------------------------------------------------- paged writes

def _seg_ws():
    return torch.zeros(kvx.kvx_segcopy_workspace_size(), dtype=torch.uint8, device="cuda")


def gpu_paged(page_len, src, s_idx, s_stride, s_off, dst, d_idx, d_stride, d_off, bulk=True):
    """Run kvx_paged_writes on copies of the host buffers; returns (status, dst)."""
    dsrc = _dev(src if src.size else np.zeros(1, np.uint8))
    ddst = _dev(dst if dst.size else np.zeros(1, np.uint8))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    n = len(s_idx)
    kvx.kvx_paged_writes(page_len, dsrc, src.size, _u32_dev(s_idx), s_stride, s_off, ddst,
                         dst.size, _u32_dev(d_idx), d_stride, d_off, n, status,
                         _seg_ws() if bulk else None)
    torch.cuda.synchronize()
    return int(status.cpu().numpy().view(np.uint32)[0]), ddst.cpu().numpy()[: dst.size]


def check_paged(page_len, src, s_idx, s_stride, s_off, dst, d_idx, d_stride, d_off):
    """Both copy paths (bulk-copy ring and registers) against the oracle."""
    want = dst.copy()
    st_o = oracle.paged_writes(page_len, src, s_idx, s_stride, s_off, want, d_idx, d_stride, d_off)
    for bulk in (True, False):
        st_g, got = gpu_paged(page_len, src, s_idx, s_stride, s_off, dst, d_idx, d_stride, d_off,
                              bulk)
        assert st_g == st_o, bulk
        assert np.array_equal(got, want), bulk
    return st_o


def _golden():
    with open(os.path.join(GOLDEN, "paged_hand.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("bulk", [True, False])
@pytest.mark.parametrize("case", _golden(), ids=lambda c: c["name"])
def test_paged_hand_fixtures_on_gpu(case, bulk):
    src = np.arange(case["src_bytes"], dtype=np.uint64).astype(np.uint8)
    dst = np.zeros(case["dst_bytes"], np.uint8)
    st, got = gpu_paged(case["page_len"], src, case["src_idx"], case["src_stride"],
                        case["src_offset"], dst, case["dst_idx"], case["dst_stride"],
                        case["dst_offset"], bulk)
    assert st == case["status"]
    assert got.tolist() == case["dst"]


# page_len, source offset, destination offset: aligned flat path, the
# uniform-length shortcut, long (> 64 KiB) segments, unaligned lengths and
# addresses (byte path)
PAGED_SHAPES = [
    (16, 0, 0), (48, 16, 32), (512, 0, 4096), (4096, 0, 0), (4096, 64, 128),
    (1024, 0, 0), (2048, 16, 0), (65536, 0, 0), (65552, 16, 0), (131072, 0, 65536),
    (4100, 0, 0), (4096, 3, 0),
    (4096, 0, 5), (1, 7, 9), (33, 1, 2),
]


@pytest.mark.parametrize("page_len,s_off,d_off", PAGED_SHAPES)
def test_paged_random_bit_exact(page_len, s_off, d_off):
    rng = np.random.default_rng(page_len * 131 + s_off * 7 + d_off)
    n = int(min(700, max(40, (24 << 20) // max(page_len, 1) // 4)))
    n += 13  # a ragged last batch of 32 pages
    ns, nd = 2 * n + 5, n + 9
    s_stride = page_len + int(rng.choice([0, 16, 4096])) * (page_len % 16 == 0)
    d_stride = page_len + int(rng.choice([0, 32])) * (page_len % 16 == 0)
    src = rng.integers(0, 256, s_off + ns * s_stride + page_len, dtype=np.uint8)
    dst = rng.integers(0, 256, d_off + nd * d_stride + page_len, dtype=np.uint8)
    s_idx = rng.integers(0, ns, n).astype(np.uint32)
    d_idx = rng.permutation(nd)[:n].astype(np.uint32)
    assert check_paged(page_len, src, s_idx, s_stride, s_off, dst, d_idx, d_stride, d_off) == 0


def test_paged_out_of_range_pages_mixed():
    """Pages past either end are skipped with their bit; the rest copy (the
    flat path's general search over batches with holes)."""
    rng = np.random.default_rng(11)
    page, n = 256, 1000
    src = rng.integers(0, 256, 600 * page, dtype=np.uint8)
    dst = rng.integers(0, 256, 1200 * page, dtype=np.uint8)
    s_idx = rng.integers(0, 640, n).astype(np.uint32)          # some past the source
    d_idx = rng.permutation(1300)[:n].astype(np.uint32)         # some past the destination
    st = check_paged(page, src, s_idx, page, 0, dst, d_idx, page, 0)
    assert st == oracle.S_SPAN | oracle.S_BOUNDS


def test_paged_wrapping_address_rejected():
    src = np.arange(64, dtype=np.uint8)
    dst = np.zeros(64, np.uint8)
    st = check_paged(4, src, [0xFFFFFFFF, 1], 1 << 63, 1 << 63, dst, [0, 1], 4, 0)
    assert st == oracle.S_SPAN


def test_paged_empty():
    src = np.arange(64, dtype=np.uint8)
    dst = np.full(64, 3, np.uint8)
    assert check_paged(16, src, [], 16, 0, dst, [], 16, 0) == 0
    assert check_paged(0, src, [1, 2], 16, 0, dst, [0, 1], 16, 0) == 0


@pytest.mark.parametrize("bulk", [True, False])
def test_paged_full_size(bulk):
    """The benchmark's paged workload (576,000 pages of 4 KiB, 2250 MiB moved
    between two page pools by permuted page tables): every byte of the
    destination pool compared with the oracle's paged write of the same
    source bytes into a canary-filled pool."""
    wl = W.paged_default()
    src = torch.empty(wl.src_bytes, dtype=torch.uint8, device="cuda")
    W.fill_pool_torch(src, wl.seed)
    dst = torch.full((wl.dst_bytes,), W.CANARY, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvx.kvx_paged_writes(wl.page_len, src, wl.src_bytes, _u32_dev(wl.src_idx), wl.src_stride,
                         wl.src_offset, dst, wl.dst_bytes, _u32_dev(wl.dst_idx), wl.dst_stride,
                         wl.dst_offset, wl.num_pages, status, _seg_ws() if bulk else None)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    host_src = host_generator_bytes(src, wl.seed)
    del src
    want = np.full(wl.dst_bytes, W.CANARY, dtype=np.uint8)
    assert oracle.paged_writes(wl.page_len, host_src, wl.src_idx, wl.src_stride, wl.src_offset,
                               want, wl.dst_idx, wl.dst_stride, wl.dst_offset) == 0
    del host_src
    assert_equal_chunked(dst, want)


# -------------------------------------------------------------------- seal

def receiver_layout(B, seg_len, rng=None, lane_major=True):
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


def check_seal(addr, B, seg_len, numa, pool_bytes, dst_addr, dst_bytes, groups=None, slab_bytes=None):
    """Plan on the GPU (itself bit-exact with the oracle), pack the oracle's
    slab, then seal on both sides from the same inputs."""
    L = addr.shape[1]
    t = oracle.encode_runs(addr)
    p = oracle.plan(t, B, seg_len, numa, pool_bytes)
    assert p.status == 0
    host_pool = W.pool_bytes_np(77, 0, pool_bytes)
    slab = np.zeros(max(1, p.slab_bytes), np.uint8)
    assert oracle.pack(host_pool, p.descs, slab[: p.slab_bytes]) == 0
    tr = gpu_plan(addr, B, seg_len, numa, pool_bytes)
    assert tr.read_status() == 0
    if groups is not None:
        tr.groups[: groups.nbytes].copy_(torch.from_numpy(groups.view(np.uint8).copy()))
    sb = p.slab_bytes if slab_bytes is None else slab_bytes
    want = np.full(max(1, dst_bytes), 0xA5, np.uint8)
    st_o = oracle.seal_blocks(t, p, B, L, seg_len, slab, dst_addr, want[:dst_bytes],
                              groups=groups, slab_bytes=sb)
    dslab = _dev(slab)
    daddr = _dev(np.ascontiguousarray(dst_addr, np.uint64).view(np.int64).reshape(-1))
    for bulk in (True, False):
        ddst = torch.full((max(1, dst_bytes),), 0xA5, dtype=torch.uint8, device="cuda")
        tr.status.zero_()
        kvx.kvx_seal_blocks(tr.lane_first, tr.run_block, tr.run_base, tr.run_stride, tr.run_group,
                            tr.run_cap, tr.groups, tr.group_cap, tr.counts, B, L, tr.seg_len, dslab,
                            sb, daddr, ddst, dst_bytes, tr.status, _seg_ws() if bulk else None)
        torch.cuda.synchronize()
        assert tr.read_status() == st_o, bulk
        assert np.array_equal(ddst.cpu().numpy(), want), bulk
    return st_o


@pytest.mark.parametrize("wl", W.small_variants(), ids=lambda w: w.name)
@pytest.mark.parametrize("layout", ["holder", "lane_major", "permuted"])
def test_seal_small_variants_bit_exact(wl, layout):
    B, L = wl.addr.shape
    if layout == "holder":
        dst_addr, size = wl.addr, wl.pool_bytes
    else:
        rng = np.random.default_rng(B * L)
        dst_addr, size = receiver_layout(B, wl.seg_len, rng if layout == "permuted" else None)
    assert check_seal(wl.addr, B, wl.seg_len, wl.numa, wl.pool_bytes, dst_addr, size) == 0


def test_seal_random_holders_bit_exact():
    rng = np.random.default_rng(99)
    for _ in range(25):
        B = int(rng.integers(1, 30))
        addr, seg_len, numa, pool = random_holder(rng, B, int(rng.integers(1, 9)), int(rng.integers(1, 4)))
        dst_addr, size = receiver_layout(B, seg_len, rng, lane_major=bool(rng.integers(0, 2)))
        assert check_seal(addr, B, seg_len, numa, pool, dst_addr, size) == 0


def test_seal_long_segments_in_rounds():
    """64 KiB and 20 KiB segments: the bulk path moves them in 16 KiB rounds."""
    B, slots = 9, 3
    L = 2 * slots
    seg_len = np.array([65536, 20480] * slots, np.uint32)
    per_block = int(seg_len.sum())
    addr = np.zeros((B, L), np.uint64)
    for b in range(B):
        addr[b] = b * per_block + np.concatenate([[0], np.cumsum(seg_len)[:-1]])
    numa = np.zeros(L, np.uint32)
    dst_addr, size = receiver_layout(B, seg_len, np.random.default_rng(5))
    assert check_seal(addr, B, seg_len, numa, B * per_block, dst_addr, size) == 0


def test_seal_per_lane_lengths():
    """K and V of different sizes (64 B and 48 B) and an odd-length lane:
    lengths differ inside one warp batch (the flat path's search) and some
    segments take the byte path."""
    B, slots = 45, 7
    L = 2 * slots
    seg_len = np.array([64, 48] * slots, np.uint32)
    seg_len[5] = 21
    addr = np.zeros((B, L), np.uint64)
    per_block = int(seg_len.sum())
    for b in range(B):
        addr[b] = b * per_block + np.concatenate([[0], np.cumsum(seg_len)[:-1]])
    numa = np.array([0] * slots + [1] * slots, np.uint32)
    rng = np.random.default_rng(3)
    dst_addr, size = receiver_layout(B, seg_len, rng)
    assert check_seal(addr, B, seg_len, numa, B * per_block, dst_addr, size) == 0


def test_seal_destination_out_of_range():
    wl = W.tiny()
    B, L = wl.addr.shape
    dst_addr, size = receiver_layout(B, wl.seg_len)
    dst_addr[3, 2] = size - 10
    dst_addr[6, 7] = 2**63
    assert check_seal(wl.addr, B, wl.seg_len, wl.numa, wl.pool_bytes, dst_addr, size) == oracle.S_BOUNDS


def test_seal_corrupt_groups():
    wl = {v.name: v for v in W.small_variants()}["default_s"]
    B, L = wl.addr.shape
    p = oracle.plan(oracle.encode_runs(wl.addr), B, wl.seg_len, wl.numa, wl.pool_bytes)
    groups = p.groups.copy()
    groups["local"][1] += np.uint64(p.slab_bytes)           # carve past the slab
    groups["count"][0] -= np.uint32(1)                      # block range too short
    dst_addr, size = receiver_layout(B, wl.seg_len)
    assert check_seal(wl.addr, B, wl.seg_len, wl.numa, wl.pool_bytes, dst_addr, size,
                      groups=groups) == oracle.S_BOUNDS


def test_seal_group_block_moved():
    """A group whose first block no longer matches its runs' first block: every
    segment of its runs is rejected, as in the oracle's seal."""
    wl = {v.name: v for v in W.small_variants()}["default_s"]
    B, L = wl.addr.shape
    p = oracle.plan(oracle.encode_runs(wl.addr), B, wl.seg_len, wl.numa, wl.pool_bytes)
    groups = p.groups.copy()
    groups["block"][0] += np.uint32(1)
    dst_addr, size = receiver_layout(B, wl.seg_len)
    assert check_seal(wl.addr, B, wl.seg_len, wl.numa, wl.pool_bytes, dst_addr, size,
                      groups=groups) == oracle.S_BOUNDS


@pytest.mark.parametrize("kind", ["dense", "nondense"])
def test_seal_group_stride_altered(kind):
    """The stride field of one group altered: on a dense group it takes no
    part in the page's formula (same bytes, no error); on a non-dense group
    the blocks after its first leave their slices.  Both copy paths match the
    oracle's seal, byte for byte and in the status word."""
    wl = {v.name: v for v in W.small_variants()}["default_s" if kind == "dense" else "worst"]
    B, L = wl.addr.shape
    p = oracle.plan(oracle.encode_runs(wl.addr), B, wl.seg_len, wl.numa, wl.pool_bytes)
    groups = p.groups.copy()
    sel = (groups["count"] > 1) & (groups["dense"] == (1 if kind == "dense" else 0))
    if kind == "nondense":
        sel &= groups["stride"] > 0
    k = int(np.flatnonzero(sel)[0])
    groups["stride"][k] += 4096
    dst_addr, size = receiver_layout(B, wl.seg_len)
    want = 0 if kind == "dense" else oracle.S_BOUNDS
    assert check_seal(wl.addr, B, wl.seg_len, wl.numa, wl.pool_bytes, dst_addr, size,
                      groups=groups) == want


@pytest.mark.parametrize("bulk", [True, False])
def test_seal_full_size_default(bulk):
    """The default workload end to end on the device: pack, then seal into a
    lane-major receiver layout; every byte of the destination compared with
    the oracle's seal of the oracle's slab (the oracle's pack of the same
    holder bytes along the oracle's plan)."""
    wl = W.default()
    B, L = wl.addr.shape
    seg = int(wl.seg_len[0])
    t = oracle.encode_runs(wl.addr)
    p = oracle.plan(t, B, wl.seg_len, wl.numa, wl.pool_bytes)
    assert p.status == 0
    tr = gpu_plan(wl.addr, B, wl.seg_len, wl.numa, wl.pool_bytes)
    assert tr.read_status() == 0
    pool = torch.empty(wl.pool_bytes, dtype=torch.uint8, device="cuda")
    W.fill_pool_torch(pool, wl.seed)
    slab = torch.empty(tr.slab_bytes, dtype=torch.uint8, device="cuda")
    tr.pack(pool, slab)
    dst_addr_np = ((np.arange(L, dtype=np.uint64)[None, :] * np.uint64(B)
                    + np.arange(B, dtype=np.uint64)[:, None]) * np.uint64(seg))
    dst_addr = torch.from_numpy(dst_addr_np.view(np.int64).reshape(-1).copy()).cuda()
    dst = torch.full((B * L * seg,), W.CANARY, dtype=torch.uint8, device="cuda")
    tr.seal(slab, dst_addr, dst, bulk=bulk)
    torch.cuda.synchronize()
    assert tr.read_status() == 0
    host_pool = host_generator_bytes(pool, wl.seed)
    del pool, slab
    want_slab = np.empty(p.slab_bytes, dtype=np.uint8)
    assert oracle.pack(host_pool, p.descs, want_slab) == 0
    del host_pool
    want = np.full(B * L * seg, W.CANARY, dtype=np.uint8)
    assert oracle.seal_blocks(t, p, B, L, wl.seg_len, want_slab, dst_addr_np, want) == 0
    del want_slab
    assert_equal_chunked(dst, want)


# ------------------------------------------------------------ verify + encode

def gpu_verify_encode(addr, size, tmpl):
    B, L = addr.shape
    pool = int(addr.max()) + int(np.max(tmpl)) + 1 if addr.size else 1
    tr = kvx.Transfer(B, tmpl, np.zeros(L, np.uint32), pool)
    tr.set_addr(addr)
    prefix = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    dsize = _u32_dev(np.ascontiguousarray(size, np.uint32).reshape(-1))
    tr.status.zero_()
    tr.verify_encode(dsize, prefix)
    torch.cuda.synchronize()
    assert tr.read_status() == 0
    return int(prefix.item()), tr


def check_verify(addr, size, tmpl):
    pre_o, t = oracle.verify_encode(addr, size, tmpl)
    pre_g, tr = gpu_verify_encode(addr, size, tmpl)
    assert pre_g == pre_o
    rpl, base, stride, count = tr.read_table()
    assert np.array_equal(rpl, t.runs_per_lane)
    assert np.array_equal(base, t.run_base)
    assert np.array_equal(stride, t.run_stride)
    assert np.array_equal(count, t.run_count)
    return pre_o


@pytest.mark.parametrize("wl", W.small_variants(), ids=lambda w: w.name)
def test_verify_encode_small_variants(wl):
    B, L = wl.addr.shape
    size = np.tile(wl.seg_len, (B, 1))
    assert check_verify(wl.addr, size, wl.seg_len) == B
    rng = np.random.default_rng(B + L)
    for _ in range(4):  # one mismatching segment somewhere: the prefix ends there
        b, l = int(rng.integers(0, B)), int(rng.integers(0, L))
        s2 = size.copy()
        s2[b, l] += 1
        if rng.random() < 0.5 and b + 1 < B:
            s2[int(rng.integers(b + 1, B)), int(rng.integers(0, L))] = 0  # later ones do not matter
        assert check_verify(wl.addr, s2, wl.seg_len) == b


def test_verify_encode_tile_edges():
    """Mismatches on every boundary the kernel cuts at (thread slices, row
    tiles, the ragged last tile) of a table that spans many tiles."""
    rng = np.random.default_rng(8)
    B, L = 2100, 70
    addr = rng.integers(0, 1 << 30, (B, L), dtype=np.uint64)
    addr[:, ::3] = (np.arange(B, dtype=np.uint64) * np.uint64(4096))[:, None]
    tmpl = np.full(L, 64, np.uint32)
    for b in [0, 1, 2, 7, 8, 63, 64, 65, 511, 512, 513, 1024, 2047, 2048, 2099]:
        size = np.tile(tmpl, (B, 1))
        size[b, int(rng.integers(0, L))] = 65
        assert check_verify(addr, size, tmpl) == b


def test_verify_encode_tall_table():
    """A table of far more row tiles than lanes (the spread lane scan) with a
    ragged last lane tile: the template check cuts it in the middle, and the
    prefix is run-encoded as the oracle encodes it."""
    rng = np.random.default_rng(30011)
    B, L = 30011, 40
    addr = rng.integers(0, 1 << 30, (B, L), dtype=np.uint64)
    addr[:, ::2] = (np.arange(B, dtype=np.uint64) * np.uint64(8192))[:, None] + np.uint64(64)
    tmpl = np.full(L, 64, np.uint32)
    for b in [17777, B - 1]:
        size = np.tile(tmpl, (B, 1))
        size[b, 37] = 0
        assert check_verify(addr, size, tmpl) == b


def test_verify_encode_full_size_default():
    wl = W.default()
    B, L = wl.addr.shape
    size = np.tile(wl.seg_len, (B, 1))
    size[700, 301] = 2048
    assert check_verify(wl.addr, size, wl.seg_len) == 700


# ------------------------------------------------------- zero-size V lanes

from gpu_helpers import check_all  # noqa: E402

K_ONLY_GPU = [
    dict(layout="bump", name="tiny", blocks=8, slots=4, seg=4096, seed=1),
    dict(layout="bump", name="bump_s", blocks=37, slots=24, seg=4096, seed=2),
    dict(layout="worst", blocks=61, slots=18, npos=128, seed=3),        # single-block planner
    dict(layout="worst", blocks=301, slots=40, npos=512, seed=4),       # cooperative planner
]


@pytest.mark.parametrize("null_v", [False, True])
@pytest.mark.parametrize("kw", K_ONLY_GPU, ids=lambda k: f'{k["layout"]}_{k["blocks"]}')
def test_k_only_bit_exact(kw, null_v):
    kw = dict(kw)
    wl = W.k_only(kw.pop("layout"), null_v=null_v, **kw)
    tr, t, p, local = check_all(wl.addr, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    assert (p.groups["chunk"] == 0).any()


@pytest.mark.parametrize("kw", K_ONLY_GPU[1:], ids=lambda k: f'{k["layout"]}_{k["blocks"]}')
def test_k_only_seal_bit_exact(kw):
    kw = dict(kw)
    wl = W.k_only(kw.pop("layout"), **kw)
    B, L = wl.addr.shape
    dst_addr, size = receiver_layout(B, wl.seg_len, np.random.default_rng(B))
    assert check_seal(wl.addr, B, wl.seg_len, wl.numa, wl.pool_bytes, dst_addr, size) == 0


@pytest.mark.parametrize("kw", [K_ONLY_GPU[0], K_ONLY_GPU[3]], ids=["small", "cooperative"])
def test_zero_size_k_rejected_on_gpu(kw):
    kw = dict(kw)
    wl = W.k_only(kw.pop("layout"), **kw)
    sl = wl.seg_len.copy()
    sl[2] = 0
    t = oracle.encode_runs(wl.addr)
    assert oracle.plan(t, wl.blocks, sl, wl.numa, wl.pool_bytes).status == oracle.S_ZERO_LEN
    tr = kvx.Transfer(wl.blocks, sl, wl.numa, wl.pool_bytes)
    tr.set_addr(wl.addr)
    tr.encode()
    tr.plan()
    torch.cuda.synchronize()
    assert tr.read_status() == oracle.S_ZERO_LEN
    assert tr.read_counts() == (0, 0, 0)


@pytest.mark.parametrize("layout", ["bump", "worst"])
def test_k_only_full_size(layout):
    """The default and worst shapes as K-only caches (288 slots, V lanes of
    size 0): every run-table, plan and rebuild array bit-exact."""
    wl = W.k_only(layout)
    check_all(wl.addr, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes, data=False)


# ------------------------------------------------------------ fuzz

@pytest.mark.parametrize("seed", range(10))
def test_seal_and_verify_random_large_holders(seed):
    """Seeded large holders (as in the parity fuzz): the seal into a permuted
    receiver layout on both copy paths, and the template check with a size
    mismatch planted at a seeded block, both equal the oracle's."""
    rng = np.random.default_rng(7000 + seed)
    addr, seg_len, numa, pool = random_holder_large(rng, max_bytes=32 << 20)
    B, L = addr.shape
    dst_addr, size = receiver_layout(B, seg_len, rng)
    assert check_seal(addr, B, seg_len, numa, pool, dst_addr, size) == 0
    sizes = np.tile(seg_len, (B, 1))
    b = int(rng.integers(0, B))
    sizes[b, int(rng.integers(0, L))] += 16
    assert check_verify(addr, sizes, seg_len) == b
