"""kvx_pack_noalloc: the pack entry point for callers that cannot allocate
device memory, whose scratch is a static array inside libkvx.

Called through the C ABI on several transfers in a row (so every call after
the first runs on scratch an earlier call left behind).  Each result is
compared byte for byte with the oracle's pack of the same holder bytes along
the oracle's own plan, and with kvx_pack given a caller workspace.  The
layouts cover the scratch's two regimes: slabs whose piece list fits in the
array (shared tiles on the bulk-copy rings) and a 377 MB scattered slab past
that limit (shared tiles on the register path).  This file is collected last
on purpose; it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_kvx_gb300 import kvx, workloads as W

pytestmark = pytest.mark.gpu

TILE = 64 * 1024
# tiles whose piece list still fits in the 4 MiB scratch: per tile 4 + 24 + 4
# bytes of lists plus 33 pieces of 24 bytes
PIECE_LIMIT_TILES = (4 << 20) // (32 + 33 * 24)


def _planned(wl):
    tr = kvx.Transfer(wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    tr.set_addr(wl.addr)
    tr.encode()
    tr.plan()
    pool = torch.empty(wl.pool_bytes, dtype=torch.uint8, device="cuda")
    W.fill_pool_torch(pool, wl.seed)
    torch.cuda.synchronize()
    assert tr.read_status() == 0
    return tr, pool


def _oracle_slab(wl, pool):
    t = oracle.encode_runs(wl.addr)
    p = oracle.plan(t, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    assert p.status == 0
    want = np.zeros(p.slab_bytes, dtype=np.uint8)
    assert oracle.pack(pool.cpu().numpy(), p.descs, want) == 0
    return want


def test_pack_noalloc_matches_oracle_and_pack_on_calls_in_a_row():
    layouts = (
        # a scattered layout: bulk-copy tiles and shared tiles, piece list in the scratch
        W.worst(blocks=61, slots=18, npos=128, seed=3),
        # 160 x 288 x 2 x 4 KiB = 377 MB = 5760 tiles of per-segment reads:
        # past the piece-list limit, shared tiles take the register path
        W.worst(blocks=160, slots=288, npos=368, seed=13),
        # a dense layout: one read per NUMA region
        W.bump("noalloc_dense", blocks=40, slots=24, seg=4096, seed=8),
    )
    tiles = [-(-wl.payload_bytes // TILE) for wl in layouts]
    assert tiles[0] <= PIECE_LIMIT_TILES < tiles[1]
    for wl in layouts:
        tr, pool = _planned(wl)
        want = _oracle_slab(wl, pool)
        assert want.size == tr.slab_bytes
        ws_slab = torch.zeros(tr.slab_bytes, dtype=torch.uint8, device="cuda")
        tr.pack(pool, ws_slab)
        got = torch.full((tr.slab_bytes,), 0x5A, dtype=torch.uint8, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        kvx.kvx_pack_noalloc(pool, pool.numel(), tr.descs, tr.counts[1:], tr.desc_cap, got,
                             got.numel(), status)
        torch.cuda.synchronize()
        assert tr.read_status() == 0
        assert int(status.item()) == 0
        got_np = got.cpu().numpy()
        assert np.array_equal(got_np, want), wl.name
        assert np.array_equal(ws_slab.cpu().numpy(), got_np), wl.name
        del tr, pool, ws_slab, got
        torch.cuda.empty_cache()


def test_pack_noalloc_rejects_a_slab_beyond_its_scratch():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dummy = torch.zeros(64, dtype=torch.uint8, device="cuda")
    n = torch.zeros(1, dtype=torch.int64, device="cuda")
    with pytest.raises(kvx.KvxError, match="KVX_ECAPACITY"):
        kvx.kvx_pack_noalloc(dummy, 64, dummy, n, 1, dummy, 64 << 30, status)
