"""kvx_pack_noalloc: the pack entry point for callers that cannot allocate
device memory, whose scratch is a static array inside libkvx.

Called through the C ABI, twice in a row on different transfers (so the
second call runs on scratch the first one left behind), each result compared
byte for byte with kvx_pack given a caller workspace.  This file is collected
last on purpose; it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_kvx_gb300 import kvx, workloads as W

pytestmark = pytest.mark.gpu


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


def test_pack_noalloc_matches_pack_on_two_calls_in_a_row():
    # a mixed layout (bulk-copy tiles and vector tiles) then a dense one
    for wl in (W.worst(blocks=61, slots=18, npos=128, seed=3),
               W.bump("noalloc_dense", blocks=40, slots=24, seg=4096, seed=8)):
        tr, pool = _planned(wl)
        want = torch.zeros(tr.slab_bytes, dtype=torch.uint8, device="cuda")
        tr.pack(pool, want)
        got = torch.full((tr.slab_bytes,), 0x5A, dtype=torch.uint8, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        kvx.kvx_pack_noalloc(pool, pool.numel(), tr.descs, tr.counts[1:], tr.desc_cap, got,
                             got.numel(), status)
        torch.cuda.synchronize()
        assert tr.read_status() == 0
        assert int(status.item()) == 0
        assert torch.equal(got, want)


def test_pack_noalloc_rejects_a_slab_beyond_its_scratch():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dummy = torch.zeros(64, dtype=torch.uint8, device="cuda")
    n = torch.zeros(1, dtype=torch.int64, device="cuda")
    with pytest.raises(kvx.KvxError, match="KVX_ECAPACITY"):
        kvx.kvx_pack_noalloc(dummy, 64, dummy, n, 1, dummy, 64 << 30, status)
