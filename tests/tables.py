"""Seeded random address tables for tests (inputs only; no method arithmetic)."""
import numpy as np


def random_holder(rng, B, slots, nodes):
    """Holder with random block placement and random per-block lane gaps:
    non-dense groups, chunk-outgrows-stride cuts and negative strides all
    occur.  Returns addr [B, L], seg_len, numa, pool_bytes."""
    L = 2 * slots
    seg = int(rng.choice([16, 32, 48]))
    numa = rng.integers(0, nodes, size=L).astype(np.uint32)
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


def random_lanes(rng, B, L, max_addr=2**40, seg=64):
    """Unstructured addresses: nearly every run is a pair."""
    addr = rng.integers(0, max_addr, size=(B, L), dtype=np.uint64) // np.uint64(seg) * np.uint64(seg)
    numa = rng.integers(0, 3, size=L).astype(np.uint32) * np.uint32(0x01010101)
    return addr, np.full(L, seg, np.uint32), numa, max_addr + seg
