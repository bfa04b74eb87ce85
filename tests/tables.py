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


def random_holder_large(rng, max_bytes=96 << 20):
    """A holder big enough for the cooperative planner and every copy path:
    a few hundred to a few thousand blocks of 8-64 slots, segments of 512 B to
    8 KiB (K and V may differ; V may be 0 B, a K-only cache), slots split over
    1-3 NUMA regions, blocks bump-allocated per region with a random share
    moved to spill positions, or fully permuted.  Returns addr [B, L],
    seg_len, numa, pool_bytes."""
    slots = int(rng.choice([8, 16, 24, 64]))
    L = 2 * slots
    k_seg = int(rng.choice([512, 2048, 4096, 8192]))
    v_seg = 0 if rng.random() < 0.2 else int(rng.choice([k_seg, 512, 4096]))
    seg_len = np.array([k_seg, v_seg] * slots, dtype=np.uint32)
    per_block = int(seg_len.sum())
    B = int(max(4, min(4000, max_bytes // max(per_block, 1) // 2)))
    B = int(rng.integers(B // 2, B + 1))
    nodes = int(rng.integers(1, 4))
    cut = np.sort(rng.choice(np.arange(1, slots), size=min(nodes - 1, slots - 1), replace=False))
    bounds = [0] + [int(c) for c in cut] + [slots]
    numa = np.zeros(L, dtype=np.uint32)
    addr = np.zeros((B, L), dtype=np.uint64)
    base = 0
    for r in range(len(bounds) - 1):
        s0, s1 = bounds[r], bounds[r + 1]
        lanes = range(2 * s0, 2 * s1)
        numa[list(lanes)] = r
        chunk = int(seg_len[2 * s0: 2 * s1].sum())
        if rng.random() < 0.3:
            pos = rng.permutation(2 * B)[:B]
        else:
            pos = np.arange(B)
            moved = rng.random(B) < rng.choice([0.0, 0.05, 0.3])
            pos[moved] = B + np.arange(int(moved.sum()))
        for b in range(B):
            off = base + int(pos[b]) * chunk
            for l in lanes:
                addr[b, l] = off
                off += int(seg_len[l])
        base += (2 * B + 1) * chunk
    return addr, seg_len, numa, base
