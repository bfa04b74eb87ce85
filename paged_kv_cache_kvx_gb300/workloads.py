"""Seeded synthetic inputs for the paged KV block-transfer path.

This module only builds inputs: a holder's per-segment address table, the slot
template (segment length and NUMA node of every lane), the holder pool size and
the payload bytes.  It holds none of the transfer method's arithmetic (no run
detection, grouping, carving or copying), so both the CPU oracle and the CUDA
path may take their inputs from here.

Layout (pegaflow PR #350 "run-encode QueryBlocksForTransfer addresses",
Problem section): a *lane* is one slot's K or V segment followed across the
block prefix; lane ``l = 2*slot + kv`` (kv 0 = K, 1 = V).  The table is
block-major: ``addr[b, l]`` is the holder-pool byte offset of block ``b``'s
segment in lane ``l``.  Slots are split into NUMA regions; inside one block,
the segments of a region's slots are back to back (same page, same section:
"within a block, all slots on the same NUMA node are contiguous").

Holder placement: region ``r`` owns a contiguous part of the pool of
``npos_r`` block positions of ``chunk_r = 2 * slots_r * seg`` bytes each; block
``b`` sits at position ``pos_r(b)``:

    addr(b, slot, kv) = region_base(r) + pos_r(b) * chunk_r
                        + ((slot - first_slot_r) * 2 + kv) * seg

Payload: the holder pool, read as little-endian uint64 words, holds
``splitmix64(seed ^ word_index)`` (Steele, Lea and Flood, "Fast Splittable
Pseudorandom Number Generators", OOPSLA 2014; the finaliser constants below are
the published ones).  A destination pool starts filled with the canary byte
0xA5, so bytes outside segments can be checked after an unpack.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

CANARY = 0xA5
KIB = 1024
MIB = 1024 * 1024

_SM_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_SM_MUL1 = np.uint64(0xBF58476D1CE4E5B9)
_SM_MUL2 = np.uint64(0x94D049BB133111EB)


@dataclass
class Workload:
    """One synthetic holder: address table, slot template and pool size."""

    name: str
    blocks: int                 # B, blocks in the prefix
    slots: int                  # slots per block; lanes L = 2 * slots
    seg: int                    # bytes per segment (every lane)
    addr: np.ndarray            # uint64 [B, L], block-major
    seg_len: np.ndarray         # uint32 [L]
    numa: np.ndarray            # uint32 [L]
    pool_bytes: int             # holder pool size in bytes
    seed: int                   # payload seed
    regions: list = field(default_factory=list)  # (first_slot, nslots, base, npos) per region
    pos: list = field(default_factory=list)      # per-region block positions (np.int64 [B])

    @property
    def lanes(self) -> int:
        return 2 * self.slots

    @property
    def segments(self) -> int:
        return self.blocks * self.lanes

    @property
    def payload_bytes(self) -> int:
        """N: the bytes a pack moves (sum of all segment lengths)."""
        return int(self.blocks) * int(self.seg_len.astype(np.uint64).sum())


def _build(name, blocks, slots, seg, region_slots, positions, npos, seed, v_seg=None):
    """Assemble a Workload from per-region slot ranges and block positions.
    v_seg (default seg) is the V segment length; 0 gives a K-only cache whose
    empty V segments sit where the next segment starts."""
    v_seg = seg if v_seg is None else v_seg
    L = 2 * slots
    addr = np.zeros((blocks, L), dtype=np.uint64)
    numa = np.zeros(L, dtype=np.uint32)
    regions = []
    base = 0
    for r, (first, nslots) in enumerate(region_slots):
        chunk = nslots * (seg + v_seg)
        pos = np.asarray(positions[r], dtype=np.uint64)
        lanes = np.arange(2 * first, 2 * (first + nslots))
        j = (lanes - 2 * first) // 2
        within = (j * (seg + v_seg) + (lanes % 2) * seg).astype(np.uint64)
        addr[:, lanes] = (np.uint64(base) + pos[:, None] * np.uint64(chunk)
                          + within[None, :])
        numa[lanes] = r
        regions.append((first, nslots, base, npos[r]))
        base += npos[r] * chunk
    seg_len = np.array([seg, v_seg] * slots, dtype=np.uint32)
    return Workload(name=name, blocks=blocks, slots=slots, seg=seg, addr=addr,
                    seg_len=seg_len, numa=numa, pool_bytes=base, seed=seed,
                    regions=regions, pos=[np.asarray(p, dtype=np.int64) for p in positions])


def _two_regions(slots):
    half = slots // 2
    return [(0, half), (half, slots - half)]


def bump(name="default", blocks=1000, slots=288, seg=4 * KIB, nregions=2, seed=2, v_seg=None):
    """Fully bump-allocated holder: pos(b) = b in every region."""
    regs = _two_regions(slots) if nregions == 2 else [(0, slots)]
    pos = [np.arange(blocks)] * len(regs)
    return _build(name, blocks, slots, seg, regs, pos, [blocks] * len(regs), seed, v_seg)


def tiny():
    """8 blocks x 4 slots x 2 x 4 KiB, slots 0-1 and 2-3 in two regions (256 KiB)."""
    return bump("tiny", blocks=8, slots=4, seg=4 * KIB, nregions=2, seed=1)


def default():
    """1000 blocks x 288 slots x 2 x 4 KiB = 576k segments, 2250 MiB, bump-allocated."""
    return bump("default", blocks=1000, slots=288, seg=4 * KIB, nregions=2, seed=2)


def wide64k():
    """200 blocks x 288 slots x 2 x 64 KiB = 7200 MiB, bump-allocated, two regions."""
    return bump("wide64k", blocks=200, slots=288, seg=64 * KIB, nregions=2, seed=6)


def worst(blocks=1000, slots=288, seg=4 * KIB, npos=2048, seed=3, v_seg=None):
    """Per-block allocation order permuted: pos(b) = first B of a seeded shuffle of
    [0, npos), the same permutation in both regions (pool = 2 * npos * chunk)."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(npos)[:blocks]
    regs = _two_regions(slots)
    return _build("worst", blocks, slots, seg, regs, [perm, perm], [npos, npos], seed, v_seg)


def mixed(blocks=4096, slots=64, seg=16 * KIB, gap_mean=56.0 / 3.0, run_mean=8.0, seed=4):
    """Two regions; alternating home gaps ~ Geom0(gap_mean) and relocated runs ~
    Geom1(run_mean) (expected 30% relocated); relocated blocks take spill
    positions B, B+1, ... in block order, identically in both regions."""
    rng = np.random.default_rng(seed)
    relocated = np.zeros(blocks, dtype=bool)
    b = 0
    while b < blocks:
        b += int(rng.geometric(1.0 / (1.0 + gap_mean))) - 1
        if b >= blocks:
            break
        n = int(rng.geometric(1.0 / run_mean))
        relocated[b:b + n] = True
        b += n
    pos = np.arange(blocks, dtype=np.int64)
    rel = np.nonzero(relocated)[0]
    pos[rel] = blocks + np.arange(rel.size)
    npos = blocks + rel.size
    regs = _two_regions(slots)
    return _build("mixed", blocks, slots, seg, regs, [pos, pos], [npos, npos], seed)


def many_small(blocks=100_000, slots=32, seg=512, nreloc=5000, seed=5):
    """One region; nreloc seeded distinct blocks moved to spill positions
    B + j in ascending block order (5% at the full size)."""
    rng = np.random.default_rng(seed)
    rel = np.sort(rng.choice(blocks, size=nreloc, replace=False))
    pos = np.arange(blocks, dtype=np.int64)
    pos[rel] = blocks + np.arange(nreloc)
    npos = blocks + nreloc
    return _build("many_small", blocks, slots, seg, [(0, slots)], [pos], [npos], seed)


def scattered(blocks=6, slots=3, seg=64, seed=7):
    """Every segment at its own seeded random slot of a pool of 4x the payload:
    no two segments adjacent by construction (the per-segment degenerate case)."""
    rng = np.random.default_rng(seed)
    L = 2 * slots
    nseg = blocks * L
    nslot = 4 * nseg
    # choose slots with a gap of at least one free slot between any two
    picks = np.sort(rng.choice(nslot // 2, size=nseg, replace=False)) * 2
    rng.shuffle(picks)
    addr = (picks.astype(np.uint64) * np.uint64(seg)).reshape(blocks, L)
    return Workload(name="scattered", blocks=blocks, slots=slots, seg=seg, addr=addr,
                    seg_len=np.full(L, seg, dtype=np.uint32),
                    numa=np.zeros(L, dtype=np.uint32), pool_bytes=nslot * seg, seed=seed)


CONFIGS = {
    "tiny": tiny,
    "default": default,
    "worst": worst,
    "mixed": mixed,
    "many_small": many_small,
    "wide64k": wide64k,
}


def k_only(layout: str, null_v: bool = False, **kw) -> Workload:
    """A K-only cache (every V segment of length 0, as in a cache that keeps a
    single latent per token), laid out like bump() or worst() with the same
    keyword arguments.  The holder either places each empty V segment where
    the next segment starts (what a bump allocator gives) or reports address
    0 for it (null_v)."""
    wl = {"bump": bump, "worst": worst}[layout](v_seg=0, **kw)
    wl.name = f"{wl.name}_konly" + ("_nullv" if null_v else "")
    if null_v:
        wl.addr[:, 1::2] = 0
    return wl


def small_variants():
    """Reduced-size versions of every configuration that still span several
    kernel tiles and end in a ragged tail (sizes are not powers of two)."""
    return [
        tiny(),
        bump("default_s", blocks=37, slots=24, seg=4 * KIB, seed=2),
        worst(blocks=61, slots=18, npos=128, seed=3),
        mixed(blocks=203, slots=10, seg=16 * KIB, seed=4),
        many_small(blocks=3001, slots=8, seg=512, nreloc=150, seed=5),
        bump("wide64k_s", blocks=9, slots=6, seg=64 * KIB, seed=6),
        scattered(),
    ]


# ------------------------------------------------------------ paged writes

@dataclass
class PagedWorkload:
    """Two page pools and the page tables of one paged write ("RDMA
    point-to-point communication for LLM systems": page sets {indices,
    stride, offset}, KvCache pages moved between a prefill and a decode
    instance).  Page i goes from source page src_idx[i] to destination page
    dst_idx[i]; each table lists distinct pages in a seeded random order, as
    a paged cache's block tables do after some churn."""

    name: str
    page_len: int
    num_pages: int
    src_idx: np.ndarray         # uint32 [num_pages]
    src_stride: int
    src_offset: int
    src_bytes: int
    dst_idx: np.ndarray         # uint32 [num_pages]
    dst_stride: int
    dst_offset: int
    dst_bytes: int
    seed: int

    @property
    def bytes_moved(self) -> int:
        return self.num_pages * self.page_len


def paged(name, num_pages, page_len, src_pages, dst_pages, src_stride=None, src_offset=0,
          dst_stride=None, dst_offset=0, seed=6):
    rng = np.random.default_rng(seed)
    src_stride = page_len if src_stride is None else src_stride
    dst_stride = page_len if dst_stride is None else dst_stride
    src_idx = rng.permutation(src_pages)[:num_pages].astype(np.uint32)
    dst_idx = rng.permutation(dst_pages)[:num_pages].astype(np.uint32)
    return PagedWorkload(name, page_len, num_pages, src_idx, src_stride, src_offset,
                         src_offset + (src_pages - 1) * src_stride + page_len, dst_idx,
                         dst_stride, dst_offset, dst_offset + (dst_pages - 1) * dst_stride + page_len,
                         seed)


def paged_default(seed=6):
    """576,000 pages of 4 KiB (2250 MiB, the default workload's bytes) from a
    pool of 720,000 pages to a pool of 640,000 pages, both tables permuted."""
    return paged("paged_default", 576_000, 4 * KIB, 720_000, 640_000, seed=seed)


# ---------------------------------------------------------------- payload bytes

def splitmix64_np(x: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser applied to uint64 counters (numpy, wrapping)."""
    with np.errstate(over="ignore"):
        z = x.astype(np.uint64) + _SM_GAMMA
        z = (z ^ (z >> np.uint64(30))) * _SM_MUL1
        z = (z ^ (z >> np.uint64(27))) * _SM_MUL2
        return z ^ (z >> np.uint64(31))


def pool_words_np(seed: int, first_word: int, nwords: int) -> np.ndarray:
    idx = np.arange(first_word, first_word + nwords, dtype=np.uint64)
    return splitmix64_np(idx ^ np.uint64(seed))


def pool_bytes_np(seed: int, start: int, nbytes: int) -> np.ndarray:
    """Holder-pool bytes [start, start + nbytes) as a uint8 array."""
    w0 = start // 8
    w1 = (start + nbytes + 7) // 8
    words = pool_words_np(seed, w0, w1 - w0)
    raw = words.view(np.uint8)
    off = start - 8 * w0
    return raw[off:off + nbytes].copy()


def holder_pool_np(wl: Workload) -> np.ndarray:
    """The whole holder pool on the host (small workloads only)."""
    return pool_bytes_np(wl.seed, 0, wl.pool_bytes)


def _logical_shr(z, k, torch):
    return (z >> k) & ((1 << (64 - k)) - 1)


def fill_pool_torch(buf, seed: int, chunk_words: int = 1 << 26):
    """Fill a uint8 torch tensor (any device, length a multiple of 8 not
    required) with the holder payload, chunk by chunk on the tensor's device.

    int64 torch arithmetic wraps modulo 2**64 like uint64; right shifts are
    made logical with a mask."""
    import torch
    n = buf.numel()
    nw = n // 8
    c1 = int(np.int64(np.uint64(0x9E3779B97F4A7C15).view(np.int64)))
    c2 = int(np.int64(np.uint64(0xBF58476D1CE4E5B9).view(np.int64)))
    c3 = int(np.int64(np.uint64(0x94D049BB133111EB).view(np.int64)))
    words = buf[: nw * 8].view(torch.int64)
    s = int(np.int64(np.uint64(seed).view(np.int64)))
    for w0 in range(0, nw, chunk_words):
        w1 = min(nw, w0 + chunk_words)
        z = torch.arange(w0, w1, dtype=torch.int64, device=buf.device) ^ s
        z = z + c1
        z = (z ^ _logical_shr(z, 30, torch)) * c2
        z = (z ^ _logical_shr(z, 27, torch)) * c3
        z = z ^ _logical_shr(z, 31, torch)
        words[w0:w1] = z
        del z
    if n % 8:
        tail = pool_bytes_np(seed, nw * 8, n % 8)
        buf[nw * 8:] = torch.from_numpy(tail).to(buf.device)
    return buf
