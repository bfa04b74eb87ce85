"""CPU oracle for the paged KV block-transfer path -- TEST INFRASTRUCTURE.

A thin ctypes shim over ``kvx_oracle.c`` (plain C, single-threaded).  Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package; the product path never does.

The structures are described here by the oracle's own numpy dtypes; they are
not imported from the CUDA library's binding.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvx_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

GROUP_DTYPE = np.dtype([("base", "<u8"), ("stride", "<i8"), ("chunk", "<u8"),
                        ("local", "<u8"), ("block", "<u4"), ("count", "<u4"),
                        ("node", "<u4"), ("dense", "<u4")])
DESC_DTYPE = np.dtype([("remote", "<u8"), ("local", "<u8"), ("len", "<u8"),
                       ("group", "<u4"), ("reserved", "<u4")])

S_LANES, S_ARRAYS, S_COVERAGE, S_ZERO_COUNT, S_ZERO_LEN = 1, 2, 4, 8, 16
S_SPAN, S_STRIDE1, S_BOUNDS, S_DESC, S_CAPACITY = 32, 64, 128, 256, 512
MAX_READ_BYTES = 32 * 1024 * 1024

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build/liboracle.so."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (force or not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-Wall", "-Wextra", "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    """The loaded oracle.  KVX_ORACLE_LIB may name another build of the same
    source (the mutation tests load deliberately broken copies that way)."""
    global _lib
    if _lib is None:
        _setup(ctypes.CDLL(os.environ.get("KVX_ORACLE_LIB") or build()))
    return _lib


def _setup(handle):
    global _lib
    _lib = handle
    u32p = ctypes.c_void_p
    _lib.kvxo_encode_runs.restype = ctypes.c_uint64
    _lib.kvxo_encode_runs.argtypes = [u32p, ctypes.c_uint32, ctypes.c_uint32, u32p, u32p,
                                      u32p, u32p, ctypes.c_uint64]
    _lib.kvxo_plan.restype = ctypes.c_uint32
    _lib.kvxo_plan.argtypes = ([u32p, ctypes.c_uint32, u32p, u32p, u32p, ctypes.c_uint64,
                                ctypes.c_uint32, u32p, u32p, ctypes.c_uint32, ctypes.c_uint64,
                                u32p, ctypes.c_uint64, u32p, ctypes.c_uint64]
                               + [u32p] * 5)
    _lib.kvxo_rebuild.restype = ctypes.c_uint32
    _lib.kvxo_rebuild.argtypes = [u32p] * 6 + [ctypes.c_uint64, ctypes.c_uint32,
                                               ctypes.c_uint32, u32p, ctypes.c_uint64, u32p]
    for name in ("kvxo_pack", "kvxo_unpack"):
        f = getattr(_lib, name)
        f.restype = ctypes.c_uint32
        f.argtypes = [u32p, ctypes.c_uint64, u32p, ctypes.c_uint64, u32p, ctypes.c_uint64]
    _lib.kvxo_verify_encode.restype = ctypes.c_uint64
    _lib.kvxo_verify_encode.argtypes = [u32p, u32p, u32p, ctypes.c_uint32, ctypes.c_uint32,
                                        u32p, u32p, u32p, u32p, ctypes.c_uint64, u32p]
    _lib.kvxo_seal_blocks.restype = ctypes.c_uint32
    _lib.kvxo_seal_blocks.argtypes = ([u32p] * 6 + [ctypes.c_uint64, ctypes.c_uint32,
                                                    ctypes.c_uint32, u32p, u32p, ctypes.c_uint64,
                                                    u32p, u32p, ctypes.c_uint64])
    _lib.kvxo_paged_writes.restype = ctypes.c_uint32
    _lib.kvxo_paged_writes.argtypes = [ctypes.c_uint64, u32p, ctypes.c_uint64, u32p,
                                       ctypes.c_uint64, ctypes.c_uint64, u32p, ctypes.c_uint64,
                                       u32p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class RunTable:
    runs_per_lane: np.ndarray   # uint32 [L]
    run_base: np.ndarray        # uint64 [R]
    run_stride: np.ndarray      # int64 [R]
    run_count: np.ndarray       # uint32 [R]

    @property
    def num_runs(self) -> int:
        return int(self.run_base.size)


@dataclass
class Plan:
    status: int
    groups: np.ndarray          # GROUP_DTYPE [G]
    descs: np.ndarray           # DESC_DTYPE [D]
    lane_first: np.ndarray      # uint32 [L + 1]
    run_block: np.ndarray       # uint32 [R]
    run_group: np.ndarray       # uint32 [R]
    run_off: np.ndarray         # uint64 [R]
    slab_bytes: int


def run_capacity(B: int, L: int) -> int:
    """Greedy runs never exceed ceil(B/2) per lane (every run but a lane's
    last one covers at least two blocks)."""
    return L * ((B + 1) // 2)


def encode_runs(addr: np.ndarray) -> RunTable:
    addr = np.ascontiguousarray(addr, dtype=np.uint64)
    B, L = addr.shape
    cap = max(1, run_capacity(B, L))
    rpl = np.zeros(L, dtype=np.uint32)
    base = np.zeros(cap, dtype=np.uint64)
    stride = np.zeros(cap, dtype=np.int64)
    count = np.zeros(cap, dtype=np.uint32)
    R = lib().kvxo_encode_runs(_p(addr), B, L, _p(rpl), _p(base), _p(stride), _p(count), cap)
    if R == 2**64 - 1:
        raise RuntimeError("oracle encode: run capacity exceeded")
    return RunTable(rpl, base[:R].copy(), stride[:R].copy(), count[:R].copy())


def desc_capacity(B: int, seg_len: np.ndarray) -> int:
    L = int(seg_len.size)
    slab = B * int(seg_len.astype(np.uint64).sum())
    return B * L + (slab + MAX_READ_BYTES - 1) // MAX_READ_BYTES + 1


def plan(table: RunTable, B: int, seg_len: np.ndarray, numa: np.ndarray, pool_bytes: int,
         group_cap: int | None = None, desc_cap: int | None = None,
         num_runs: int | None = None) -> Plan:
    rpl = np.ascontiguousarray(table.runs_per_lane, dtype=np.uint32)
    base = np.ascontiguousarray(table.run_base, dtype=np.uint64)
    stride = np.ascontiguousarray(table.run_stride, dtype=np.int64)
    count = np.ascontiguousarray(table.run_count, dtype=np.uint32)
    seg_len = np.ascontiguousarray(seg_len, dtype=np.uint32)
    numa = np.ascontiguousarray(numa, dtype=np.uint32)
    R = table.num_runs if num_runs is None else num_runs
    Lt = int(rpl.size)
    if group_cap is None:
        group_cap = max(1, R)
    if desc_cap is None:
        desc_cap = desc_capacity(B, seg_len) if int(seg_len.size) else 1
    groups = np.zeros(max(1, group_cap), dtype=GROUP_DTYPE)
    descs = np.zeros(max(1, desc_cap), dtype=DESC_DTYPE)
    lane_first = np.zeros(Lt + 1, dtype=np.uint32)
    n = max(1, base.size)
    run_block = np.zeros(n, dtype=np.uint32)
    run_group = np.zeros(n, dtype=np.uint32)
    run_off = np.zeros(n, dtype=np.uint64)
    counts = np.zeros(3, dtype=np.uint64)
    st = lib().kvxo_plan(_p(rpl), Lt, _p(base if base.size else np.zeros(1, np.uint64)),
                         _p(stride if stride.size else np.zeros(1, np.int64)),
                         _p(count if count.size else np.zeros(1, np.uint32)), R, B,
                         _p(seg_len if seg_len.size else np.zeros(1, np.uint32)),
                         _p(numa if numa.size else np.zeros(1, np.uint32)), int(seg_len.size),
                         pool_bytes, _p(groups), group_cap, _p(descs), desc_cap,
                         _p(lane_first), _p(run_block), _p(run_group), _p(run_off), _p(counts))
    ng, nd, slab = (int(x) for x in counts)
    return Plan(int(st), groups[:ng].copy(), descs[:nd].copy(), lane_first,
                run_block[:R].copy(), run_group[:R].copy(), run_off[:R].copy(), slab)


def rebuild(table: RunTable, p: Plan, B: int, L: int, seg_len: np.ndarray,
            slab_bytes: int | None = None, groups: np.ndarray | None = None,
            run_group: np.ndarray | None = None):
    """Returns (status, local uint64 [B, L])."""
    groups = p.groups if groups is None else groups
    run_group = p.run_group if run_group is None else run_group
    slab_bytes = p.slab_bytes if slab_bytes is None else slab_bytes
    local = np.full((B, L), np.uint64(0xDEADBEEFDEADBEEF), dtype=np.uint64)
    g = np.ascontiguousarray(groups if groups.size else np.zeros(1, GROUP_DTYPE))
    rg = np.ascontiguousarray(run_group if run_group.size else np.zeros(1, np.uint32),
                              dtype=np.uint32)
    st = lib().kvxo_rebuild(_p(np.ascontiguousarray(table.runs_per_lane, dtype=np.uint32)),
                            _p(np.ascontiguousarray(table.run_base if table.num_runs else np.zeros(1, np.uint64))),
                            _p(np.ascontiguousarray(table.run_stride if table.num_runs else np.zeros(1, np.int64))),
                            _p(np.ascontiguousarray(table.run_count if table.num_runs else np.zeros(1, np.uint32))),
                            _p(rg), _p(g), int(groups.size), B, L,
                            _p(np.ascontiguousarray(seg_len, dtype=np.uint32) if L else np.zeros(1, np.uint32)),
                            slab_bytes, _p(local if local.size else np.zeros(1, np.uint64)))
    return int(st), local


def pack(pool: np.ndarray, descs: np.ndarray, slab: np.ndarray) -> int:
    d = np.ascontiguousarray(descs if descs.size else np.zeros(1, DESC_DTYPE))
    return int(lib().kvxo_pack(_p(pool), pool.size, _p(d), int(descs.size), _p(slab), slab.size))


def unpack(slab: np.ndarray, descs: np.ndarray, dst_pool: np.ndarray) -> int:
    d = np.ascontiguousarray(descs if descs.size else np.zeros(1, DESC_DTYPE))
    return int(lib().kvxo_unpack(_p(slab), slab.size, _p(d), int(descs.size), _p(dst_pool),
                                 dst_pool.size))


def _nz(a: np.ndarray, dtype) -> np.ndarray:
    """A contiguous array of dtype, never empty (ctypes wants a real pointer)."""
    a = np.ascontiguousarray(a, dtype=dtype)
    return a if a.size else np.zeros(1, dtype=dtype)


def verify_encode(addr: np.ndarray, size: np.ndarray, tmpl_len: np.ndarray):
    """Holder prefix scan with the slot-template check.  Returns (prefix
    blocks, RunTable of those blocks)."""
    addr = np.ascontiguousarray(addr, dtype=np.uint64)
    B, L = addr.shape
    size = np.ascontiguousarray(size, dtype=np.uint32)
    assert size.shape == (B, L)
    cap = max(1, run_capacity(B, L))
    rpl = np.zeros(max(1, L), dtype=np.uint32)
    base = np.zeros(cap, dtype=np.uint64)
    stride = np.zeros(cap, dtype=np.int64)
    count = np.zeros(cap, dtype=np.uint32)
    prefix = np.zeros(1, dtype=np.uint32)
    R = lib().kvxo_verify_encode(_p(_nz(addr, np.uint64)), _p(_nz(size, np.uint32)),
                                 _p(_nz(tmpl_len, np.uint32)), B, L, _p(rpl), _p(base),
                                 _p(stride), _p(count), cap, _p(prefix))
    if R == 2**64 - 1:
        raise RuntimeError("oracle verify_encode: run capacity exceeded")
    return int(prefix[0]), RunTable(rpl[:L].copy(), base[:R].copy(), stride[:R].copy(),
                                    count[:R].copy())


def seal_blocks(table: RunTable, p: Plan, B: int, L: int, seg_len: np.ndarray,
                slab: np.ndarray, dst_addr: np.ndarray, dst: np.ndarray,
                groups: np.ndarray | None = None, run_group: np.ndarray | None = None,
                slab_bytes: int | None = None) -> int:
    """Install every segment from the slab at dst[dst_addr[b][l]] (in place on
    dst).  Returns the status bitmask."""
    groups = p.groups if groups is None else groups
    run_group = p.run_group if run_group is None else run_group
    slab_bytes = slab.size if slab_bytes is None else slab_bytes
    assert slab_bytes <= slab.size
    dst_addr = np.ascontiguousarray(dst_addr, dtype=np.uint64)
    assert dst_addr.shape == (B, L)
    return int(lib().kvxo_seal_blocks(
        _p(_nz(table.runs_per_lane, np.uint32)), _p(_nz(table.run_base, np.uint64)),
        _p(_nz(table.run_stride, np.int64)), _p(_nz(table.run_count, np.uint32)),
        _p(_nz(run_group, np.uint32)), _p(_nz(groups, GROUP_DTYPE)), int(groups.size), B, L,
        _p(_nz(seg_len, np.uint32)), _p(_nz(slab, np.uint8)), slab_bytes,
        _p(_nz(dst_addr, np.uint64)), _p(dst), dst.size))


def paged_writes(page_len: int, src: np.ndarray, src_idx: np.ndarray, src_stride: int,
                 src_offset: int, dst: np.ndarray, dst_idx: np.ndarray, dst_stride: int,
                 dst_offset: int) -> int:
    """Copy page i of the source page set to page i of the destination set
    (in place on dst).  Returns the status bitmask."""
    src_idx = np.ascontiguousarray(src_idx, dtype=np.uint32)
    dst_idx = np.ascontiguousarray(dst_idx, dtype=np.uint32)
    assert src_idx.size == dst_idx.size
    assert dst.flags["C_CONTIGUOUS"] and dst.dtype == np.uint8
    return int(lib().kvxo_paged_writes(page_len, _p(_nz(src, np.uint8)), src.size,
                                       _p(_nz(src_idx, np.uint32)), src_stride, src_offset,
                                       _p(dst if dst.size else np.zeros(1, np.uint8)), dst.size,
                                       _p(_nz(dst_idx, np.uint32)), dst_stride, dst_offset,
                                       int(src_idx.size)))
