"""Thin Python binding of libkvx (ctypes; argument marshalling only).

Every function below has the name of the C entry point it calls and passes
device pointers of torch tensors straight through.  PyTorch provides device
memory and streams; every step of the transfer runs in libkvx's kernels.
There is no fallback: if the library is missing, loading raises.

``Transfer`` bundles the buffers of one block-prefix transfer (allocated with
torch, sized from the library's capacity and workspace queries) and runs the
five calls in order on one stream, with no host synchronisation in between.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import build as _build

# struct kvx_group / kvx_desc (include/kvx.h)
GROUP_DTYPE = np.dtype([("base", "<u8"), ("stride", "<i8"), ("chunk", "<u8"), ("local", "<u8"),
                        ("block", "<u4"), ("count", "<u4"), ("node", "<u4"), ("dense", "<u4")])
DESC_DTYPE = np.dtype([("remote", "<u8"), ("local", "<u8"), ("len", "<u8"), ("group", "<u4"),
                       ("reserved", "<u4")])
assert GROUP_DTYPE.itemsize == 48 and DESC_DTYPE.itemsize == 32

KVX_OK, KVX_EINVAL, KVX_ECAPACITY, KVX_ECUDA = 0, 1, 3, 4
S_LANES, S_ARRAYS, S_COVERAGE, S_ZERO_COUNT, S_ZERO_LEN = 1, 2, 4, 8, 16
S_SPAN, S_STRIDE1, S_BOUNDS, S_DESC, S_CAPACITY, S_TIMEOUT = 32, 64, 128, 256, 512, 1024
MAX_READ_BYTES = 32 * 1024 * 1024

_ERR = {KVX_EINVAL: "KVX_EINVAL", KVX_ECAPACITY: "KVX_ECAPACITY", KVX_ECUDA: "KVX_ECUDA"}

_lib = None
_P = ctypes.c_void_p
_U32 = ctypes.c_uint32
_U64 = ctypes.c_uint64
_SZ = ctypes.c_size_t

_SIGS = {
    "kvx_run_capacity": (_U64, [_U32, _U32]),
    "kvx_encode_workspace_size": (_SZ, [_U32, _U32]),
    "kvx_encode_runs": (ctypes.c_int, [_P, _U32, _U32, _P, _P, _P, _P, _U64, _P, _P, _P, _SZ, _P]),
    "kvx_desc_capacity": (_U64, [_U32, _U32, _U64]),
    "kvx_plan_bounds": (ctypes.c_int, [_U32, _U32, _U64, _U64, _P, _P]),
    "kvx_plan_workspace_size": (_SZ, [_U32, _U64, _U64]),
    "kvx_plan_set_sm_share": (ctypes.c_int, [_U32]),
    "kvx_plan_groups": (ctypes.c_int, [_P, _U32, _P, _P, _P, _P, _U64, _U32, _P, _P, _U32, _U64,
                                       _P, _U64, _P, _U64, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "kvx_rebuild": (ctypes.c_int, [_P, _P, _P, _P, _P, _U64, _P, _U64, _P, _U32, _U32, _P, _U64,
                                   _P, _P, _P]),
    "kvx_copy_workspace_size": (_SZ, [_U64]),
    "kvx_pack": (ctypes.c_int, [_P, _U64, _P, _P, _U64, _P, _U64, _P, _P, _SZ, _P]),
    "kvx_unpack": (ctypes.c_int, [_P, _U64, _P, _P, _U64, _P, _U64, _P, _P, _SZ, _P]),
    "kvx_pack_noalloc": (ctypes.c_int, [_P, _U64, _P, _P, _U64, _P, _U64, _P, _P]),
    "kvx_copy_prepare": (ctypes.c_int, [_P, _U64, _P, _P, _U64, _P, _U64, _P, _P, _SZ, _P]),
    "kvx_pack_prepared": (ctypes.c_int, [_P, _U64, _P, _P, _U64, _P, _U64, _P, _P, _SZ, _P]),
    "kvx_unpack_prepared": (ctypes.c_int, [_P, _U64, _P, _P, _U64, _P, _U64, _P, _P, _SZ, _P]),
    "kvx_verify_encode": (ctypes.c_int, [_P, _P, _P, _U32, _U32, _P, _P, _P, _P, _P, _U64, _P, _P,
                                         _P, _SZ, _P]),
    "kvx_segcopy_workspace_size": (_SZ, []),
    "kvx_seal_blocks": (ctypes.c_int, [_P, _P, _P, _P, _P, _U64, _P, _U64, _P, _U32, _U32, _P, _P,
                                       _U64, _P, _P, _U64, _P, _P, _SZ, _P]),
    "kvx_paged_writes": (ctypes.c_int, [_U64, _P, _U64, _P, _U64, _U64, _P, _U64, _P, _U64, _U64,
                                        _U64, _P, _P, _SZ, _P]),
    "kvx_selftest_timeouts": (ctypes.c_int, [_P, _P]),
    "kvx_launch_count": (_U64, []),
    "kvx_version": (_U32, []),
}


class KvxError(RuntimeError):
    pass


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded libkvx.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise KvxError("libkvx.so is not built (%s); run paged_kv_cache_kvx_gb300.build.build()" % path)
        handle = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            f = getattr(handle, name)
            f.restype = res
            f.argtypes = args
        _lib = handle
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, name: str):
    if code != KVX_OK:
        raise KvxError("%s returned %s" % (name, _ERR.get(code, str(code))))


# ------------------------------------------------------------ entry points

def kvx_run_capacity(B: int, L: int) -> int:
    return int(lib().kvx_run_capacity(B, L))


def kvx_encode_workspace_size(B: int, L: int) -> int:
    return int(lib().kvx_encode_workspace_size(B, L))


def kvx_encode_runs(addr, B, L, runs_per_lane, run_base, run_stride, run_count, run_capacity,
                    num_runs, status, ws, stream=None):
    _check(lib().kvx_encode_runs(_ptr(addr), B, L, _ptr(runs_per_lane), _ptr(run_base),
                                 _ptr(run_stride), _ptr(run_count), run_capacity, _ptr(num_runs),
                                 _ptr(status), _ptr(ws), ws.numel(), _stream(stream)),
           "kvx_encode_runs")


def kvx_desc_capacity(B: int, L: int, seg_bytes_sum: int) -> int:
    return int(lib().kvx_desc_capacity(B, L, seg_bytes_sum))


def kvx_plan_bounds(B: int, L: int, num_runs: int, max_seg_bytes_total: int):
    """(group_cap, desc_cap) for kvx_plan_groups; num_runs 0 = unknown."""
    g, d = ctypes.c_uint64(0), ctypes.c_uint64(0)
    _check(lib().kvx_plan_bounds(B, L, num_runs, max_seg_bytes_total, ctypes.addressof(g),
                                 ctypes.addressof(d)), "kvx_plan_bounds")
    return int(g.value), int(d.value)


def kvx_plan_set_sm_share(blocks_per_sm: int) -> None:
    """Blocks per SM the planner's grid may take on the current device: 1 (the
    default; it fits beside a running bulk copy) or 2 (an otherwise idle
    device)."""
    _check(lib().kvx_plan_set_sm_share(blocks_per_sm), "kvx_plan_set_sm_share")


def kvx_plan_workspace_size(L: int, run_capacity: int, pool_bytes: int) -> int:
    return int(lib().kvx_plan_workspace_size(L, run_capacity, pool_bytes))


def kvx_plan_groups(runs_per_lane, table_lanes, run_base, run_stride, run_count, num_runs,
                    run_capacity, B, seg_len, numa, template_lanes, pool_bytes, groups,
                    group_capacity, descs, desc_capacity, lane_first, run_block, run_group,
                    run_off, counts, status, ws, stream=None):
    _check(lib().kvx_plan_groups(_ptr(runs_per_lane), table_lanes, _ptr(run_base),
                                 _ptr(run_stride), _ptr(run_count), _ptr(num_runs), run_capacity,
                                 B, _ptr(seg_len), _ptr(numa), template_lanes, pool_bytes,
                                 _ptr(groups), group_capacity, _ptr(descs), desc_capacity,
                                 _ptr(lane_first), _ptr(run_block), _ptr(run_group), _ptr(run_off),
                                 _ptr(counts), _ptr(status), _ptr(ws), ws.numel(),
                                 _stream(stream)), "kvx_plan_groups")


def kvx_rebuild(lane_first, run_block, run_base, run_stride, run_group, run_capacity, groups,
                group_capacity, counts, B, L, seg_len, slab_bytes, local, status, stream=None):
    _check(lib().kvx_rebuild(_ptr(lane_first), _ptr(run_block), _ptr(run_base), _ptr(run_stride),
                             _ptr(run_group), run_capacity, _ptr(groups), group_capacity,
                             _ptr(counts), B, L, _ptr(seg_len), slab_bytes, _ptr(local),
                             _ptr(status), _stream(stream)), "kvx_rebuild")


def kvx_copy_workspace_size(slab_bytes: int) -> int:
    return int(lib().kvx_copy_workspace_size(slab_bytes))


def kvx_pack(pool, pool_bytes, descs, num_descs, desc_capacity, slab, slab_bytes, status, ws,
             stream=None):
    _check(lib().kvx_pack(_ptr(pool), pool_bytes, _ptr(descs), _ptr(num_descs), desc_capacity,
                          _ptr(slab), slab_bytes, _ptr(status), _ptr(ws), ws.numel(),
                          _stream(stream)), "kvx_pack")


def kvx_unpack(slab, slab_bytes, descs, num_descs, desc_capacity, dst_pool, pool_bytes, status, ws,
               stream=None):
    _check(lib().kvx_unpack(_ptr(slab), slab_bytes, _ptr(descs), _ptr(num_descs), desc_capacity,
                            _ptr(dst_pool), pool_bytes, _ptr(status), _ptr(ws), ws.numel(),
                            _stream(stream)), "kvx_unpack")


def kvx_copy_prepare(pool, pool_bytes, descs, num_descs, desc_capacity, slab, slab_bytes, status, ws,
                     stream=None):
    _check(lib().kvx_copy_prepare(_ptr(pool), pool_bytes, _ptr(descs), _ptr(num_descs), desc_capacity,
                                  _ptr(slab), slab_bytes, _ptr(status), _ptr(ws), ws.numel(),
                                  _stream(stream)), "kvx_copy_prepare")


def kvx_pack_prepared(pool, pool_bytes, descs, num_descs, desc_capacity, slab, slab_bytes, status, ws,
                      stream=None):
    _check(lib().kvx_pack_prepared(_ptr(pool), pool_bytes, _ptr(descs), _ptr(num_descs), desc_capacity,
                                   _ptr(slab), slab_bytes, _ptr(status), _ptr(ws), ws.numel(),
                                   _stream(stream)), "kvx_pack_prepared")


def kvx_unpack_prepared(slab, slab_bytes, descs, num_descs, desc_capacity, dst_pool, pool_bytes, status,
                        ws, stream=None):
    _check(lib().kvx_unpack_prepared(_ptr(slab), slab_bytes, _ptr(descs), _ptr(num_descs), desc_capacity,
                                     _ptr(dst_pool), pool_bytes, _ptr(status), _ptr(ws), ws.numel(),
                                     _stream(stream)), "kvx_unpack_prepared")


def kvx_pack_noalloc(pool, pool_bytes, descs, num_descs, desc_capacity, slab, slab_bytes, status,
                     stream=None):
    """kvx_pack with the library's own static scratch (no workspace argument)."""
    _check(lib().kvx_pack_noalloc(_ptr(pool), pool_bytes, _ptr(descs), _ptr(num_descs),
                                  desc_capacity, _ptr(slab), slab_bytes, _ptr(status),
                                  _stream(stream)), "kvx_pack_noalloc")


def kvx_verify_encode(addr, seg_size, seg_len, B, L, prefix_blocks, runs_per_lane, run_base,
                      run_stride, run_count, run_capacity, num_runs, status, ws, stream=None):
    _check(lib().kvx_verify_encode(_ptr(addr), _ptr(seg_size), _ptr(seg_len), B, L,
                                   _ptr(prefix_blocks), _ptr(runs_per_lane), _ptr(run_base),
                                   _ptr(run_stride), _ptr(run_count), run_capacity, _ptr(num_runs),
                                   _ptr(status), _ptr(ws), ws.numel(), _stream(stream)),
           "kvx_verify_encode")


def kvx_segcopy_workspace_size() -> int:
    return int(lib().kvx_segcopy_workspace_size())


def kvx_seal_blocks(lane_first, run_block, run_base, run_stride, run_group, run_capacity, groups,
                    group_capacity, counts, B, L, seg_len, slab, slab_bytes, dst_addr, dst,
                    dst_bytes, status, ws=None, stream=None):
    """ws (a uint8 device tensor of kvx_segcopy_workspace_size() bytes) selects the
    bulk-copy path; None the register path."""
    _check(lib().kvx_seal_blocks(_ptr(lane_first), _ptr(run_block), _ptr(run_base),
                                 _ptr(run_stride), _ptr(run_group), run_capacity, _ptr(groups),
                                 group_capacity, _ptr(counts), B, L, _ptr(seg_len), _ptr(slab),
                                 slab_bytes, _ptr(dst_addr), _ptr(dst),
                                 dst_bytes, _ptr(status), _ptr(ws), 0 if ws is None else ws.numel(),
                                 _stream(stream)), "kvx_seal_blocks")


def kvx_paged_writes(page_len, src, src_bytes, src_indices, src_stride, src_offset, dst, dst_bytes,
                     dst_indices, dst_stride, dst_offset, num_pages, status, ws=None, stream=None):
    """ws as for kvx_seal_blocks."""
    _check(lib().kvx_paged_writes(page_len, _ptr(src), src_bytes, _ptr(src_indices), src_stride,
                                  src_offset, _ptr(dst), dst_bytes, _ptr(dst_indices), dst_stride,
                                  dst_offset, num_pages, _ptr(status), _ptr(ws),
                                  0 if ws is None else ws.numel(), _stream(stream)),
           "kvx_paged_writes")


def kvx_selftest_timeouts(status, stream=None):
    _check(lib().kvx_selftest_timeouts(_ptr(status), _stream(stream)), "kvx_selftest_timeouts")


def kvx_launch_count() -> int:
    return int(lib().kvx_launch_count())


def kvx_version() -> int:
    return int(lib().kvx_version())


# ------------------------------------------------------------ buffers

def _u64_np(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint64)


def _u32_np(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


class Transfer:
    """Device buffers for one block-prefix transfer of B blocks with the given
    slot template (seg_len, numa: one entry per lane) from a holder pool of
    pool_bytes bytes.  All memory comes from torch; libkvx allocates nothing.
    """

    def __init__(self, B: int, seg_len, numa, pool_bytes: int, device="cuda"):
        seg_len = np.asarray(seg_len, dtype=np.uint32)
        numa = np.asarray(numa, dtype=np.uint32)
        self.B = int(B)
        self.L = int(seg_len.size)
        self.seg_len_host = seg_len.copy()
        self.pool_bytes = int(pool_bytes)
        self.device = torch.device(device)
        L, dev = self.L, self.device
        seg_sum = int(seg_len.astype(np.uint64).sum())
        self.slab_bytes = self.B * seg_sum
        self.run_cap = kvx_run_capacity(self.B, L)
        group_cap, desc_cap = kvx_plan_bounds(self.B, L, 0, seg_sum)
        self.group_cap = max(1, group_cap)
        self.desc_cap = max(1, desc_cap)
        i32, i64, u8 = torch.int32, torch.int64, torch.uint8
        n = max(1, self.run_cap)
        self.seg_len = torch.from_numpy(seg_len.view(np.int32).copy()).to(dev)
        self.numa = torch.from_numpy(numa.view(np.int32).copy()).to(dev)
        self.addr = torch.empty(max(1, self.B * L), dtype=i64, device=dev)
        self.runs_per_lane = torch.empty(max(1, L), dtype=i32, device=dev)
        self.run_base = torch.empty(n, dtype=i64, device=dev)
        self.run_stride = torch.empty(n, dtype=i64, device=dev)
        self.run_count = torch.empty(n, dtype=i32, device=dev)
        self.num_runs = torch.zeros(1, dtype=i64, device=dev)
        self.groups = torch.empty(self.group_cap * GROUP_DTYPE.itemsize, dtype=u8, device=dev)
        self.descs = torch.empty(self.desc_cap * DESC_DTYPE.itemsize, dtype=u8, device=dev)
        self.lane_first = torch.empty(L + 1, dtype=i32, device=dev)
        self.run_block = torch.empty(n, dtype=i32, device=dev)
        self.run_group = torch.empty(n, dtype=i32, device=dev)
        self.run_off = torch.empty(n, dtype=i64, device=dev)
        self.counts = torch.zeros(3, dtype=i64, device=dev)
        self.status = torch.zeros(1, dtype=i32, device=dev)
        self.local = torch.empty(max(1, self.B * L), dtype=i64, device=dev)
        self.enc_ws = torch.empty(kvx_encode_workspace_size(self.B, L), dtype=u8, device=dev)
        self.plan_ws = torch.empty(kvx_plan_workspace_size(L, self.run_cap, self.pool_bytes),
                                   dtype=u8, device=dev)
        self.copy_ws = torch.empty(kvx_copy_workspace_size(self.slab_bytes), dtype=u8, device=dev)
        self.unpack_ws = torch.empty_like(self.copy_ws)  # an unpack prepared while a pack runs
        self.seg_ws = torch.empty(kvx_segcopy_workspace_size(), dtype=u8, device=dev)

    # -- the five calls ------------------------------------------------
    def encode(self, addr=None, stream=None):
        a = self.addr if addr is None else addr
        kvx_encode_runs(a, self.B, self.L, self.runs_per_lane, self.run_base, self.run_stride,
                        self.run_count, self.run_cap, self.num_runs, self.status, self.enc_ws,
                        stream)

    def verify_encode(self, seg_size, prefix, addr=None, stream=None):
        """Holder prefix scan: blocks checked against the template (seg_size
        [B][L] observed sizes), then the passing prefix run-encoded.  The
        prefix length lands in prefix (a device uint32)."""
        a = self.addr if addr is None else addr
        kvx_verify_encode(a, seg_size, self.seg_len, self.B, self.L, prefix, self.runs_per_lane,
                          self.run_base, self.run_stride, self.run_count, self.run_cap,
                          self.num_runs, self.status, self.enc_ws, stream)

    def plan(self, stream=None, table_lanes=None, group_cap=None, desc_cap=None):
        kvx_plan_groups(self.runs_per_lane, self.L if table_lanes is None else table_lanes,
                        self.run_base, self.run_stride, self.run_count, self.num_runs,
                        self.run_cap, self.B, self.seg_len, self.numa, self.L, self.pool_bytes,
                        self.groups, self.group_cap if group_cap is None else group_cap,
                        self.descs, self.desc_cap if desc_cap is None else desc_cap,
                        self.lane_first, self.run_block, self.run_group, self.run_off,
                        self.counts, self.status, self.plan_ws, stream)

    def rebuild(self, stream=None, slab_bytes=None):
        kvx_rebuild(self.lane_first, self.run_block, self.run_base, self.run_stride, self.run_group,
                    self.run_cap, self.groups, self.group_cap, self.counts, self.B, self.L,
                    self.seg_len, self.slab_bytes if slab_bytes is None else slab_bytes,
                    self.local, self.status, stream)

    def pack(self, pool, slab, stream=None):
        kvx_pack(pool, pool.numel(), self.descs, self.counts[1:], self.desc_cap, slab,
                 slab.numel(), self.status, self.copy_ws, stream)

    def unpack(self, slab, dst_pool, stream=None):
        kvx_unpack(slab, slab.numel(), self.descs, self.counts[1:], self.desc_cap, dst_pool,
                   dst_pool.numel(), self.status, self.copy_ws, stream)

    def prepare_pack(self, pool, slab, stream=None):
        """Checks and tile lists of the next pack (kvx_copy_prepare)."""
        kvx_copy_prepare(pool, pool.numel(), self.descs, self.counts[1:], self.desc_cap, slab,
                         slab.numel(), self.status, self.copy_ws, stream)

    def prepare_unpack(self, slab, dst_pool, stream=None):
        """Checks and tile lists of the next unpack, in their own workspace."""
        kvx_copy_prepare(dst_pool, dst_pool.numel(), self.descs, self.counts[1:], self.desc_cap, slab,
                         slab.numel(), self.status, self.unpack_ws, stream)

    def pack_prepared(self, pool, slab, stream=None):
        kvx_pack_prepared(pool, pool.numel(), self.descs, self.counts[1:], self.desc_cap, slab,
                          slab.numel(), self.status, self.copy_ws, stream)

    def unpack_prepared(self, slab, dst_pool, stream=None):
        kvx_unpack_prepared(slab, slab.numel(), self.descs, self.counts[1:], self.desc_cap, dst_pool,
                            dst_pool.numel(), self.status, self.unpack_ws, stream)

    def seal(self, slab, dst_addr, dst, stream=None, bulk=None):
        """Install every segment from the slab at dst[dst_addr[b][l]] (seal
        from template metadata; no local table is written).  bulk selects the
        bulk-copy path (True) or the register path (False); by default the
        bulk path when every non-empty segment is at least 2 KiB."""
        if bulk is None:
            sl = self.seg_len_host[self.seg_len_host > 0]
            bulk = bool(sl.size) and int(sl.min()) >= 2048
        kvx_seal_blocks(self.lane_first, self.run_block, self.run_base, self.run_stride,
                        self.run_group, self.run_cap, self.groups, self.group_cap, self.counts,
                        self.B, self.L, self.seg_len, slab, slab.numel(), dst_addr, dst,
                        dst.numel(), self.status, self.seg_ws if bulk else None, stream)

    def step(self, pool, slab, dst_pool, stream=None, side=None):
        """One pass of the whole path: encode, plan, rebuild, pack, unpack.
        With a side stream, the unpack's preparation and the rebuild (which
        need only the plan) run there alongside pack and join before the
        unpack and the end of the step."""
        main = torch.cuda.current_stream(self.device) if stream is None else stream
        self.encode(stream=main)
        self.plan(stream=main)
        if side is None:
            self.rebuild(stream=main)
            self.pack(pool, slab, stream=main)
            self.unpack(slab, dst_pool, stream=main)
            return
        planned = torch.cuda.Event()
        planned.record(main)
        side.wait_event(planned)
        self.prepare_unpack(slab, dst_pool, stream=side)
        prepared = torch.cuda.Event()
        prepared.record(side)
        self.rebuild(stream=side)
        rebuilt = torch.cuda.Event()
        rebuilt.record(side)
        self.pack(pool, slab, stream=main)
        main.wait_event(prepared)
        self.unpack_prepared(slab, dst_pool, stream=main)
        main.wait_event(rebuilt)

    def set_addr(self, addr_np: np.ndarray):
        a = np.ascontiguousarray(addr_np, dtype=np.uint64).reshape(-1)
        if a.size:
            self.addr[: a.size].copy_(torch.from_numpy(a.view(np.int64)))

    # -- host readback (tests, bench) ----------------------------------
    def read_status(self) -> int:
        return int(_u32_np(self.status)[0])

    def read_counts(self):
        c = _u64_np(self.counts)
        return int(c[0]), int(c[1]), int(c[2])

    def read_table(self):
        R = int(_u64_np(self.num_runs)[0])
        return (_u32_np(self.runs_per_lane)[: self.L].copy(), _u64_np(self.run_base)[:R].copy(),
                self.run_stride.cpu().numpy()[:R].copy(), _u32_np(self.run_count)[:R].copy())

    def read_plan(self):
        ng, nd, slab = self.read_counts()
        R = int(_u64_np(self.num_runs)[0])
        groups = self.groups.cpu().numpy()[: ng * GROUP_DTYPE.itemsize].view(GROUP_DTYPE).copy()
        descs = self.descs.cpu().numpy()[: nd * DESC_DTYPE.itemsize].view(DESC_DTYPE).copy()
        return dict(groups=groups, descs=descs, slab_bytes=slab,
                    lane_first=_u32_np(self.lane_first)[: self.L + 1].copy(),
                    run_block=_u32_np(self.run_block)[:R].copy(),
                    run_group=_u32_np(self.run_group)[:R].copy(),
                    run_off=_u64_np(self.run_off)[:R].copy())

    def read_local(self) -> np.ndarray:
        return _u64_np(self.local)[: self.B * self.L].reshape(self.B, self.L).copy()


def overlapped_steps(transfers, pool, slab, dst_pool, n, main, ctl, side):
    """n passes of the whole path over a stream of transfers, taking the
    Transfer objects in turn (at least two, each with its own metadata and
    the same table): the control path of a pass (encode, plan) runs on the
    ctl stream while the previous pass copies on main; rebuild and the two
    copies' preparations (checks and tile lists) run on side; main only moves
    bytes.  A Transfer's next encode waits until its previous pass's copies
    are done (they read its plan and its tile lists).  Every pass does all
    five calls; only independent passes overlap."""
    k = len(transfers)
    assert k >= 2
    copied = [None] * k
    start = torch.cuda.Event()  # ctl and side fork from main (also what a graph capture needs)
    start.record(main)
    ctl.wait_event(start)
    side.wait_event(start)
    for i in range(n):
        tr = transfers[i % k]
        if copied[i % k] is not None:
            ctl.wait_event(copied[i % k])
        tr.encode(stream=ctl)
        tr.plan(stream=ctl)
        planned = torch.cuda.Event()
        planned.record(ctl)
        side.wait_event(planned)
        tr.prepare_pack(pool, slab, stream=side)
        tr.prepare_unpack(slab, dst_pool, stream=side)
        prepared = torch.cuda.Event()
        prepared.record(side)
        tr.rebuild(stream=side)
        rebuilt = torch.cuda.Event()
        rebuilt.record(side)
        main.wait_event(prepared)
        tr.pack_prepared(pool, slab, stream=main)
        tr.unpack_prepared(slab, dst_pool, stream=main)
        main.wait_event(rebuilt)
        done = torch.cuda.Event()
        done.record(main)
        copied[i % k] = done
    # the last pass's preparations and rebuild were joined into main above, so
    # every operation on ctl and side is ordered before main's end
