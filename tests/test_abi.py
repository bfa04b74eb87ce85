"""The C ABI library builds, loads and exports every entry point that
include/kvx.h declares (no GPU needed: nothing is launched)."""
import os
import re
import subprocess

from conftest import ROOT


def _declared():
    src = open(os.path.join(ROOT, "include", "kvx.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvx_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_five_calls():
    names = _declared()
    for n in ("kvx_encode_runs", "kvx_plan_bounds", "kvx_plan_groups", "kvx_rebuild", "kvx_pack",
              "kvx_unpack"):
        assert n in names


def test_library_exports_every_declared_symbol():
    from paged_kv_cache_kvx_gb300 import build
    path = build.build()
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (kvx_[a-z_0-9]+)$", out, flags=re.M))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing


def test_library_loads_and_answers_host_queries():
    from paged_kv_cache_kvx_gb300 import kvx
    assert kvx.kvx_version() >= 100
    assert kvx.kvx_run_capacity(1000, 576) == 576 * 500
    assert kvx.kvx_run_capacity(7, 3) == 12
    # 576k spans plus one extra piece per 32 MiB of slab
    assert kvx.kvx_desc_capacity(1000, 576, 576 * 4096) == 576000 + 71
    assert kvx.kvx_encode_workspace_size(1000, 576) > 0
    assert kvx.kvx_plan_workspace_size(576, 288000, 2**31) > 0
    assert kvx.kvx_copy_workspace_size(2**31) >= 4 * (2**31 // 32768)


def test_plan_bounds_through_the_c_abi():
    """kvx_plan_bounds: one group per run at most (the greedy bound when the
    run count is unknown), one read per segment plus one piece per 32 MiB."""
    import ctypes
    from paged_kv_cache_kvx_gb300 import kvx
    L = kvx.lib()
    g, d = ctypes.c_uint64(7), ctypes.c_uint64(7)
    assert L.kvx_plan_bounds(1000, 576, 0, 576 * 4096, ctypes.addressof(g), ctypes.addressof(d)) == 0
    assert (g.value, d.value) == (576 * 500, 576000 + 71)
    # the default table's 576 runs (one per lane)
    assert kvx.kvx_plan_bounds(1000, 576, 576, 576 * 4096) == (576, 576000 + 71)
    assert kvx.kvx_plan_bounds(0, 0, 0, 0) == (0, 0)
    # more runs than any greedy encoding of B blocks has, or a missing output
    assert L.kvx_plan_bounds(1000, 576, 576 * 500 + 1, 4096, ctypes.addressof(g),
                             ctypes.addressof(d)) == EINVAL
    assert L.kvx_plan_bounds(1000, 576, 576, 4096, None, ctypes.addressof(d)) == EINVAL
    assert L.kvx_plan_bounds(1000, 576, 576, 4096, ctypes.addressof(g), None) == EINVAL


def test_plan_sm_share_rejects_other_values():
    """kvx_plan_set_sm_share takes 1 or 2 blocks per SM; anything else is
    KVX_EINVAL before the device is looked at."""
    from paged_kv_cache_kvx_gb300 import kvx
    L = kvx.lib()
    for bad in (0, 3, 4, 2**32 - 1):
        assert L.kvx_plan_set_sm_share(bad) == EINVAL


def test_binding_has_no_cpu_fallback():
    """The product path refuses to run without its CUDA library."""
    from paged_kv_cache_kvx_gb300 import kvx
    saved = kvx._lib
    try:
        kvx._lib = None
        orig = kvx.lib_path
        kvx.lib_path = lambda: "/nonexistent/libkvx.so"
        try:
            kvx.lib()
            raised = False
        except kvx.KvxError:
            raised = True
        assert raised
    finally:
        kvx.lib_path = orig
        kvx._lib = saved


# Host-side argument checks return before any CUDA call, so they run here
# without a GPU.  Pointers are dummy non-null addresses that are never
# dereferenced; KVX_EINVAL = 1, KVX_ECAPACITY = 3.
EINVAL, ECAPACITY = 1, 3
P = 0x1000  # a non-null dummy device pointer


def _lib():
    from paged_kv_cache_kvx_gb300 import kvx
    return kvx.lib()


def test_encode_rejects_small_capacity_and_workspace():
    L = _lib()
    B, Ln = 1000, 576
    cap = int(L.kvx_run_capacity(B, Ln))
    ws = int(L.kvx_encode_workspace_size(B, Ln))
    assert L.kvx_encode_runs(P, B, Ln, P, P, P, P, cap - 1, P, P, P, ws, None) == ECAPACITY
    assert L.kvx_encode_runs(P, B, Ln, P, P, P, P, cap, P, P, P, ws - 1, None) == EINVAL
    assert L.kvx_encode_runs(P, B, Ln, P, P, P, P, cap, P, None, P, ws, None) == EINVAL  # no status
    assert L.kvx_verify_encode(P, None, P, B, Ln, P, P, P, P, P, cap, P, P, P, ws, None) == EINVAL


def test_plan_rejects_oversized_run_capacity():
    L = _lib()
    args = [P, 4, P, P, P, P, (1 << 31) + 1, 10, P, P, 4, 1 << 20, P, 1, P, 1, P, P, P, P, P, P, P,
            1 << 40, None]
    assert L.kvx_plan_groups(*args) == EINVAL


def test_copies_reject_small_workspaces():
    L = _lib()
    slab = 1 << 30
    ws = int(L.kvx_copy_workspace_size(slab))
    # below even the tile lists
    assert L.kvx_pack(P, 1 << 31, P, P, 10, P, slab, P, P, 64, None) == EINVAL
    assert L.kvx_unpack(P, slab, P, P, 10, P, 1 << 31, P, P, 64, None) == EINVAL
    # the segment copies: a workspace, if given, must hold the claim counter
    seg_ws = int(L.kvx_segcopy_workspace_size())
    assert seg_ws >= 4
    assert L.kvx_paged_writes(4096, P, 1 << 20, P, 4096, 0, P, 1 << 20, P, 4096, 0, 10, P, P,
                              seg_ws - 1, None) == EINVAL
    assert L.kvx_paged_writes(4096, P, 1 << 20, P, 4096, 0, P, 1 << 20, P, 4096, 0, 10, None, P,
                              seg_ws, None) == EINVAL  # no status word
    # nothing to copy: returns at once, no launch
    assert L.kvx_paged_writes(4096, P, 1 << 20, P, 4096, 0, P, 1 << 20, P, 4096, 0, 0, P, None, 0,
                              None) == 0
    assert L.kvx_seal_blocks(P, P, P, P, P, 10, P, 10, P, 4, 4, P, P, 1 << 20, P, P, 1 << 20, P, P,
                             seg_ws - 1, None) == EINVAL
    assert ws > 0


def test_prepared_copies_reject_bad_arguments():
    L = _lib()
    slab = 1 << 30
    ws = int(L.kvx_copy_workspace_size(slab))
    for fn in (L.kvx_copy_prepare, L.kvx_pack_prepared, L.kvx_unpack_prepared):
        assert fn(P, 1 << 31, P, P, 10, P, slab, P, P, 64, None) == EINVAL      # workspace too small
        assert fn(P, 1 << 31, P, P, 10, P, slab, None, P, ws, None) == EINVAL   # no status word
        assert fn(P, 1 << 31, None, P, 10, P, slab, P, P, ws, None) == EINVAL   # no descriptors
        assert fn(None, 1 << 31, P, P, 10, P, slab, P, P, ws, None) == EINVAL   # pool bytes, no pool


def test_noalloc_pack_rejects_slabs_beyond_its_scratch():
    L = _lib()
    assert L.kvx_pack_noalloc(P, 1 << 40, P, P, 10, P, 1 << 34, P, None) == ECAPACITY
