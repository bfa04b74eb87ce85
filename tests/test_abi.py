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
    for n in ("kvx_encode_runs", "kvx_plan_groups", "kvx_rebuild", "kvx_pack", "kvx_unpack"):
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
