"""The oracle's pins catch plausible mistakes.

Each mutant below is one plausible slip in the oracle (a dropped term, a wrong
sign, index or operand, an off-by-one, a transposed copy).  It is planted in a
temporary copy of the C source on the CPU, compiled, and the pin suites
(test_oracle_pins.py, test_oracle_pins_next.py) are run against it in a
child process; every mutant must make at least one pin fail (or crash the
child).
"""
import os
import subprocess
import sys
import tempfile

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "oracle", "kvx_oracle.c")

MUTANTS = [
    ("encode_stride_sign", "stride = addr[(s + 1) * L + l] - base;", "stride = base - addr[(s + 1) * L + l];"),
    ("encode_extend_bound", "while (last + 1 < B &&", "while (last + 2 < B &&"),
    ("encode_diff_index", "addr[(last + 1) * L + l] - addr[last * L + l] == stride",
     "addr[(last + 1) * L + l] - addr[s * L + l] == stride"),
    ("encode_count_off_by_one", "run_count[R] = (uint32_t)(last - s + 1);", "run_count[R] = (uint32_t)(last - s);"),
    ("sort_drops_node", "if (a->node != b->node) return a->node < b->node ? -1 : 1;", ""),
    ("sort_base_descending", "if (a->base != b->base) return a->base < b->base ? -1 : 1;",
     "if (a->base != b->base) return a->base < b->base ? 1 : -1;"),
    ("fits_strict", "grown <= (uint64_t)g->stride", "grown < (uint64_t)g->stride"),
    ("fits_dropped", "return g->stride > 0 && grown <= (uint64_t)g->stride;", "return 1;"),
    ("adjacency_dropped_term", "r->base == g->base + g->chunk", "r->base >= g->base"),
    ("accepts_ignores_block", "r->block == g->block && ", ""),
    ("accepts_ignores_stride", "r->stride == g->stride && ", ""),
    ("dense_rule", "g->chunk == (uint64_t)g->stride", "g->chunk <= (uint64_t)g->stride"),
    ("carve_drops_count", "cursor += (uint64_t)g->count * g->chunk;", "cursor += g->chunk;"),
    ("desc_remote_uses_chunk", "uint64_t remote = g->base + i * (uint64_t)g->stride;",
     "uint64_t remote = g->base + i * g->chunk;"),
    ("desc_local_uses_stride", "uint64_t local = g->local + i * g->chunk;",
     "uint64_t local = g->local + i * (uint64_t)g->stride;"),
    ("split_16mib", "#define KVXO_MAX_READ_BYTES ((uint64_t)32 * 1024 * 1024)",
     "#define KVXO_MAX_READ_BYTES ((uint64_t)16 * 1024 * 1024)"),
    ("span_drops_len", "hi + (i128)x->len > (i128)pool_bytes", "hi > (i128)pool_bytes"),
    ("span_first_only", "i128 hi = last > first ? last : first;", "i128 hi = first;"),
    ("coverage_one_sided", "if (blk != B)", "if (blk > B)"),
    ("decode_block_step", "            blk += x->count;", "            blk += 1;"),
    ("stride1_dropped", "if (x->count == 1 && x->stride != 0)", "if (0)"),
    ("zero_count_dropped", "st |= KVXO_S_ZERO_COUNT;", ";"),
    ("rebuild_dense_drops_group_remote", "loc = (i128)g->local + ((i128)remote - (i128)g->base);",
     "loc = (i128)g->local + (i128)remote;"),
    ("rebuild_mirror_uses_stride", "loc = (i128)g->local + gb * (i128)g->chunk +",
     "loc = (i128)g->local + gb * (i128)g->stride +"),
    ("rebuild_remote_sign", "uint64_t remote = run_base[r] + i * (uint64_t)run_stride[r];",
     "uint64_t remote = run_base[r] - i * (uint64_t)run_stride[r];"),
    ("rebuild_bounds_drops_len", "loc + (i128)seg_len[l] <= slice + (i128)g->chunk", "loc <= slice + (i128)g->chunk"),
    ("pack_transposed", "memcpy(slab + d[k].local, pool + d[k].remote, d[k].len);",
     "memcpy(slab + d[k].remote, pool + d[k].local, d[k].len);"),
    ("unpack_transposed", "memcpy(dst_pool + d[k].remote, slab + d[k].local, d[k].len);",
     "memcpy(dst_pool + d[k].local, slab + d[k].remote, d[k].len);"),
    ("tiling_check_dropped", "if (d[k].local != expect || d[k].len == 0)", "if (d[k].len == 0)"),
    ("zero_len_any_lane", "if (seg_len[l] == 0 && l % 2 == 0)", "if (seg_len[l] == 0)"),
    ("zero_len_v_lanes", "if (seg_len[l] == 0 && l % 2 == 0)", "if (seg_len[l] == 0 && l % 2 == 1)"),
    ("empty_runs_not_last", "    if ((a->len == 0) != (b->len == 0)) return a->len == 0 ? 1 : -1;  /* empty runs last */\n", ""),
    ("empty_runs_first", "return a->len == 0 ? 1 : -1;  /* empty runs last */", "return a->len == 0 ? -1 : 1;"),
    ("verify_skips_instead_of_stopping", "        if (!ok)\n            break;", "        if (!ok)\n            continue;"),
    ("verify_checks_lane0_only", "for (uint32_t l = 0; l < L && ok; l++)", "for (uint32_t l = 0; l < 1 && ok; l++)"),
    ("verify_prefix_off_by_one", "taken = b + 1;", "taken = b;"),
    ("seal_drops_dst_check", "if (!in_range(dst_addr[k], seg_len[l], dst_bytes)) {", "if (0) {"),
    ("seal_lane0_length", "memcpy(dst + dst_addr[k], slab + local[k], seg_len[l]);",
     "memcpy(dst + dst_addr[k], slab + local[k], seg_len[0] - 1);"),
    ("seal_ignores_rebuild_flag", "            if (local[k] == UINT64_MAX)\n                continue;",
     "            if (local[k] == UINT64_MAX)\n                local[k] = 0;"),
    ("paged_src_uses_dst_stride", "(i128)src_idx[i] * (i128)src_stride;", "(i128)src_idx[i] * (i128)dst_stride;"),
    ("paged_drops_dst_offset", "i128 d = (i128)dst_offset + ", "i128 d = "),
    ("paged_64bit_arithmetic", "i128 s = (i128)src_offset + (i128)src_idx[i] * (i128)src_stride;",
     "i128 s = (uint64_t)(src_offset + (uint64_t)src_idx[i] * src_stride);"),
    ("paged_bounds_off_by_one", "if (d + (i128)page_len > (i128)dst_bytes) {", "if (d + (i128)page_len >= (i128)dst_bytes) {"),
    ("paged_indices_swapped", "(i128)dst_idx[i] * (i128)dst_stride;", "(i128)src_idx[i] * (i128)dst_stride;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutated = src.replace(old, new)
    c = tmp_path / "mutant.c"
    c.write_text(mutated)
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-w", "-o", str(so), str(c)])
    env = dict(os.environ, KVX_ORACLE_LIB=str(so))
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                          os.path.join(ROOT, "tests", "test_oracle_pins_next.py")],
                         env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode != 0, f"mutant {name} survived the pins:\n{res.stdout[-2000:]}"
