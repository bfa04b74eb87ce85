#!/usr/bin/env python
"""Benchmark of the paged KV block-transfer path on GB300.

One step = one pass of the whole path over the default workload (1000 blocks
x 288 slots x 2 x 4 KiB = 576k segments, 2250 MiB, bump-allocated holder in
two NUMA regions): kvx_encode_runs, kvx_plan_groups, kvx_rebuild, kvx_pack,
kvx_unpack, all on one stream with inputs resident in HBM.  The headline
value is pack+unpack bytes (read + write: 4 N per step) over the step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kvx|reference]

--impl reference times the CPU oracle (the method as plain single-threaded
C) on a bounded sample of the same workload.  Under torchrun every rank runs
its own replica (independent transfers: weak scaling, no collective on the
data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV pack+unpack GB/s (fraction of HBM peak); run-encode Msegments/s"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0      # the ~8 TB/s nominal HBM3e figure
FALLBACK_HBM_GBS = 6800.0     # profiling recipe's fallback when no measured peak exists
WORKLOAD = ("default: 1000 blocks x 288 slots x 2 segments (K,V) x 4 KiB uint8 = 576,000 "
            "segments, 2250 MiB, bump-allocated holder, slots 0-143 / 144-287 in two NUMA regions")
# the copy kernels' translation units: the kernel file, then the headers it
# compiles with (a change to any of them can change the kernel)
COPY_SRC = [os.path.join(ROOT, "paged_kv_cache_kvx_gb300", "csrc", f)
            for f in ("kvx_copy.cu", "kvx_ring.cuh", "kvx_common.cuh")]
PROFILE = os.path.join(ROOT, "profiles", "copy_default.md")
SEGCOPY_SRC = [os.path.join(ROOT, "paged_kv_cache_kvx_gb300", "csrc", f)
               for f in ("kvx_segcopy.cu", "kvx_ring.cuh", "kvx_common.cuh")]


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, device=None) -> float:
    """The largest of every rank's x (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def step_value(payload_bytes: int, steps: int, world: int, total_ms: float) -> float:
    """Whole-job GB/s: every rank moves 4 N bytes per step (pack and unpack
    each read and write N), over the slowest rank's time."""
    return 4.0 * payload_bytes * steps * world / (total_ms / 1e3) / 1e9


def host_info():
    """The host the CPU baseline ran on: logical cores and CPU model."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware") and ":" in line:
                    model = line.split(":", 1)[1].strip()
                    break
                if key == "cpu part" and not model:
                    model = "cpu part " + line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return {"nproc": os.cpu_count(), "cpu": model or platform.processor() or platform.machine()}


def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def copy_kernel_hash(src=COPY_SRC):
    """First 16 hex digits of the SHA-256 of a source file (or of several,
    concatenated in order)."""
    h = hashlib.sha256()
    for path in ([src] if isinstance(src, str) else src):
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def stage_roofline(med_ms, S, R, G, D, L, N, peak):
    """Every stage of one pass against the HBM roofline: its algorithmic bytes
    (what the step must read and write at least), those bytes over the
    stage's median time, and that rate as a fraction of the measured peak.
    encode: the address table read (8 B per segment), the run table written
    (20 B per run, 4 B per lane); plan: the run table read, lane_first,
    run_block / run_group / run_off (16 B per run), groups (48 B) and reads
    (32 B) written; rebuild: a pointer per segment written (8 B), the per-run
    records (first block, group, base, stride: 24 B) and groups read; pack,
    unpack: N read and N written."""
    nbytes = {
        "encode": 8 * S + 20 * R + 4 * L,
        "plan": 20 * R + 4 * L + 4 * (L + 1) + 16 * R + 48 * G + 32 * D + 24,
        "rebuild": 8 * S + 24 * R + 48 * G + 4 * (L + 1),
        "pack": 2 * N,
        "unpack": 2 * N,
    }
    out = {}
    for i, name in enumerate(["encode", "plan", "rebuild", "pack", "unpack"]):
        gbs = nbytes[name] / (float(med_ms[i]) / 1e3) / 1e9
        out[name] = {"algorithmic_bytes": int(nbytes[name]), "gbs": gbs, "frac": gbs / peak,
                     "bound": "hbm" if name in ("pack", "unpack") else "latency"}
    return out


def profiled_traffic(profile=PROFILE, src=COPY_SRC):
    """DRAM bytes per launch from a committed ncu summary, only while the
    kernel's source is the one that was profiled."""
    try:
        text = open(profile).read()
    except OSError:
        return None
    m = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", text)
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m or not t or m.group(1) != copy_kernel_hash(src):
        return None
    return float(t.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="kvx_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------- oracle arm

def oracle_sample_step(wl, host_pool):
    """One pass of the whole path through the CPU oracle; returns seconds."""
    import oracle
    t0 = time.perf_counter()
    t = oracle.encode_runs(wl.addr)
    p = oracle.plan(t, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    st, local = oracle.rebuild(t, p, wl.blocks, wl.lanes, wl.seg_len)
    slab = np.empty(p.slab_bytes, dtype=np.uint8)
    s1 = oracle.pack(host_pool, p.descs, slab)
    dst = np.empty(wl.pool_bytes, dtype=np.uint8)
    s2 = oracle.unpack(slab, p.descs, dst)
    dt = time.perf_counter() - t0
    if p.status or st or s1 or s2:
        raise RuntimeError("oracle sample failed")
    return dt


def oracle_sample_workload(name: str):
    """A bounded sample of a workload for the CPU oracle: the same generator
    with fewer blocks (the table's per-block structure, slot template and
    address pattern kept).  Returns (workload, full-size block count)."""
    from paged_kv_cache_kvx_gb300 import workloads as W
    if name == "default":
        return W.bump("default_sample", blocks=100, slots=288, seg=4096, seed=2), 1000
    if name == "tiny":
        return W.tiny(), 8
    if name == "worst":
        return W.worst(blocks=100, npos=248), 1000
    if name == "mixed":
        return W.mixed(blocks=256), 4096
    if name == "many_small":
        return W.many_small(blocks=5000, nreloc=250), 100_000
    if name == "wide64k":
        return W.bump("wide64k_sample", blocks=10, slots=288, seg=64 * 1024, nregions=2, seed=6), 200
    if name == "konly":
        return W.k_only("bump", name="default_sample", blocks=100), 1000
    raise ValueError(name)


def oracle_baseline(target_s: float, workload: str = "default"):
    """The oracle on a bounded sample of the workload, repeated for about
    target_s seconds.  Returns (GB/s, description, steps, seconds per pass)."""
    from paged_kv_cache_kvx_gb300 import workloads as W
    wl, full_blocks = oracle_sample_workload(workload)
    pool = W.holder_pool_np(wl)
    first = oracle_sample_step(wl, pool)
    n = max(1, int(target_s / max(first, 1e-6)))
    times = [oracle_sample_step(wl, pool) for _ in range(n)]
    per = statistics.median(times)
    gbs = 4 * wl.payload_bytes / per / 1e9
    desc = ("oracle encode+plan+rebuild+pack+unpack on %d of the %d blocks of the %s workload's "
            "generator (%d segments, %.0f MiB), median of %d passes, single thread"
            % (wl.blocks, full_blocks, workload, wl.segments, wl.payload_bytes / 2**20, n))
    return gbs, desc, n, per


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from paged_kv_cache_kvx_gb300 import workloads as W
    import oracle
    oracle.build()
    # size the sample so warm-up + timed passes take about a minute
    probe = W.bump("default_probe", blocks=20, slots=288, seg=4096, seed=2)
    ppool = W.holder_pool_np(probe)
    t_probe = oracle_sample_step(probe, ppool) / 20.0
    target_s = 60.0
    blocks = int(max(2, min(1000, target_s / max(1e-9, t_probe * (args.steps + args.warmup)))))
    wl = W.bump("default_sample", blocks=blocks, slots=288, seg=4096, seed=2)
    pool = W.holder_pool_np(wl)
    for _ in range(args.warmup):
        oracle_sample_step(wl, pool)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_step(wl, pool)
    dt = time.perf_counter() - t0
    value = 4 * wl.payload_bytes * args.steps / dt / 1e9
    sample = ("first %d of 1000 blocks of the default workload per step (%d segments, %.1f MiB), "
              "single-threaded C oracle" % (blocks, wl.segments, wl.payload_bytes / 2**20))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample_blocks": blocks},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "host": host_info(),
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------------- kvx arm

def check_parity(tr, wl, pool, slab, dst, local_dev_np=None):
    """The same process checks the CUDA path against the oracle first."""
    import oracle
    import torch
    from paged_kv_cache_kvx_gb300 import workloads as W
    t = oracle.encode_runs(wl.addr)
    p = oracle.plan(t, wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes)
    st, local = oracle.rebuild(t, p, wl.blocks, wl.lanes, wl.seg_len)
    assert p.status == 0 and st == 0
    assert tr.read_status() == 0, "device status %#x" % tr.read_status()
    rpl, base, stride, count = tr.read_table()
    assert np.array_equal(rpl, t.runs_per_lane) and np.array_equal(base, t.run_base)
    assert np.array_equal(stride, t.run_stride) and np.array_equal(count, t.run_count)
    g = tr.read_plan()
    assert g["groups"].tobytes() == p.groups.tobytes()
    assert g["descs"].tobytes() == p.descs.tobytes()
    assert np.array_equal(tr.read_local(), local)
    rng = np.random.default_rng(0)
    for b, l in zip(rng.integers(0, wl.blocks, 64), rng.integers(0, wl.lanes, 64)):
        a, lo, n = int(wl.addr[b, l]), int(local[b, l]), int(wl.seg_len[l])
        assert np.array_equal(slab[lo:lo + n].cpu().numpy(), W.pool_bytes_np(wl.seed, a, n))
    assert pool_identity(wl, pool, dst)
    return len(p.descs), len(p.groups), t.num_runs


def pool_identity(wl, pool, dst):
    """Every block position in use holds the same bytes in pool and dst (the
    segments tile each used position, so this covers every segment byte)."""
    import torch
    for (first, nslots, base, npos), pos in zip(wl.regions, wl.pos):
        chunk = int(wl.seg_len[2 * first:2 * (first + nslots)].astype(np.int64).sum())
        used = np.zeros(npos, dtype=bool)
        used[pos] = True
        u = torch.from_numpy(used).to(pool.device)
        a = pool[base:base + npos * chunk].view(npos, chunk)
        d = dst[base:base + npos * chunk].view(npos, chunk)
        if not torch.equal(a[u], d[u]):
            return False
    return True


# the workloads the default run also measures (each its own entry of
# per_workload), then the calls beyond the main path
PER_WORKLOAD = ["worst", "mixed", "many_small", "wide64k", "tiny", "konly"]
PER_CALL = ["seal", "paged", "verify"]


def make_workload(name: str, blocks: int = 1000):
    """A workload by name (blocks != 1000 gives the reduced tables used for
    profiler captures)."""
    from paged_kv_cache_kvx_gb300 import workloads as W
    if name == "konly":
        return W.k_only("bump", name="default")
    if blocks != 1000:
        if name == "worst":
            return W.worst(blocks=blocks, npos=2 * blocks + 48)
        if name == "many_small":
            return W.many_small(blocks=blocks, nreloc=blocks // 20)
        if name == "mixed":
            return W.mixed(blocks=blocks)
        if name == "default":
            return W.bump("default", blocks=blocks, slots=288, seg=4096, nregions=2, seed=2)
    return W.CONFIGS[name]()


def describe(name: str, wl) -> str:
    if name == "default":
        return WORKLOAD
    if name == "konly":
        return ("konly: the default shape as a K-only cache (1000 blocks x 288 slots, K 4 KiB, "
                "V 0 B), 1125 MiB per copy")
    return "%s: %d blocks x %d slots x 2 x %d B, %d segments, %.1f MiB payload" % (
        name, wl.blocks, wl.slots, wl.seg, wl.segments, wl.payload_bytes / 2**20)


def l2_note(wl) -> str:
    N = wl.payload_bytes
    if min(wl.pool_bytes, N) > 129e6:
        return ("inputs larger than L2 (%.0f MiB pool, %.0f MiB slab vs 129 MB), no flush"
                % (wl.pool_bytes / 2**20, N / 2**20))
    return ("inputs of %.2f MiB pool, %.2f MiB slab stay in L2 (not flushed: a parity configuration, "
            "not the headline)" % (wl.pool_bytes / 2**20, N / 2**20))


# Blocks per SM of the planner's grid (kvx_plan_set_sm_share) in each launch
# mode: two where a pass runs alone on the device (stream-launched steps, one
# transfer at a time), one where each pass is planned beside the previous
# pass's copies (the overlapped graph: its grid must be resident beside them).
PLAN_SHARE = {"stream": 2, "graph": 2, "overlapped": 1}


def measure_path(wl, K, warmup, dev, world, sample_clocks):
    """The whole path on one workload: one step checked against the oracle
    first, then K steps launched call by call with an event between calls, K
    replays of one captured step, and K independent transfers back to back
    (overlapped graph).  Returns the buffers and every raw figure."""
    import torch
    from paged_kv_cache_kvx_gb300 import kvx, workloads as W
    kvx.kvx_plan_set_sm_share(PLAN_SHARE["stream"])
    tr = kvx.Transfer(wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes, device=dev)
    tr.set_addr(wl.addr)
    pool = torch.empty(wl.pool_bytes, dtype=torch.uint8, device=dev)
    W.fill_pool_torch(pool, wl.seed)
    slab = torch.empty(tr.slab_bytes, dtype=torch.uint8, device=dev)
    dst = torch.full((wl.pool_bytes,), W.CANARY, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        tr.step(pool, slab, dst, stream=stream)
    torch.cuda.synchronize()
    ndescs, ngroups, nruns = check_parity(tr, wl, pool, slab, dst)

    for _ in range(max(3, warmup)):
        tr.step(pool, slab, dst, stream=stream)
    torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index or 0) if sample_clocks else None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    launches0 = kvx.kvx_launch_count()
    start.record(stream)
    for i in range(K):
        e = ev[i]
        e[0].record(stream)
        tr.encode(stream=stream)
        e[1].record(stream)
        tr.plan(stream=stream)
        e[2].record(stream)
        tr.rebuild(stream=stream)
        e[3].record(stream)
        tr.pack(pool, slab, stream=stream)
        e[4].record(stream)
        tr.unpack(slab, dst, stream=stream)
        e[5].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    launches = kvx.kvx_launch_count() - launches0
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    total_ms = start.elapsed_time(end)
    stage = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(5)] for e in ev])  # ms
    total_ms = max_over_ranks(total_ms, device=dev)
    assert tr.read_status() == 0
    assert pool_identity(wl, pool, dst)

    # The same step captured once as a CUDA graph and replayed K times (the
    # path keeps its counts on the device, so one capture replays every step).
    kvx.kvx_plan_set_sm_share(PLAN_SHARE["graph"])
    graph_ms, graph_launches = measure_graph(tr, wl, pool, slab, dst, K, world, dev)
    if graph_ms is not None:
        graph_ms = max_over_ranks(graph_ms, device=dev)
    # Independent transfers back to back, as a server streams them: a second
    # set of metadata lets each pass's encode and plan run while the previous
    # pass copies (every pass still does all five calls).
    tr2 = kvx.Transfer(wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes, device=dev)
    tr2.set_addr(wl.addr)
    kvx.kvx_plan_set_sm_share(PLAN_SHARE["overlapped"])
    over_ms, over_launches = measure_graph_overlapped([tr, tr2], wl, pool, slab, dst, K, world, dev)
    kvx.kvx_plan_set_sm_share(PLAN_SHARE["stream"])  # e2e and later calls run one transfer at a time
    if over_ms is not None:
        over_ms = max_over_ranks(over_ms, device=dev)
    clocks = sampler.stop() if sampler else None  # sampled over all three timed regions
    del tr2
    return dict(tr=tr, pool=pool, slab=slab, dst=dst, stream=stream, nruns=nruns, ngroups=ngroups,
                ndescs=ndescs, total_ms=total_ms, stage=stage, launches=launches,
                graph_ms=graph_ms, graph_launches=graph_launches, over_ms=over_ms,
                over_launches=over_launches, clocks=clocks)


def path_figures(wl, m, K, world, peak, peak_kind):
    """Every figure of one measured workload: the fastest of the three launch
    modes as the value, each stage's mean and median time, pack and unpack
    against the HBM roofline (2 N bytes over the call's mean time) and as
    payload rates (N over the call's mean time), encode and rebuild
    Msegments/s and every stage against its algorithmic bytes."""
    N, S = wl.payload_bytes, wl.segments
    total_ms, launch_mode, launches = m["total_ms"], "stream", m["launches"]
    stream_value = step_value(N, K, world, total_ms)
    graph_ms, over_ms = m["graph_ms"], m["over_ms"]
    graph_value = step_value(N, K, world, graph_ms) if graph_ms is not None else None
    if graph_ms is not None and graph_ms < total_ms:
        total_ms, launch_mode, launches = graph_ms, "cuda_graph", m["graph_launches"]
    if over_ms is not None and over_ms < total_ms:
        total_ms, launch_mode, launches = over_ms, "cuda_graph_overlapped", m["over_launches"]
    med = np.median(m["stage"], axis=0)
    mean = m["stage"].mean(axis=0)
    pack_gbs = 2.0 * N / (mean[3] / 1e3) / 1e9
    unpack_gbs = 2.0 * N / (mean[4] / 1e3) / 1e9
    both = 4.0 * N / ((mean[3] + mean[4]) / 1e3) / 1e9
    dom = 3 if mean[3] >= mean[4] else 4
    achieved = 2.0 * N / (mean[dom] / 1e3) / 1e9
    names = ["encode", "plan", "rebuild", "pack", "unpack"]
    return {
        "value": step_value(N, K, world, total_ms), "ms_per_step": total_ms / K,
        "launch_mode": launch_mode, "gpu_launches": int(launches), "plan_sm_share": dict(PLAN_SHARE),
        "value_stream_launched": stream_value, "value_graph_one_transfer_at_a_time": graph_value,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "kvx_pack" if dom == 3 else "kvx_unpack",
                     "peak_source": "%s hbm_gbs" % peak_kind},
        "pack_gbs": pack_gbs, "unpack_gbs": unpack_gbs, "pack_unpack_gbs": both,
        "frac_of_%s_peak" % peak_kind: both / peak,
        "frac_of_nominal_8tbs": both / NOMINAL_HBM_GBS,
        "encode_msegs_per_s": S / (mean[0] / 1e3) / 1e6,
        "rebuild_msegs_per_s": S / (mean[2] / 1e3) / 1e6,
        "pack_payload_gbs": N / (mean[3] / 1e3) / 1e9,
        "unpack_payload_gbs": N / (mean[4] / 1e3) / 1e9,
        "stage_ms_mean": dict(zip(names, map(float, mean))),
        "stage_ms_median": dict(zip(names, map(float, med))),
        "stage_roofline": stage_roofline(med, S, m["nruns"], m["ngroups"], m["ndescs"], wl.lanes, N,
                                         peak),
    }


def workload_entry(name, args, dev, peak, peak_kind):
    """One entry of per_workload: the workload's full step checked against
    the oracle, measured as the headline is, with the oracle's rate on a
    bounded sample of the same generator."""
    import torch
    wl = make_workload(name)
    m = measure_path(wl, args.steps, args.warmup, dev, 1, True)
    entry = {"workload": describe(name, wl), "segments": wl.segments,
             "payload_bytes": wl.payload_bytes, "bytes_moved_per_step": 4 * wl.payload_bytes,
             "runs": m["nruns"], "groups": m["ngroups"], "descs": m["ndescs"],
             "parity": ("run table, plan and rebuilt pointers equal to the oracle's; sampled slab "
                        "segments equal to the generator's bytes; every used pool position "
                        "restored by unpack"),
             "l2": l2_note(wl)}
    entry.update(path_figures(wl, m, args.steps, 1, peak, peak_kind))
    entry["clocks"] = m["clocks"]
    for k in ("tr", "pool", "slab", "dst"):
        m.pop(k)
    del m
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    cb, desc, n, per = oracle_baseline(target_s=args.aux_cpu_seconds, workload=name)
    entry["cpu_baseline"] = {"value": cb, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "host": host_info(), "sample": desc}
    return entry


def run_kvx(args):
    import torch
    import torch.distributed as dist
    from paged_kv_cache_kvx_gb300 import build

    rank, world, local_rank = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    build.build()
    reduced = args.blocks != 1000
    # e2e, the memcpy comparator and the oracle leg are measured on the
    # default workload's own line; profiler captures (--no-aux, reduced
    # tables) skip them
    headline = args.workload == "default" and not reduced
    aux = headline and not args.no_aux
    oracle_leg = not args.no_aux and not reduced
    wl = make_workload(args.workload, args.blocks)
    N = wl.payload_bytes
    K = args.steps
    m = measure_path(wl, K, args.warmup, dev, world, rank == 0)
    tr, pool, slab, dst, stream = m["tr"], m["pool"], m["slab"], m["dst"], m["stream"]

    # end to end through the same calls with host buffers
    e2e = measure_e2e(tr, wl, pool, slab, dst, stream, args, dev) if aux else None
    # comparator: one plain device-to-device copy of N bytes
    memcpy_gbs = measure_memcpy(pool, slab, N, stream) if aux else None

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    peak, peak_kind = load_peak()
    fig = path_figures(wl, m, K, world, peak, peak_kind)
    # the committed counters are per launch of the default workload only
    fig["roofline"]["traffic"] = profiled_traffic() if headline else None
    line = {
        "metric": METRIC, "value": fig.pop("value"), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": fig.pop("ms_per_step"), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": describe(args.workload, wl), "bytes_moved_per_step": 4 * N,
                   "l2": l2_note(wl), "runs": m["nruns"], "groups": m["ngroups"],
                   "descs": m["ndescs"]},
    }
    line["roofline"] = fig.pop("roofline")
    line.update(fig)
    line["memcpy_d2d_gbs"] = memcpy_gbs
    line["e2e"] = e2e
    line["clocks"] = m["clocks"]
    if reduced:
        line["config"]["workload"] = "reduced for profiling: %s with %d blocks" % (args.workload,
                                                                                   args.blocks)
    if world == 1 and oracle_leg:
        cb, desc, n, per = oracle_baseline(target_s=args.cpu_seconds, workload=args.workload)
        line["cpu_baseline"] = {"value": cb, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "host": host_info(),
                                "sample": desc}
    if world == 1 and aux and not args.headline_only:
        # every other configuration and the calls beyond the main path, each
        # checked against the oracle first, in the same run as the headline
        for k in ("tr", "pool", "slab", "dst"):
            m.pop(k)
        del tr, pool, slab, dst
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        per = {}
        for name in PER_WORKLOAD:
            per[name] = workload_entry(name, args, dev, peak, peak_kind)
        for name in PER_CALL:
            per[name] = measure_next(name, args, dev, args.aux_cpu_seconds)
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
        line["per_workload"] = per
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def measure_graph(tr, wl, pool, slab, dst, K, world, dev):
    """K replays of one captured step, timed with CUDA events on the replay
    stream; returns (ms, library kernels launched per K steps) or (None, 0)
    when capture is not possible."""
    import torch
    from paged_kv_cache_kvx_gb300 import kvx
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device=dev)
        torch.cuda.synchronize()
        before = kvx.kvx_launch_count()
        side = torch.cuda.Stream(device=dev)
        with torch.cuda.graph(g, stream=cap):
            tr.step(pool, slab, dst, side=side)
        per_step = kvx.kvx_launch_count() - before
    except Exception as e:  # capture unsupported here: report the stream-launched figure only
        print("graph capture unavailable: %s" % e, file=sys.stderr)
        return None, 0
    rs = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(rs):
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    dst.fill_(0)
    tr.status.zero_()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    with torch.cuda.stream(rs):
        a.record(rs)
        for _ in range(K):
            g.replay()
        b.record(rs)
    torch.cuda.synchronize()
    assert tr.read_status() == 0 and pool_identity(wl, pool, dst), "graph replay broke parity"
    return a.elapsed_time(b), per_step * K


def measure_graph_overlapped(trs, wl, pool, slab, dst, K, world, dev, per_graph=8):
    """K passes of the path as replays of one captured graph of per_graph
    passes over the transfers in trs (kvx.overlapped_steps: each pass's
    encode and plan overlap the previous pass's copies).  Returns (ms for K
    passes, library kernels launched) or (None, 0) when capture fails."""
    import torch
    from paged_kv_cache_kvx_gb300 import kvx
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device=dev)
        ctl = torch.cuda.Stream(device=dev)
        side = torch.cuda.Stream(device=dev)
        torch.cuda.synchronize()
        before = kvx.kvx_launch_count()
        with torch.cuda.graph(g, stream=cap):
            kvx.overlapped_steps(trs, pool, slab, dst, per_graph, cap, ctl, side)
        per_replay = kvx.kvx_launch_count() - before
    except Exception as e:
        print("overlapped graph capture unavailable: %s" % e, file=sys.stderr)
        return None, 0
    reps = max(1, K // per_graph)
    rs = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(rs):
        for _ in range(2):
            g.replay()
    torch.cuda.synchronize()
    dst.fill_(0)
    for tr in trs:
        tr.status.zero_()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    with torch.cuda.stream(rs):
        a.record(rs)
        for _ in range(reps):
            g.replay()
        b.record(rs)
    torch.cuda.synchronize()
    assert all(tr.read_status() == 0 for tr in trs) and pool_identity(wl, pool, dst), \
        "overlapped replay broke parity"
    # per K passes
    return a.elapsed_time(b) * K / (reps * per_graph), per_replay * reps * K // (reps * per_graph)


def measure_e2e(tr, wl, pool, slab, dst, stream, args, dev):
    """Same metric through the same calls with HOST buffers.  Every step
    copies its address table and holder pool in from pinned memory, runs the
    five calls, and copies the unpacked pool and the rebuilt pointers back to
    pinned memory.  Steps are pipelined over two buffer sets on three streams
    (copy-in of step i+1 and copy-out of step i overlap the compute), as a
    caller streaming transfers would run them; the timed region spans the
    first copy-in to the last copy-out."""
    import torch
    h_addr = torch.from_numpy(wl.addr.reshape(-1).view(np.int64).copy()).pin_memory()
    h_pool = torch.empty(wl.pool_bytes, dtype=torch.uint8).pin_memory()
    h_pool.copy_(pool, non_blocking=False)
    nset = 2
    d_addr = [tr.addr] + [torch.empty_like(tr.addr) for _ in range(nset - 1)]
    d_pool = [pool] + [torch.empty_like(pool) for _ in range(nset - 1)]
    d_dst = [dst] + [torch.empty_like(dst) for _ in range(nset - 1)]
    d_local = [tr.local] + [torch.empty_like(tr.local) for _ in range(nset - 1)]
    h_dst = [torch.empty(wl.pool_bytes, dtype=torch.uint8).pin_memory() for _ in range(nset)]
    h_local = [torch.empty(wl.blocks * wl.lanes, dtype=torch.int64).pin_memory() for _ in range(nset)]
    n_in = h_addr.numel() * 8 + h_pool.numel()
    n_out = h_dst[0].numel() + h_local[0].numel() * 8
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    nchunk = 4  # each direction split over four streams, so several copy engines share it
    c_in = [torch.cuda.Stream(device=dev) for _ in range(nchunk)]
    c_out = [torch.cuda.Stream(device=dev) for _ in range(nchunk)]
    bounds = [wl.pool_bytes * i // nchunk for i in range(nchunk + 1)]

    def chunked(streams, head, dst_t, src_t):
        """dst_t <- src_t in nchunk pieces on `streams`, ordered after `head`
        and joined back into `head`."""
        ev0 = torch.cuda.Event()
        ev0.record(head)
        done = []
        for i, cs in enumerate(streams):
            cs.wait_event(ev0)
            with torch.cuda.stream(cs):
                dst_t[bounds[i]:bounds[i + 1]].copy_(src_t[bounds[i]:bounds[i + 1]], non_blocking=True)
            e = torch.cuda.Event()
            e.record(cs)
            done.append(e)
        for e in done:
            head.wait_event(e)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_done = [ev() for _ in range(nset)]
    comp_done = [ev() for _ in range(nset)]
    out_done = [ev() for _ in range(nset)]
    used = [False] * nset

    def one(i):
        k = i % nset
        with torch.cuda.stream(s_in):
            if used[k]:
                s_in.wait_event(comp_done[k])  # step i-2 finished reading set k's inputs
            d_addr[k][: h_addr.numel()].copy_(h_addr, non_blocking=True)
            chunked(c_in, s_in, d_pool[k], h_pool)
            in_done[k].record(s_in)
        stream.wait_event(in_done[k])
        if used[k]:
            stream.wait_event(out_done[k])  # step i-2's results were copied out
        tr.local = d_local[k]  # rebuilt pointers of this step go to set k
        with torch.cuda.stream(stream):
            tr.encode(addr=d_addr[k], stream=stream)
            tr.plan(stream=stream)
            tr.rebuild(stream=stream)
            tr.pack(d_pool[k], slab, stream=stream)
            tr.unpack(slab, d_dst[k], stream=stream)
            comp_done[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[k])
            chunked(c_out, s_out, h_dst[k], d_dst[k])
            h_local[k].copy_(d_local[k][: h_local[k].numel()], non_blocking=True)
            out_done[k].record(s_out)
        used[k] = True

    for i in range(2):
        one(i)
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 24))
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(steps):
        one(i)
    b.record(s_out)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    tr.local = d_local[0]
    ok = all(bool(torch.equal(h, h_pool)) for h in h_dst)
    ok = ok and all(bool(torch.equal(h, h_local[0])) for h in h_local)
    return {"value": 4.0 * wl.payload_bytes / (ms / 1e3) / 1e9, "unit": UNIT,
            "h2d_bytes_per_step": int(n_in), "d2h_bytes_per_step": int(n_out),
            "ms_per_step": ms, "steps": steps, "pipelined_buffer_sets": nset,
            "copy_streams_per_direction": nchunk, "verified": ok}


# ------------------------------------------------- rows beyond the main path

def _events_loop(fn, K, stream):
    """K calls of fn on stream between two events; returns ms."""
    import torch
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(K):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def _timed_cpu(fn, target_s):
    fn()
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < target_s:
        fn()
        n += 1
    return (time.perf_counter() - t0) / max(n, 1), n


def run_next(args):
    """--workload paged | seal | verify as a line of its own."""
    import torch
    from paged_kv_cache_kvx_gb300 import build
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    print(json.dumps(measure_next(args.workload, args, dev, args.cpu_seconds)), flush=True)
    return 0


def measure_next(name, args, dev, cpu_seconds):
    """paged | seal | verify: the calls that widen the path, each on a
    full-size input, checked against the oracle / the generator first, then
    K launches timed with CUDA events on one stream.  Returns the line."""
    import torch
    import oracle
    from paged_kv_cache_kvx_gb300 import kvx, workloads as W

    oracle.build()
    stream = torch.cuda.Stream(device=dev)
    K = args.steps
    peak, peak_kind = load_peak()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sampler = ClockSampler(0)
    line = {"metric": METRIC, "n_gpus": 1, "steps": K, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
            "data": "synthetic", "e2e": None}

    # a reduced case for profiler captures (seal and paged only)
    reduced = args.blocks != 1000 and args.workload == name and name in ("seal", "paged")
    if name == "paged":
        # full size: 576,000 pages; reduced: 576 pages per block of --blocks
        wl = W.paged("paged", 576 * args.blocks, 4096, 720 * args.blocks, 640 * args.blocks,
                     seed=6) if reduced else W.paged_default()
        src = torch.empty(wl.src_bytes, dtype=torch.uint8, device=dev)
        W.fill_pool_torch(src, wl.seed)
        dst = torch.full((wl.dst_bytes,), W.CANARY, dtype=torch.uint8, device=dev)
        si = torch.from_numpy(wl.src_idx.view(np.int32)).to(dev)
        di = torch.from_numpy(wl.dst_idx.view(np.int32)).to(dev)

        seg_ws = torch.zeros(kvx.kvx_segcopy_workspace_size(), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()  # the buffers were filled on torch's stream, the calls run on ours

        def call():
            kvx.kvx_paged_writes(wl.page_len, src, wl.src_bytes, si, wl.src_stride, wl.src_offset,
                                 dst, wl.dst_bytes, di, wl.dst_stride, wl.dst_offset, wl.num_pages,
                                 status, seg_ws, stream)
        call()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        rng = np.random.default_rng(1)
        for i in rng.integers(0, wl.num_pages, 256):  # sampled pages against the generator
            d = wl.dst_offset + int(wl.dst_idx[i]) * wl.dst_stride
            s_ = wl.src_offset + int(wl.src_idx[i]) * wl.src_stride
            assert np.array_equal(dst[d:d + wl.page_len].cpu().numpy(),
                                  W.pool_bytes_np(wl.seed, s_, wl.page_len)), i
        N = wl.bytes_moved
        unit_bytes = 2 * N
        cfg = ("paged: 576,000 pages of 4 KiB (2250 MiB) from a 720,000-page pool to a 640,000-page "
               "pool through seeded permuted page tables (kvx_paged_writes)")
        kernel = "kvx_paged_writes"

        def cpu_leg():
            n = 20000  # 80 MiB of 4 KiB pages between two 20,000-page pools, permuted tables
            small = W.paged("paged_sample", n, wl.page_len, n, n, seed=wl.seed)
            s_np = W.pool_bytes_np(wl.seed, 0, small.src_bytes)
            d_np = np.zeros(small.dst_bytes, np.uint8)
            per, reps = _timed_cpu(lambda: oracle.paged_writes(
                small.page_len, s_np, small.src_idx, small.src_stride, 0, d_np, small.dst_idx,
                small.dst_stride, 0), cpu_seconds)
            return (2 * n * wl.page_len / per / 1e9,
                    "oracle paged_writes, %d pages of 4 KiB between two %d-page pools, %d passes"
                    % (n, n, reps))

        def status_ok():
            return int(status.item()) == 0
    elif name == "seal":
        wl = make_workload("default", args.blocks if reduced else 1000)
        tr = kvx.Transfer(wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes, device=dev)
        tr.set_addr(wl.addr)
        pool = torch.empty(wl.pool_bytes, dtype=torch.uint8, device=dev)
        W.fill_pool_torch(pool, wl.seed)
        slab = torch.empty(tr.slab_bytes, dtype=torch.uint8, device=dev)
        B, L, seg = wl.blocks, wl.lanes, wl.seg
        b = torch.arange(B, dtype=torch.int64, device=dev)[:, None]
        l = torch.arange(L, dtype=torch.int64, device=dev)[None, :]
        dst_addr = ((l * B + b) * seg).reshape(-1).contiguous()   # receiver: lane-major
        dst = torch.full((B * L * seg,), W.CANARY, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()  # the buffers were filled on torch's stream, the calls run on ours
        tr.encode(stream=stream)
        tr.plan(stream=stream)
        tr.pack(pool, slab, stream=stream)

        def call():
            tr.seal(slab, dst_addr, dst, stream=stream)
        call()
        torch.cuda.synchronize()
        assert tr.read_status() == 0
        rng = np.random.default_rng(2)
        for bb, ll in zip(rng.integers(0, B, 256), rng.integers(0, L, 256)):
            o = (int(ll) * B + int(bb)) * seg
            assert np.array_equal(dst[o:o + seg].cpu().numpy(),
                                  W.pool_bytes_np(wl.seed, int(wl.addr[bb, ll]), seg)), (bb, ll)
        N = wl.payload_bytes
        unit_bytes = 2 * N
        cfg = ("seal: the default workload's slab (2250 MiB) installed into a lane-major receiver "
               "layout with local offsets computed on the fly (kvx_seal_blocks)")
        kernel = "kvx_seal_blocks"

        def cpu_leg():
            small = W.bump("seal_sample", blocks=40, slots=288, seg=4096, seed=2)
            t = oracle.encode_runs(small.addr)
            p = oracle.plan(t, small.blocks, small.seg_len, small.numa, small.pool_bytes)
            hp = W.holder_pool_np(small)
            sl = np.zeros(p.slab_bytes, np.uint8)
            oracle.pack(hp, p.descs, sl)
            da = ((np.arange(small.lanes)[None, :] * small.blocks + np.arange(small.blocks)[:, None])
                  * small.seg).astype(np.uint64)
            d_np = np.zeros(small.payload_bytes, np.uint8)
            per, reps = _timed_cpu(lambda: oracle.seal_blocks(
                t, p, small.blocks, small.lanes, small.seg_len, sl, da, d_np), cpu_seconds)
            return 2 * small.payload_bytes / per / 1e9, "oracle seal_blocks on the first 40 of 1000 blocks, %d passes" % reps

        def status_ok():
            return tr.read_status() == 0
    else:  # verify
        wl = W.default()
        tr = kvx.Transfer(wl.blocks, wl.seg_len, wl.numa, wl.pool_bytes, device=dev)
        tr.set_addr(wl.addr)
        size_np = np.tile(wl.seg_len, (wl.blocks, 1))
        size = torch.from_numpy(size_np.view(np.int32).reshape(-1).copy()).to(dev)
        prefix = torch.zeros(1, dtype=torch.int32, device=dev)
        torch.cuda.synchronize()  # the buffers were filled on torch's stream, the calls run on ours

        def call():
            tr.verify_encode(size, prefix, stream=stream)
        # parity: every block passes here; one mismatch at block 700 ends the prefix there
        bad = size_np.copy()
        bad[700, 301] = 1
        dbad = torch.from_numpy(bad.view(np.int32).reshape(-1).copy()).to(dev)
        torch.cuda.synchronize()
        tr.verify_encode(dbad, prefix, stream=stream)
        torch.cuda.synchronize()
        pre_o, t_o = oracle.verify_encode(wl.addr, bad, wl.seg_len)
        assert int(prefix.item()) == pre_o == 700
        rpl, base, stride, count = tr.read_table()
        assert np.array_equal(count, t_o.run_count) and np.array_equal(base, t_o.run_base)
        call()
        torch.cuda.synchronize()
        assert int(prefix.item()) == wl.blocks and tr.read_status() == 0
        N = wl.segments
        unit_bytes = None
        cfg = ("verify: the default table (576,000 segments) checked block by block against the slot "
               "template and run-encoded in one cooperative launch (kvx_verify_encode)")
        kernel = "kvx_verify_encode"

        def cpu_leg():
            per, reps = _timed_cpu(lambda: oracle.verify_encode(wl.addr, size_np, wl.seg_len),
                                   cpu_seconds)
            return wl.segments / per / 1e6, "oracle verify_encode on the whole default table, %d passes" % reps

        def status_ok():
            return tr.read_status() == 0 and int(prefix.item()) == wl.blocks

    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    sampler.start()
    l0 = kvx.kvx_launch_count()
    with torch.cuda.stream(stream):
        ms = _events_loop(call, K, stream)
    launches = kvx.kvx_launch_count() - l0
    clocks = sampler.stop()
    assert status_ok()
    per_ms = ms / K
    if unit_bytes is not None:
        value = unit_bytes * K / (ms / 1e3) / 1e9
        line.update({"value": value, "unit": "GB/s",
                     "roofline": {"bound": "hbm", "achieved": value, "peak": peak, "unit": "GB/s",
                                  "frac": value / peak, "traffic": profiled_traffic(
                                      os.path.join(ROOT, "profiles", "%s_default.md" % name),
                                      SEGCOPY_SRC), "kernel": kernel,
                                  "peak_source": "%s hbm_gbs" % peak_kind}})
    else:
        value = N * K / (ms / 1e3) / 1e6
        line.update({"value": value, "unit": "Msegments/s", "roofline": None})
    if reduced:
        cfg = "reduced for profiling: %s with %d blocks (%s)" % (name, args.blocks, cfg)
    line.update({"ms_per_step": per_ms, "gpu_launches": int(launches), "clocks": clocks,
                 "launch_mode": "stream",
                 "config": {"workload": cfg, "l2": "inputs larger than L2, no flush"
                            if unit_bytes else "4.6 MB table (fits L2): latency-bound"}})
    cb, desc = cpu_leg()
    line["cpu_baseline"] = {"value": cb, "unit": line["unit"], "cores": 1, "kind": "oracle",
                            "host": host_info(),
                            "sample": desc}
    return line


def measure_memcpy(pool, slab, N, stream):
    import torch
    src = pool[:N]
    with torch.cuda.stream(stream):
        for _ in range(3):
            slab.copy_(src, non_blocking=True)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    n = 20
    with torch.cuda.stream(stream):
        for _ in range(n):
            slab.copy_(src, non_blocking=True)
    b.record(stream)
    torch.cuda.synchronize()
    return 2.0 * N * n / (a.elapsed_time(b) / 1e3) / 1e9


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["kvx", "reference"], default="kvx")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work for the oracle baseline leg of the kvx arm")
    ap.add_argument("--blocks", type=int, default=1000,
                    help="blocks of the default, worst, mixed or many_small shape (fewer only for profiler "
                         "captures; the full table otherwise)")
    ap.add_argument("--workload", default="default",
                    choices=["default", "tiny", "worst", "mixed", "many_small", "wide64k", "konly",
                             "paged", "seal", "verify"],
                    help="the default workload is the benchmark; the others are parity "
                         "configurations (konly: the default shape as a K-only cache) and the "
                         "calls beyond the main path (paged, seal, verify)")
    ap.add_argument("--no-aux", action="store_true",
                    help="skip the e2e, memcpy, CPU-baseline and per-workload legs (profiler captures)")
    ap.add_argument("--headline-only", action="store_true",
                    help="measure the default workload only (no per_workload entries)")
    ap.add_argument("--aux-cpu-seconds", type=float, default=3.0,
                    help="CPU work for the oracle leg of each per_workload entry")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.workload in ("paged", "seal", "verify"):
        return run_next(args)
    return run_kvx(args)


if __name__ == "__main__":
    sys.exit(main())
