/*
 * kvx.h -- C ABI of libkvx, the GB300 (sm_103a) paged KV-cache block-transfer
 * path.
 *
 * The method is the one of pegaflow PR #350, "perf(transfer)!: run-encode
 * QueryBlocksForTransfer addresses and coalesce RDMA READs":
 *
 *   kvx_encode_runs  the holder's per-lane run encoding of the block prefix's
 *                    segment addresses (Holder paragraph; Wire format
 *                    paragraph: runs_per_lane / run_base / run_stride /
 *                    run_count parallel arrays)
 *   kvx_plan_groups  the requester's plan_transfer, steps 1-4 (validate;
 *                    decode, bucket per NUMA node, sort by remote base; dense
 *                    grouping; slab carve and one read per dense group or per
 *                    block) and the READ splitting paragraph (32 MiB pieces)
 *   kvx_rebuild      step 5: local(b) = group_local + (remote(b) -
 *                    group_remote), every pointer bounds-checked
 *   kvx_pack         the data movement of the planned reads: scattered holder
 *                    segments -> dense staging slab
 *   kvx_unpack       the inverse copy: slab -> a pool with the holder's layout
 *                    (not on the page; it closes the round trip)
 *   kvx_copy_prepare, kvx_pack_prepared, kvx_unpack_prepared
 *                    the same two copies split into a preparation (checks,
 *                    tile lists) and the byte movement, so one copy can be
 *                    prepared while another runs
 *
 * and the steps around it that the pages name next:
 *
 *   kvx_verify_encode  the holder's prefix scan with its two-phase check of
 *                    each block against the slot template, fused with the
 *                    run encoding (Holder paragraph)
 *   kvx_seal_blocks  seal from template metadata: fetched segments installed
 *                    at the receiver's addresses straight from the slab, the
 *                    local offsets computed on the fly (the PR's follow-up)
 *   kvx_paged_writes page-index driven copies, the paged write of the
 *                    TransferEngine API ("RDMA point-to-point communication
 *                    for LLM systems", Perplexity)
 *
 * Conventions for every call:
 *   - Array arguments are DEVICE pointers, allocated and owned by the caller.
 *     The library allocates nothing; scratch memory is the caller's `ws`
 *     buffer of at least the size the matching *_workspace_size() returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream).  They return after enqueueing.
 *   - The return value reports host-detectable problems only: KVX_EINVAL
 *     (null pointer, bad size, too-small workspace), KVX_ECAPACITY (an output
 *     capacity below the bound the call needs), KVX_ECUDA (a launch failed).
 *     Nothing is enqueued when the return value is not KVX_OK.
 *   - Data-dependent problems are OR-ed as KVX_S_* bits into the caller's
 *     device word `status` (never cleared by the library; the caller zeroes it
 *     and reads it after synchronising).  A nonzero status means the outputs
 *     of that call are undefined, except as stated per call.  No call traps
 *     or asserts.  Thread blocks wait on one another only at the grid
 *     barriers of cooperative launches (encode, verify-encode, plan), each
 *     bounded by one second of wall time, after which the kernel ORs
 *     KVX_S_TIMEOUT and returns: bad input cannot hang or fault the GPU;
 *     every global access is checked against the capacities passed in.
 *   - Co-scheduling: the grid of a cooperative launch is sized to fit on
 *     the device, but while other kernels occupy SMs (the library's own
 *     copies included: these calls are meant to run beside them) some of its
 *     blocks start only when room frees up.  If other work keeps the SMs so full
 *     that some block of kvx_encode_runs, kvx_verify_encode or
 *     kvx_plan_groups waits more than a second for room while the others
 *     wait at a grid barrier, the call ends with KVX_S_TIMEOUT and invalid
 *     outputs (reported, never silent).  Callers that run kernels lasting
 *     a second or more beside these calls should order them (a stream or
 *     an event) or re-run the call when KVX_S_TIMEOUT comes back.
 *   - Outputs must not alias inputs.
 *
 * Layouts: the address table and the rebuilt local pointers are block-major,
 * element [b][l] at b*L + l.  Lane l = 2*slot + kv (kv 0 = K, 1 = V): one
 * slot's K or V segment followed across the block prefix.  Addresses are byte
 * offsets into the holder pool; local pointers are byte offsets into the slab.
 */
#ifndef KVX_H
#define KVX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvx_status {
    KVX_OK = 0,
    KVX_EINVAL = 1,
    KVX_ECAPACITY = 3,
    KVX_ECUDA = 4
} kvx_status;

/* Device status bits: the plan's validation classes follow the page's Trust
 * boundary list (wrong lane count, bad coverage, zero-count runs, zero-size
 * slots, span overflow) and its step 1 (parallel arrays in sync). */
#define KVX_S_LANES      1u    /* table lane count != template lane count */
#define KVX_S_ARRAYS     2u    /* per-lane run counts do not add up to the run arrays' length */
#define KVX_S_COVERAGE   4u    /* a lane's run counts do not add up to the block count */
#define KVX_S_ZERO_COUNT 8u    /* a run covers zero blocks */
#define KVX_S_ZERO_LEN   16u   /* a K lane (even lane) has segment length 0 */
#define KVX_S_SPAN       32u   /* a run's remote span wraps or leaves the holder pool */
#define KVX_S_STRIDE1    64u   /* a one-block run with a nonzero stride */
#define KVX_S_BOUNDS     128u  /* a pointer or copy outside its slab/pool/group range */
#define KVX_S_DESC       256u  /* descriptors do not tile the slab in order, or a prepared
                                  copy's lists were not made for it (kvx_copy_prepare) */
#define KVX_S_CAPACITY   512u  /* a plan output exceeds its capacity, or the slab 2^63 bytes */
#define KVX_S_TIMEOUT    1024u /* a copy kernel's bounded wait on its own bulk copy gave up
                                  (the GPU did not deliver the bytes; the copy is incomplete) */

/* READ splitting: planned descriptors are split into pieces of at most
 * MAX_RDMA_READ_BYTES = 32 MiB. */
#define KVX_MAX_READ_BYTES ((uint64_t)32 * 1024 * 1024)

/* One dense group (Requester step 3): runs that share NUMA node, block range
 * and stride and whose bases are adjacent, while their summed segment length
 * (chunk) still fits the stride.  48 bytes. */
typedef struct kvx_group {
    uint64_t base;    /* remote address of the group's bytes in its first block */
    int64_t  stride;  /* remote distance between consecutive blocks */
    uint64_t chunk;   /* bytes per block = sum of member segment lengths */
    uint64_t local;   /* slab offset of the group's first byte (the carve) */
    uint32_t block;   /* first block */
    uint32_t count;   /* number of blocks */
    uint32_t node;    /* NUMA node of every member lane */
    uint32_t dense;   /* 1 when count == 1 or chunk == stride: one remote span */
} kvx_group;

/* One planned read: slab[local, local+len) <-> pool[remote, remote+len).
 * 32 bytes.  Descriptors come in group, block, piece order; their local
 * ranges tile [0, slab bytes) back to back. */
typedef struct kvx_desc {
    uint64_t remote;
    uint64_t local;
    uint64_t len;      /* 1 .. KVX_MAX_READ_BYTES */
    uint32_t group;
    uint32_t reserved; /* 0 */
} kvx_desc;

/* ------------------------------------------------------------ run encoding */

/* Greedy bound: every run but a lane's last covers >= 2 blocks, so a lane
 * has at most ceil(B/2) runs.  Returns L * ceil(B/2). */
uint64_t kvx_run_capacity(uint32_t B, uint32_t L);

size_t kvx_encode_workspace_size(uint32_t B, uint32_t L);

/*
 * Run-encode the per-segment address table (Holder paragraph, Problem
 * section: per lane the bump-allocated addresses form addr(i) = base +
 * i*stride).  Per lane, greedily: a run starts at block s, its stride is the
 * wrapping difference addr(s+1) - addr(s) (0 when s is the lane's last
 * block), and it grows while the next difference equals the stride.
 *
 *   addr           [B][L] uint64, holder-pool byte offsets (block-major).
 *   runs_per_lane  [L] out: runs of each lane.
 *   run_base, run_stride, run_count
 *                  [run_capacity] out, lane-major, blocks ascending: first
 *                  address, stride (int64 bit pattern of the uint64
 *                  difference), blocks covered.
 *   run_capacity   must be >= kvx_run_capacity(B, L) (else KVX_ECAPACITY).
 *   num_runs       [1] out: total runs R (device).
 *   status         [1] device word; encoding cannot fail on data, so the
 *                  only bit it can OR in is KVX_S_TIMEOUT (a grid barrier
 *                  of the one cooperative launch waited more than a
 *                  second; the run table is then invalid).
 *   ws, ws_bytes   scratch, >= kvx_encode_workspace_size(B, L).
 */
kvx_status kvx_encode_runs(const uint64_t *addr, uint32_t B, uint32_t L,
                           uint32_t *runs_per_lane, uint64_t *run_base,
                           int64_t *run_stride, uint32_t *run_count,
                           uint64_t run_capacity, uint64_t *num_runs,
                           uint32_t *status, void *ws, size_t ws_bytes,
                           void *stream);

/*
 * The holder's prefix scan with its slot-template check, fused with the run
 * encoding (Holder paragraph: each block is verified against the slot
 * template first and only then feeds its addresses to the per-lane run
 * accumulators, two-phase per block, so a mid-block mismatch never leaks
 * part of a block into the table).  Block b passes when seg_size[b][l] ==
 * seg_len[l] for every lane l; the prefix is the blocks before the first
 * block that fails (all B when every block passes), and the run table is
 * exactly what kvx_encode_runs writes for those blocks.
 *
 *   seg_size       [B][L] uint32, the sizes the holder's blocks actually
 *                  have (block-major, like addr).
 *   seg_len        [L] uint32, the slot template's segment lengths.
 *   prefix_blocks  [1] out (device): blocks in the prefix, B' <= B.  The
 *                  plan of this table takes B' as its block count.
 * Every other argument as for kvx_encode_runs (workspace:
 * kvx_encode_workspace_size(B, L); runs of blocks >= B' are never written).
 * One cooperative launch; a template mismatch is not an error (it only ends
 * the prefix), so status gets KVX_S_TIMEOUT at most.
 */
kvx_status kvx_verify_encode(const uint64_t *addr, const uint32_t *seg_size,
                             const uint32_t *seg_len, uint32_t B, uint32_t L,
                             uint32_t *prefix_blocks, uint32_t *runs_per_lane,
                             uint64_t *run_base, int64_t *run_stride,
                             uint32_t *run_count, uint64_t run_capacity,
                             uint64_t *num_runs, uint32_t *status, void *ws,
                             size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------ plan */

/* Bound on descriptors for a valid table: at most one span per segment
 * plus one extra piece per 32 MiB of slab.  seg_bytes_sum = sum of the
 * template's segment lengths. */
uint64_t kvx_desc_capacity(uint32_t B, uint32_t L, uint64_t seg_bytes_sum);

/*
 * Host-only helper, no device work: the output capacities kvx_plan_groups
 * needs for a table of B blocks and L lanes (Requester steps 3-4: at most one
 * group per run; at most one read per segment plus one extra piece per
 * 32 MiB of slab).
 *
 *   num_runs             the table's run count when the host knows it, or 0
 *                        for "unknown" (the greedy bound kvx_run_capacity(B,
 *                        L) is used instead).
 *   max_seg_bytes_total  sum of the template's segment lengths (bytes per
 *                        block).
 *   group_cap, desc_cap  out (host pointers): groups and descriptors to
 *                        allocate; equal to the bounds the plan checks.
 * Returns KVX_EINVAL for a null output pointer or a num_runs above
 * kvx_run_capacity(B, L) (no greedy encoding of B blocks has that many).
 */
kvx_status kvx_plan_bounds(uint32_t B, uint32_t L, uint64_t num_runs,
                           uint64_t max_seg_bytes_total, uint64_t *group_cap,
                           uint64_t *desc_cap);

size_t kvx_plan_workspace_size(uint32_t L, uint64_t run_capacity, uint64_t pool_bytes);

/*
 * Plan the transfer (Requester steps 1-4 and READ splitting).
 *
 * Step 1, validate: table_lanes == template_lanes (else KVX_S_LANES, nothing
 * else checked); per-lane run counts add up to *num_runs, which must be <=
 * run_capacity (KVX_S_ARRAYS); every K lane (even lane, l = 2*slot + kv)
 * has a segment length > 0 (KVX_S_ZERO_LEN; a V lane of length 0 is a
 * K-only cache and is accepted); every lane's counts add up to B
 * (KVX_S_COVERAGE); every
 * count > 0 (KVX_S_ZERO_COUNT); a one-block run has stride 0
 * (KVX_S_STRIDE1); base + i*stride for i in [0, count) plus the segment
 * length stays inside [0, pool_bytes) with exact arithmetic (KVX_S_SPAN).
 * All failing classes are reported together.  On any failure the counts are
 * 0 and nothing else is planned.
 * Step 2: decode each run (lane, first block, node = numa[lane], length =
 * seg_len[lane]) and sort by (node, empty, base, lane, first block), where
 * empty = (length == 0): runs that move no byte come after the node's other
 * runs, so they never split a coalescable stretch.
 * Step 3: walk the sorted runs; a run joins the open group when it has the
 * same node, first block, count and stride, its base equals group base +
 * chunk, and the grown chunk still fits the stride (count == 1, or stride > 0
 * and chunk <= stride); otherwise it opens a new group.
 * Step 4: carve the slab: groups back to back in order (so each NUMA node's
 * groups form one contiguous partition).  A dense group is one read of
 * count*chunk bytes; a non-dense group is one read of chunk bytes per block
 * into a dense local mirror.  Every read is split into 32 MiB pieces.  A
 * group of empty runs has chunk 0: no slab bytes and no read.
 *
 * Inputs: the run table as kvx_encode_runs writes it (num_runs on the
 * device); B; the slot template seg_len[template_lanes], numa[template_lanes];
 * the holder pool size.
 * Outputs: groups[group_capacity], descs[desc_capacity];
 * lane_first[table_lanes + 1] (index of each lane's first run, exclusive
 * prefix of runs_per_lane); per run run_block (decoded first block),
 * run_group, run_off (run base - group base);
 * counts[3] = {groups, descriptors, slab bytes} (device).  groups and descs
 * need their structs' 8-byte alignment; 16-byte aligned arrays are written in
 * 16-byte pieces.  run_capacity must be <= 2^31 (else KVX_EINVAL).  Capacities below
 * run_capacity groups or kvx_desc_capacity() descriptors may end in
 * KVX_S_CAPACITY on the device.
 */
kvx_status kvx_plan_groups(const uint32_t *runs_per_lane, uint32_t table_lanes,
                           const uint64_t *run_base, const int64_t *run_stride,
                           const uint32_t *run_count, const uint64_t *num_runs,
                           uint64_t run_capacity, uint32_t B,
                           const uint32_t *seg_len, const uint32_t *numa,
                           uint32_t template_lanes, uint64_t pool_bytes,
                           kvx_group *groups, uint64_t group_capacity,
                           kvx_desc *descs, uint64_t desc_capacity,
                           uint32_t *lane_first, uint32_t *run_block,
                           uint32_t *run_group, uint64_t *run_off,
                           uint64_t *counts, uint32_t *status,
                           void *ws, size_t ws_bytes, void *stream);

/*
 * The share of the device kvx_plan_groups may use for its cooperative grid,
 * in blocks per SM (default 1).  One setting per device for the whole
 * process: set for the calling thread's current device, it applies to every
 * later call on that device, from any thread.
 *   1  one block per SM: the whole grid can be resident beside a running
 *      kvx_pack / kvx_unpack bulk copy (one planner block fits next to a
 *      copy block), so a transfer is planned while another one copies.
 *   2  two blocks per SM, for a device that runs nothing else meanwhile:
 *      tables of more than one 2048-run tile per SM then give each block
 *      one tile instead of two (the many_small table plans ~18 % faster);
 *      smaller tables still work one block per SM (the first block to
 *      start on each distinct SM).  Beside a bulk copy half the grid would
 *      wait for the copy to end; if other work keeps whole SMs from hosting
 *      any planner block while fewer such SMs remain than the table has
 *      tiles, the call ends in KVX_S_TIMEOUT after about a second, like any
 *      cooperative call whose grid cannot become resident.
 * Any other value: KVX_EINVAL, setting unchanged.  The grid size is fixed
 * when a call is made (a captured graph keeps the share it was captured
 * with).
 */
kvx_status kvx_plan_set_sm_share(uint32_t blocks_per_sm);

/* ---------------------------------------------------------------- rebuild */

/*
 * Rebuild every segment's slab pointer arithmetically (Requester step 5).
 * With r the run of lane l covering block b, G its group, i = b - G.block
 * and remote(b) = run_base[r] + (b - run_block[r]) * run_stride[r] (the run
 * arithmetic, wrapping in 64 bits): a dense group gives the page's local =
 * group_local + (remote(b) - group_remote) = G.local + (remote(b) - G.base);
 * a non-dense group gives its dense local mirror, G.local + i * G.chunk +
 * (remote(b) - (G.base + i * G.stride)).  Both are evaluated exactly.  Each
 * pointer is checked: the group index is below counts[0], b lies in the
 * group's block range, the segment [local, local + seg_len[l]) lies inside
 * block i's chunk of the group carve, and the carve ends within slab_bytes.
 * A failing entry is set to UINT64_MAX and KVX_S_BOUNDS is raised.
 *
 * Inputs: lane_first [L + 1], run_block, run_group [run_capacity] and groups
 * as kvx_plan_groups wrote them; run_base, run_stride [run_capacity] as
 * kvx_encode_runs wrote them (the table that was planned); counts (device,
 * [0] = groups); seg_len [L]; slab_bytes (the slab buffer's size).
 * Output: local [B][L] uint64 (block-major).
 */
kvx_status kvx_rebuild(const uint32_t *lane_first, const uint32_t *run_block,
                       const uint64_t *run_base, const int64_t *run_stride,
                       const uint32_t *run_group, uint64_t run_capacity,
                       const kvx_group *groups, uint64_t group_capacity,
                       const uint64_t *counts, uint32_t B, uint32_t L,
                       const uint32_t *seg_len, uint64_t slab_bytes,
                       uint64_t *local, uint32_t *status, void *stream);

/* ------------------------------------------------------------ pack/unpack */

/* Scratch for kvx_pack / kvx_unpack: the slab's 64 KiB tile lists plus a
 * list of descriptor pieces (about 24 B per 2 KiB of slab).  A workspace of
 * at least the tile lists' size but below this size is accepted too: tiles
 * shared by several descriptors then all take the register path. */
size_t kvx_copy_workspace_size(uint64_t slab_bytes);

/*
 * Pack: slab[d.local, +d.len) = pool[d.remote, +d.len) for every planned
 * descriptor (the bytes of the page's coalesced reads).
 *
 *   pool, pool_bytes       holder pool (read).
 *   descs, num_descs       descriptors as kvx_plan_groups wrote them;
 *                          num_descs is a device pointer (counts + 1 of the
 *                          plan); at most desc_capacity are read.
 *   slab, slab_bytes       destination slab.
 * The descriptors must tile the slab in order (each local == previous local
 * + previous len, first local 0, every len > 0); otherwise KVX_S_DESC is
 * raised and nothing is copied.  A descriptor whose range leaves the pool or
 * the slab is skipped with KVX_S_BOUNDS; the others are copied.
 */
kvx_status kvx_pack(const uint8_t *pool, uint64_t pool_bytes,
                    const kvx_desc *descs, const uint64_t *num_descs,
                    uint64_t desc_capacity, uint8_t *slab, uint64_t slab_bytes,
                    uint32_t *status, void *ws, size_t ws_bytes, void *stream);

/*
 * Unpack, the inverse copy: dst_pool[d.remote, +d.len) = slab[d.local,
 * +d.len).  Same descriptor rules as kvx_pack.  Destination ranges of
 * different descriptors must not overlap (a valid plan of a table whose
 * segments do not overlap guarantees it); overlapping ranges give undefined
 * bytes in the overlap.  Pool bytes outside the descriptors are untouched.
 */
kvx_status kvx_unpack(const uint8_t *slab, uint64_t slab_bytes,
                      const kvx_desc *descs, const uint64_t *num_descs,
                      uint64_t desc_capacity, uint8_t *dst_pool,
                      uint64_t pool_bytes, uint32_t *status,
                      void *ws, size_t ws_bytes, void *stream);

/* -------------------------------------------- seal from template metadata */

/* Scratch for kvx_seal_blocks / kvx_paged_writes on their bulk-copy path. */
size_t kvx_segcopy_workspace_size(void);

/*
 * Seal the fetched blocks into the receiver's cache (pegaflow PR #350: the
 * follow-up named after the stage breakdown, "seal from template metadata",
 * which removes the per-segment pointer construction of step 5).  For every
 * block b < B and lane l < L: dst[dst_addr[b][l], + seg_len[l]) =
 * slab[local(b, l), + seg_len[l]), where local(b, l) is computed on the fly
 * exactly as kvx_rebuild defines it (same arithmetic, same checks) and never
 * stored.  A segment whose local offset fails a check, or whose destination
 * range leaves [0, dst_bytes), is not copied and raises KVX_S_BOUNDS; the
 * others are copied.  dst_addr = the holder table gives the bytes kvx_unpack
 * writes.
 *
 * Inputs: the run table and plan outputs as for kvx_rebuild; the slab
 * (read, slab_bytes);
 * dst_addr [B][L] uint64 byte offsets into dst (block-major); dst, dst_bytes.
 * Destination ranges must not overlap each other (else the overlap holds
 * undefined bytes) and must not overlap the slab.
 *
 * ws, ws_bytes: optional scratch of kvx_segcopy_workspace_size() bytes.
 * With it the copy runs through the SM's bulk-copy engine (shared-memory
 * rings fed by cp.async.bulk, batches claimed from a counter in ws, which
 * the call zeroes); with ws == NULL through registers (16-byte vectors),
 * allocation-free.  Both give the same bytes.  On GB300 the bulk path is the
 * faster one for segments of 2 KiB and more, the register path for shorter
 * ones.  One launch (plus a memset of ws).
 */
kvx_status kvx_seal_blocks(const uint32_t *lane_first, const uint32_t *run_block,
                           const uint64_t *run_base, const int64_t *run_stride,
                           const uint32_t *run_group, uint64_t run_capacity,
                           const kvx_group *groups,
                           uint64_t group_capacity, const uint64_t *counts,
                           uint32_t B, uint32_t L, const uint32_t *seg_len,
                           const uint8_t *slab, uint64_t slab_bytes,
                           const uint64_t *dst_addr, uint8_t *dst,
                           uint64_t dst_bytes, uint32_t *status, void *ws,
                           size_t ws_bytes, void *stream);

/* ------------------------------------------------------------ paged writes */

/*
 * Paged write by page indices ("RDMA point-to-point communication for LLM
 * systems", Perplexity: the TransferEngine API's page sets {indices, stride,
 * offset} and its paged-write call), as a device-to-device copy.  For i in
 * [0, num_pages): page_len bytes from src at src_offset + src_indices[i] *
 * src_stride go to dst at dst_offset + dst_indices[i] * dst_stride.
 * Addresses are computed exactly (no 64-bit wrap).  A page whose source
 * range leaves [0, src_bytes) raises KVX_S_SPAN, one whose destination range
 * leaves [0, dst_bytes) raises KVX_S_BOUNDS; such a page is not copied, the
 * others are.  Pages are copied in no particular order; destination pages
 * must not overlap each other or the source (else undefined bytes there).
 *
 *   src_indices, dst_indices  [num_pages] uint32 (device).
 *   src, dst                  device buffers of src_bytes / dst_bytes.
 *   ws, ws_bytes              optional, as for kvx_seal_blocks: with it, pages
 *                             of 2 KiB or more take the bulk-copy path; without
 *                             it, or for shorter pages, the register path.
 * One launch.  num_pages == 0 enqueues nothing.
 */
kvx_status kvx_paged_writes(uint64_t page_len,
                            const uint8_t *src, uint64_t src_bytes,
                            const uint32_t *src_indices, uint64_t src_stride,
                            uint64_t src_offset,
                            uint8_t *dst, uint64_t dst_bytes,
                            const uint32_t *dst_indices, uint64_t dst_stride,
                            uint64_t dst_offset,
                            uint64_t num_pages, uint32_t *status,
                            void *ws, size_t ws_bytes, void *stream);

/*
 * kvx_pack / kvx_unpack in two stages, so that the descriptor checks and the
 * tile lists of a copy can be made while another copy runs (a receiver can
 * prepare its unpack as soon as the plan is known, before the bytes arrive).
 * No counterpart in the paper: a packaging of the same data movement (Requester
 * step 4).
 *
 * kvx_copy_prepare runs the checks of kvx_pack / kvx_unpack (KVX_S_DESC,
 * KVX_S_BOUNDS into *status) and writes the tile lists into ws.  pool and slab
 * (device pointers, not dereferenced here) only decide whether the 16-byte
 * bulk paths may be used; pass the buffers the copy will use, or any with the
 * same alignment.  A following kvx_pack_prepared or kvx_unpack_prepared with
 * the same descs, num_descs, desc_capacity, pool_bytes, slab_bytes and ws moves
 * the bytes exactly as kvx_pack / kvx_unpack would; it must be ordered after
 * the preparation (same stream, or an event), and the descriptors must not
 * change in between.  One preparation serves one copy.  A copy along lists
 * that were made for other arguments, or that another copy already used,
 * moves nothing and raises KVX_S_DESC.  Arguments, sizes, ownership and
 * return codes as for kvx_pack / kvx_unpack; ws is sized by
 * kvx_copy_workspace_size(slab_bytes).
 */
kvx_status kvx_copy_prepare(const void *pool, uint64_t pool_bytes,
                            const kvx_desc *descs, const uint64_t *num_descs,
                            uint64_t desc_capacity, const void *slab, uint64_t slab_bytes,
                            uint32_t *status, void *ws, size_t ws_bytes, void *stream);
kvx_status kvx_pack_prepared(const uint8_t *pool, uint64_t pool_bytes,
                             const kvx_desc *descs, const uint64_t *num_descs,
                             uint64_t desc_capacity, uint8_t *slab, uint64_t slab_bytes,
                             uint32_t *status, void *ws, size_t ws_bytes, void *stream);
kvx_status kvx_unpack_prepared(const uint8_t *slab, uint64_t slab_bytes,
                               const kvx_desc *descs, const uint64_t *num_descs,
                               uint64_t desc_capacity, uint8_t *dst_pool, uint64_t pool_bytes,
                               uint32_t *status, void *ws, size_t ws_bytes, void *stream);

/*
 * kvx_pack without a caller workspace, for callers that cannot allocate
 * device memory (code where cudaMalloc is forbidden or would stall, such as
 * an allocation-free serving loop, or a language binding with no device
 * allocator).  The paper has no counterpart: it is a packaging variant of
 * kvx_pack.  Same arguments and results as kvx_pack, minus ws / ws_bytes.
 *
 * Its scratch is a 4 MiB file-scope device array inside libkvx, held on
 * every GPU that loads the library until the process exits.  It always
 * holds the slab's tile lists, which covers slabs up to 131,048 tiles of
 * 64 KiB (about 8 GiB); a larger slab_bytes returns KVX_ECAPACITY and
 * enqueues nothing.  For slabs up to about 5,000 tiles (about 330 MB) it
 * also holds the piece list, so tiles shared by several descriptors take the
 * bulk-copy rings as in kvx_pack; above that they take the register path
 * (same bytes).
 * Every call looks up the array's device address in the current context
 * (the caller's device and context must be current), so a context that was
 * reset, or another context on the same device, gets its own copy.  The
 * first call in a context may load this part of the library's device code
 * into that context, which the CUDA driver does with an allocation of its
 * own: make one call (or any other kvx_pack call) at initialisation, before
 * any stream capture and before the phase that must not allocate.  Every
 * call shares the array: calls that overlap on the GPU race and must be
 * serialised by the caller.  Apart from that first module load, the call
 * allocates nothing and calls no allocating routine.
 */
kvx_status kvx_pack_noalloc(const uint8_t *pool, uint64_t pool_bytes,
                            const kvx_desc *descs, const uint64_t *num_descs,
                            uint64_t desc_capacity, uint8_t *slab, uint64_t slab_bytes,
                            uint32_t *status, void *stream);

/*
 * Diagnostic, no counterpart in the paper: shows that the library's bounded
 * waits give up instead of hanging.  Launches, in order on the stream, a grid
 * barrier that waits for one block more than is launched, an mbarrier wait
 * for bytes no copy will deliver, and the planner's cross-block flag wait on
 * a flag nothing sets; each polls to its limit (about one second), then ORs
 * KVX_S_TIMEOUT into its own word of status[3] (device words: barrier,
 * mbarrier, flag) and returns.  Nothing is copied and nothing faults.
 */
kvx_status kvx_selftest_timeouts(uint32_t *status, void *stream);

/* ---------------------------------------------------------------- utility */

/* Number of kernels this library has launched in this process. */
uint64_t kvx_launch_count(void);

/* Library version, major * 10000 + minor * 100 + patch. */
uint32_t kvx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVX_H */
