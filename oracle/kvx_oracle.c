/*
 * kvx_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU statement of the paged KV block-transfer
 * path of pegaflow PR #350 ("perf(transfer)!: run-encode
 * QueryBlocksForTransfer addresses and coalesce RDMA READs").  It exists so
 * that the CUDA library can be checked against it byte for byte; nothing in
 * the product may call it.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg load it.
 *
 * It shares no code, header, table or helper with the CUDA library: every
 * structure and constant below is restated here from the page.
 *
 * Every function follows the page's steps in the page's order:
 *   kvxo_encode_runs  -- Holder paragraph: per-lane greedy arithmetic runs
 *                        (RunTableBuilder), written as the sequential rule.
 *   kvxo_plan         -- Requester steps 1-4 and "READ splitting":
 *                        validate, decode/bucket/sort, dense grouping
 *                        (group_accepts), slab carve, descriptors split at
 *                        32 MiB.
 *   kvxo_rebuild      -- Requester step 5: local(b) = group_local +
 *                        (remote(b) - group_remote), every pointer checked.
 *   kvxo_pack/unpack  -- the data movement ("data itself moves"), one memcpy
 *                        per descriptor; unpack is the inverse copy.
 *   kvxo_verify_encode -- Holder paragraph: the prefix scan checks each block
 *                        against the slot template before its addresses
 *                        enter the run accumulators (two-phase per block).
 *   kvxo_seal_blocks  -- the follow-up the PR names after its stage
 *                        breakdown (seal from template metadata): every
 *                        segment is installed from the slab at its rebuilt
 *                        offset, with no per-segment pointer table kept.
 *   kvxo_paged_writes -- "RDMA point-to-point communication for LLM
 *                        systems" (Perplexity), TransferEngine API listing:
 *                        pages named by {indices, stride, offset}, the
 *                        paged-write call copying page_len bytes per page.
 *
 * Readings where the page is silent (each is also listed in the design notes):
 *   - stride is the uint64 wrapping difference addr(s+1) - addr(s), stored as
 *     its int64 bit pattern; a run of length 1 has stride 0.
 *   - runs are emitted lane-major, blocks ascending.
 *   - sort key (node, base, lane, first block), all ascending (with empty
 *     runs after the others of their node, see below).
 *   - "grown chunk still fits the stride": fits(c) <=> count == 1 or
 *     (stride > 0 and c <= stride); a run that fails it alone still forms a
 *     one-run group.
 *   - a group is dense when count == 1 or chunk == stride: its bytes are then
 *     one contiguous remote span.
 *   - non-dense rebuild: local = G.local + i*G.chunk + (remote - (G.base +
 *     i*G.stride)), the "dense local mirror" of step 4.
 *   - descriptors split into 32 MiB pieces, remainder last; order = group,
 *     block, piece.
 *   - zero-size slots: lane l = 2*slot + kv; only a zero-size K slot (even
 *     lane) is rejected, as the page lists.  A zero-size V lane (a K-only
 *     cache) is accepted: its runs are validated like any other, but as they
 *     move no byte they must not decide how byte-carrying runs group, so
 *     they sort after every non-empty run of their NUMA node (key: node,
 *     empty, base, lane, block).  There the same grouping rule gives them
 *     groups of chunk 0 -- no slab bytes, no descriptor -- and their rebuilt
 *     pointers are empty ranges at the end of the node's partition.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status bits (one per rejected class of the page's trust boundary). */
#define KVXO_S_LANES      1u    /* table lane count != template lane count */
#define KVXO_S_ARRAYS     2u    /* parallel arrays not in sync */
#define KVXO_S_COVERAGE   4u    /* a lane's run counts do not add up to B */
#define KVXO_S_ZERO_COUNT 8u    /* a run with count 0 */
#define KVXO_S_ZERO_LEN   16u   /* a K lane (even lane) with segment length 0 */
#define KVXO_S_SPAN       32u   /* a remote span overflows / leaves the pool */
#define KVXO_S_STRIDE1    64u   /* a one-block run with nonzero stride */
#define KVXO_S_BOUNDS     128u  /* a local pointer / copy outside its range */
#define KVXO_S_DESC       256u  /* descriptors do not tile the slab in order */
#define KVXO_S_CAPACITY   512u  /* an output array is too small */

/* "planned descs are split at MAX_RDMA_READ_BYTES = 32 MiB" */
#define KVXO_MAX_READ_BYTES ((uint64_t)32 * 1024 * 1024)

typedef struct {
    uint64_t base;    /* remote address of the group's bytes in its first block */
    int64_t  stride;  /* remote distance between consecutive blocks */
    uint64_t chunk;   /* bytes per block: sum of member segment lengths */
    uint64_t local;   /* slab offset of the group's first byte */
    uint32_t block;   /* first block */
    uint32_t count;   /* number of blocks */
    uint32_t node;    /* NUMA node */
    uint32_t dense;   /* 1: count*chunk bytes form one remote span */
} kvxo_group;

typedef struct {
    uint64_t remote;
    uint64_t local;
    uint64_t len;
    uint32_t group;
    uint32_t reserved;
} kvxo_desc;

typedef __int128 i128;

/* ------------------------------------------------------------------ encode */

/*
 * Greedy per-lane run encoding (Holder paragraph; the response's parallel
 * arrays runs_per_lane / run_base / run_stride / run_count of the Wire
 * format paragraph).  A run starts at element s; its stride is
 * addr(s+1) - addr(s) (0 if s is the lane's last element); it grows while the
 * next difference equals that stride.
 *
 * addr is block-major [B][L].  Returns the number of runs written, or
 * UINT64_MAX if cap is too small.
 */
uint64_t kvxo_encode_runs(const uint64_t *addr, uint32_t B, uint32_t L,
                          uint32_t *runs_per_lane, uint64_t *run_base,
                          int64_t *run_stride, uint32_t *run_count, uint64_t cap)
{
    uint64_t R = 0;
    for (uint32_t l = 0; l < L; l++) {
        uint32_t nruns = 0;
        uint64_t s = 0;
        while (s < B) {
            uint64_t base = addr[s * L + l];
            uint64_t stride = 0;
            uint64_t last = s;           /* last element of this run */
            if (s + 1 < B) {
                stride = addr[(s + 1) * L + l] - base;
                last = s + 1;
                while (last + 1 < B &&
                       addr[(last + 1) * L + l] - addr[last * L + l] == stride)
                    last++;
            }
            if (R >= cap)
                return UINT64_MAX;
            run_base[R] = base;
            run_stride[R] = (int64_t)stride;
            run_count[R] = (uint32_t)(last - s + 1);
            R++;
            nruns++;
            s = last + 1;
        }
        runs_per_lane[l] = nruns;
    }
    return R;
}

/* -------------------------------------------------------------------- plan */

typedef struct {
    uint64_t base;
    int64_t stride;
    uint64_t len;
    uint32_t lane;
    uint32_t block;
    uint32_t count;
    uint32_t node;
} run_rec;

static const run_rec *g_sort_recs;   /* qsort has no context argument */

static int cmp_run(const void *pa, const void *pb)
{
    const run_rec *a = &g_sort_recs[*(const uint64_t *)pa];
    const run_rec *b = &g_sort_recs[*(const uint64_t *)pb];
    if (a->node != b->node) return a->node < b->node ? -1 : 1;
    if ((a->len == 0) != (b->len == 0)) return a->len == 0 ? 1 : -1;  /* empty runs last */
    if (a->base != b->base) return a->base < b->base ? -1 : 1;
    if (a->lane != b->lane) return a->lane < b->lane ? -1 : 1;
    if (a->block != b->block) return a->block < b->block ? -1 : 1;
    return 0;
}

/* "grown chunk still fits the stride" */
static int fits(const kvxo_group *g, uint64_t grown)
{
    if (g->count == 1)
        return 1;
    return g->stride > 0 && grown <= (uint64_t)g->stride;
}

/* group_accepts: same block range, same stride, base-adjacent, still fits. */
static int group_accepts(const kvxo_group *g, const run_rec *r)
{
    return r->node == g->node && r->block == g->block && r->count == g->count &&
           r->stride == g->stride && r->base == g->base + g->chunk &&
           fits(g, g->chunk + r->len);
}

/*
 * Requester plan (steps 1-4 + READ splitting).
 *
 * Inputs: the run table (runs_per_lane[table_lanes]; run_base, run_stride,
 * run_count each num_runs long), the block count B, the slot template
 * (seg_len and numa, template_lanes entries each) and the holder pool size.
 * Outputs: groups, descs, lane_first[table_lanes + 1], and per run run_block
 * (decoded first block), run_group, run_off (= run base - group base);
 * counts[0..2] = groups, descs, slab bytes.  Returns the status bitmask; on a
 * nonzero status counts are 0 and the other outputs are undefined.
 */
uint32_t kvxo_plan(const uint32_t *runs_per_lane, uint32_t table_lanes,
                   const uint64_t *run_base, const int64_t *run_stride,
                   const uint32_t *run_count, uint64_t num_runs, uint32_t B,
                   const uint32_t *seg_len, const uint32_t *numa,
                   uint32_t template_lanes, uint64_t pool_bytes,
                   kvxo_group *groups, uint64_t group_cap,
                   kvxo_desc *descs, uint64_t desc_cap,
                   uint32_t *lane_first, uint32_t *run_block,
                   uint32_t *run_group, uint64_t *run_off, uint64_t *counts)
{
    counts[0] = counts[1] = counts[2] = 0;

    /* Step 1: validate. */
    if (table_lanes != template_lanes)
        return KVXO_S_LANES;
    uint32_t st = 0;
    uint64_t total_len = 0;
    for (uint32_t l = 0; l < table_lanes; l++) {
        if (seg_len[l] == 0 && l % 2 == 0)     /* a zero-size K slot */
            st |= KVXO_S_ZERO_LEN;
        if (runs_per_lane[l] == 0 && B > 0)
            st |= KVXO_S_COVERAGE;
        total_len += seg_len[l];
    }
    uint64_t sum_runs = 0;
    for (uint32_t l = 0; l < table_lanes; l++)
        sum_runs += runs_per_lane[l];
    if (sum_runs != num_runs)
        return st | KVXO_S_ARRAYS;
    if ((i128)B * (i128)total_len >= ((i128)1 << 63))
        return st | KVXO_S_CAPACITY;

    /* Step 2: decode runs (lane, first block, node, segment length). */
    run_rec *rec = (run_rec *)malloc(sizeof(run_rec) * (num_runs ? num_runs : 1));
    uint64_t r = 0;
    for (uint32_t l = 0; l < table_lanes; l++) {
        lane_first[l] = (uint32_t)r;
        uint64_t blk = 0;
        for (uint32_t j = 0; j < runs_per_lane[l]; j++, r++) {
            run_rec *x = &rec[r];
            x->base = run_base[r];
            x->stride = run_stride[r];
            x->len = seg_len[l];
            x->lane = l;
            x->block = (uint32_t)blk;
            x->count = run_count[r];
            x->node = numa[l];
            run_block[r] = (uint32_t)blk;
            if (x->count == 0)
                st |= KVXO_S_ZERO_COUNT;
            if (x->count == 1 && x->stride != 0)
                st |= KVXO_S_STRIDE1;
            if (x->count >= 1) {
                /* the run touches base + i*stride for i in [0, count) */
                i128 first = (i128)x->base;
                i128 last = first + (i128)(x->count - 1) * (i128)x->stride;
                i128 hi = last > first ? last : first;
                if (last < 0 || hi + (i128)x->len > (i128)pool_bytes)
                    st |= KVXO_S_SPAN;
            }
            blk += x->count;
        }
        if (blk != B)
            st |= KVXO_S_COVERAGE;
    }
    lane_first[table_lanes] = (uint32_t)r;
    if (st) {
        free(rec);
        return st;
    }

    /* Step 2 (cont.): bucket per NUMA node, sort by remote base. */
    uint64_t *order = (uint64_t *)malloc(sizeof(uint64_t) * (num_runs ? num_runs : 1));
    for (uint64_t i = 0; i < num_runs; i++)
        order[i] = i;
    g_sort_recs = rec;
    qsort(order, num_runs, sizeof(uint64_t), cmp_run);

    /* Step 3: dense grouping with group_accepts. */
    uint64_t ng = 0;
    for (uint64_t p = 0; p < num_runs; p++) {
        const run_rec *x = &rec[order[p]];
        if (ng > 0 && group_accepts(&groups[ng - 1], x)) {
            kvxo_group *g = &groups[ng - 1];
            run_group[order[p]] = (uint32_t)(ng - 1);
            run_off[order[p]] = x->base - g->base;
            g->chunk += x->len;
            continue;
        }
        if (ng >= group_cap) {
            free(order);
            free(rec);
            return KVXO_S_CAPACITY;
        }
        kvxo_group *g = &groups[ng];
        g->base = x->base;
        g->stride = x->stride;
        g->chunk = x->len;
        g->local = 0;
        g->block = x->block;
        g->count = x->count;
        g->node = x->node;
        g->dense = 0;
        run_group[order[p]] = (uint32_t)ng;
        run_off[order[p]] = 0;
        ng++;
    }

    /* Step 4: slab carve (groups back to back in planner order) and one
     * descriptor per dense group / per block of a non-dense group, each
     * split into 32 MiB pieces. */
    uint64_t cursor = 0, nd = 0;
    for (uint64_t gi = 0; gi < ng; gi++) {
        kvxo_group *g = &groups[gi];
        g->dense = (g->count == 1 || (g->stride > 0 && g->chunk == (uint64_t)g->stride));
        g->local = cursor;
        uint64_t spans = g->dense ? 1 : g->count;
        uint64_t span_len = g->dense ? (uint64_t)g->count * g->chunk : g->chunk;
        for (uint64_t i = 0; i < spans; i++) {
            uint64_t remote = g->base + i * (uint64_t)g->stride;
            uint64_t local = g->local + i * g->chunk;
            for (uint64_t done = 0; done < span_len; done += KVXO_MAX_READ_BYTES) {
                if (nd >= desc_cap) {
                    free(order);
                    free(rec);
                    return KVXO_S_CAPACITY;
                }
                uint64_t piece = span_len - done;
                if (piece > KVXO_MAX_READ_BYTES)
                    piece = KVXO_MAX_READ_BYTES;
                descs[nd].remote = remote + done;
                descs[nd].local = local + done;
                descs[nd].len = piece;
                descs[nd].group = (uint32_t)gi;
                descs[nd].reserved = 0;
                nd++;
            }
        }
        cursor += (uint64_t)g->count * g->chunk;
    }
    counts[0] = ng;
    counts[1] = nd;
    counts[2] = cursor;
    free(order);
    free(rec);
    return 0;
}

/* ----------------------------------------------------------------- rebuild */

/*
 * Step 5: local(b) = group_local + (remote(b) - group_remote) for a dense
 * group; a non-dense group keeps one dense local block per remote block, so
 * its block i starts at G.local + i*G.chunk and the segment sits at its
 * remote offset from that block's remote start.  remote(b) comes from the run
 * arithmetic base + i*stride.  Every pointer is checked: the group index is in
 * range, the segment lies inside its block's slice of the group's carve, and
 * the carve lies inside the slab.  A failing entry gets UINT64_MAX.
 *
 * local is block-major [B][L].  Returns the status bitmask.
 */
uint32_t kvxo_rebuild(const uint32_t *runs_per_lane, const uint64_t *run_base,
                      const int64_t *run_stride, const uint32_t *run_count,
                      const uint32_t *run_group, const kvxo_group *groups,
                      uint64_t num_groups, uint32_t B, uint32_t L,
                      const uint32_t *seg_len, uint64_t slab_bytes, uint64_t *local)
{
    uint32_t st = 0;
    uint64_t r = 0;
    for (uint32_t l = 0; l < L; l++) {
        uint64_t blk = 0;
        for (uint32_t j = 0; j < runs_per_lane[l]; j++, r++) {
            for (uint64_t i = 0; i < run_count[r]; i++) {
                uint64_t b = blk + i;
                if (b >= B)
                    continue;
                uint64_t remote = run_base[r] + i * (uint64_t)run_stride[r];
                uint64_t out = UINT64_MAX;
                uint32_t gi = run_group[r];
                if (gi < num_groups) {
                    const kvxo_group *g = &groups[gi];
                    i128 gb = (i128)b - (i128)g->block;  /* block index inside the group */
                    i128 loc;
                    if (g->dense)
                        loc = (i128)g->local + ((i128)remote - (i128)g->base);
                    else
                        loc = (i128)g->local + gb * (i128)g->chunk +
                              ((i128)remote - ((i128)g->base + gb * (i128)g->stride));
                    i128 slice = (i128)g->local + gb * (i128)g->chunk;
                    int ok = gb >= 0 && gb < (i128)g->count && loc >= slice &&
                             loc + (i128)seg_len[l] <= slice + (i128)g->chunk &&
                             (i128)g->local + (i128)g->count * (i128)g->chunk <= (i128)slab_bytes;
                    if (ok)
                        out = (uint64_t)loc;
                }
                if (out == UINT64_MAX)
                    st |= KVXO_S_BOUNDS;
                local[b * L + l] = out;
            }
            blk += run_count[r];
        }
    }
    return st;
}

/* ------------------------------------------------------------ pack/unpack */

static uint32_t check_tiling(const kvxo_desc *d, uint64_t n)
{
    uint64_t expect = 0;
    for (uint64_t k = 0; k < n; k++) {
        if (d[k].local != expect || d[k].len == 0)
            return KVXO_S_DESC;
        expect += d[k].len;
        if (expect < d[k].len)
            return KVXO_S_DESC;
    }
    return 0;
}

static int in_range(uint64_t off, uint64_t len, uint64_t size)
{
    return off <= size && len <= size - off;
}

/* Gather: slab[local .. +len) = pool[remote .. +len) for every descriptor. */
uint32_t kvxo_pack(const uint8_t *pool, uint64_t pool_bytes, const kvxo_desc *d,
                   uint64_t n, uint8_t *slab, uint64_t slab_bytes)
{
    uint32_t st = check_tiling(d, n);
    if (st)
        return st;
    for (uint64_t k = 0; k < n; k++) {
        if (!in_range(d[k].remote, d[k].len, pool_bytes) ||
            !in_range(d[k].local, d[k].len, slab_bytes)) {
            st |= KVXO_S_BOUNDS;
            continue;
        }
        memcpy(slab + d[k].local, pool + d[k].remote, d[k].len);
    }
    return st;
}

/* Scatter, the inverse: dst_pool[remote .. +len) = slab[local .. +len). */
uint32_t kvxo_unpack(const uint8_t *slab, uint64_t slab_bytes, const kvxo_desc *d,
                     uint64_t n, uint8_t *dst_pool, uint64_t pool_bytes)
{
    uint32_t st = check_tiling(d, n);
    if (st)
        return st;
    for (uint64_t k = 0; k < n; k++) {
        if (!in_range(d[k].remote, d[k].len, pool_bytes) ||
            !in_range(d[k].local, d[k].len, slab_bytes)) {
            st |= KVXO_S_BOUNDS;
            continue;
        }
        memcpy(dst_pool + d[k].remote, slab + d[k].local, d[k].len);
    }
    return st;
}

/* ------------------------------------------------ holder verify + encode */

/*
 * Holder prefix scan with the slot-template check (Holder paragraph): blocks
 * are taken in order; a block is first checked as a whole -- every lane's
 * segment size equals the template's length for that lane -- and only a
 * block that passes contributes its addresses, so a mismatch in the middle
 * of a block leaves nothing of that block in the table.  The scan stops at
 * the first block that fails; *prefix receives the number of blocks taken.
 * The run table is the greedy encoding (kvxo_encode_runs) of those blocks:
 * addr is block-major, so they are its first *prefix rows.
 */
uint64_t kvxo_verify_encode(const uint64_t *addr, const uint32_t *size,
                            const uint32_t *tmpl_len, uint32_t B, uint32_t L,
                            uint32_t *runs_per_lane, uint64_t *run_base,
                            int64_t *run_stride, uint32_t *run_count,
                            uint64_t cap, uint32_t *prefix)
{
    uint32_t taken = 0;
    for (uint32_t b = 0; b < B; b++) {
        int ok = 1;                              /* phase 1: the whole block */
        for (uint32_t l = 0; l < L && ok; l++)
            if (size[(uint64_t)b * L + l] != tmpl_len[l])
                ok = 0;
        if (!ok)
            break;
        taken = b + 1;                           /* phase 2: its addresses join */
    }
    *prefix = taken;
    return kvxo_encode_runs(addr, taken, L, runs_per_lane, run_base, run_stride,
                            run_count, cap);
}

/* ------------------------------------------------------------------ seal */

/*
 * Seal from template metadata: segment (b, l) is copied from the slab at its
 * rebuilt offset local(b, l) (kvxo_rebuild) to dst[dst_addr[b][l] ..
 * + seg_len[l]), the receiver's own placement of that segment.  A segment
 * whose rebuilt offset failed its checks, or whose destination range leaves
 * dst, is not copied and raises KVXO_S_BOUNDS.  dst_addr is block-major
 * [B][L].  Returns the status bitmask (0 on a clean run; UINT32_MAX when the
 * scratch table cannot be allocated).
 */
uint32_t kvxo_seal_blocks(const uint32_t *runs_per_lane, const uint64_t *run_base,
                          const int64_t *run_stride, const uint32_t *run_count,
                          const uint32_t *run_group, const kvxo_group *groups,
                          uint64_t num_groups, uint32_t B, uint32_t L,
                          const uint32_t *seg_len, const uint8_t *slab,
                          uint64_t slab_bytes, const uint64_t *dst_addr,
                          uint8_t *dst, uint64_t dst_bytes)
{
    uint64_t n = (uint64_t)B * L;
    uint64_t *local = (uint64_t *)malloc((n ? n : 1) * sizeof(uint64_t));
    if (!local)
        return UINT32_MAX;
    uint32_t st = kvxo_rebuild(runs_per_lane, run_base, run_stride, run_count, run_group,
                               groups, num_groups, B, L, seg_len, slab_bytes, local);
    for (uint32_t b = 0; b < B; b++) {
        for (uint32_t l = 0; l < L; l++) {
            uint64_t k = (uint64_t)b * L + l;
            if (local[k] == UINT64_MAX)
                continue;                        /* flagged by the rebuild */
            if (!in_range(dst_addr[k], seg_len[l], dst_bytes)) {
                st |= KVXO_S_BOUNDS;
                continue;
            }
            memcpy(dst + dst_addr[k], slab + local[k], seg_len[l]);
        }
    }
    free(local);
    return st;
}

/* ---------------------------------------------------------- paged writes */

/*
 * Paged write (TransferEngine API listing): a page set is {indices, stride,
 * offset}; page i of the source set begins at src_offset + src_idx[i] *
 * src_stride and is copied, page_len bytes, to page i of the destination set
 * at dst_offset + dst_idx[i] * dst_stride.  Addresses are computed exactly;
 * a page that does not lie inside its buffer is not copied (KVXO_S_SPAN for
 * the source side, KVXO_S_BOUNDS for the destination side).  Destination
 * pages are expected not to overlap.
 */
uint32_t kvxo_paged_writes(uint64_t page_len, const uint8_t *src, uint64_t src_bytes,
                           const uint32_t *src_idx, uint64_t src_stride, uint64_t src_offset,
                           uint8_t *dst, uint64_t dst_bytes, const uint32_t *dst_idx,
                           uint64_t dst_stride, uint64_t dst_offset, uint64_t n)
{
    uint32_t st = 0;
    for (uint64_t i = 0; i < n; i++) {
        i128 s = (i128)src_offset + (i128)src_idx[i] * (i128)src_stride;
        i128 d = (i128)dst_offset + (i128)dst_idx[i] * (i128)dst_stride;
        int ok = 1;
        if (s + (i128)page_len > (i128)src_bytes) {
            st |= KVXO_S_SPAN;
            ok = 0;
        }
        if (d + (i128)page_len > (i128)dst_bytes) {
            st |= KVXO_S_BOUNDS;
            ok = 0;
        }
        if (ok)
            memcpy(dst + (uint64_t)d, src + (uint64_t)s, page_len);
    }
    return st;
}
