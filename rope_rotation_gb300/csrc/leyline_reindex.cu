// leyline_reindex.cu -- re-index splices on GB300 (sm_103a): survivors that shift by a
// multiple of the block size keep their pages, their rope bands turn in place, and the
// other blocks' rows are written into fresh pages.
//
// "Leyline: KV Cache Directives for Agentic Inference", sections 2.2-2.3 (the rotation
// and re-index of every downstream slot) and 3 (block-level storage).
#include <type_traits>

#include "leyline_device.cuh"

namespace leyline {
namespace {

// -------------------------------------------------------------------------
// Re-index mode (pool flag LEYLINE_POOL_REINDEX; block size 1, or a call whose
// directives all lie on block boundaries): a surviving downstream block keeps its
// page.  Up to four kernels, each a programmatic dependent of the one before:
//   prep + R      one launch of two parts.  Prep CTAs stage the page of every
//                 rewritten table entry (the kept block's old page, or a fresh page)
//                 and return the pages of dropped blocks to the ring; they read the old
//                 table and write only the staging array, the ring's push region and
//                 (lazy pools) the counts of kept and returned pages.  The other CTAs
//                 copy the call's rows of R into their fresh pages, which they find in
//                 the ring's pop region by prep's own rule, so the parts do not wait on
//                 each other;
//   fresh rows    survivor and prefix rows of boundary blocks into their staged fresh
//                 pages (if any);
//   rotate        turns the rope bands of every turned row in place (128 bytes read
//                 and written per band and layer; the latent is not touched; if any);
//   commit        installs the staged entries, clears entries past the new end,
//                 writes the new length.
// One prep item i: the page of new block i of its request (the kept block's old page,
// or its fresh page), or the return of one dropped old block to the ring.
__device__ __forceinline__ void prep_item(const SpliceArgs& a, const PlanView& pv, long long i)
{
    const long long B = a.g.block_size;
    const ReqPlan& rp = pv.reqs[find_req(pv.reqs, a.n_reqs, i, BY_PREP)];
    const long long k = i - rp.prep_begin;
    const long long blocks = (rp.new_len + B - 1) / B - rp.b0;  // new blocks from b0 on
    const int32_t* trow = a.table + (long long)rp.req * a.max_blocks;
    if (k < blocks) {
        const long long jb = rp.b0 + k;  // new block
        const long long p = jb * B;      // its first row
        const long long valid = rp.new_len - p < B ? rp.new_len - p : B;
        const Seg* sg = pv.segs + rp.seg_begin;
        const Seg s = sg[find_seg(sg, rp.seg_count, p)];
        int page;
        if (jb >= s.kb0 && jb < s.kb1) {  // kept: the old block holding exactly these rows
            const long long ob = (s.src_start + (p - s.new_start)) / B;
            page = (ob >= 0 && ob < a.max_blocks) ? trow[ob] : -1;
            if (page < 0 || page >= a.g.num_pages) {
                raise_status(a.status, ST_BAD_PAGE);
                page = -1;
            }
            if (a.pending && page >= 0 && s.turn != 0)  // the valid slots turn; the others stay 0
                for (long long sl = 0; sl < valid; ++sl) a.pending[(long long)page * B + sl] += s.turn;
        } else {  // fresh: the new block's position among the request's fresh blocks
            const long long kept_before = s.kept_before + (jb < s.kb0 ? 0 : (long long)s.kb1 - s.kb0);
            page = a.free_q[ring(a.pop_base + rp.pop_off + (k - kept_before), a.q_cap)];
            if (page < 0 || page >= a.g.num_pages) {
                raise_status(a.status, ST_BAD_FRESH);
                page = -1;
            }
        }
        a.stage[rp.stage_begin + k] = page;
    } else {
        const long long j = k - blocks;  // j-th returned old block of the request
        const Seg* dg = pv.segs + rp.drop_seg_begin;
        int q = 0;
        for (int x = 1; x < rp.drop_seg_count; ++x)
            if (dg[x].aux <= j) q = x;
        const long long ob = dg[q].src_start + (j - dg[q].aux);
        int page = (ob >= 0 && ob < a.max_blocks) ? trow[ob] : -1;
        if (page < 0 || page >= a.g.num_pages) {
            raise_status(a.status, ST_BAD_OLD);
            page = -1;
        }
        a.free_q[ring(a.push_base + rp.push_off + j, a.q_cap)] = page;
        // a free page carries no pending turn; when the fresh-rows kernel still reads
        // survivors from the request's returned pages, the commit clears them instead
        if (a.pending && page >= 0 && rp.fresh_seg_count == 0)
            for (long long sl = 0; sl < B; ++sl) a.pending[(long long)page * B + sl] = 0;
    }
}

// Re-index mode writes fresh rows and turns kept bands.
//   prep_repl_reindex (its row-of-R part): the call's rows of R form one list; items
//   of (row, 8 layers) are spread over every warp of its CTAs, the warp moving the
//   item's (layer, vector) list with kReplVecs vectors per lane in flight.  A row of R
//   moves 9 times the bytes of a turned band, so rows of R are not tied to one CTA's
//   share of the tiles.
//   copy_fresh_reindex: the other rows of blocks that get fresh pages (survivors and
//   prefix rows of boundary blocks), likewise spread over warps, read through the old
//   table and turned by their segment's cos/sin.
//   rotate_in_place: the kept rows of each turned (ROT) segment are cut into 16-row
//   tiles of their own (the planner numbers them in Seg::tile_off); survivors that
//   keep their encoding -- every survivor of a lazy pool -- cost nothing.  Work unit
//   = (tile, group of layers).  The threads' work items (4 per band and layer for
//   half-split pairs, 8 interleaved; at most kMaxItems per thread) are decoded once
//   at kernel start, and the unit loop advances tile and layer group by counters, so
//   a unit costs only its loads, its arithmetic and its stores.
constexpr int kMaxRopeDim = 256;
constexpr int kMaxItems = 4;    // work items per thread: rope_heads * rope_dim <= 512
constexpr int kFreshLayers = 8;  // layers per item of the fresh-rows kernel
#ifndef LEYLINE_REPL_VECS
#define LEYLINE_REPL_VECS 4
#endif
constexpr int kReplVecs = LEYLINE_REPL_VECS;  // vectors per lane in flight in a row-of-R item
#ifndef LEYLINE_REPL_LAYERS
#define LEYLINE_REPL_LAYERS 8
#endif
constexpr int kReplLayers = LEYLINE_REPL_LAYERS;  // layers per row-of-R item

// Layers per work unit of the re-index rotate kernel: as many as give each of the
// CTA's threads kItems work items (at least one layer).
__host__ __device__ __forceinline__ int reindex_layers_per_unit(int per_layer, int items)
{
    const int l = items * kMoveThreads / per_layer;
    return l > 0 ? l : 1;
}

// An uploaded plan's requests and segments in shared memory, for the kernels that look up a
// request and a segment per work item (prep, rows of R, fresh rows, commit).  They are
// contiguous in the upload (requests, segments, then the cos / sin), so a CTA copies them
// once and its lookups then read shared memory instead of a chain of global loads.  The
// launch passes their bytes as dynamic shared memory, or 0 when they exceed
// kStagedPlanMax (the lookups then read global memory); a plan that travels as a kernel
// parameter is read where it is.
constexpr unsigned kStagedPlanMax = 48u << 10;
extern __shared__ uint4 staged_plan_smem[];

__device__ __forceinline__ PlanView staged_plan_view(const SpliceArgs& a, const ParamPlan& plan)
{
    return plan_view(a, plan);
}

__device__ __forceinline__ PlanView staged_plan_view(const SpliceArgs& a, const NoParamPlan& plan)
{
    unsigned bytes;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(bytes));
    if (bytes == 0) return plan_view(a, plan);
    const uint4* src = reinterpret_cast<const uint4*>(a.reqs);
    for (unsigned v = threadIdx.x; v < bytes / 16; v += blockDim.x) staged_plan_smem[v] = src[v];
    __syncthreads();
    const char* base = reinterpret_cast<const char*>(staged_plan_smem);
    return PlanView{reinterpret_cast<const ReqPlan*>(base),
                    reinterpret_cast<const Seg*>(base + (reinterpret_cast<const char*>(a.segs) -
                                                         reinterpret_cast<const char*>(a.reqs))),
                    a.trig};
}

// Dynamic shared memory of a launch that stages the plan: the bytes of its requests and
// segments when the plan is uploaded and they fit, else 0.
template <class PlanSrc>
unsigned staged_plan_bytes(const SpliceArgs& a)
{
    if (std::is_same<PlanSrc, ParamPlan>::value) return 0;
    const size_t bytes = (size_t)(reinterpret_cast<const char*>(a.trig) - reinterpret_cast<const char*>(a.reqs));
    return bytes <= kStagedPlanMax && bytes % 16 == 0 ? (unsigned)bytes : 0u;
}

// One row-of-R item: row rrow of the call's rows of R, layers [l0, l0 + kReplLayers),
// moved by one warp into the row's fresh page.  The page is the one prep stages for
// the row's block (a block holding a row of R is never kept): the block's position
// among its request's fresh blocks, read from the ring's pop region.
__device__ __forceinline__ void repl_item(const SpliceArgs& a, const PlanView& pv, long long rrow, long long l0,
                                          int lane)
{
    const long long L = a.g.num_layers;
    const int row_vecs = a.g.row_vecs, lv = a.g.latent_vecs;
    uint4* kv = static_cast<uint4*>(a.kv);
    const ReqPlan& rp = pv.reqs[find_req(pv.reqs, a.n_reqs, rrow, BY_REPL)];
    long long j = rrow - rp.repl_begin;  // row within the request's rows of R
    const Seg* sg = pv.segs + rp.seg_begin;
    int k = -1;
    for (int q = 0; q < rp.seg_count && k < 0; ++q) {
        if (sg[q].kind != SEG_REPL) continue;
        if (j < sg[q].n_repl) k = q;
        else j -= sg[q].n_repl;
    }
    if (k < 0) {
        if (lane == 0) raise_status(a.status, ST_BAD_FRESH);
        return;
    }
    const Seg s = sg[k];
    const long long p = s.new_start + j;  // rows fit 32 bits (the planner checks lengths)
    const unsigned B = (unsigned)a.g.block_size, pb = (unsigned)p / B;
    const Seg sb = sg[find_seg(sg, rp.seg_count, (long long)pb * B)];  // segment of the block's first row
    const long long kept_before = sb.kept_before + ((long long)pb < sb.kb0 ? 0 : (long long)sb.kb1 - sb.kb0);
    const int page = a.free_q[ring(a.pop_base + rp.pop_off + ((long long)pb - rp.b0 - kept_before), a.q_cap)];
    if (page < 0 || page >= a.g.num_pages) {
        if (lane == 0) raise_status(a.status, ST_BAD_FRESH);
        return;
    }
    const long long slot = (long long)page * B + ((unsigned)p - pb * B);
    if (a.pending && l0 == 0 && lane == 0) a.pending[slot] = 0;  // R is encoded at its final position
    const long long rstride = (long long)s.n_repl * row_vecs;
    const uint4* src = static_cast<const uint4*>(s.repl) + j * row_vecs;
    const long long l1 = l0 + kReplLayers < L ? l0 + kReplLayers : L;
    // the item's (layer, vector) pairs as one list, kReplVecs vectors per lane in flight
    // before any store (a warp moves up to 32 * kReplVecs * 16 bytes at a time)
    const int n = (int)(l1 - l0) * row_vecs;
    for (int e0 = 0; e0 < n; e0 += 32 * kReplVecs) {
        uint4 v[kReplVecs];
        int dl[kReplVecs], dc[kReplVecs];
#pragma unroll
        for (int q = 0; q < kReplVecs; ++q) {
            const int e = e0 + 32 * q + lane;
            dl[q] = e / row_vecs;
            dc[q] = e - dl[q] * row_vecs;
            if (e < n) v[q] = ld_stream(src + (l0 + dl[q]) * rstride + dc[q]);
        }
#pragma unroll
        for (int q = 0; q < kReplVecs; ++q) {
            const int e = e0 + 32 * q + lane;
            const long long layer = l0 + dl[q];
            const int c = dc[q];
            if (e < n)
                st_stream(kv + (c < lv ? lat_off(a.g, layer, slot) + c : band_off(a.g, layer, slot) + (c - lv)), v[q]);
        }
    }
}

// Prep and the rows of R in one launch: CTAs [0, a.prep_ctas) take the prep items
// (one per thread), the others the row-of-R items (one per warp).  The two parts
// write disjoint memory (staging array, ring push region and the counts of kept and
// returned pages; fresh pages and their counts), so neither waits for the other.
template <class PlanSrc>
__global__ void __launch_bounds__(kMoveThreads) prep_repl_reindex(const __grid_constant__ SpliceArgs a,
                                                                  const __grid_constant__ PlanSrc plan)
{
    wait_for_previous_grid();
    allow_next_grid();
    const PlanView pv = staged_plan_view(a, plan);
    const long long prep_ctas = a.prep_ctas;
    if ((long long)blockIdx.x < prep_ctas) {
        const long long stride = prep_ctas * blockDim.x;
        for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < a.total_prep; i += stride)
            prep_item(a, pv, i);
        return;
    }
    const int lane = threadIdx.x & 31;
    const long long gw = (((long long)blockIdx.x - prep_ctas) * blockDim.x + threadIdx.x) >> 5;
    const long long nw = (((long long)gridDim.x - prep_ctas) * blockDim.x) >> 5;
    const long long chunks = (a.g.num_layers + kReplLayers - 1) / kReplLayers;
    for (long long w = gw; w < a.total_repl * chunks; w += nw) {
        const long long rrow = w / chunks;
        repl_item(a, pv, rrow, (w - rrow * chunks) * kReplLayers, lane);
    }
}


// The part of a fresh row beyond the first 64 latent vectors and the first 32 band
// items (wider rows than MLA), out of line so the common path keeps its registers.
template <int kLayout, bool kBf16>
__device__ __forceinline__ void copy_fresh_rest(const Geometry& g, const uint4* sl, uint4* dl, const uint4* sb,
                                             uint4* db, const float* trig_table, int trig, int lane)
{
    constexpr int kPairs = kLayout == 0 ? 8 : 4;
    const int lv = g.latent_vecs, hv = g.head_vecs, half = g.rope_dim / 2;
    const int head_items = kLayout == 0 ? hv / 2 : hv;
    const int band_items = g.rope_heads * head_items;
    for (int c = 64 + lane; c < lv; c += 32) st_stream(dl + c, ld_stream(sl + c));
    for (int it = 32 + lane; it < band_items; it += 32) {
        const int head = it / head_items, qi = it - head * head_items;
        float cs[8], sn[8];
        const float* tp = trig_table ? trig_table + 2 * ((long long)trig * half + kPairs * qi) : nullptr;
        if (tp) {
#pragma unroll
            for (int u = 0; u < kPairs; ++u) {
                cs[u] = tp[2 * u];
                sn[u] = tp[2 * u + 1];
            }
        }
        if (kLayout == 0) {
            uint4 x = ld_stream(sb + head * hv + qi), y = ld_stream(sb + head * hv + qi + hv / 2);
            if (tp) rotate_half_split<kBf16>(x, y, cs, sn);
            st_stream(db + head * hv + qi, x);
            st_stream(db + head * hv + qi + hv / 2, y);
        } else {
            uint4 x = ld_stream(sb + head * hv + qi);
            if (tp) rotate_interleaved<kBf16>(x, cs, sn);
            st_stream(db + head * hv + qi, x);
        }
    }
}

// Fresh rows of a re-indexed call other than rows of R: the survivors and prefix rows
// of blocks that do not keep their pages, written into the fresh page prep staged for
// their block.  A survivor is read through the old table and
// turned by its segment's cos/sin; in a lazy pool its pending count moves with it.
template <int kLayout, bool kBf16, class PlanSrc>
__global__ void __launch_bounds__(kMoveThreads, 3) copy_fresh_reindex(const __grid_constant__ SpliceArgs a,
                                                                   const __grid_constant__ PlanSrc plan)
{
    wait_for_previous_grid();
    allow_next_grid();
    const PlanView pv = staged_plan_view(a, plan);
    const int lane = threadIdx.x & 31;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long L = a.g.num_layers;
    const int chunks = (int)((L + kFreshLayers - 1) / kFreshLayers);
    const int row_vecs = a.g.row_vecs, lv = a.g.latent_vecs, hv = a.g.head_vecs, half = a.g.rope_dim / 2;
    constexpr int kPairs = kLayout == 0 ? 8 : 4;  // pairs per work item
    const int head_items = kLayout == 0 ? hv / 2 : hv;
    const int band_items = a.g.rope_heads * head_items;
    const unsigned B = (unsigned)a.g.block_size;
    uint4* kv = static_cast<uint4*>(a.kv);
    for (long long w = gw; w < a.total_fresh * chunks; w += nw) {
        const long long frow = w / chunks;
        const long long l0 = (w - frow * chunks) * kFreshLayers;
        const ReqPlan& rp = pv.reqs[find_req(pv.reqs, a.n_reqs, frow, BY_FRESH)];
        const long long f = frow - rp.fresh_begin;  // fresh row within the request
        const Seg* fg = pv.segs + rp.fresh_seg_begin;
        int q = 0;
        for (int x = 1; x < rp.fresh_seg_count; ++x)
            if (fg[x].aux <= f) q = x;
        const long long p = fg[q].new_start + (f - fg[q].aux);  // its new row (rows fit 32 bits)
        const Seg* sg = pv.segs + rp.seg_begin;
        const Seg s = sg[find_seg(sg, rp.seg_count, p)];
        const unsigned pb = (unsigned)p / B;
        const int dpage = a.stage[rp.stage_begin + ((long long)pb - rp.b0)];
        if (dpage < 0 || dpage >= a.g.num_pages) continue;  // prep has recorded a bad fresh page
        const long long dslot = (long long)dpage * B + ((unsigned)p - pb * B);
        const uint4 *src_lat, *src_band;
        long long lat_stride, band_stride, sslot = -1;
        if (s.kind == SEG_REPL) {
            src_lat = static_cast<const uint4*>(s.repl) + (p - s.new_start) * row_vecs;
            src_band = src_lat + lv;
            lat_stride = band_stride = (long long)s.n_repl * row_vecs;
        } else {
            const long long t = s.src_start + (p - s.new_start);  // old row
            const unsigned tb = (unsigned)t / B;
            const int spage = (t >= 0 && (long long)tb < a.max_blocks) ? a.table[(long long)rp.req * a.max_blocks + tb]
                                                                      : -1;
            if (spage < 0 || spage >= a.g.num_pages) {
                if (lane == 0) raise_status(a.status, ST_BAD_PAGE);
                continue;
            }
            sslot = (long long)spage * B + ((unsigned)t - tb * B);
            src_lat = kv + lat_off(a.g, 0, sslot);
            src_band = kv + band_off(a.g, 0, sslot);
            lat_stride = a.g.lat_layer_vecs;
            band_stride = a.g.rope_layer_vecs;
        }
        if (a.pending && l0 == 0 && lane == 0)  // once per row: R at its final position, survivors carried
            a.pending[dslot] = sslot < 0 ? 0 : a.pending[sslot] + s.turn;
        const int trig = s.kind == SEG_ROT ? s.trig : -1;
        const long long l1 = l0 + kFreshLayers < L ? l0 + kFreshLayers : L;
        const bool band_lane = lane < band_items;  // this lane's first band item: it = lane
        const int head0 = band_lane ? lane / head_items : 0, q0 = lane - head0 * head_items;
        const float* tp0 = trig >= 0 ? pv.trig + 2 * ((long long)trig * half + kPairs * q0) : nullptr;
#pragma unroll 1
        for (long long layer = l0; layer < l1; ++layer) {
            // one round per layer: the first 64 latent vectors (the MLA latent) and the first
            // band item of every lane are loaded before anything is stored
            const uint4* sl = src_lat + layer * lat_stride;
            uint4* dl = kv + lat_off(a.g, layer, dslot);
            const uint4* sb = src_band + layer * band_stride + head0 * hv + q0;
            uint4* db = kv + band_off(a.g, layer, dslot) + head0 * hv + q0;
            uint4 v0, v1, x, y;
            if (lane < lv) v0 = ld_stream(sl + lane);
            if (32 + lane < lv) v1 = ld_stream(sl + 32 + lane);
            if (band_lane) {
                x = ld_stream(sb);
                if (kLayout == 0) y = ld_stream(sb + hv / 2);
            }
            if (lane < lv) st_stream(dl + lane, v0);
            if (32 + lane < lv) st_stream(dl + 32 + lane, v1);
            if (band_lane) {
                float cs[8], sn[8];
                if (tp0) {
#pragma unroll
                    for (int u = 0; u < kPairs; ++u) {
                        cs[u] = tp0[2 * u];
                        sn[u] = tp0[2 * u + 1];
                    }
                }
                if (kLayout == 0) {
                    if (tp0) rotate_half_split<kBf16>(x, y, cs, sn);
                    st_stream(db, x);
                    st_stream(db + hv / 2, y);
                } else {
                    if (tp0) rotate_interleaved<kBf16>(x, cs, sn);
                    st_stream(db, x);
                }
            }
            if (lv > 64 || band_items > 32)  // wider latents, more than 32 band items: out of line
                copy_fresh_rest<kLayout, kBf16>(a.g, sl, dl, src_band + layer * band_stride,
                                                kv + band_off(a.g, layer, dslot), trig >= 0 ? pv.trig : nullptr,
                                                trig, lane);
        }
    }
}

// kItems: work items per thread.  1 for the MLA row (16 rows x 4 or 8 items per
// layer: a unit covers 4 or 2 layers), with 8 CTAs per SM; kMaxItems for wider rows.
template <int kLayout, bool kBf16, int kItems, class PlanSrc>
__global__ void __launch_bounds__(kMoveThreads, kItems == 1 ? 5 : 2) rotate_in_place(const __grid_constant__ SpliceArgs a,
                                                                const __grid_constant__ PlanSrc plan)
{
    __shared__ uint4* band_s[kTileRows];                  // the tile's rows' bands (layer 0); nullptr: none
    __shared__ __align__(16) float trig_s[kMaxRopeDim];  // (cos, sin) per pair of the tile's segment
    wait_for_previous_grid();
    allow_next_grid();
    const PlanView pv = plan_view(a, plan);
    const long long L = a.g.num_layers;
    const int hv = a.g.head_vecs;
    const int rope_dim = a.g.rope_dim;
    constexpr int kPairs = kLayout == 0 ? 8 : 4;        // pairs per work item
    const int head_items = kLayout == 0 ? hv / 2 : hv;  // work items per RoPE band
    const int ipr = a.g.rope_heads * head_items;        // work items per row and layer
    const int per_layer = kTileRows * ipr;
    const int lpu = reindex_layers_per_unit(per_layer, kItems);
    const long long groups = (L + lpu - 1) / lpu;
    // this thread's items: row i, layer offset lo, vector offset in the bands, pair group q
    int it_row[kItems], it_lo[kItems], it_off[kItems], it_q[kItems];
    int n_items = 0;
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
        const int e = threadIdx.x + k * kMoveThreads;
        it_row[k] = it_lo[k] = it_off[k] = it_q[k] = 0;
        if (e < lpu * per_layer) {
            const int lo = e / per_layer, it = e - lo * per_layer;
            const int i = it / ipr, hq = it - i * ipr;
            const int head = hq / head_items, q = hq - head * head_items;
            it_row[k] = i;
            it_lo[k] = lo;
            it_off[k] = head * hv + q;
            it_q[k] = q;
            n_items = k + 1;
        }
    }
    long long u0, u1;
    my_units(a.total_tiles * groups, u0, u1);
    long long tile = u0 / groups, grp = u0 - (u0 / groups) * groups;
    long long cur_tile = -1;
    for (long long u = u0; u < u1; ++u) {
        if (tile != cur_tile) {
            __syncthreads();
            if (threadIdx.x < kTileRows) {
                uint4* band = nullptr;
                const ReqPlan& rp = pv.reqs[find_req(pv.reqs, a.n_reqs, tile, BY_TILE)];
                const long long lt = tile - rp.tile_begin;
                const Seg* sg = pv.segs + rp.seg_begin;
                int k = 0;
                for (int q = 0; q < rp.seg_count; ++q)
                    if (sg[q].tile_off >= 0 && sg[q].tile_off <= lt) k = q;
                const Seg s = sg[k];
                const long long B0 = a.g.block_size;
                const long long seg_end = k + 1 < rp.seg_count ? sg[k + 1].new_start : rp.new_len;
                const long long kept_end = (long long)s.kb1 * B0 < seg_end ? (long long)s.kb1 * B0 : seg_end;
                const long long p = (long long)s.kb0 * B0 + (lt - s.tile_off) * kTileRows + threadIdx.x;
                if (p < kept_end) {  // rows and block sizes fit 32 bits (the planner checks lengths)
                    const unsigned B = (unsigned)a.g.block_size, pb = (unsigned)p / B;
                    const int page = a.stage[rp.stage_begin + ((long long)pb - rp.b0)];
                    if (page >= 0 && page < a.g.num_pages)
                        band = static_cast<uint4*>(a.kv) + band_off(a.g, 0, (long long)page * B + ((unsigned)p - pb * B));
                }
                band_s[threadIdx.x] = band;
                for (int c = threadIdx.x; c < rope_dim; c += kTileRows)  // the segment's cos/sin
                    trig_s[c] = pv.trig[(long long)s.trig * rope_dim + c];
            }
            __syncthreads();
            cur_tile = tile;
        }
        const long long layer0 = grp * lpu;
        if (kItems == 1) {
            // one item per thread: when the next unit is the same tile's next layer group,
            // both units' loads are issued before either unit's stores
            const bool two = grp + 1 < groups && u + 1 < u1;
            uint4* band = n_items ? band_s[it_row[0]] : nullptr;
            const long long la = layer0 + it_lo[0], lb = la + lpu;
            const bool da = band && la < L, db = two && band && lb < L;
            uint4* ra = band + la * a.g.rope_layer_vecs + it_off[0];
            uint4* rb = band + lb * a.g.rope_layer_vecs + it_off[0];
            uint4 xa, ya, xb, yb;
            if (da) {
                xa = ld_rw(ra);
                if (kLayout == 0) ya = ld_rw(ra + hv / 2);
            }
            if (db) {
                xb = ld_rw(rb);
                if (kLayout == 0) yb = ld_rw(rb + hv / 2);
            }
            if (da || db) {
                float cs[8], sn[8];
                const float* tp = &trig_s[2 * kPairs * it_q[0]];
#pragma unroll
                for (int w = 0; w < kPairs; ++w) {
                    cs[w] = tp[2 * w];
                    sn[w] = tp[2 * w + 1];
                }
                if (kLayout == 0) {
                    if (da) {
                        rotate_half_split<kBf16>(xa, ya, cs, sn);
                        st_stream(ra, xa);
                        st_stream(ra + hv / 2, ya);
                    }
                    if (db) {
                        rotate_half_split<kBf16>(xb, yb, cs, sn);
                        st_stream(rb, xb);
                        st_stream(rb + hv / 2, yb);
                    }
                } else {
                    if (da) {
                        rotate_interleaved<kBf16>(xa, cs, sn);
                        st_stream(ra, xa);
                    }
                    if (db) {
                        rotate_interleaved<kBf16>(xb, cs, sn);
                        st_stream(rb, xb);
                    }
                }
            }
            if (two) {
                ++u;
                ++grp;
            }
        } else {
#pragma unroll
        for (int k = 0; k < kItems; ++k) {
            if (k >= n_items) break;
            const long long layer = layer0 + it_lo[k];
            uint4* band = band_s[it_row[k]];
            if (layer >= L || !band) continue;
            uint4* r = band + layer * a.g.rope_layer_vecs + it_off[k];
            float cs[8], sn[8];
            const float* tp = &trig_s[2 * kPairs * it_q[k]];
#pragma unroll
            for (int w = 0; w < kPairs; ++w) {
                cs[w] = tp[2 * w];
                sn[w] = tp[2 * w + 1];
            }
            if (kLayout == 0) {
                uint4 x = ld_rw(r), y = ld_rw(r + hv / 2);
                rotate_half_split<kBf16>(x, y, cs, sn);
                st_stream(r, x);
                st_stream(r + hv / 2, y);
            } else {
                uint4 x = ld_rw(r);
                rotate_interleaved<kBf16>(x, cs, sn);
                st_stream(r, x);
            }
        }
        }
        if (++grp == groups) {
            grp = 0;
            ++tile;
        }
    }
}

// In-place rotation of rows whose rope bands fill 8 vectors (MLA: one 64-wide band; GQA:
// 2 bands of 32 or 4 of 16).  Each band is turned by 8 lanes, one 16-byte chunk each, so
// that a warp instruction covers four whole 128-byte bands (half-split: the partner half
// comes from lane ^ head_vecs / 2).  The CTA's 256 threads cover 16 rows x 8 chunks x 2
// layers, and each thread issues the loads of kRotPasses layers (2 apart) before any
// store: a unit is (16-row tile, 2 * kRotPasses layers).  Tiles, their lookup and the
// cos / sin of their segment are as in rotate_in_place.
constexpr int kRotPasses = 4;
#ifndef LEYLINE_LINES_MIN_CTAS
#define LEYLINE_LINES_MIN_CTAS 4
#endif
constexpr int kRotUnitLayers = 2 * kRotPasses;

template <int kLayout, bool kBf16, class PlanSrc>
__global__ void __launch_bounds__(kMoveThreads, LEYLINE_LINES_MIN_CTAS) rotate_in_place_lines(const __grid_constant__ SpliceArgs a,
                                                                         const __grid_constant__ PlanSrc plan)
{
    __shared__ uint4* band_s[kTileRows];                  // the tile's rows' bands (layer 0); nullptr: none
    __shared__ __align__(16) float trig_s[kMaxRopeDim];  // (cos, sin) per pair of the tile's segment
    wait_for_previous_grid();
    allow_next_grid();
    const PlanView pv = plan_view(a, plan);
    const long long L = a.g.num_layers;
    const long long rope_layer = a.g.rope_layer_vecs;
    const int hv = a.g.head_vecs;
    const int rope_dim = a.g.rope_dim;
    constexpr int kPairs = kLayout == 0 ? 8 : 4;
    const int row = (threadIdx.x >> 3) & (kTileRows - 1);  // this thread's row of a tile
    const int c = threadIdx.x & 7;                         // its chunk of the row's bands
    const int lo = threadIdx.x / (8 * kTileRows);          // its layer of each pair of layers
    const int q = c & (hv - 1);                            // chunk within its band
    const int j0 = kLayout == 0 ? kPairs * (q & (hv / 2 - 1)) : kPairs * q;  // first pair of the chunk
    const bool y_half = kLayout == 0 && q >= hv / 2;
    const long long groups = (L + kRotUnitLayers - 1) / kRotUnitLayers;
    long long u0, u1;
    my_units(a.total_tiles * groups, u0, u1);
    long long tile = u0 / groups, grp = u0 - (u0 / groups) * groups;
    long long cur_tile = -1;
    float cs[8], sn[8];
    for (long long u = u0; u < u1; ++u) {
        if (tile != cur_tile) {
            __syncthreads();
            if (threadIdx.x < kTileRows) {
                uint4* band = nullptr;
                const ReqPlan& rp = pv.reqs[find_req(pv.reqs, a.n_reqs, tile, BY_TILE)];
                const long long lt = tile - rp.tile_begin;
                const Seg* sg = pv.segs + rp.seg_begin;
                int k = 0;
                for (int qq = 0; qq < rp.seg_count; ++qq)
                    if (sg[qq].tile_off >= 0 && sg[qq].tile_off <= lt) k = qq;
                const Seg sgk = sg[k];
                const long long B0 = a.g.block_size;
                const long long seg_end = k + 1 < rp.seg_count ? sg[k + 1].new_start : rp.new_len;
                const long long kept_end = (long long)sgk.kb1 * B0 < seg_end ? (long long)sgk.kb1 * B0 : seg_end;
                const long long p = (long long)sgk.kb0 * B0 + (lt - sgk.tile_off) * kTileRows + threadIdx.x;
                if (p < kept_end) {  // rows and block sizes fit 32 bits (the planner checks lengths)
                    const unsigned B = (unsigned)a.g.block_size, pb = (unsigned)p / B;
                    const int page = a.stage[rp.stage_begin + ((long long)pb - rp.b0)];
                    if (page >= 0 && page < a.g.num_pages)
                        band = static_cast<uint4*>(a.kv) + band_off(a.g, 0, (long long)page * B + ((unsigned)p - pb * B));
                }
                band_s[threadIdx.x] = band;
                for (int e = threadIdx.x; e < rope_dim; e += kTileRows)  // the segment's cos/sin
                    trig_s[e] = pv.trig[(long long)sgk.trig * rope_dim + e];
            }
            __syncthreads();
            cur_tile = tile;
#pragma unroll
            for (int w = 0; w < kPairs; ++w) {
                cs[w] = trig_s[2 * (j0 + w)];
                sn[w] = trig_s[2 * (j0 + w) + 1];
            }
        }
        uint4* band = band_s[row];
        const long long layer0 = grp * kRotUnitLayers + lo;
        uint4 v[kRotPasses];
        uint4* ptr[kRotPasses];
#pragma unroll
        for (int k = 0; k < kRotPasses; ++k) {
            const long long layer = layer0 + 2 * k;
            ptr[k] = band + layer * rope_layer + c;
            v[k] = make_uint4(0u, 0u, 0u, 0u);
            if (band && layer < L) v[k] = ld_rw(ptr[k]);
        }
#pragma unroll
        for (int k = 0; k < kRotPasses; ++k) {
            const bool ok = band && layer0 + 2 * k < L;
            if (kLayout == 0) {
                const uint4 o = shfl_xor_vec(v[k], hv / 2);  // every lane takes part
                if (ok) st_stream(ptr[k], turn_own_half<kBf16>(v[k], o, y_half, cs, sn));
            } else if (ok) {
                rotate_interleaved<kBf16>(v[k], cs, sn);
                st_stream(ptr[k], v[k]);
            }
        }
        if (++grp == groups) {
            grp = 0;
            ++tile;
        }
    }
}

// Commit of a re-indexed call: staged entries into the new blocks [b0, new end),
// -1 into the blocks past the new end, the new length, and (lazy pools) pending
// counts of 0 on the returned pages.  The staged values are final once prep has
// finished.  When a fresh-rows or rotate kernel runs between prep and this one, that
// kernel waited for prep before it let this one launch, so the values are loaded before
// griddepcontrol.wait; when prep itself is the previous kernel (a call that turns no
// band and writes no other fresh rows: every lazy block-1 call), they are loaded after.
template <class PlanSrc>
__global__ void __launch_bounds__(kCommitThreads) commit_reindex(const __grid_constant__ SpliceArgs a,
                                                                 const __grid_constant__ PlanSrc plan)
{
    const PlanView pv = staged_plan_view(a, plan);  // the plan is final before the previous kernel
    const long long stride = (long long)gridDim.x * blockDim.x;
    long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    int val = -1;
    const ReqPlan* rp = nullptr;
    long long k = 0;
    const long long B = a.g.block_size;
    const bool early = a.total_fresh > 0 || a.total_tiles > 0;  // a kernel between prep and this one
    if (i < a.total_commit) {
        rp = &pv.reqs[find_req(pv.reqs, a.n_reqs, i, BY_COMMIT)];
        k = i - rp->commit_begin;
        if (early && k < (rp->new_len + B - 1) / B - rp->b0) val = a.stage[rp->stage_begin + k];
    }
    wait_for_previous_grid();
    allow_next_grid();
    if (!early && i < a.total_commit && k < (rp->new_len + B - 1) / B - rp->b0) val = a.stage[rp->stage_begin + k];
    while (i < a.total_commit) {
        int32_t* trow = a.table_w + (long long)rp->req * a.max_blocks;
        const long long nb_new = (rp->new_len + B - 1) / B, nb_old = (rp->old_len + B - 1) / B;
        const long long blocks = nb_new - rp->b0;
        const long long tail = nb_old > nb_new ? nb_old - nb_new : 0;
        if (k == 0) a.seq_lens_dev[rp->req] = (int32_t)rp->new_len;
        if (k < blocks) {
            trow[rp->b0 + k] = val;
        } else if (k < blocks + tail) {
            trow[nb_new + (k - blocks)] = -1;
        } else if (a.pending && rp->fresh_seg_count > 0 && k < blocks + tail + rp->drop_count) {
            // a returned page carries no pending turn (its rows have been read by now)
            const int page = a.free_q[ring(a.push_base + rp->push_off + (k - blocks - tail), a.q_cap)];
            if (page >= 0 && page < a.g.num_pages)
                for (long long sl = 0; sl < B; ++sl) a.pending[(long long)page * B + sl] = 0;
        }
        i += stride;
        if (i >= a.total_commit) break;
        rp = &pv.reqs[find_req(pv.reqs, a.n_reqs, i, BY_COMMIT)];
        k = i - rp->commit_begin;
        val = k < (rp->new_len + B - 1) / B - rp->b0 ? a.stage[rp->stage_begin + k] : -1;
    }
}

template <class PlanSrc>
int launch_reindex(const SpliceArgs& a, const PlanSrc& plan, int grid, cudaStream_t s, cudaEvent_t t0, cudaEvent_t t1)
{
    cudaError_t e = cudaSuccess;
    // prep and the rows of R: one launch, prep CTAs first
    const int prep_ctas = a.total_prep > 0 ? grid_for(a.total_prep, kMoveThreads, 8192) : 0;
    const long long repl_items = a.total_repl * ((a.g.num_layers + kReplLayers - 1) / kReplLayers);
    const int repl_ctas = repl_items > 0 ? grid_for(repl_items * 32, kMoveThreads, 8192) : 0;
    // Timing events bracket the in-place rotation when there is one (the call's dominant
    // kernel), else the launches before the commit.
    const bool rotates = a.total_tiles > 0;
    if (t0 && !rotates) e = cudaEventRecord(t0, s);
    if (e == cudaSuccess && prep_ctas + repl_ctas > 0) {
        SpliceArgs b = a;
        b.prep_ctas = prep_ctas;
        e = launch_dependent_smem(prep_repl_reindex<PlanSrc>, prep_ctas + repl_ctas, kMoveThreads,
                                  staged_plan_bytes<PlanSrc>(a), s, b, plan);
    }
    const bool bf16 = a.g.precision == LEYLINE_ROTATE_BF16_NAIVE;
    const bool split = a.g.pair_layout == LEYLINE_PAIRS_HALF_SPLIT;
    const int ipr = a.g.rope_heads * (split ? a.g.head_vecs / 2 : a.g.head_vecs);
    const int per_layer = kTileRows * ipr;
    const bool lines = a.g.rope_heads * a.g.head_vecs == 8;  // bands of 8 vectors: whole-line kernel
    const bool mla = per_layer <= kMoveThreads;               // one item per thread; else kMaxItems
    const int lpu = lines ? kRotUnitLayers : reindex_layers_per_unit(per_layer, mla ? 1 : kMaxItems);
    const long long units = a.total_tiles * ((a.g.num_layers + lpu - 1) / lpu);
    if (grid > units) grid = (int)std::max<long long>(units, 1);
    if (e == cudaSuccess && a.total_fresh > 0) {  // other fresh rows: items of (row, kFreshLayers layers)
        const long long items = a.total_fresh * ((a.g.num_layers + kFreshLayers - 1) / kFreshLayers);
        const int fgrid = grid_for(items * 32, kMoveThreads, 8192);
        auto k = split ? (bf16 ? copy_fresh_reindex<0, true, PlanSrc> : copy_fresh_reindex<0, false, PlanSrc>)
                       : (bf16 ? copy_fresh_reindex<1, true, PlanSrc> : copy_fresh_reindex<1, false, PlanSrc>);
        e = launch_dependent_smem(k, fgrid, kMoveThreads, staged_plan_bytes<PlanSrc>(a), s, a, plan);
    }
    if (e == cudaSuccess && t0 && rotates) e = cudaEventRecord(t0, s);
    if (e == cudaSuccess && units > 0 && lines) {
        e = split ? (bf16 ? launch_dependent(rotate_in_place_lines<0, true, PlanSrc>, grid, kMoveThreads, s, a, plan)
                          : launch_dependent(rotate_in_place_lines<0, false, PlanSrc>, grid, kMoveThreads, s, a, plan))
                  : (bf16 ? launch_dependent(rotate_in_place_lines<1, true, PlanSrc>, grid, kMoveThreads, s, a, plan)
                          : launch_dependent(rotate_in_place_lines<1, false, PlanSrc>, grid, kMoveThreads, s, a, plan));
    } else if (e == cudaSuccess && units > 0) {
        if (split)
            e = bf16 ? (mla ? launch_dependent(rotate_in_place<0, true, 1, PlanSrc>, grid, kMoveThreads, s, a, plan)
                            : launch_dependent(rotate_in_place<0, true, kMaxItems, PlanSrc>, grid, kMoveThreads, s, a,
                                               plan))
                     : (mla ? launch_dependent(rotate_in_place<0, false, 1, PlanSrc>, grid, kMoveThreads, s, a, plan)
                            : launch_dependent(rotate_in_place<0, false, kMaxItems, PlanSrc>, grid, kMoveThreads, s,
                                               a, plan));
        else
            e = bf16 ? (mla ? launch_dependent(rotate_in_place<1, true, 1, PlanSrc>, grid, kMoveThreads, s, a, plan)
                            : launch_dependent(rotate_in_place<1, true, kMaxItems, PlanSrc>, grid, kMoveThreads, s, a,
                                               plan))
                     : (mla ? launch_dependent(rotate_in_place<1, false, 1, PlanSrc>, grid, kMoveThreads, s, a, plan)
                            : launch_dependent(rotate_in_place<1, false, kMaxItems, PlanSrc>, grid, kMoveThreads, s,
                                               a, plan));
    }
    if (e == cudaSuccess && t1) e = cudaEventRecord(t1, s);
    if (e == cudaSuccess && a.total_commit > 0)
        e = launch_dependent_smem(commit_reindex<PlanSrc>, grid_for(a.total_commit, kCommitThreads, 8192),
                                  kCommitThreads, staged_plan_bytes<PlanSrc>(a), s, a, plan);
    if (e == cudaSuccess) e = cudaGetLastError();
    return (int)e;
}

}  // namespace

int launch_reindex_call(const SpliceArgs& a, const ParamPlan* pp, int grid, void* stream, cudaEvent_t t0,
                        cudaEvent_t t1)
{
    cudaStream_t s = (cudaStream_t)stream;
    if (pp) return launch_reindex(a, *pp, grid, s, t0, t1);
    return launch_reindex(a, NoParamPlan{0}, grid, s, t0, t1);
}

int rotate_in_place_blocks_per_sm(int* blocks)
{
    int a = 0, b = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, rotate_in_place<0, false, 1, ParamPlan>,
                                                                  kMoveThreads, 0);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, rotate_in_place_lines<0, false, ParamPlan>, kMoveThreads,
                                                          0);
    *blocks = a < b ? a : b;  // a grid that both rotate kernels hold at once
    return (int)e;
}

}  // namespace leyline
