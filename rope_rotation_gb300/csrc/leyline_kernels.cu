// leyline_kernels.cu -- device side of the GB300 Leyline AMORTIZE splice (sm_103a).
//
// "Leyline: KV Cache Directives for Agentic Inference":
//   section 2.2  every downstream slot's RoPE band gets K_pe_new = R(Delta) K_pe
//                (one 2x2 rotation per pair); K_nope and V (here: the compressed
//                latent they derive from) are kept.
//   section 2.3  the rotation kernel re-indexes and rotates every downstream slot.
//   section 4.3  the rotation is computed in fp32 and stored in bf16.
//
// Kernels of one splice, in stream order:
//   move+rotate  every rewritten row x layer is read once and written once into a
//                fresh page: latent and R rows copied as 16-byte vectors, the rope
//                band turned in fp32 with the segment's cos/sin and rounded to
//                bf16 (the HBM-bound hot loop);
//   commit       new block-table entries, new lengths, old pages returned to the
//                free-page ring.
// The commit kernel is launched as a programmatic dependent of move+rotate, so its
// launch overlaps the move; it waits (griddepcontrol.wait) for the move to finish
// before it touches the table.  The path is bandwidth-bound (about 64 fp32 FMAs per
// 2304 bytes moved), so it uses no tensor cores.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "leyline_internal.h"

namespace leyline {
namespace {

constexpr int kMoveThreads = 256;  // 8 warps x 2 rows = one 16-row tile
constexpr int kRowsPerWarp = 2;
static_assert(kTileRows == (kMoveThreads / 32) * kRowsPerWarp, "tile shape");

// device status bits (leyline_sync_status)
enum : int32_t { ST_BAD_PAGE = 1, ST_BAD_BLOCK = 2, ST_BAD_FRESH = 4, ST_BAD_OLD = 8 };

__device__ __forceinline__ void raise_status(int32_t* status, int32_t bit) { atomicOr(status, bit); }

// Programmatic dependent launch: wait until the preceding kernel in the stream has
// finished and its writes are visible; allow the next kernel to be launched now.
__device__ __forceinline__ void wait_for_previous_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 16-byte streaming load through the non-coherent path, not kept in L1: every
// source row is read exactly once and is never written during the kernel.
__device__ __forceinline__ uint4 ld_stream(const uint4* p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// 16-byte store with the evict-first (streaming) policy.
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// One pair turned by (c, s):  x' = x c - y s,  y' = x s + y c.
__device__ __forceinline__ void turn_fp32(float x, float y, float c, float s, float& xo, float& yo)
{
    xo = fmaf(x, c, -(y * s));
    yo = fmaf(x, s, y * c);
}

// The naive all-bf16 arm: products and sums each rounded to bf16 (c, s are bf16 values).
__device__ __forceinline__ void turn_bf16(float x, float y, float c, float s, float& xo, float& yo)
{
    const float xc = round_bf16(x * c), ys = round_bf16(y * s);
    const float xs = round_bf16(x * s), yc = round_bf16(y * c);
    xo = xc - ys;
    yo = xs + yc;
}

// Half-split layout: xv holds x of pairs j0..j0+7, yv holds y of the same pairs.
template <bool kBf16>
__device__ __forceinline__ void rotate_half_split(uint4& xv, uint4& yv, const float* c, const float* s)
{
    uint32_t* xw = reinterpret_cast<uint32_t*>(&xv);
    uint32_t* yw = reinterpret_cast<uint32_t*>(&yv);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        float x0 = bf16_lo(xw[w]), x1 = bf16_hi(xw[w]);
        float y0 = bf16_lo(yw[w]), y1 = bf16_hi(yw[w]);
        float a0, b0, a1, b1;
        if (kBf16) {
            turn_bf16(x0, y0, c[2 * w], s[2 * w], a0, b0);
            turn_bf16(x1, y1, c[2 * w + 1], s[2 * w + 1], a1, b1);
        } else {
            turn_fp32(x0, y0, c[2 * w], s[2 * w], a0, b0);
            turn_fp32(x1, y1, c[2 * w + 1], s[2 * w + 1], a1, b1);
        }
        xw[w] = pack_bf16x2(a0, a1);
        yw[w] = pack_bf16x2(b0, b1);
    }
}

// Interleaved layout: word w of v holds pair (x, y) of pair j0 + w.
template <bool kBf16>
__device__ __forceinline__ void rotate_interleaved(uint4& v, const float* c, const float* s)
{
    uint32_t* vw = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        float x = bf16_lo(vw[w]), y = bf16_hi(vw[w]);
        float a, b;
        if (kBf16) turn_bf16(x, y, c[w], s[w], a, b);
        else turn_fp32(x, y, c[w], s[w], a, b);
        vw[w] = pack_bf16x2(a, b);
    }
}

// ------------------------------------------------------------- plan access --
// The plan is either a __grid_constant__ kernel parameter (small plans) or in
// device memory; both are read through the same three pointers.
struct NoParamPlan {
    int32_t unused;
};

struct PlanView {
    const ReqPlan* reqs;
    const Seg* segs;
    const float* trig;
};

__device__ __forceinline__ PlanView plan_view(const SpliceArgs&, const ParamPlan& p)
{
    return PlanView{p.reqs, p.segs, p.trig};
}
__device__ __forceinline__ PlanView plan_view(const SpliceArgs& a, const NoParamPlan&)
{
    return PlanView{a.reqs, a.segs, a.trig};
}

// Where one destination row of a tile comes from and goes to (layer 0).
struct RowDesc {
    const uint4* src;        // latent of the source row (layer 0); nullptr: row is not written
    uint4* dst;              // latent of the destination row (layer 0)
    long long src_lstride;   // 16-byte vectors between consecutive layers of the source latent
    const uint4* src_band;   // rope bands of the source row (layer 0)
    uint4* dst_band;         // rope bands of the destination row (layer 0)
    long long band_lstride;  // 16-byte vectors between consecutive layers of the source bands
    int trig;                // trig entry, -1: no rotation
    int pad;
};

// Offsets (16-byte vectors from the pool base) of the latent and of the rope bands of
// the row of (layer, slot).
__device__ __forceinline__ long long lat_off(const Geometry& g, long long layer, long long slot)
{
    return layer * g.lat_layer_vecs + slot * g.lat_row_vecs;
}
__device__ __forceinline__ long long band_off(const Geometry& g, long long layer, long long slot)
{
    return g.rope_base_vecs + layer * g.rope_layer_vecs + slot * g.rope_row_vecs;
}

enum ReqKey : int { BY_TILE = 0, BY_COMMIT = 1, BY_PREP = 2, BY_FRESH = 3, BY_REPL = 4 };

// Last request whose first tile / commit item / prep item / fresh row / row of R is <= v.
__device__ __forceinline__ int find_req(const ReqPlan* reqs, int n, long long v, int key_kind)
{
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        const long long key = key_kind == BY_TILE     ? reqs[mid].tile_begin
                              : key_kind == BY_COMMIT ? reqs[mid].commit_begin
                              : key_kind == BY_PREP   ? reqs[mid].prep_begin
                              : key_kind == BY_FRESH  ? reqs[mid].fresh_begin
                                                      : reqs[mid].repl_begin;
        if (key <= v) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Segment of destination row p among a request's row segments (linear: at most
// 2 per directive plus one).
__device__ __forceinline__ int find_seg(const Seg* sg, int count, long long p)
{
    int k = 0;
    for (int q = 1; q < count; ++q)
        if (sg[q].new_start <= p) k = q;
    return k;
}

__device__ __forceinline__ long long ring(long long i, long long cap) { return i % cap; }

// Slot map of destination row i of a tile: segment lookup, then the source row
// through the old block table (or the rows of R), the destination row in its
// fresh page.  Every page id and block index is checked; a bad one is recorded
// in the status word and the row is skipped.
__device__ RowDesc make_desc(const SpliceArgs& a, const PlanView& pv, long long tile, int i)
{
    RowDesc d{nullptr, nullptr, 0, nullptr, nullptr, 0, -1, 0};
    const ReqPlan& rp = pv.reqs[find_req(pv.reqs, a.n_reqs, tile, BY_TILE)];
    const long long p = rp.row0 + (tile - rp.tile_begin) * kTileRows + i;
    if (p >= rp.new_len) return d;
    const Seg* sg = pv.segs + rp.seg_begin;
    int k = 0;
    for (int q = 1; q < rp.seg_count; ++q)
        if (sg[q].new_start <= p) k = q;
    const Seg s = sg[k];
    const long long off = p - s.new_start;
    const long long B = a.g.block_size;
    const long long rv = a.g.row_vecs;
    uint4* kv = static_cast<uint4*>(a.kv);
    const long long dblk = p / B;
    const bool from_cache = s.kind != SEG_REPL;
    const long long t = s.src_start + off;
    const long long blk = t / B;
    const bool blk_ok = !from_cache || (t >= 0 && blk < a.max_blocks);
    // both global loads are issued before either result is checked
    const int fresh = a.free_q[ring(a.pop_base + rp.pop_off + (dblk - rp.b0), a.q_cap)];
    const int page = (from_cache && blk_ok) ? a.table[(long long)rp.req * a.max_blocks + blk] : 0;
    if (!blk_ok) {
        raise_status(a.status, ST_BAD_BLOCK);
        return d;
    }
    if (from_cache && (page < 0 || page >= a.g.num_pages)) {
        raise_status(a.status, ST_BAD_PAGE);
        return d;
    }
    if (fresh < 0 || fresh >= a.g.num_pages) {
        raise_status(a.status, ST_BAD_FRESH);
        return d;
    }
    if (from_cache) {
        const long long sslot = (long long)page * B + (t - blk * B);
        d.src = kv + lat_off(a.g, 0, sslot);
        d.src_band = kv + band_off(a.g, 0, sslot);
        d.src_lstride = a.g.lat_layer_vecs;
        d.band_lstride = a.g.rope_layer_vecs;
        d.trig = s.kind == SEG_ROT ? s.trig : -1;
    } else {  // rows of R are whole rows [latent | bands]
        d.src = static_cast<const uint4*>(s.repl) + (s.src_start + off) * rv;
        d.src_band = d.src + a.g.latent_vecs;
        d.src_lstride = d.band_lstride = (long long)s.n_repl * rv;
    }
    const long long dslot = (long long)fresh * B + (p - dblk * B);
    d.dst = kv + lat_off(a.g, 0, dslot);
    d.dst_band = kv + band_off(a.g, 0, dslot);
    if (a.pending)  // lazy pool: the destination slot carries the source's pending turn plus this one
        a.pending[dslot] = from_cache ? a.pending[(long long)page * B + (t - blk * B)] + s.turn : 0;
    return d;
}

// Contiguous share [u0, u1) of `units` for this CTA (sizes differ by at most one).
__device__ __forceinline__ void my_units(long long units, long long& u0, long long& u1)
{
    const long long per = units / gridDim.x, rem = units % gridDim.x;
    const long long b = blockIdx.x;
    u0 = b * per + (b < rem ? b : rem);
    u1 = u0 + per + (b < rem ? 1 : 0);
}

// -------------------------------------------------------------------------
// Move+rotate, MLA shape (latent 512 = 64 vectors, rope 64 = 8 vectors).
// Work unit = (16-row tile, layer); a CTA takes a contiguous run of units, so it
// walks the layers of one tile and computes the tile's slot map once.  Warp w
// owns rows 2w and 2w+1: each lane moves 4 latent vectors (a warp instruction
// covers 512 contiguous bytes), and 8 (half-split) or 16 (interleaved) lanes
// move the rope band with the pair's cos/sin held in registers.
template <int kLayout, bool kBf16, class PlanSrc>
__global__ void __launch_bounds__(kMoveThreads, 3) move_rotate_mla(const __grid_constant__ SpliceArgs a,
                                                                const __grid_constant__ PlanSrc plan)
{
    constexpr int kRopeVecs = 8;
    __shared__ RowDesc desc[kTileRows];
    wait_for_previous_grid();
    allow_next_grid();
    const PlanView pv = plan_view(a, plan);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long L = a.g.num_layers;
    const long long lat_layer = a.g.lat_layer_vecs, rope_layer = a.g.rope_layer_vecs;
    const int half = 4 * kRopeVecs;  // pairs per row
    constexpr int kRopeLanesPerRow = kLayout == 0 ? kRopeVecs / 2 : kRopeVecs;  // 4 or 8
    const bool rope_lane = lane < kRowsPerWarp * kRopeLanesPerRow;
    const int rope_row = warp * kRowsPerWarp + lane / kRopeLanesPerRow;
    const int rope_q = lane % kRopeLanesPerRow;
    float cs[8], sn[8];
    int trig = -1;

    long long u0, u1;
    my_units(a.total_tiles * L, u0, u1);
    long long cur_tile = -1;
    for (long long u = u0; u < u1; ++u) {
        const long long tile = u / L;
        const long long layer = u - tile * L;
        if (tile != cur_tile) {
            __syncthreads();
            if (threadIdx.x < kTileRows) desc[threadIdx.x] = make_desc(a, pv, tile, threadIdx.x);
            __syncthreads();
            cur_tile = tile;
            trig = rope_lane ? desc[rope_row].trig : -1;
            if (trig >= 0) {
                // pairs covered by this lane: 8 (half-split) or 4 (interleaved)
                const int j0 = kLayout == 0 ? 8 * rope_q : 4 * rope_q;
                const float* tp = pv.trig + 2 * ((long long)trig * half + j0);
#pragma unroll
                for (int w = 0; w < (kLayout == 0 ? 8 : 4); ++w) {
                    cs[w] = tp[2 * w];
                    sn[w] = tp[2 * w + 1];
                }
            }
        }
        const RowDesc d0 = desc[warp * kRowsPerWarp];
        const RowDesc d1 = desc[warp * kRowsPerWarp + 1];
        uint4 v[4];
        if (d0.src) {
            const uint4* s0 = d0.src + layer * d0.src_lstride;
            v[0] = ld_stream(s0 + lane);
            v[1] = ld_stream(s0 + lane + 32);
        }
        if (d1.src) {
            const uint4* s1 = d1.src + layer * d1.src_lstride;
            v[2] = ld_stream(s1 + lane);
            v[3] = ld_stream(s1 + lane + 32);
        }
        const RowDesc dr = rope_lane ? desc[rope_row] : d0;
        const bool do_rope = rope_lane && dr.src != nullptr;
        uint4 rx, ry;
        if (do_rope) {
            const uint4* rs = dr.src_band + layer * dr.band_lstride;
            rx = ld_stream(rs + rope_q);
            if (kLayout == 0) ry = ld_stream(rs + rope_q + kRopeVecs / 2);
        }
        if (d0.src) {
            uint4* t0 = d0.dst + layer * lat_layer;
            st_stream(t0 + lane, v[0]);
            st_stream(t0 + lane + 32, v[1]);
        }
        if (d1.src) {
            uint4* t1 = d1.dst + layer * lat_layer;
            st_stream(t1 + lane, v[2]);
            st_stream(t1 + lane + 32, v[3]);
        }
        if (do_rope) {
            uint4* rd = dr.dst_band + layer * rope_layer;
            if (kLayout == 0) {
                if (trig >= 0) rotate_half_split<kBf16>(rx, ry, cs, sn);
                st_stream(rd + rope_q, rx);
                st_stream(rd + rope_q + kRopeVecs / 2, ry);
            } else {
                if (trig >= 0) rotate_interleaved<kBf16>(rx, cs, sn);
                st_stream(rd + rope_q, rx);
            }
        }
    }
}

// -------------------------------------------------------------------------
// Move+rotate for any latent_dim (multiple of 8) and rope_dim (multiple of 16):
// the same slot map, with plain strided loops over the vectors of the tile.
template <bool kBf16, class PlanSrc>
__global__ void __launch_bounds__(kMoveThreads) move_rotate_generic(const __grid_constant__ SpliceArgs a,
                                                                    const __grid_constant__ PlanSrc plan)
{
    __shared__ RowDesc desc[kTileRows];
    wait_for_previous_grid();
    allow_next_grid();
    const PlanView pv = plan_view(a, plan);
    const long long L = a.g.num_layers;
    const int lv = a.g.latent_vecs, hv = a.g.head_vecs, half = a.g.rope_dim / 2;
    const bool split = a.g.pair_layout == LEYLINE_PAIRS_HALF_SPLIT;
    const int head_items = split ? hv / 2 : hv;  // work items per RoPE band
    const int rope_items = a.g.rope_heads * head_items;
    long long u0, u1;
    my_units(a.total_tiles * L, u0, u1);
    long long cur_tile = -1;
    for (long long u = u0; u < u1; ++u) {
        const long long tile = u / L;
        const long long layer = u - tile * L;
        if (tile != cur_tile) {
            __syncthreads();
            if (threadIdx.x < kTileRows) desc[threadIdx.x] = make_desc(a, pv, tile, threadIdx.x);
            __syncthreads();
            cur_tile = tile;
        }
        for (int it = threadIdx.x; it < kTileRows * lv; it += blockDim.x) {
            const RowDesc d = desc[it / lv];
            if (!d.src) continue;
            const int c = it % lv;
            st_stream(d.dst + layer * a.g.lat_layer_vecs + c, ld_stream(d.src + layer * d.src_lstride + c));
        }
        for (int it = threadIdx.x; it < kTileRows * rope_items; it += blockDim.x) {
            const RowDesc d = desc[it / rope_items];
            if (!d.src) continue;
            const int hq = it % rope_items;
            const int head = hq / head_items, q = hq - head * head_items;
            const uint4* rs = d.src_band + layer * d.band_lstride + head * hv;
            uint4* rd = d.dst_band + layer * a.g.rope_layer_vecs + head * hv;
            float cs[8], sn[8];
            const int j0 = split ? 8 * q : 4 * q;
            const int np = split ? 8 : 4;
            if (d.trig >= 0) {
                for (int w = 0; w < np; ++w) {
                    cs[w] = pv.trig[2 * ((long long)d.trig * half + j0 + w)];
                    sn[w] = pv.trig[2 * ((long long)d.trig * half + j0 + w) + 1];
                }
            }
            if (split) {
                uint4 x = ld_stream(rs + q), y = ld_stream(rs + q + hv / 2);
                if (d.trig >= 0) rotate_half_split<kBf16>(x, y, cs, sn);
                st_stream(rd + q, x);
                st_stream(rd + q + hv / 2, y);
            } else {
                uint4 x = ld_stream(rs + q);
                if (d.trig >= 0) rotate_interleaved<kBf16>(x, cs, sn);
                st_stream(rd + q, x);
            }
        }
    }
}

// -------------------------------------------------------------------------
// Move+rotate with bulk-copy (TMA) loads, warp-specialized.
// A CTA walks its contiguous run of (16-row tile, layer) units through a ring of
// kBulkStages shared-memory stages, each guarded by a "full" and an "empty"
// mbarrier.  Warp 0 is the producer: for every unit it waits until the stage is
// empty, then one lane issues one cp.async.bulk load per run of rows whose
// sources are contiguous in global memory (up to a whole 16-token page); the
// load completes the stage's full barrier.  It also computes each tile's slot map
// into a small ring in shared memory.  Warps 1..4 are consumers: each waits for
// the stage to be full, reads its 4 rows back as 16-byte vectors, turns the rope
// band in registers, writes the rows to their fresh pages with streaming stores,
// and arrives on the stage's empty barrier.  No CTA-wide barrier sits in the
// loop, so the producer runs up to kBulkStages units ahead and the loads need no
// registers while in flight.  Every wait is bounded by the global timer: on
// timeout the CTA records ST_TIMEOUT, sets a shared abort flag that makes every
// warp leave its loop, and the producer waits (bounded) for its own loads still
// in flight before the CTA exits.
constexpr int kBulkConsumerWarps = 4;
constexpr int kBulkThreads = 32 * (1 + kBulkConsumerWarps);
constexpr int kBulkStages = 5;
constexpr int kDescSlots = kBulkStages + 1;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s
enum : int32_t { ST_TIMEOUT = 32 };

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of the given parity; false after kWaitLimitNs or once the
// CTA's abort flag is set.
__device__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, const volatile int* abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort_flag && *abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ uint4 lds16(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__host__ __device__ constexpr size_t bulk_smem_bytes(uint32_t row_bytes)
{
    return (size_t)kBulkStages * kTileRows * row_bytes + (size_t)kDescSlots * kTileRows * sizeof(RowDesc) +
           (size_t)2 * kBulkStages * sizeof(uint64_t) + 16;
}

// Stage one unit (one thread): expect its bytes on the stage's full barrier and
// issue one bulk load per run of rows with contiguous sources.
__device__ __forceinline__ void stage_unit(const RowDesc* rd, long long layer, long long rv, uint32_t row_bytes,
                                           uint32_t sbase, uint32_t bar)
{
    uint32_t bytes = 0;
    for (int i = 0; i < kTileRows; ++i)
        if (rd[i].src) bytes += row_bytes;
    mbar_expect_tx(bar, bytes);
    int i = 0;
    while (i < kTileRows) {
        if (!rd[i].src) {
            ++i;
            continue;
        }
        int j = i + 1;
        while (j < kTileRows && rd[j].src && rd[j].src == rd[j - 1].src + rv && rd[j].src_lstride == rd[i].src_lstride)
            ++j;
        bulk_load(sbase + (uint32_t)i * row_bytes, rd[i].src + layer * rd[i].src_lstride, (uint32_t)(j - i) * row_bytes,
                  bar);
        i = j;
    }
}

// MLA shape (latent 64 vectors, rope 8 vectors per row).
template <int kLayout, bool kBf16, class PlanSrc>
__global__ void __launch_bounds__(kBulkThreads) move_rotate_bulk(const __grid_constant__ SpliceArgs a,
                                                                 const __grid_constant__ PlanSrc plan)
{
    constexpr int kLatentVecs = 64, kRopeVecs = 8, kRowVecs = kLatentVecs + kRopeVecs;
    constexpr uint32_t kRowBytes = kRowVecs * 16;
    constexpr uint32_t kStageBytes = kTileRows * kRowBytes;
    constexpr int kRowsPerConsumer = kTileRows / kBulkConsumerWarps;  // 4
    constexpr int kRopeLanesPerRow = kLayout == 0 ? kRopeVecs / 2 : kRopeVecs;
    extern __shared__ __align__(128) unsigned char smem[];
    wait_for_previous_grid();
    allow_next_grid();
    const PlanView pv = plan_view(a, plan);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long L = a.g.num_layers;
    RowDesc* ring = reinterpret_cast<RowDesc*>(smem + (size_t)kBulkStages * kStageBytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + kDescSlots * kTileRows);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kBulkStages);
    const uint32_t smem0 = smem_addr(smem);
    const uint32_t full0 = smem_addr(bars);
    const uint32_t empty0 = full0 + 8 * kBulkStages;

    long long u0, u1;
    my_units(a.total_tiles * L, u0, u1);
    if (u0 >= u1) return;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kBulkStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kBulkConsumerWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        long long desc_tile = -1;
        long long v = u0;
        for (; v < u1; ++v) {
            const long long k = v - u0;
            const int s = (int)(k % kBulkStages);
            if (k >= kBulkStages &&
                !mbar_wait_bounded(empty0 + 8 * s, (uint32_t)(((k / kBulkStages) - 1) & 1), abort_flag)) {
                if (lane == 0 && !*abort_flag) {
                    *abort_flag = 1;
                    raise_status(a.status, ST_TIMEOUT);
                }
                break;
            }
            const long long tile = v / L;
            RowDesc* rd = ring + (tile % kDescSlots) * kTileRows;
            if (tile != desc_tile) {
                if (lane < kTileRows) rd[lane] = make_desc(a, pv, tile, lane);
                __threadfence_block();  // the slot map is published by lane 0's arrive on the full barrier
                __syncwarp();
                desc_tile = tile;
            }
            if (lane == 0) stage_unit(rd, v - tile * L, kRowVecs, kRowBytes, smem0 + (uint32_t)s * kStageBytes, full0 + 8 * s);
            __syncwarp();
        }
        if (v < u1 && lane == 0) {
            // aborted: loads of units [v - kBulkStages, v) may still be landing; the
            // consumers stop at the abort flag, so wait for those loads here
            for (long long w = (v - kBulkStages > u0 ? v - kBulkStages : u0); w < v; ++w) {
                const long long k = w - u0;
                mbar_wait_bounded(full0 + 8 * (int)(k % kBulkStages), (uint32_t)((k / kBulkStages) & 1), nullptr);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const long long layer_vecs = a.g.layer_vecs;
    const int half = 4 * kRopeVecs;
    const bool rope_lane = lane < kRowsPerConsumer * kRopeLanesPerRow;
    const int rope_row = cw * kRowsPerConsumer + lane / kRopeLanesPerRow;
    const int rope_q = lane % kRopeLanesPerRow;
    float cs[8], sn[8];
    int trig = -1;
    long long cur_tile = -1;
    for (long long u = u0; u < u1; ++u) {
        const long long k = u - u0;
        const int s = (int)(k % kBulkStages);
        if (!mbar_wait_bounded(full0 + 8 * s, (uint32_t)((k / kBulkStages) & 1), abort_flag)) {
            if (lane == 0 && !*abort_flag) {
                *abort_flag = 1;
                raise_status(a.status, ST_TIMEOUT);
            }
            break;
        }
        const long long tile = u / L;
        const long long layer = u - tile * L;
        const RowDesc* rd = ring + (tile % kDescSlots) * kTileRows;
        if (tile != cur_tile) {
            cur_tile = tile;
            trig = rope_lane ? rd[rope_row].trig : -1;
            if (trig >= 0) {
                const int j0 = kLayout == 0 ? 8 * rope_q : 4 * rope_q;
                const float* tp = pv.trig + 2 * ((long long)trig * half + j0);
#pragma unroll
                for (int w = 0; w < (kLayout == 0 ? 8 : 4); ++w) {
                    cs[w] = tp[2 * w];
                    sn[w] = tp[2 * w + 1];
                }
            }
        }
        const uint32_t sbase = smem0 + (uint32_t)s * kStageBytes;
#pragma unroll
        for (int r = 0; r < kRowsPerConsumer; ++r) {
            const int i = cw * kRowsPerConsumer + r;
            const RowDesc d = rd[i];
            if (!d.src) continue;
            uint4* dst = d.dst + layer * layer_vecs;
            const uint32_t srow = sbase + (uint32_t)i * kRowBytes;
            const uint4 v0 = lds16(srow + 16u * lane);
            const uint4 v1 = lds16(srow + 16u * (lane + 32));
            st_stream(dst + lane, v0);
            st_stream(dst + lane + 32, v1);
        }
        if (rope_lane && rd[rope_row].src) {
            const RowDesc d = rd[rope_row];
            uint4* dst = d.dst + layer * layer_vecs + kLatentVecs;
            const uint32_t srow = sbase + (uint32_t)rope_row * kRowBytes + kLatentVecs * 16u;
            if (kLayout == 0) {
                uint4 x = lds16(srow + 16u * rope_q), y = lds16(srow + 16u * (rope_q + kRopeVecs / 2));
                if (trig >= 0) rotate_half_split<kBf16>(x, y, cs, sn);
                st_stream(dst + rope_q, x);
                st_stream(dst + rope_q + kRopeVecs / 2, y);
            } else {
                uint4 x = lds16(srow + 16u * rope_q);
                if (trig >= 0) rotate_interleaved<kBf16>(x, cs, sn);
                st_stream(dst + rope_q, x);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);  // this warp is done reading stage s
    }
}

// -------------------------------------------------------------------------
// Commit: block-table entries [b0, b0 + n_new) take the fresh pages, entries
// [b0 + n_new, b0 + n_old) become -1, the old pages of [b0, b0 + n_old) go back
// onto the free-page ring, and seq_lens_dev takes the new length.  One thread
// owns one table entry, so reading the old id and writing the new one cannot
// race; the pages taken ([pop_base, +total_pop) of the ring) and the slots
// written ([push_base, +total_push)) never overlap.
// The kernel runs as a programmatic dependent of move+rotate.  What it reads
// (plan, table, ring) was final before move+rotate started and move+rotate never
// writes it, so each thread loads its first entry before griddepcontrol.wait and
// only its writes wait for move+rotate to finish reading the table.  Its CTAs
// are small (128 threads) so that they fit beside the move kernel's CTAs.
constexpr int kCommitThreads = 128;

template <class PlanSrc>
__global__ void __launch_bounds__(kCommitThreads) commit_kernel(const __grid_constant__ SpliceArgs a,
                                                                const __grid_constant__ PlanSrc plan)
{
    const PlanView pv = plan_view(a, plan);
    const long long stride = (long long)gridDim.x * blockDim.x;
    long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    const ReqPlan* rp = nullptr;
    long long k = 0;
    int old = -1, fresh = -1;
    if (i < a.total_commit) {
        rp = &pv.reqs[find_req(pv.reqs, a.n_reqs, i, BY_COMMIT)];
        k = i - rp->commit_begin;
        if (k < rp->n_old) old = a.table_w[(long long)rp->req * a.max_blocks + rp->b0 + k];
        if (k < rp->n_new) fresh = a.free_q[ring(a.pop_base + rp->pop_off + k, a.q_cap)];
    }
    wait_for_previous_grid();
    allow_next_grid();
    while (i < a.total_commit) {
        int32_t* row = a.table_w + (long long)rp->req * a.max_blocks + rp->b0;
        if (k == 0) a.seq_lens_dev[rp->req] = (int32_t)rp->new_len;
        if (k < rp->n_new) row[k] = fresh;
        else if (k < rp->n_old) row[k] = -1;
        if (k < rp->n_old) {
            if (old < 0 || old >= a.g.num_pages) {
                raise_status(a.status, ST_BAD_OLD);
                old = -1;
            }
            a.free_q[ring(a.push_base + rp->push_off + k, a.q_cap)] = old;
            if (a.pending && old >= 0)  // a free page carries no pending turn
                for (int j = 0; j < a.g.block_size; ++j) a.pending[(long long)old * a.g.block_size + j] = 0;
        }
        i += stride;
        if (i >= a.total_commit) break;
        rp = &pv.reqs[find_req(pv.reqs, a.n_reqs, i, BY_COMMIT)];
        k = i - rp->commit_begin;
        old = k < rp->n_old ? a.table_w[(long long)rp->req * a.max_blocks + rp->b0 + k] : -1;
        fresh = k < rp->n_new ? a.free_q[ring(a.pop_base + rp->pop_off + k, a.q_cap)] : -1;
    }
}

// -------------------------------------------------------------------------
// Re-index mode (pool flag LEYLINE_POOL_REINDEX; block size 1, or a call whose
// directives all lie on block boundaries): a surviving downstream block keeps its
// page.  Up to four kernels, each a programmatic dependent of the one before:
//   prep          stages the page of every rewritten table entry (the kept block's
//                 old page, or a fresh page for a block of R) and returns the pages
//                 of dropped blocks to the ring; it reads the old table and writes
//                 only the staging array and the ring's push region;
//   rows of R     copies the call's rows of R into their fresh pages (if any);
//   rotate        turns the rope bands of every turned row in place (128 bytes read
//                 and written per band and layer; the latent is not touched; if any);
//   commit        installs the staged entries, clears entries past the new end,
//                 writes the new length.
template <class PlanSrc>
__global__ void prep_reindex(const __grid_constant__ SpliceArgs a, const __grid_constant__ PlanSrc plan)
{
    wait_for_previous_grid();
    allow_next_grid();
    const PlanView pv = plan_view(a, plan);
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long B = a.g.block_size;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < a.total_prep; i += stride) {
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
}

// 16-byte load that may be followed by a store to the same address (no .nc path).
__device__ __forceinline__ uint4 ld_rw(const uint4* p)
{
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Re-index mode writes fresh rows and turns kept bands.
//   copy_repl_reindex: the call's rows of R form one list; items of (row, 8 layers)
//   are spread over every warp of the grid, a lane moving every 32nd vector of the
//   row with four loads in flight.  A row of R moves 9 times the bytes of a turned
//   band, so rows of R are not tied to one CTA's share of the tiles.
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

// Layers per work unit of the re-index rotate kernel: as many as give each of the
// CTA's threads kItems work items (at least one layer).
__host__ __device__ __forceinline__ int reindex_layers_per_unit(int per_layer, int items)
{
    const int l = items * kMoveThreads / per_layer;
    return l > 0 ? l : 1;
}

// Rows of R of a re-indexed call into their fresh pages (the pages prep staged).
template <class PlanSrc>
__global__ void __launch_bounds__(kMoveThreads) copy_repl_reindex(const __grid_constant__ SpliceArgs a,
                                                                  const __grid_constant__ PlanSrc plan)
{
    wait_for_previous_grid();
    allow_next_grid();
    const PlanView pv = plan_view(a, plan);
    const int lane = threadIdx.x & 31;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long L = a.g.num_layers;
    const int chunks = (int)((L + kFreshLayers - 1) / kFreshLayers);
    const int row_vecs = a.g.row_vecs, lv = a.g.latent_vecs;
    uint4* kv = static_cast<uint4*>(a.kv);
    for (long long w = gw; w < a.total_repl * chunks; w += nw) {
        const long long rrow = w / chunks;
        const long long l0 = (w - rrow * chunks) * kFreshLayers;
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
            continue;
        }
        const Seg s = sg[k];
        const long long p = s.new_start + j;  // rows fit 32 bits (the planner checks lengths)
        const unsigned B = (unsigned)a.g.block_size, pb = (unsigned)p / B;
        const int page = a.stage[rp.stage_begin + ((long long)pb - rp.b0)];
        if (page < 0 || page >= a.g.num_pages) continue;  // prep has recorded a bad fresh page
        const long long slot = (long long)page * B + ((unsigned)p - pb * B);
        if (a.pending && l0 == 0 && lane == 0) a.pending[slot] = 0;  // R is encoded at its final position
        const long long rstride = (long long)s.n_repl * row_vecs;
        const uint4* src = static_cast<const uint4*>(s.repl) + j * row_vecs;
        const long long l1 = l0 + kFreshLayers < L ? l0 + kFreshLayers : L;
        for (long long layer = l0; layer < l1; ++layer) {
            for (int c0 = 0; c0 < row_vecs; c0 += 4 * 32) {
                uint4 v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c = c0 + 32 * q + lane;
                    if (c < row_vecs) v[q] = ld_stream(src + layer * rstride + c);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c = c0 + 32 * q + lane;
                    if (c < row_vecs)
                        st_stream(kv + (c < lv ? lat_off(a.g, layer, slot) + c : band_off(a.g, layer, slot) + (c - lv)),
                                  v[q]);
                }
            }
        }
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
    const PlanView pv = plan_view(a, plan);
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
__global__ void __launch_bounds__(kMoveThreads, kItems == 1 ? 8 : 2) rotate_in_place(const __grid_constant__ SpliceArgs a,
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
        if (++grp == groups) {
            grp = 0;
            ++tile;
        }
    }
}

// Commit of a re-indexed call: staged entries into the new blocks [b0, new end),
// -1 into the blocks past the new end, the new length, and (lazy pools) pending
// counts of 0 on the returned pages.  The staged values are final before the
// rotate kernel starts and it never writes them, so they are loaded before
// griddepcontrol.wait.
template <class PlanSrc>
__global__ void __launch_bounds__(kCommitThreads) commit_reindex(const __grid_constant__ SpliceArgs a,
                                                                 const __grid_constant__ PlanSrc plan)
{
    const PlanView pv = plan_view(a, plan);
    const long long stride = (long long)gridDim.x * blockDim.x;
    long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    int val = -1;
    const ReqPlan* rp = nullptr;
    long long k = 0;
    const long long B = a.g.block_size;
    if (i < a.total_commit) {
        rp = &pv.reqs[find_req(pv.reqs, a.n_reqs, i, BY_COMMIT)];
        k = i - rp->commit_begin;
        if (k < (rp->new_len + B - 1) / B - rp->b0) val = a.stage[rp->stage_begin + k];
    }
    wait_for_previous_grid();
    allow_next_grid();
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

__global__ void init_queue_kernel(int32_t* q, long long num_pages)
{
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < 2 * num_pages;
         i += (long long)gridDim.x * blockDim.x)
        q[i] = i < num_pages ? (int32_t)i : -1;
}

// Gather logical rows [t0, t1) of one request and layer into a contiguous buffer.
__global__ void gather_kernel(const uint4* kv, const int32_t* table_row, const Geometry g, long long layer,
                              long long t0, long long n, uint4* out, int32_t* status)
{
    const long long row_vecs = g.row_vecs, lv = g.latent_vecs, B = g.block_size;
    const long long total = n * row_vecs;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long r = i / row_vecs, c = i - r * row_vecs;
        const long long t = t0 + r;
        const int page = table_row[t / B];
        if (page < 0 || page >= g.num_pages) {
            raise_status(status, ST_BAD_PAGE);
            continue;
        }
        const long long slot = (long long)page * B + t % B;
        out[i] = c < lv ? kv[lat_off(g, layer, slot) + c] : kv[band_off(g, layer, slot) + (c - lv)];
    }
}

// -------------------------------------------------------------------------
// Lazy pools.  cos / sin of pending * theta_j: the angle is formed in fp64 and the
// fp64 sincos reduces it, then it is rounded once to the rotation's arithmetic,
// exactly as the host does for an eager splice.
__device__ __forceinline__ void pending_trig(int pend, double theta_j, bool bf16, float& c, float& s)
{
    double sd, cd;
    sincos((double)pend * theta_j, &sd, &cd);
    if (bf16) {
        c = __bfloat162float(__double2bfloat16(cd));
        s = __bfloat162float(__double2bfloat16(sd));
    } else {
        c = (float)cd;
        s = (float)sd;
    }
}

// cos / sin of the pairs of item q of a band: 8 pairs j = 8q.. (half-split) or 4
// pairs j = 4q.. (interleaved).
template <int kLayout>
__device__ __forceinline__ void item_trig(int pend, int q, const double* theta_j, bool bf16, float* c, float* s)
{
    constexpr int kPairs = kLayout == 0 ? 8 : 4;
#pragma unroll
    for (int w = 0; w < kPairs; ++w) pending_trig(pend, theta_j[kPairs * q + w], bf16, c[w], s[w]);
}

// Item q of the band at `band` (x at q, y at q + head_vecs / 2 for half-split),
// turned by (c, s) and written to `dst`.
template <int kLayout>
__device__ __forceinline__ void turn_item(const uint4* band, uint4* dst, int q, int hv, bool bf16, const float* c,
                                          const float* s)
{
    if (kLayout == 0) {
        uint4 x = band[q], y = band[q + hv / 2];
        if (bf16) rotate_half_split<true>(x, y, c, s);
        else rotate_half_split<false>(x, y, c, s);
        dst[q] = x;
        dst[q + hv / 2] = y;
    } else {
        uint4 x = band[q];
        if (bf16) rotate_interleaved<true>(x, c, s);
        else rotate_interleaved<false>(x, c, s);
        dst[q] = x;
    }
}

// Gather from a lazy pool: one warp per row.  The latent is copied; item q of each
// rope band is turned by the slot's pending count on the way out.
template <int kLayout>
__global__ void gather_lazy_kernel(const uint4* kv, const int32_t* table_row, const Geometry g, long long layer,
                                   long long t0, long long n, uint4* out, const int32_t* pending,
                                   const double* theta_j, int32_t* status)
{
    const int lane = threadIdx.x & 31;
    const bool bf16 = g.precision == LEYLINE_ROTATE_BF16_NAIVE;
    const int hv = g.head_vecs;
    const int head_items = kLayout == 0 ? hv / 2 : hv;
    const long long warps = (long long)gridDim.x * (blockDim.x / 32);
    for (long long r = blockIdx.x * (long long)(blockDim.x / 32) + threadIdx.x / 32; r < n; r += warps) {
        const long long t = t0 + r;
        const long long B = g.block_size;
        const int page = table_row[t / B];
        if (page < 0 || page >= g.num_pages) {
            if (lane == 0) raise_status(status, ST_BAD_PAGE);
            continue;
        }
        const long long slot = (long long)page * B + t % B;
        const uint4* lat = kv + lat_off(g, layer, slot);
        const uint4* bands = kv + band_off(g, layer, slot);
        uint4* o = out + r * g.row_vecs;
        for (int c = lane; c < g.latent_vecs; c += 32) o[c] = lat[c];
        const int pend = pending[slot];
        for (int it = lane; it < g.rope_heads * head_items; it += 32) {
            const int head = it / head_items, q = it - head * head_items;
            const uint4* band = bands + head * hv;
            uint4* dst = o + g.latent_vecs + head * hv;
            if (pend == 0) {
                dst[q] = band[q];
                if (kLayout == 0) dst[q + hv / 2] = band[q + hv / 2];
                continue;
            }
            float c[8], s[8];
            item_trig<kLayout>(pend, q, theta_j, bf16, c, s);
            turn_item<kLayout>(band, dst, q, hv, bf16, c, s);
        }
    }
}

// Materialize a lazy request: one warp per row.  Lanes take the row's (layer,
// band item) pairs in turn, so the pair group q of a lane, and the cos / sin held
// for it, change only when the items per layer do not divide 32.  The count is
// read before and cleared after every layer of the row is turned in place.
template <int kLayout>
__global__ void materialize_kernel(uint4* kv, const int32_t* table_row, const Geometry g, long long len,
                                   int32_t* pending, const double* theta_j, int32_t* status)
{
    const int lane = threadIdx.x & 31;
    const bool bf16 = g.precision == LEYLINE_ROTATE_BF16_NAIVE;
    const int hv = g.head_vecs;
    const int head_items = kLayout == 0 ? hv / 2 : hv;
    const int items = g.rope_heads * head_items;  // per layer
    const long long warps = (long long)gridDim.x * (blockDim.x / 32);
    for (long long t = blockIdx.x * (long long)(blockDim.x / 32) + threadIdx.x / 32; t < len; t += warps) {
        const long long B = g.block_size;
        const int page = table_row[t / B];
        if (page < 0 || page >= g.num_pages) {
            if (lane == 0) raise_status(status, ST_BAD_PAGE);
            continue;
        }
        const long long slot = (long long)page * B + t % B;
        const int pend = pending[slot];
        if (pend == 0) continue;
        float c[8], s[8];
        int have_q = -1;
        for (long long idx = lane; idx < (long long)g.num_layers * items; idx += 32) {
            const long long layer = idx / items;
            const int it = (int)(idx - layer * items);
            const int head = it / head_items, q = it - head * head_items;
            if (q != have_q) {
                item_trig<kLayout>(pend, q, theta_j, bf16, c, s);
                have_q = q;
            }
            uint4* band = kv + band_off(g, layer, slot) + head * hv;
            turn_item<kLayout>(band, band, q, hv, bf16, c, s);
        }
        __syncwarp();
        if (lane == 0) pending[slot] = 0;
    }
}

__global__ void clear_pending_kernel(int32_t* pending, const int32_t* page_ids, long long n, int block_size)
{
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n * block_size;
         i += (long long)gridDim.x * blockDim.x)
        pending[(long long)page_ids[i / block_size] * block_size + i % block_size] = 0;
}

int grid_for(long long items, int threads, int cap)
{
    long long g = (items + threads - 1) / threads;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return (int)g;
}

bool mla_shape(const Geometry& g) { return g.latent_vecs == 64 && g.rope_vecs == 8 && g.rope_heads == 1; }

// Launch with programmatic stream serialization: the kernel may start before the
// previous kernel in the stream ends; it calls griddepcontrol.wait before it
// reads anything that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), int grid, int block, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Launch with programmatic stream serialization and dynamic shared memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent_smem(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t s,
                                  Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <class PlanSrc>
cudaError_t launch_bulk(const SpliceArgs& a, const PlanSrc& plan, int grid, cudaStream_t s)
{
    const bool bf16 = a.g.precision == LEYLINE_ROTATE_BF16_NAIVE;
    const size_t smem = bulk_smem_bytes((uint32_t)a.g.row_vecs * 16u);
    if (a.g.pair_layout == LEYLINE_PAIRS_HALF_SPLIT)
        return bf16 ? launch_dependent_smem(move_rotate_bulk<0, true, PlanSrc>, grid, kBulkThreads, smem, s, a, plan)
                    : launch_dependent_smem(move_rotate_bulk<0, false, PlanSrc>, grid, kBulkThreads, smem, s, a, plan);
    return bf16 ? launch_dependent_smem(move_rotate_bulk<1, true, PlanSrc>, grid, kBulkThreads, smem, s, a, plan)
                : launch_dependent_smem(move_rotate_bulk<1, false, PlanSrc>, grid, kBulkThreads, smem, s, a, plan);
}

template <class PlanSrc>
cudaError_t launch_move(const SpliceArgs& a, const PlanSrc& plan, int grid, cudaStream_t s)
{
    // the bulk kernel copies whole rows: pools of whole rows only
    if (a.move_kernel == MOVE_BULK && mla_shape(a.g) && !(a.g.flags & LEYLINE_POOL_SPLIT_ROPE))
        return launch_bulk(a, plan, grid, s);
    const bool bf16 = a.g.precision == LEYLINE_ROTATE_BF16_NAIVE;
    if (mla_shape(a.g)) {
        if (a.g.pair_layout == LEYLINE_PAIRS_HALF_SPLIT)
            return bf16 ? launch_dependent(move_rotate_mla<0, true, PlanSrc>, grid, kMoveThreads, s, a, plan)
                        : launch_dependent(move_rotate_mla<0, false, PlanSrc>, grid, kMoveThreads, s, a, plan);
        return bf16 ? launch_dependent(move_rotate_mla<1, true, PlanSrc>, grid, kMoveThreads, s, a, plan)
                    : launch_dependent(move_rotate_mla<1, false, PlanSrc>, grid, kMoveThreads, s, a, plan);
    }
    return bf16 ? launch_dependent(move_rotate_generic<true, PlanSrc>, grid, kMoveThreads, s, a, plan)
                : launch_dependent(move_rotate_generic<false, PlanSrc>, grid, kMoveThreads, s, a, plan);
}

template <class PlanSrc>
int launch_reindex(const SpliceArgs& a, const PlanSrc& plan, int grid, cudaStream_t s, cudaEvent_t t0, cudaEvent_t t1)
{
    cudaError_t e = cudaSuccess;
    if (a.total_prep > 0)
        e = launch_dependent(prep_reindex<PlanSrc>, grid_for(a.total_prep, 256, 8192), 256, s, a, plan);
    const bool bf16 = a.g.precision == LEYLINE_ROTATE_BF16_NAIVE;
    const bool split = a.g.pair_layout == LEYLINE_PAIRS_HALF_SPLIT;
    const int ipr = a.g.rope_heads * (split ? a.g.head_vecs / 2 : a.g.head_vecs);
    const int per_layer = kTileRows * ipr;
    const bool mla = per_layer <= kMoveThreads;  // one item per thread; else kMaxItems
    const int lpu = reindex_layers_per_unit(per_layer, mla ? 1 : kMaxItems);
    const long long units = a.total_tiles * ((a.g.num_layers + lpu - 1) / lpu);
    if (grid > units) grid = (int)std::max<long long>(units, 1);
    if (e == cudaSuccess && t0) e = cudaEventRecord(t0, s);
    if (e == cudaSuccess && a.total_repl > 0) {  // rows of R: items of (row, kFreshLayers layers), a warp each
        const long long items = a.total_repl * ((a.g.num_layers + kFreshLayers - 1) / kFreshLayers);
        e = launch_dependent(copy_repl_reindex<PlanSrc>, grid_for(items * 32, kMoveThreads, 8192), kMoveThreads, s,
                             a, plan);
    }
    if (e == cudaSuccess && a.total_fresh > 0) {  // other fresh rows: items of (row, kFreshLayers layers)
        const long long items = a.total_fresh * ((a.g.num_layers + kFreshLayers - 1) / kFreshLayers);
        const int fgrid = grid_for(items * 32, kMoveThreads, 8192);
        auto k = split ? (bf16 ? copy_fresh_reindex<0, true, PlanSrc> : copy_fresh_reindex<0, false, PlanSrc>)
                       : (bf16 ? copy_fresh_reindex<1, true, PlanSrc> : copy_fresh_reindex<1, false, PlanSrc>);
        e = launch_dependent(k, fgrid, kMoveThreads, s, a, plan);
    }
    if (e == cudaSuccess && units > 0) {
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
        e = launch_dependent(commit_reindex<PlanSrc>, grid_for(a.total_commit, kCommitThreads, 8192), kCommitThreads, s,
                             a, plan);
    if (e == cudaSuccess) e = cudaGetLastError();
    return (int)e;
}

template <class PlanSrc>
int launch_both(const SpliceArgs& a, const PlanSrc& plan, int grid, cudaStream_t s, cudaEvent_t t0, cudaEvent_t t1)
{
    if (a.reindex) return launch_reindex(a, plan, grid, s, t0, t1);
    const long long units = a.total_tiles * a.g.num_layers;
    if (grid > units) grid = (int)std::max<long long>(units, 1);
    cudaError_t e = cudaSuccess;
    if (t0) e = cudaEventRecord(t0, s);
    if (e == cudaSuccess && units > 0) e = launch_move(a, plan, grid, s);
    if (e == cudaSuccess && t1) e = cudaEventRecord(t1, s);
    if (e == cudaSuccess && a.total_commit > 0) {
        const int cgrid = grid_for(a.total_commit, kCommitThreads, 8192);
        if (units > 0) {
            e = launch_dependent(commit_kernel<PlanSrc>, cgrid, kCommitThreads, s, a, plan);
        } else {  // no move kernel before it: a plain launch, so its early reads see all earlier work
            commit_kernel<PlanSrc><<<cgrid, kCommitThreads, 0, s>>>(a, plan);
            e = cudaGetLastError();
        }
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    return (int)e;
}

}  // namespace

int launch_init_queue(int32_t* q, int64_t num_pages, void* stream)
{
    init_queue_kernel<<<grid_for(2 * num_pages, 256, 4096), 256, 0, (cudaStream_t)stream>>>(q, num_pages);
    return (int)cudaGetLastError();
}

int launch_splice(const SpliceArgs& a, const ParamPlan* pp, int grid, void* stream, cudaEvent_t t0, cudaEvent_t t1)
{
    cudaStream_t s = (cudaStream_t)stream;
    if (pp) return launch_both(a, *pp, grid, s, t0, t1);
    return launch_both(a, NoParamPlan{0}, grid, s, t0, t1);
}

int launch_gather(const void* kv, const int32_t* table_row, const Geometry& g, int32_t layer, int64_t t0,
                  int64_t t1, void* out, int32_t* status, void* stream)
{
    const long long n = t1 - t0;
    if (n <= 0) return 0;
    gather_kernel<<<grid_for(n * g.row_vecs, 256, 8192), 256, 0, (cudaStream_t)stream>>>(
        static_cast<const uint4*>(kv), table_row, g, layer, t0, n, static_cast<uint4*>(out), status);
    return (int)cudaGetLastError();
}

int rotate_in_place_blocks_per_sm(int* blocks)
{
    return (int)cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, rotate_in_place<0, false, 1, ParamPlan>,
                                                              kMoveThreads, 0);
}

int launch_gather_lazy(const void* kv, const int32_t* table_row, const Geometry& g, int32_t layer, int64_t t0,
                       int64_t t1, void* out, const int32_t* pending, const double* theta_j, int32_t* status,
                       void* stream)
{
    const long long n = t1 - t0;
    if (n <= 0) return 0;
    auto k = g.pair_layout == LEYLINE_PAIRS_HALF_SPLIT ? gather_lazy_kernel<0> : gather_lazy_kernel<1>;
    k<<<grid_for(n * 32, 256, 8192), 256, 0, (cudaStream_t)stream>>>(static_cast<const uint4*>(kv), table_row, g,
                                                                      layer, t0, n, static_cast<uint4*>(out),
                                                                      pending, theta_j, status);
    return (int)cudaGetLastError();
}

int launch_materialize(void* kv, const int32_t* table_row, const Geometry& g, int64_t len, int32_t* pending,
                       const double* theta_j, int32_t* status, void* stream)
{
    if (len <= 0) return 0;
    auto k = g.pair_layout == LEYLINE_PAIRS_HALF_SPLIT ? materialize_kernel<0> : materialize_kernel<1>;
    k<<<grid_for(len * 32, 256, 8192), 256, 0, (cudaStream_t)stream>>>(static_cast<uint4*>(kv), table_row, g, len,
                                                                        pending, theta_j, status);
    return (int)cudaGetLastError();
}

int launch_clear_pending(int32_t* pending, const int32_t* page_ids, int64_t n, int32_t block_size, void* stream)
{
    if (n <= 0) return 0;
    clear_pending_kernel<<<grid_for(n * block_size, 256, 4096), 256, 0, (cudaStream_t)stream>>>(pending, page_ids, n,
                                                                                             block_size);
    return (int)cudaGetLastError();
}

int move_rotate_blocks_per_sm(int* blocks)
{
    return (int)cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, move_rotate_mla<0, false, ParamPlan>,
                                                              kMoveThreads, 0);
}

namespace {
template <class K>
cudaError_t allow_smem(K kernel, size_t smem)
{
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}
}  // namespace

int bulk_prepare(int32_t row_bytes, int* blocks)
{
    *blocks = 0;
    const size_t smem = bulk_smem_bytes((uint32_t)row_bytes);
    int dev = 0, limit = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&limit, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return (int)e;
    if (smem > (size_t)limit) return 0;  // rows too wide for the staged kernel: *blocks stays 0
    e = allow_smem(move_rotate_bulk<0, false, ParamPlan>, smem);
    if (e == cudaSuccess) e = allow_smem(move_rotate_bulk<0, true, ParamPlan>, smem);
    if (e == cudaSuccess) e = allow_smem(move_rotate_bulk<1, false, ParamPlan>, smem);
    if (e == cudaSuccess) e = allow_smem(move_rotate_bulk<1, true, ParamPlan>, smem);
    if (e == cudaSuccess) e = allow_smem(move_rotate_bulk<0, false, NoParamPlan>, smem);
    if (e == cudaSuccess) e = allow_smem(move_rotate_bulk<0, true, NoParamPlan>, smem);
    if (e == cudaSuccess) e = allow_smem(move_rotate_bulk<1, false, NoParamPlan>, smem);
    if (e == cudaSuccess) e = allow_smem(move_rotate_bulk<1, true, NoParamPlan>, smem);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, move_rotate_bulk<0, false, ParamPlan>, kBulkThreads,
                                                          smem);
    return (int)e;
}

}  // namespace leyline
