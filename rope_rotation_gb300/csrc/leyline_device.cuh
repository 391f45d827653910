// leyline_device.cuh -- device helpers shared by the kernel translation units of the GB300
// Leyline AMORTIZE splice (sm_103a): leyline_move.cu (rewrite: move+rotate, commit),
// leyline_reindex.cu (re-index pools), leyline_read.cu (gathers, lazy reads, queues).
//
// "Leyline: KV Cache Directives for Agentic Inference":
//   section 2.2  every downstream slot's RoPE band gets K_pe_new = R(Delta) K_pe
//                (one 2x2 rotation per pair); K_nope and V (here: the compressed
//                latent they derive from) are kept.
//   section 4.3  the rotation is computed in fp32 and stored in bf16.
//
// Everything here lives in an unnamed namespace: each translation unit has its own
// copy, and the kernels of one unit see only their own instantiations.
#pragma once

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

// A 16-byte vector from lane ^ m (every lane of the warp takes part).
__device__ __forceinline__ uint4 shfl_xor_vec(uint4 v, int m)
{
    v.x = __shfl_xor_sync(0xffffffffu, v.x, m);
    v.y = __shfl_xor_sync(0xffffffffu, v.y, m);
    v.z = __shfl_xor_sync(0xffffffffu, v.z, m);
    v.w = __shfl_xor_sync(0xffffffffu, v.w, m);
    return v;
}

// Half-split pairs, one half only: the lane holding x (pairs j0..j0+7) returns
// x' = x c - y s, the lane holding y returns y' = x s + y c, each with the arithmetic of
// rotate_half_split (fp32: one FMA per output; bf16 arm: products and sum rounded).
template <bool kBf16>
__device__ __forceinline__ uint4 turn_own_half(const uint4& mine, const uint4& other, bool y_half, const float* c,
                                               const float* s)
{
    const uint32_t* mw = reinterpret_cast<const uint32_t*>(&mine);
    const uint32_t* ow = reinterpret_cast<const uint32_t*>(&other);
    uint4 out;
    uint32_t* rw = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        float r[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float m = h ? bf16_hi(mw[w]) : bf16_lo(mw[w]);
            const float o = h ? bf16_hi(ow[w]) : bf16_lo(ow[w]);
            const float x = y_half ? o : m, y = y_half ? m : o;
            const float cc = c[2 * w + h], ss = s[2 * w + h];
            if (kBf16) {
                r[h] = y_half ? round_bf16(x * ss) + round_bf16(y * cc) : round_bf16(x * cc) - round_bf16(y * ss);
            } else {
                r[h] = y_half ? fmaf(x, ss, y * cc) : fmaf(x, cc, -(y * ss));
            }
        }
        rw[w] = pack_bf16x2(r[0], r[1]);
    }
    return out;
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

// CTAs of the commit kernels are small (128 threads) so that they fit beside the
// CTAs of the kernel before them.
constexpr int kCommitThreads = 128;

// 16-byte load that may be followed by a store to the same address (no .nc path).
__device__ __forceinline__ uint4 ld_rw(const uint4* p)
{
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ------------------------------------------------------------ launches --
inline int grid_for(long long items, int threads, int cap)
{
    long long g = (items + threads - 1) / threads;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return (int)g;
}

inline bool mla_shape(const Geometry& g) { return g.latent_vecs == 64 && g.rope_vecs == 8 && g.rope_heads == 1; }

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

}  // namespace
}  // namespace leyline
