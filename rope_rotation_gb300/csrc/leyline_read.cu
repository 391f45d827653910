// leyline_read.cu -- reads and bookkeeping kernels of the GB300 Leyline splice library
// (sm_103a): the free-page ring's initial fill, gathers of logical rows (lazy pools turn
// each row's bands by its pending count on the way out), materialize, pending clears.
//
// "Leyline: KV Cache Directives for Agentic Inference", section 2.2: R(a) R(b) = R(a + b),
// so a lazy pool's summed turn is applied once when a row is read.
#include "leyline_device.cuh"

namespace leyline {
namespace {

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
// Lazy pools.  cos / sin of pending * theta_j, formed in fp64 and rounded once to the
// rotation's arithmetic, as the host does for an eager splice.  A count below
// kTurnSpan^2 in magnitude takes the angle-addition product of the pool's two turn
// tables (R(a) R(b) = R(a + b): 2 loads and 6 fp64 operations); a larger one, fp64
// sincos of the angle.
__device__ __forceinline__ void pending_trig(int pend, const double* turn, int half, int j, bool bf16, float& c,
                                             float& s)
{
    const long long a = pend < 0 ? -(long long)pend : (long long)pend;
    double sd, cd;
    if (a < (long long)kTurnSpan * kTurnSpan) {
        const double2* lo = reinterpret_cast<const double2*>(turn + (half + 1) / 2 * 2);
        const double2* hi = lo + (size_t)half * kTurnSpan;
        const double2 l = lo[(size_t)j * kTurnSpan + (a % kTurnSpan)];
        const double2 h = hi[(size_t)j * kTurnSpan + (a / kTurnSpan)];
        cd = fma(h.x, l.x, -(h.y * l.y));
        sd = fma(h.y, l.x, h.x * l.y);
        if (pend < 0) sd = -sd;
    } else {
        sincos((double)pend * turn[j], &sd, &cd);
    }
    if (bf16) {
        c = __bfloat162float(__double2bfloat16(cd));
        s = __bfloat162float(__double2bfloat16(sd));
    } else {
        c = (float)cd;
        s = (float)sd;
    }
}

// The read kernels run one warp per row.  A warp forms the cos / sin of every pair
// of a band once per pending count -- a lane per pair, into the warp's slice of
// shared memory -- and keeps them while the count stays the same (after a splice a
// segment's survivors share one count); each lane then reads the pairs of its items.
constexpr int kReadThreads = 256;
constexpr int kMaxPairs = 128;  // rope_dim <= 256

struct WarpTrig {
    float2* cs;     // this warp's [kMaxPairs] (cos, sin)
    int pend = 0;   // count the slice holds
    bool valid = false;

    __device__ __forceinline__ void ensure(int count, const double* turn, int half, bool bf16)
    {
        if (valid && count == pend) return;  // warp-uniform: the count is the row's
        __syncwarp();                        // lanes are done reading the previous count's values
        for (int j = threadIdx.x & 31; j < half; j += 32) {
            float c, s;
            pending_trig(count, turn, half, j, bf16, c, s);
            cs[j] = make_float2(c, s);
        }
        __syncwarp();
        pend = count;
        valid = true;
    }
};

// cos / sin of the pairs of item q of a band: 8 pairs j = 8q.. (half-split) or 4
// pairs j = 4q.. (interleaved).
template <int kLayout>
__device__ __forceinline__ void item_trig(const float2* cs, int q, float* c, float* s)
{
    constexpr int kPairs = kLayout == 0 ? 8 : 4;
#pragma unroll
    for (int w = 0; w < kPairs; ++w) {
        const float2 v = cs[kPairs * q + w];
        c[w] = v.x;
        s[w] = v.y;
    }
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
                                   const double* turn, int32_t* status)
{
    __shared__ float2 trig_smem[kReadThreads / 32][kMaxPairs];
    const int lane = threadIdx.x & 31;
    const bool bf16 = g.precision == LEYLINE_ROTATE_BF16_NAIVE;
    const int hv = g.head_vecs;
    const int head_items = kLayout == 0 ? hv / 2 : hv;
    const int half = g.rope_dim / 2;
    WarpTrig wt;
    wt.cs = trig_smem[threadIdx.x / 32];
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
        if (pend != 0) wt.ensure(pend, turn, half, bf16);
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
            item_trig<kLayout>(wt.cs, q, c, s);
            turn_item<kLayout>(band, dst, q, hv, bf16, c, s);
        }
    }
}

// Materialize lazy requests: the rows of the set's requests form one list, one warp per
// row (its request found by binary search over the cumulative row ends), its lanes walking
// the row's (layer, band item) pairs.  When the items per layer divide 32 -- MLA bands, and 1, 2, 4 or 8
// GQA heads -- a lane's item is the same in every layer, so its cos / sin are read
// once per row and two layers' loads are in flight before either layer's stores.  The
// count is read before and cleared after every layer of the row is turned in place.
template <int kLayout>
__global__ void materialize_kernel(uint4* kv, const int32_t* table, int max_blocks,
                                   const __grid_constant__ MaterializeSet set, const Geometry g, int32_t* pending,
                                   const double* turn, int32_t* status)
{
    __shared__ float2 trig_smem[kReadThreads / 32][kMaxPairs];
    const int lane = threadIdx.x & 31;
    const bool bf16 = g.precision == LEYLINE_ROTATE_BF16_NAIVE;
    const int hv = g.head_vecs;
    const int head_items = kLayout == 0 ? hv / 2 : hv;
    const int items = g.rope_heads * head_items;  // per layer
    const int half = g.rope_dim / 2;
    const long long n_it = (long long)g.num_layers * items;
    const bool fixed_item = 32 % items == 0;
    WarpTrig wt;
    wt.cs = trig_smem[threadIdx.x / 32];
    const long long warps = (long long)gridDim.x * (blockDim.x / 32);
    const long long rows = set.row_end[set.n - 1];
    for (long long f = blockIdx.x * (long long)(blockDim.x / 32) + threadIdx.x / 32; f < rows; f += warps) {
        int lo = 0, hi = set.n - 1;  // first request whose rows end after f
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (set.row_end[mid] > f) hi = mid;
            else lo = mid + 1;
        }
        const long long t = f - (lo ? set.row_end[lo - 1] : 0);
        const int32_t* table_row = table + (long long)set.req[lo] * max_blocks;
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
        if (fixed_item) {
            const int it = lane % items;
            const int head = it / head_items, q = it - head * head_items;
            uint4 x0, y0, x1, y1;
            uint4 *b0 = nullptr, *b1 = nullptr;
            bool one = false, two = false;
            auto load = [&](long long idx) {
                one = idx < n_it;
                two = idx + 32 < n_it;
                b0 = kv + band_off(g, idx / items, slot) + head * hv;
                b1 = kv + band_off(g, (idx + 32) / items, slot) + head * hv;
                if (one) {
                    x0 = b0[q];
                    if (kLayout == 0) y0 = b0[q + hv / 2];
                }
                if (two) {
                    x1 = b1[q];
                    if (kLayout == 0) y1 = b1[q + hv / 2];
                }
            };
            load(lane);  // the first two layers' loads are in flight while the cos / sin form
            wt.ensure(pend, turn, half, bf16);
            item_trig<kLayout>(wt.cs, q, c, s);
            for (long long idx = lane; idx < n_it; idx += 64) {
                if (idx != lane) load(idx);
                if (kLayout == 0) {
                    if (bf16) rotate_half_split<true>(x0, y0, c, s);
                    else rotate_half_split<false>(x0, y0, c, s);
                    b0[q] = x0;
                    b0[q + hv / 2] = y0;
                    if (two) {
                        if (bf16) rotate_half_split<true>(x1, y1, c, s);
                        else rotate_half_split<false>(x1, y1, c, s);
                        b1[q] = x1;
                        b1[q + hv / 2] = y1;
                    }
                } else {
                    if (bf16) rotate_interleaved<true>(x0, c, s);
                    else rotate_interleaved<false>(x0, c, s);
                    b0[q] = x0;
                    if (two) {
                        if (bf16) rotate_interleaved<true>(x1, c, s);
                        else rotate_interleaved<false>(x1, c, s);
                        b1[q] = x1;
                    }
                }
            }
        } else {
            wt.ensure(pend, turn, half, bf16);
            int have_q = -1;
            for (long long idx = lane; idx < n_it; idx += 32) {
                const long long layer = idx / items;
                const int it = (int)(idx - layer * items);
                const int head = it / head_items, q = it - head * head_items;
                if (q != have_q) {
                    item_trig<kLayout>(wt.cs, q, c, s);
                    have_q = q;
                }
                uint4* band = kv + band_off(g, layer, slot) + head * hv;
                turn_item<kLayout>(band, band, q, hv, bf16, c, s);
            }
        }
        __syncwarp();
        if (lane == 0) pending[slot] = 0;
    }
}

// -------------------------------------------------------------------------
// Materialize, rows whose rope bands fill 8 vectors (MLA: one 64-wide band; GQA: 2 bands
// of 32 or 4 of 16), in two kernels.  compact_pending_kernel lists the set's rows whose
// count is not 0 (slot and count; the order of rows is kept within each block of 256), so
// that the band pass splits only rows with work among its CTAs: after a splice the turned
// rows of a request are one contiguous stretch, and an even split of all rows would leave
// most CTAs idle.  materialize_band8_kernel cuts the list into tiles of 32 rows, and a unit
// is (tile, kMatLayers layers); the CTAs take contiguous runs of units.  In a unit each
// row's band is moved by 8 lanes, one 16-byte chunk each (a warp instruction covers four
// whole 128-byte bands; half-split: the partner half comes from lane ^ head_vecs/2), with
// the loads of all kMatLayers layers issued before any store.
//
// A prologue per chunk of up to 8 tiles reads the list (warp w: tile w of the chunk) and
// clears the rows' counts (the band pass reads counts from the list only).  Consecutive
// rows mostly share their count (a splice's survivors of one segment), so each warp forms
// the cos / sin once per run of equal counts in its tile, for the first kMatRuns runs;
// rows of later runs (more than kMatRuns distinct counts in 32 rows) form their own.
constexpr int kMatThreads = 256;
constexpr int kMatTileRows = 32;  // 8 lanes per row
#ifndef LEYLINE_MAT_LAYERS
#define LEYLINE_MAT_LAYERS 4
#endif
#ifndef LEYLINE_MAT_MIN_CTAS
#define LEYLINE_MAT_MIN_CTAS 3
#endif
constexpr int kMatLayers = LEYLINE_MAT_LAYERS;  // layers in flight per unit
constexpr int kMatChunkTiles = kMatThreads / 32;
constexpr int kMatRuns = 4;

// (cos, sin) of pair j of one count, out of line: the rare path of rows whose count has
// no shared slot (returned by value, so the caller keeps its arrays in registers).
__device__ __noinline__ float2 pair_trig(int pend, const double* turn, int half, int j, bool bf16)
{
    float c, s;
    pending_trig(pend, turn, half, j, bf16, c, s);
    return make_float2(c, s);
}

// Slot of flat row f of the set (-1 with the status bit raised when its page is bad).
__device__ __forceinline__ long long set_row_slot(const MaterializeSet& set, const int32_t* table, int max_blocks,
                                                  const Geometry& g, long long f, int32_t* status)
{
    int lo = 0, hi = set.n - 1;  // first request whose rows end after f
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (set.row_end[mid] > f) hi = mid;
        else lo = mid + 1;
    }
    const long long t = f - (lo ? set.row_end[lo - 1] : 0);
    const long long B = g.block_size;
    const int page = table[(long long)set.req[lo] * max_blocks + t / B];
    if (page < 0 || page >= g.num_pages) {
        raise_status(status, ST_BAD_PAGE);
        return -1;
    }
    return (long long)page * B + t % B;
}

// The set's rows with a count other than 0, appended to (slot, count) lists at *n.
__global__ void __launch_bounds__(kMatThreads) compact_pending_kernel(const int32_t* table, int max_blocks,
                                                                      const __grid_constant__ MaterializeSet set,
                                                                      const Geometry g, const int32_t* pending,
                                                                      long long* out_slot, int32_t* out_pend,
                                                                      unsigned long long* n, int32_t* status)
{
    __shared__ int warp_n[kMatThreads / 32];
    __shared__ unsigned long long base;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long rows = set.row_end[set.n - 1];
    // every CTA runs the same number of rounds, so that all its threads reach the barriers
    for (long long f0 = (long long)blockIdx.x * kMatThreads; f0 < rows; f0 += (long long)gridDim.x * kMatThreads) {
        const long long f = f0 + threadIdx.x;
        long long slot = -1;
        int pend = 0;
        if (f < rows) {
            slot = set_row_slot(set, table, max_blocks, g, f, status);
            if (slot >= 0) pend = pending[slot];
        }
        const unsigned has = __ballot_sync(0xffffffffu, pend != 0);
        if (lane == 0) warp_n[warp] = __popc(has);
        __syncthreads();
        if (threadIdx.x == 0) {
            int total = 0;
            for (int w = 0; w < kMatThreads / 32; ++w) {
                const int c = warp_n[w];
                warp_n[w] = total;  // exclusive prefix
                total += c;
            }
            base = total ? atomicAdd(n, (unsigned long long)total) : 0ull;
        }
        __syncthreads();
        if (pend != 0) {
            const unsigned long long at = base + warp_n[warp] + __popc(has & ((1u << lane) - 1u));
            out_slot[at] = slot;
            out_pend[at] = pend;
        }
        __syncthreads();  // warp_n and base are rewritten in the next round
    }
    allow_next_grid();  // the band pass may launch; it waits for this grid before reading the lists
}

template <int kLayout, bool kBf16>
__global__ void __launch_bounds__(kMatThreads, LEYLINE_MAT_MIN_CTAS) materialize_band8_kernel(uint4* kv, const Geometry g,
                                                                        const long long* list_slot,
                                                                        const int32_t* list_pend,
                                                                        const unsigned long long* list_n,
                                                                        unsigned long long* next_n, int32_t* pending,
                                                                        const double* turn)
{
    __shared__ long long slot_s[kMatChunkTiles][kMatTileRows];  // -1: nothing to turn
    __shared__ int cnt_s[kMatChunkTiles][kMatTileRows];         // the row's count
    __shared__ int run_s[kMatChunkTiles][kMatTileRows];         // its run among the tile's counts
    __shared__ float2 cs_s[kMatChunkTiles][kMatRuns][32];        // (cos, sin) per pair of the first runs
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int hv = g.head_vecs;
    const int half = g.rope_dim / 2;  // <= 32: the row's bands fill 8 vectors
    const int row = threadIdx.x >> 3, c = threadIdx.x & 7;  // this thread's row of a tile and chunk of it
    const int q = c & (hv - 1);                              // chunk within its band
    constexpr int kPairs = kLayout == 0 ? 8 : 4;
    const int j0 = kLayout == 0 ? kPairs * (q & (hv / 2 - 1)) : kPairs * q;  // first pair of the chunk
    const bool y_half = kLayout == 0 && q >= hv / 2;
    const long long L = g.num_layers;
    const long long groups = (L + kMatLayers - 1) / kMatLayers;
    wait_for_previous_grid();  // the lists are complete
    const long long rows = (long long)*list_n;
    if (blockIdx.x == 0 && threadIdx.x == 0) *next_n = 0;  // the next launch's counter (its lists are not in use)
    const long long tiles = (rows + kMatTileRows - 1) / kMatTileRows;
    long long u0, u1;
    my_units(tiles * groups, u0, u1);
    long long u = u0;
    while (u < u1) {
        // prologue of a chunk: the tiles from the current unit's on
        const long long t0 = u / groups;
        const long long t_end = (u1 - 1) / groups + 1 < t0 + kMatChunkTiles ? (u1 - 1) / groups + 1 : t0 + kMatChunkTiles;
        __syncthreads();  // the previous chunk's shared values are no longer read
        {
            const long long tile = t0 + warp;
            const long long f = tile * kMatTileRows + lane;
            long long slot = -1;
            int pend = 0;
            if (tile < t_end && f < rows) {
                slot = list_slot[f];
                pend = list_pend[f];
                pending[slot] = 0;  // a slot is listed once; the band pass reads counts from the list
            }
            const int prev = __shfl_up_sync(0xffffffffu, pend, 1);
            const bool start = pend != 0 && (lane == 0 || prev != pend);
            const unsigned starts = __ballot_sync(0xffffffffu, start);
            const int run = pend != 0 ? __popc(starts & (0xffffffffu >> (31 - lane))) - 1 : -1;
            slot_s[warp][lane] = pend != 0 ? slot : -1;
            cnt_s[warp][lane] = pend;
            run_s[warp][lane] = run;
            const int runs = __popc(starts);
            unsigned rest = starts;
            for (int r = 0; r < runs && r < kMatRuns; ++r) {
                const int src = __ffs(rest) - 1;  // lane where run r starts
                rest &= rest - 1;
                const int cnt = __shfl_sync(0xffffffffu, pend, src);
                if (lane < half) {
                    float cc, ss;
                    pending_trig(cnt, turn, half, lane, kBf16, cc, ss);
                    cs_s[warp][r][lane] = make_float2(cc, ss);
                }
            }
        }
        __syncthreads();
        // the chunk's units
        const long long u_end = t_end * groups < u1 ? t_end * groups : u1;
        long long cur_tile = -1;
        long long slot = -1;
        float cs[8], sn[8];
        long long tile = t0, grp = u - t0 * groups;  // advanced by counters, not divisions
        for (; u < u_end; ++u) {
            const long long layer0 = grp * kMatLayers;
            if (tile != cur_tile) {
                cur_tile = tile;
                const int ti = (int)(tile - t0);
                slot = slot_s[ti][row];
                if (slot >= 0) {
                    const int run = run_s[ti][row];
                    if (run < kMatRuns) {
#pragma unroll
                        for (int w = 0; w < kPairs; ++w) {
                            const float2 v = cs_s[ti][run][j0 + w];
                            cs[w] = v.x;
                            sn[w] = v.y;
                        }
                    } else {  // more distinct counts in this tile than the shared slots hold
#pragma unroll
                        for (int w = 0; w < kPairs; ++w) {
                            const float2 t = pair_trig(cnt_s[ti][row], turn, half, j0 + w, kBf16);
                            cs[w] = t.x;
                            sn[w] = t.y;
                        }
                    }
                }
            }
            uint4 v[kMatLayers];
            uint4* p[kMatLayers];
#pragma unroll
            for (int k = 0; k < kMatLayers; ++k) {
                v[k] = make_uint4(0u, 0u, 0u, 0u);
                p[k] = kv + band_off(g, layer0 + k, slot < 0 ? 0 : slot) + c;
                if (slot >= 0 && layer0 + k < L) v[k] = ld_rw(p[k]);
            }
#pragma unroll
            for (int k = 0; k < kMatLayers; ++k) {
                if (kLayout == 0) {
                    const uint4 o = shfl_xor_vec(v[k], hv / 2);  // every lane takes part
                    if (slot >= 0 && layer0 + k < L) st_stream(p[k], turn_own_half<kBf16>(v[k], o, y_half, cs, sn));
                } else if (slot >= 0 && layer0 + k < L) {
                    rotate_interleaved<kBf16>(v[k], cs, sn);
                    st_stream(p[k], v[k]);
                }
            }
            if (++grp == groups) {
                grp = 0;
                ++tile;
            }
        }
    }
}

__global__ void clear_pending_kernel(int32_t* pending, const int32_t* page_ids, long long n, int block_size)
{
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n * block_size;
         i += (long long)gridDim.x * blockDim.x)
        pending[(long long)page_ids[i / block_size] * block_size + i % block_size] = 0;
}

}  // namespace

// A plan too large for a kernel parameter, copied from its pinned host staging slot into
// the slot's device buffer by a kernel that reads host memory directly.  As a dependent
// launch it keeps the call in the chain of dependent launches, where a copy-engine
// transfer would break it: the copy would start only once the kernel before it had ended,
// and the next kernel could launch only once the copy had.  The copy may run beside the
// previous call's last kernel: the slot's buffer was last read by the call that used the
// slot 8 uploaded calls back, and that call has ended, since the copy kernel of the
// uploaded call after it waited for every earlier kernel before any later one launched.
// It then waits for the previous kernel before the next kernel may launch, so every
// kernel after it starts after all earlier calls have ended, as after a stream-ordered
// copy; the next kernel reads the plan only after its own wait.
__global__ void upload_plan_kernel(const uint4* src, uint4* dst, long long n)
{
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        dst[i] = src[i];
    wait_for_previous_grid();
    allow_next_grid();
}

int launch_upload_plan(const void* host_src, void* dev_dst, size_t bytes, void* stream)
{
    if (bytes == 0 || bytes % 16 != 0) return (int)cudaErrorInvalidValue;
    const long long n = (long long)(bytes / 16);
    return (int)launch_dependent(upload_plan_kernel, grid_for(n, 256, 64), 256, (cudaStream_t)stream,
                                 static_cast<const uint4*>(host_src), static_cast<uint4*>(dev_dst), n);
}

int launch_init_queue(int32_t* q, int64_t num_pages, void* stream)
{
    init_queue_kernel<<<grid_for(2 * num_pages, 256, 4096), 256, 0, (cudaStream_t)stream>>>(q, num_pages);
    return (int)cudaGetLastError();
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

int launch_gather_lazy(const void* kv, const int32_t* table_row, const Geometry& g, int32_t layer, int64_t t0,
                       int64_t t1, void* out, const int32_t* pending, const double* turn, int32_t* status,
                       void* stream)
{
    const long long n = t1 - t0;
    if (n <= 0) return 0;
    auto k = g.pair_layout == LEYLINE_PAIRS_HALF_SPLIT ? gather_lazy_kernel<0> : gather_lazy_kernel<1>;
    k<<<grid_for(n * 32, kReadThreads, 8192), kReadThreads, 0, (cudaStream_t)stream>>>(static_cast<const uint4*>(kv), table_row, g,
                                                                      layer, t0, n, static_cast<uint4*>(out),
                                                                      pending, turn, status);
    return (int)cudaGetLastError();
}

int launch_materialize(void* kv, const int32_t* table, int32_t max_blocks, const MaterializeSet& set,
                       const Geometry& g, int32_t* pending, const double* turn, int32_t* status,
                       const MaterializeScratch& scratch, void* stream)
{
    if (set.n <= 0 || set.row_end[set.n - 1] <= 0) return 0;
    const long long rows = set.row_end[set.n - 1];
    if (materialize_uses_list(g)) {  // the row's bands fill 8 vectors: the listed rows in tiles of 32
        const cudaStream_t s = (cudaStream_t)stream;
        const bool split = g.pair_layout == LEYLINE_PAIRS_HALF_SPLIT;
        const bool bf16 = g.precision == LEYLINE_ROTATE_BF16_NAIVE;
        auto k = split ? (bf16 ? materialize_band8_kernel<0, true> : materialize_band8_kernel<0, false>)
                       : (bf16 ? materialize_band8_kernel<1, true> : materialize_band8_kernel<1, false>);
        int dev = 0, sms = 0, per_sm = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kMatThreads, 0);
        if (e != cudaSuccess) return (int)e;
        compact_pending_kernel<<<grid_for(rows, kMatThreads, 4096), kMatThreads, 0, s>>>(
            table, max_blocks, set, g, pending, scratch.slot, scratch.pend, scratch.n, status);
        e = cudaGetLastError();
        if (e == cudaSuccess)
            e = launch_dependent(k, sms * std::max(per_sm, 1), kMatThreads, s, static_cast<uint4*>(kv), g,
                                 static_cast<const long long*>(scratch.slot), static_cast<const int32_t*>(scratch.pend),
                                 static_cast<const unsigned long long*>(scratch.n), scratch.n_next, pending, turn);
        return (int)e;
    }
    auto k = g.pair_layout == LEYLINE_PAIRS_HALF_SPLIT ? materialize_kernel<0> : materialize_kernel<1>;
    k<<<grid_for(rows * 32, kReadThreads, 8192), kReadThreads, 0, (cudaStream_t)stream>>>(
        static_cast<uint4*>(kv), table, max_blocks, set, g, pending, turn, status);
    return (int)cudaGetLastError();
}

int launch_clear_pending(int32_t* pending, const int32_t* page_ids, int64_t n, int32_t block_size, void* stream)
{
    if (n <= 0) return 0;
    clear_pending_kernel<<<grid_for(n * block_size, 256, 4096), 256, 0, (cudaStream_t)stream>>>(pending, page_ids, n,
                                                                                             block_size);
    return (int)cudaGetLastError();
}

}  // namespace leyline
