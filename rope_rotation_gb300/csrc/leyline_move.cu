// leyline_move.cu -- rewrite splices on GB300 (sm_103a): the move+rotate kernels and the
// commit kernel.
//
// "Leyline: KV Cache Directives for Agentic Inference", section 2.3: the rotation kernel
// re-indexes and rotates every downstream slot.
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
// before it touches the table.  Calls enqueued back to back may overlap as well: when
// the host has shown that a call shares no request with the calls still running and
// takes no page they returned, its move kernel starts before they end (SpliceArgs::
// overlap_prev).  The path is bandwidth-bound (about 64 fp32 FMAs per 2304 bytes
// moved), so it uses no tensor cores.
#include "leyline_device.cuh"

namespace leyline {
namespace {

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
    constexpr int kWarps = kMoveThreads / 32;
    __shared__ RowDesc desc[kTileRows];
    // An overlapped call (a.overlap_prev) reads nothing the calls still running write, so it
    // starts at once and waits for the previous kernel only at its end, which keeps the
    // completion of calls in stream order.
    if (!a.overlap_prev) wait_for_previous_grid();
    allow_next_grid();
    const PlanView pv = plan_view(a, plan);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long L = a.g.num_layers;
    const long long lat_layer = a.g.lat_layer_vecs, rope_layer = a.g.rope_layer_vecs;
    const int half = 4 * kRopeVecs;  // pairs per row
    // 8 lanes per row's band, one 16-byte chunk each: a warp's loads cover whole lines
    // (half-split: the partner half comes from lane ^ 4)
    constexpr int kRopeLanesPerRow = kRopeVecs;
    const bool rope_lane = lane < kRowsPerWarp * kRopeLanesPerRow;
    const int rope_row = warp * kRowsPerWarp + lane / kRopeLanesPerRow;
    const int rope_c = lane % kRopeLanesPerRow;                 // this lane's chunk
    const int rope_q = kLayout == 0 ? rope_c % (kRopeVecs / 2) : rope_c;  // its pair group
    float cs[8], sn[8];
    int trig = -1;

    // The split is by warp unit (one warp's two rows of a tile in one layer): CTA runs
    // then differ by one warp unit, not by a whole (tile, layer) unit, so the CTAs that
    // finish last hold 1/8 of a unit more work than the rest.  A warp outside this
    // CTA's run skips the unit's loads and stores but still joins its barriers.
    // The run is walked with 32-bit counters: k counts its units, and (tile, layer)
    // advance by one layer per unit.  Units [k_first, k_last) are this warp's.
    int n, k_first, k_last, layer;
    long long tile;
    {
        long long w0, w1;
        my_units(a.total_tiles * L * kWarps, w0, w1);
        const long long u0 = w0 / kWarps, u1 = (w1 + kWarps - 1) / kWarps;
        n = (int)(u1 - u0);
        k_first = warp >= (int)(w0 - u0 * kWarps) ? 0 : 1;
        k_last = warp < (int)(w1 - (u1 - 1) * kWarps) ? n : n - 1;
        tile = u0 / L;
        layer = (int)(u0 - tile * L);
    }
    long long cur_tile = -1;
    for (int k = 0; k < n; ++k, ++layer) {
        if (layer == L) {
            layer = 0;
            ++tile;
        }
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
        const bool mine = k >= k_first && k < k_last;
        const RowDesc d0 = desc[warp * kRowsPerWarp];
        const RowDesc d1 = desc[warp * kRowsPerWarp + 1];
        const bool has0 = mine && d0.src != nullptr, has1 = mine && d1.src != nullptr;
        uint4 v[4];
        if (has0) {
            const uint4* s0 = d0.src + layer * d0.src_lstride;
            v[0] = ld_stream(s0 + lane);
            v[1] = ld_stream(s0 + lane + 32);
        }
        if (has1) {
            const uint4* s1 = d1.src + layer * d1.src_lstride;
            v[2] = ld_stream(s1 + lane);
            v[3] = ld_stream(s1 + lane + 32);
        }
        const RowDesc dr = rope_lane ? desc[rope_row] : d0;
        const bool do_rope = mine && rope_lane && dr.src != nullptr;
        uint4 rx = make_uint4(0u, 0u, 0u, 0u);
        if (do_rope) {
            const uint4* rs = dr.src_band + layer * dr.band_lstride;
            rx = ld_stream(rs + rope_c);
        }
        const uint4 rp = kLayout == 0 ? shfl_xor_vec(rx, kRopeVecs / 2) : rx;  // every lane takes part
        if (has0) {
            uint4* t0 = d0.dst + layer * lat_layer;
            st_stream(t0 + lane, v[0]);
            st_stream(t0 + lane + 32, v[1]);
        }
        if (has1) {
            uint4* t1 = d1.dst + layer * lat_layer;
            st_stream(t1 + lane, v[2]);
            st_stream(t1 + lane + 32, v[3]);
        }
        if (do_rope) {
            uint4* rd = dr.dst_band + layer * rope_layer;
            if (kLayout == 0) {
                const bool hi = rope_c >= kRopeVecs / 2;  // this lane holds the y half
                uint4 x = hi ? rp : rx, y = hi ? rx : rp;
                if (trig >= 0) rotate_half_split<kBf16>(x, y, cs, sn);
                st_stream(rd + rope_c, hi ? y : x);
            } else {
                if (trig >= 0) rotate_interleaved<kBf16>(rx, cs, sn);
                st_stream(rd + rope_c, rx);
            }
        }
    }
    if (a.overlap_prev) wait_for_previous_grid();
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

template <class PlanSrc>
__global__ void __launch_bounds__(kCommitThreads) commit_kernel(const __grid_constant__ SpliceArgs a,
                                                                const __grid_constant__ PlanSrc plan)
{
    // The next call's first kernel may launch at once: it waits for this grid before it
    // reads anything, unless the host has let it overlap (it then reads nothing this
    // grid writes).
    allow_next_grid();
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
int launch_both(const SpliceArgs& a, const PlanSrc& plan, int grid, cudaStream_t s, cudaEvent_t t0, cudaEvent_t t1)
{
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

int launch_splice(const SpliceArgs& a, const ParamPlan* pp, int grid, void* stream, cudaEvent_t t0, cudaEvent_t t1)
{
    if (a.reindex) return launch_reindex_call(a, pp, grid, stream, t0, t1);
    cudaStream_t s = (cudaStream_t)stream;
    if (pp) return launch_both(a, *pp, grid, s, t0, t1);
    return launch_both(a, NoParamPlan{0}, grid, s, t0, t1);
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
