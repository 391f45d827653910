// leyline_pool_state.h -- host-side state of a pool (the opaque leyline_pool_t).
// Shared by the C ABI translation units (leyline_pool.cpp, leyline_noalloc.cu);
// no kernel reads it.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <utility>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "leyline_internal.h"

namespace leyline {
// A named NVTX range for the host side of an entry point (shown by profilers that record
// NVTX, such as ncu --nvtx; close to free when no tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace leyline

// State of one pool (opaque to callers as leyline_pool_t).
struct leyline_pool {
    leyline_pool_desc_t desc{};
    leyline::Geometry g{};
    void* kv = nullptr;
    int device = 0;
    int sm_count = 0;
    int move_blocks_per_sm = 1;
    int bulk_blocks_per_sm = 0;
    int reindex_blocks_per_sm = 1;
    int32_t move_kernel = 0;  // MoveKernel used by this pool
    int32_t* d_stage = nullptr;  // re-index: staged table entries
    int32_t* d_pending = nullptr;  // lazy: pending turns per slot
    double* d_theta_j = nullptr;   // lazy: the readers' turn table (layout at kTurnSpan)
    size_t d_stage_cap = 0;      // entries
    int32_t* d_queue = nullptr;  // free-page ring, 2 * num_pages entries
    int64_t q_cap = 0;
    int64_t q_head = 0;          // monotonic: next page to take is d_queue[q_head % q_cap]
    int64_t q_tail = 0;          // monotonic: next free slot is d_queue[q_tail % q_cap]
    int32_t* d_status = nullptr;
    // uploaded plans: a ring of slots, each a pinned host staging buffer and a device
    // buffer, so the host can plan several calls ahead of the GPU and a call's upload may
    // run beside the previous call's last kernel.  The host rewrites a slot's staging
    // buffer once the slot's last upload event has completed.  The device buffer is
    // rewritten by the slot's next copy kernel, which may start before the previous call
    // has ended, but not before the call that last read the buffer has: that call is 8
    // uploaded calls back, and the copy kernel of the uploaded call after it waited for
    // every earlier kernel before any later kernel could launch.
    static constexpr int kPlanSlots = 8;
    char* d_plan[kPlanSlots] = {};
    size_t d_plan_cap[kPlanSlots] = {};
    char* h_plan[kPlanSlots] = {};
    size_t h_plan_cap[kPlanSlots] = {};
    cudaEvent_t plan_uploaded[kPlanSlots] = {};
    bool slot_used[kPlanSlots] = {};
    int next_slot = 0;
    cudaEvent_t done = nullptr;           // last enqueued work of the pool
    bool has_work = false;
    cudaStream_t last_stream = nullptr;
    leyline_stats_t last_stats{};
    bool timing = false;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> tev;
    size_t tev_used = 0;
    // Rewrite splices enqueued back to back on one stream may overlap: a call's move kernel
    // may start while the calls before it still run.  The window holds the calls that may
    // still run: those since the last call whose move kernel waited at its start.
    static constexpr int kOverlapWindow = 8;
    bool window_open = false;          // the last work on last_stream was a rewrite splice's commit
    int window_calls = 0;
    int64_t window_tail = 0;           // ring tail when the window's first call was planned
    std::vector<int32_t> window_reqs;  // requests the window's calls rewrite
    // lazy pools: the lists of rows a materialize launch turns (one entry per slot of the pool)
    long long* d_mat_slot = nullptr;
    int32_t* d_mat_pend = nullptr;
    unsigned long long* d_mat_n = nullptr;  // two counters, used by launches in turn
    int mat_turn = 0;                        // the counter the next launch uses
    // Checkpoint of the page accounting (leyline_pool_checkpoint / leyline_pool_rollback):
    // copies of the ring and, in lazy pools, of the pending counts, with the ring positions.
    int32_t* d_ckpt_queue = nullptr;
    int32_t* d_ckpt_pending = nullptr;
    bool has_ckpt = false;
    int64_t ckpt_head = 0;
    int64_t ckpt_tail = 0;
    bool ckpt_turned = false;  // stored bands were turned in place since the checkpoint
};
