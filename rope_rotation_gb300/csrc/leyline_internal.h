// leyline_internal.h -- declarations shared by the host planner, the pool / C ABI
// and the kernel launchers.  Not installed; the public surface is include/leyline.h.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <string>
#include <utility>
#include <vector>

#include "leyline.h"
#include "leyline_plan.h"

namespace leyline {

// Thread-local message for leyline_last_error().
int set_error(int code, const std::string& msg);
void clear_error();

// Validate a pool descriptor and derive the geometry.  Returns LEYLINE_OK or INVALID_ARG.
int make_geometry(const leyline_pool_desc_t* desc, Geometry* g);

// Output of the host planner for one splice call.
struct Plan {
    std::vector<ReqPlan> reqs;
    std::vector<Seg> segs;
    std::vector<int64_t> trig_delta;  // accumulated Delta of every ROT segment
    int64_t total_tiles = 0;          // move+rotate tiles over all requests
    int64_t total_commit = 0;         // commit work items over all requests
    int64_t total_pop = 0;            // fresh pages
    int64_t total_push = 0;           // pages returned
    leyline_stats_t stats{};
};

// Validate the directives against the host length mirror and build the plan.
// free_pages < 0 skips the page check.  Returns LEYLINE_OK or an error code
// (the message is set); on error *plan is unspecified and nothing else changed.
int build_plan(const Geometry& g, const int64_t* seq_lens_host, int32_t num_reqs, int32_t max_blocks,
               const leyline_directive_t* dirs, int32_t n, int64_t free_pages, Plan* plan);

// Kernel arguments (passed by value).
struct SpliceArgs {
    void* kv;                      // pool base
    const int32_t* table;          // [num_reqs][max_blocks], read by the move+rotate kernel
    int32_t* table_w;              // same table, written by the commit kernel
    int32_t* seq_lens_dev;
    int32_t* free_stack;           // [num_pages]
    const ReqPlan* reqs;
    const Seg* segs;
    const int64_t* trig_delta;
    float* trig;                   // [n_trig][rope_dim / 2][2] (cos, sin)
    int32_t* staged;               // [total_pop] fresh page ids in pop order
    int32_t* status;               // device status word
    int64_t pop_top;               // free-stack top before the call
    int64_t push_base;             // pop_top - total_pop
    int64_t total_tiles;
    int64_t total_commit;
    int64_t total_pop;
    int32_t n_reqs;
    int32_t n_trig;
    int32_t max_blocks;
    int32_t pad;
    Geometry g;
};

// Launchers (leyline_kernels.cu).  Each returns the cudaError_t of the launch as int.
int launch_init_stack(int32_t* stack, int64_t num_pages, void* stream);
int launch_plan_kernel(const SpliceArgs& a, void* stream);
int launch_move_rotate(const SpliceArgs& a, int grid, void* stream);
int launch_commit(const SpliceArgs& a, void* stream);
int launch_gather(const void* kv, const int32_t* table_row, const Geometry& g, int32_t layer, int64_t t0,
                  int64_t t1, void* out, int32_t* status, void* stream);
// Resident CTAs per SM of the move+rotate kernel (occupancy query).
int move_rotate_blocks_per_sm(int* blocks);

}  // namespace leyline

// State of one pool (opaque to callers as leyline_pool_t).
struct leyline_pool {
    leyline_pool_desc_t desc{};
    leyline::Geometry g{};
    void* kv = nullptr;
    int device = 0;
    int sm_count = 0;
    int move_blocks_per_sm = 1;
    int32_t* d_stack = nullptr;
    int64_t free_top = 0;
    int32_t* d_status = nullptr;
    char* d_plan = nullptr;
    size_t d_plan_cap = 0;
    char* h_plan = nullptr;  // pinned
    size_t h_plan_cap = 0;
    cudaEvent_t plan_uploaded = nullptr;  // staging buffer reusable once this completes
    cudaEvent_t done = nullptr;           // last enqueued work of the pool
    bool has_work = false;
    cudaStream_t last_stream = nullptr;
    leyline_stats_t last_stats{};
    bool timing = false;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> tev;
    size_t tev_used = 0;
};
