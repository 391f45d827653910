// leyline_internal.h -- declarations shared by the host planner, the pool / C ABI
// and the kernel launchers.  Not installed; the public surface is include/leyline.h.
#pragma once

#include <cuda_runtime.h>

#include <chrono>
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
    std::vector<float> trig;  // per ROT segment: rope_dim / 2 pairs of (cos, sin) of Delta * theta_j
    int32_t n_trig = 0;       // ROT segments
    bool reindex = false;     // the call re-indexes (block size 1, LEYLINE_POOL_REINDEX)
    int64_t total_prep = 0;   // re-index: prep items (staged entries + dropped tokens)
    int64_t total_stage = 0;  // re-index: staged table entries
    int64_t total_repl = 0;   // re-index: rows of R of the call
    int64_t total_fresh = 0;  // re-index: survivor and prefix rows written into fresh pages
    int64_t total_tiles = 0;  // move+rotate tiles over all requests
    int64_t total_commit = 0; // commit work items over all requests
    int64_t total_pop = 0;    // fresh pages
    int64_t total_push = 0;   // pages returned
    leyline_stats_t stats{};
};

// Validate the directives against the host length mirror and build the plan.
// free_pages < 0 skips the page check.  Returns LEYLINE_OK or an error code
// (the message is set); on error *plan is unspecified and nothing else changed.
int build_plan(const Geometry& g, const int64_t* seq_lens_host, int32_t num_reqs, int32_t max_blocks,
               const leyline_directive_t* dirs, int32_t n, int64_t free_pages, Plan* plan);

// A plan small enough to travel as a kernel parameter (__grid_constant__): no
// host-to-device copy and no plan buffer on the path.
constexpr int kParamReqs = 8;  // 128 bytes each
constexpr int kParamSegs = 24;
constexpr int kParamTrigFloats = 640;  // 10 rotated segments of a 64-wide rope band
struct alignas(16) ParamPlan {
    ReqPlan reqs[kParamReqs];
    Seg segs[kParamSegs];
    float trig[kParamTrigFloats];
};
bool plan_fits_params(const Plan& plan);
void pack_param_plan(const Plan& plan, ParamPlan* pp);

// Which move+rotate kernel runs: 16-byte vector loads/stores through registers, or
// bulk copies (TMA) staged through shared memory.
enum MoveKernel : int32_t { MOVE_VECTOR = 0, MOVE_BULK = 1 };

// Kernel arguments (passed by value).
struct SpliceArgs {
    void* kv;                 // pool base
    const int32_t* table;     // [num_reqs][max_blocks], read by the move+rotate kernel
    int32_t* table_w;         // same table, written by the commit kernel
    int32_t* seq_lens_dev;
    int32_t* free_q;          // free-page ring, q_cap entries
    int64_t q_cap;
    int64_t pop_base;         // ring position of the first page this call takes (mod q_cap)
    int64_t push_base;        // ring position of the first page this call returns (mod q_cap)
    const ReqPlan* reqs;      // plan in device memory (when it is not a kernel parameter)
    const Seg* segs;
    const float* trig;
    int32_t* stage;           // re-index: staged table entries [total_stage]
    int32_t* pending;         // lazy pools: pending turns [num_pages * block_size], else nullptr
    int32_t* status;          // device status word
    int64_t total_prep;
    int64_t total_repl;       // re-index: rows of R of the call
    int64_t total_fresh;      // re-index: survivor and prefix rows written into fresh pages
    int64_t total_tiles;
    int64_t total_commit;
    int32_t n_reqs;
    int32_t n_trig;
    int32_t max_blocks;
    int32_t move_kernel;      // MoveKernel
    int32_t reindex;          // 1: prep + in-place rotation + staged commit
    int32_t prep_ctas;        // re-index: CTAs of the prep part of the prep + rows-of-R launch
    int32_t overlap_prev;     // 1: the move kernel starts without waiting for the previous kernel
                              // and waits for it at its end (the host has ruled out hazards)
    int32_t pad3;
    Geometry g;
};

// Launchers (leyline_move.cu, leyline_reindex.cu, leyline_read.cu).  Each returns the
// cudaError_t of the launches as int.
int launch_init_queue(int32_t* q, int64_t num_pages, void* stream);
// Copy an uploaded plan (bytes a multiple of 16) from pinned host memory into device
// memory by a dependent launch on `stream`.
int launch_upload_plan(const void* host_src, void* dev_dst, size_t bytes, void* stream);
// Enqueue a re-indexed call's kernels (prep, rows of R, fresh rows, rotation, commit):
// leyline_reindex.cu.  launch_splice calls it for plans with reindex set.
int launch_reindex_call(const SpliceArgs& a, const ParamPlan* pp, int grid, void* stream, cudaEvent_t t0,
                        cudaEvent_t t1);
// Enqueue move+rotate then commit.  pp != nullptr: the plan travels in pp (a.reqs,
// a.segs, a.trig unused); else it is read from a.reqs / a.segs / a.trig.  With
// timing events, they bracket the move+rotate kernel.
int launch_splice(const SpliceArgs& a, const ParamPlan* pp, int grid, void* stream, cudaEvent_t t0,
                  cudaEvent_t t1);
int launch_gather(const void* kv, const int32_t* table_row, const Geometry& g, int32_t layer, int64_t t0,
                  int64_t t1, void* out, int32_t* status, void* stream);
// Lazy pools: gather turning each row's rope bands by its pending count; turn is the
// pool's device turn table (see kTurnSpan below).
int launch_gather_lazy(const void* kv, const int32_t* table_row, const Geometry& g, int32_t layer, int64_t t0,
                       int64_t t1, void* out, const int32_t* pending, const double* turn, int32_t* status,
                       void* stream);
// Lazy pools: the requests one materialize launch turns, and the cumulative ends of their
// rows in the launch's flat row list (request k holds rows [row_end[k - 1], row_end[k])).
constexpr int kMaterializeReqs = 64;
struct MaterializeSet {
    int32_t n;
    int32_t pad;
    int32_t req[kMaterializeReqs];
    int64_t row_end[kMaterializeReqs];
};
// Device lists of the rows a materialize launch turns (pool-owned, one entry per slot of
// the pool): slot and count of each listed row, and the number listed.  Launches use two
// counters in turn: n (0 when the launch starts) and n_next, which the launch's band pass
// sets to 0 for the next launch.
struct MaterializeScratch {
    long long* slot;
    int32_t* pend;
    unsigned long long* n;
    unsigned long long* n_next;
};
// Whether launch_materialize lists the rows first (and so needs MaterializeScratch of the
// set's row count): rows whose rope bands fill 8 vectors.
inline bool materialize_uses_list(const Geometry& g) { return g.rope_heads * g.head_vecs == 8; }
// Lazy pools: turn every row of the set's requests by its pending count, in place, and
// clear the counts; table is the block table [num_reqs][max_blocks].
int launch_materialize(void* kv, const int32_t* table, int32_t max_blocks, const MaterializeSet& set,
                       const Geometry& g, int32_t* pending, const double* turn, int32_t* status,
                       const MaterializeScratch& scratch, void* stream);
// Lazy pools: set the pending counts of n pages (device ids) to 0.
int launch_clear_pending(int32_t* pending, const int32_t* page_ids, int64_t n, int32_t block_size, void* stream);
// Device access to a caller buffer.  Memory of `device` and managed memory are
// used as they are; pinned host memory (cudaHostAlloc, cudaHostRegister) is used
// through its device alias, so kernels read or write it in place over the host
// link (NVLink-C2C on Grace hosts).  Pageable host memory and memory of another
// device are refused (LEYLINE_ERR_INVALID_ARG, message naming `what`).
int resolve_access(const void* ptr, int device, const char* what, void** alias, bool* is_host);

// Lazy pools' turn table (device, fp64), read by the kernels that apply pending
// counts: theta_j for the `half` pairs (padded to an even count), then
//   lo[j][m] = (cos, sin)(m * theta_j)              m < kTurnSpan
//   hi[j][m] = (cos, sin)(m * kTurnSpan * theta_j)  m < kTurnSpan
// so that a count p < kTurnSpan^2 turns by the product of hi[j][p / kTurnSpan] and
// lo[j][p % kTurnSpan] (angle addition) instead of a sincos.
constexpr int kTurnSpan = 2048;
inline size_t turn_table_doubles(int half) { return (size_t)(half + 1) / 2 * 2 + (size_t)4 * half * kTurnSpan; }

// Host time of a splice call, reported in leyline_stats_t.
using HostClock = std::chrono::steady_clock::time_point;
inline HostClock host_now() { return std::chrono::steady_clock::now(); }
inline void set_host_times(leyline_stats_t* st, HostClock enter, HostClock resolved, HostClock planned)
{
    using std::chrono::duration_cast;
    using std::chrono::nanoseconds;
    st->host_ns = duration_cast<nanoseconds>(host_now() - enter).count();
    st->resolve_ns = duration_cast<nanoseconds>(resolved - enter).count();
    st->plan_ns = duration_cast<nanoseconds>(planned - resolved).count();
}
// resolve_access for every directive's rows of R.  *out points at the directives
// to plan from: `dirs` itself, or a copy in *work with aliases substituted.
// *host_rows is set when any rows of R live in host memory.
int resolve_repl_rows(const leyline_directive_t* dirs, int32_t n, int device, std::vector<leyline_directive_t>* work,
                      const leyline_directive_t** out, bool* host_rows);
// Resident CTAs per SM of the vector move+rotate kernel (occupancy query).
int move_rotate_blocks_per_sm(int* blocks);
// Resident CTAs per SM of the in-place rotation kernel of re-index mode.
int rotate_in_place_blocks_per_sm(int* blocks);
// Allow the bulk kernel its shared memory for rows of row_bytes and report its
// resident CTAs per SM (0 if the rows are too wide for it).
int bulk_prepare(int32_t row_bytes, int* blocks);

}  // namespace leyline
