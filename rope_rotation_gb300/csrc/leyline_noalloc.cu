// leyline_noalloc.cu -- leyline_splice_noalloc: the splice without any device or
// pinned-memory allocation.
//
// Who needs it.  leyline_splice keeps its per-call plan in a buffer that the pool
// grows with cudaMalloc / cudaHostAlloc when a call needs more room than any
// earlier one.  Some callers must never trigger that: a serving process whose
// framework has already reserved nearly all device memory in its own caching
// allocator (a cudaMalloc behind its back can fail or fragment the pool it
// manages), or a process that forbids device allocations after start-up so
// that its memory footprint stays fixed.  This entry point runs the same
// kernels, but its scratch lives in a file-scope static device array of fixed
// size, and the plan is staged through a static host array.
//
// The scratch.  g_splice_scratch holds kNoallocScratchBytes (4 MiB) on every GPU
// on which this library's device code is loaded, from then until the process
// exits.  Its device address is looked up once per device with
// cudaGetSymbolAddress on the first call made on that device (with the device
// current).  Every call shares
// the array: calls that overlap on the GPU (on different streams, or from
// different pools, without ordering between them) race on it.  Calls on one pool
// are ordered by the pool, as for leyline_splice.  Each call writes every byte
// its kernels read (the uploaded plan; in re-index mode also the staged table
// entries, written by the prep kernel before anything reads them), so nothing has
// to start at zero and what the previous call left behind is never read.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "leyline_internal.h"
#include "leyline_pool_state.h"

using namespace leyline;

namespace {

constexpr size_t kNoallocScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_splice_scratch[kNoallocScratchBytes];

// Host staging of the uploaded part of the plan (pageable, static).
alignas(256) static unsigned char g_host_plan[kNoallocScratchBytes];

std::mutex g_mutex;                     // guards g_host_plan and g_scratch_addr
void* g_scratch_addr[kMaxDevices] = {};  // device address of g_splice_scratch, per device

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int cuda_fail(cudaError_t e, const char* what)
{
    char msg[256];
    snprintf(msg, sizeof msg, "%s: %s", what, cudaGetErrorString(e));
    return set_error(LEYLINE_ERR_CUDA, msg);
}

// Device address of the static scratch on `device` (which must be current).
int scratch_address(int device, void** out)
{
    if (device < 0 || device >= kMaxDevices) return set_error(LEYLINE_ERR_INVALID_ARG, "device ordinal too large");
    if (!g_scratch_addr[device]) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_splice_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "looking up the static splice scratch");
        g_scratch_addr[device] = ptr;
    }
    *out = g_scratch_addr[device];
    return LEYLINE_OK;
}

}  // namespace

extern "C" int leyline_splice_noalloc(leyline_pool_t* p, leyline_block_table_t* bt, const leyline_directive_t* dirs,
                                      int32_t n, void* stream_v)
{
    NvtxRange range("leyline_splice_noalloc");
    clear_error();
    const HostClock t_enter = host_now();
    if (!p) return set_error(LEYLINE_ERR_INVALID_ARG, "null pool");
    if (!bt || !bt->table || !bt->seq_lens_dev || !bt->seq_lens_host || bt->num_reqs < 0 || bt->max_blocks < 0)
        return set_error(LEYLINE_ERR_INVALID_ARG, "incomplete block table");
    for (int32_t r = 0; r < bt->num_reqs; ++r)
        if (bt->seq_lens_host[r] < 0 || bt->seq_lens_host[r] > (int64_t)bt->max_blocks * p->g.block_size)
            return set_error(LEYLINE_ERR_INVALID_ARG, "seq_lens_host entry outside [0, max_blocks * block_size]");
    std::vector<leyline_directive_t> resolved;  // filled only when a host alias differs from its pointer
    const leyline_directive_t* use = dirs;
    bool host_rows = false;
    int rc = resolve_repl_rows(dirs, n, p->device, &resolved, &use, &host_rows);
    if (rc != LEYLINE_OK) return rc;
    const HostClock t_resolved = host_now();
    Plan plan;
    const int64_t free_now = p->q_tail - p->q_head;
    rc = build_plan(p->g, bt->seq_lens_host, bt->num_reqs, bt->max_blocks, use, n, free_now, &plan);
    if (rc != LEYLINE_OK) return rc;
    const HostClock t_planned = host_now();
    if (plan.reqs.empty()) {
        p->last_stats = plan.stats;
        set_host_times(&p->last_stats, t_enter, t_resolved, t_planned);
        return LEYLINE_OK;
    }
    if (free_now - plan.total_pop + plan.total_push > p->g.num_pages)
        return set_error(LEYLINE_ERR_INVALID_ARG,
                         "the rewritten requests hold more pages than the pool has free slots for: "
                         "their tables were not filled from this pool");

    // scratch layout: reqs | segs | trig (cos, sin per pair of every rotated segment)
    //                 | staged table entries (re-index mode)
    const size_t off_segs = align_up(sizeof(ReqPlan) * plan.reqs.size(), 16);
    const size_t off_trig = align_up(off_segs + sizeof(Seg) * plan.segs.size(), 16);
    const size_t upload = off_trig + sizeof(float) * plan.trig.size();
    const size_t off_stage = align_up(upload, 16);
    const size_t total = off_stage + sizeof(int32_t) * (size_t)plan.total_stage;
    if (total > kNoallocScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "this splice needs %zu bytes of scratch; the static scratch of leyline_splice_noalloc holds %zu "
                 "(split the directives over several calls, or use leyline_splice)",
                 total, kNoallocScratchBytes);
        return set_error(LEYLINE_ERR_SCRATCH, msg);
    }

    std::lock_guard<std::mutex> lock(g_mutex);
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(p->device) != cudaSuccess)
        return set_error(LEYLINE_ERR_CUDA, "cannot select the pool's device");
    struct Restore {
        int dev;
        ~Restore()
        {
            if (dev >= 0) cudaSetDevice(dev);
        }
    } restore{prev};

    void* scratch_v = nullptr;
    rc = scratch_address(p->device, &scratch_v);
    if (rc != LEYLINE_OK) return rc;
    char* scratch = static_cast<char*>(scratch_v);
    cudaStream_t stream = (cudaStream_t)stream_v;
    cudaError_t e;
    if (p->has_work && p->last_stream != stream) {
        e = cudaStreamWaitEvent(stream, p->done, 0);
        if (e != cudaSuccess) return cuda_fail(e, "ordering after the previous splice");
    }
    memcpy(g_host_plan, plan.reqs.data(), sizeof(ReqPlan) * plan.reqs.size());
    memcpy(g_host_plan + off_segs, plan.segs.data(), sizeof(Seg) * plan.segs.size());
    if (!plan.trig.empty()) memcpy(g_host_plan + off_trig, plan.trig.data(), sizeof(float) * plan.trig.size());
    // From pageable memory: the copy is staged before the call returns, so the
    // static host buffer may be reused by the next call.
    e = cudaMemcpyAsync(scratch, g_host_plan, upload, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "uploading the plan");

    SpliceArgs a{};
    a.kv = p->kv;
    a.table = bt->table;
    a.table_w = bt->table;
    a.seq_lens_dev = bt->seq_lens_dev;
    a.free_q = p->d_queue;
    a.q_cap = p->q_cap;
    a.pop_base = p->q_head;
    a.push_base = p->q_tail;
    a.reqs = reinterpret_cast<const ReqPlan*>(scratch);
    a.segs = reinterpret_cast<const Seg*>(scratch + off_segs);
    a.trig = reinterpret_cast<const float*>(scratch + off_trig);
    if (plan.reindex) {
        a.stage = reinterpret_cast<int32_t*>(scratch + off_stage);
        a.total_prep = plan.total_prep;
        a.total_repl = plan.total_repl;
        a.total_fresh = plan.total_fresh;
        a.reindex = 1;
    }
    a.status = p->d_status;
    a.total_tiles = plan.total_tiles;
    a.total_commit = plan.total_commit;
    a.n_reqs = (int32_t)plan.reqs.size();
    a.n_trig = plan.n_trig;
    a.max_blocks = bt->max_blocks;
    a.pending = p->d_pending;
    a.g = p->g;

    a.move_kernel = host_rows ? MOVE_VECTOR : p->move_kernel;  // rows of R in host memory: plain loads
    const int grid = p->sm_count * (plan.reindex                    ? p->reindex_blocks_per_sm
                                    : a.move_kernel == MOVE_BULK ? p->bulk_blocks_per_sm
                                                                 : p->move_blocks_per_sm);
    // kernel timing uses the events leyline_kernel_timing_enable created up front; a call
    // past those goes untimed rather than create more
    cudaEvent_t t0 = nullptr, t1 = nullptr;
    if (p->timing && p->tev_used < p->tev.size()) {
        t0 = p->tev[p->tev_used].first;
        t1 = p->tev[p->tev_used].second;
        ++p->tev_used;
    }
    int err = launch_splice(a, nullptr, grid, stream, t0, t1);
    if (err != 0) return cuda_fail((cudaError_t)err, "launching the splice kernels");
    e = cudaEventRecord(p->done, stream);
    if (e != cudaSuccess) return cuda_fail(e, "recording completion event");
    p->has_work = true;
    p->last_stream = stream;
    p->window_open = false;  // this entry point does not overlap; the next splice waits for it
    if (plan.reindex && !p->d_pending) p->ckpt_turned = true;  // bands turned in place

    for (const ReqPlan& rp : plan.reqs) bt->seq_lens_host[rp.req] = rp.new_len;
    p->q_head += plan.total_pop;
    p->q_tail += plan.total_push;
    p->last_stats = plan.stats;
    set_host_times(&p->last_stats, t_enter, t_resolved, t_planned);
    return LEYLINE_OK;
}
