// leyline_pool.cpp -- pool, free-page list, splice / gather entry points (C ABI).
//
// The pool borrows the caller's KV memory and block tables.  It owns the
// free-page list (a device ring of 2 * num_pages page ids; head and tail are
// counted on the host), device plan and staging buffers, a pinned host buffer
// for plans too large to travel as a kernel parameter, a status word and a few
// events.  A splice call:
//   1. validates and plans on the host (leyline_planner.cpp) -- on error nothing
//      is enqueued and nothing changes;
//   2. passes the plan to the kernels as a __grid_constant__ parameter when it
//      is small, else uploads it with one async host-to-device copy;
//   3. enqueues the move+rotate and commit kernels (re-index mode: prep, rotate,
//      commit) on the caller's stream, each a programmatic dependent of the last;
//   4. updates the host mirrors (lengths, free-page count) at enqueue time.
// In the default mode source pages are only read and fresh pages only written,
// so a splice whose spans shift downstream rows left (Delta < 0) or right
// (Delta > 0) has no read/write overlap; the old pages are recycled by the
// commit kernel.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "leyline_internal.h"
#include "leyline_pool_state.h"

namespace leyline {
const char* last_error_cstr();
}

using namespace leyline;

namespace {

constexpr size_t kPlanSlotBytes = 64 << 10;  // pinned plan staging per slot (grown on demand)

// Timing event pairs created when kernel timing is switched on (more are made on demand).
constexpr size_t kTimingEventsUpFront = 256;

struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) == cudaSuccess && cudaSetDevice(dev) == cudaSuccess) ok = true;
    }
    ~DeviceGuard()
    {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

int cuda_error(cudaError_t e, const char* what)
{
    char msg[256];
    snprintf(msg, sizeof msg, "%s: %s", what, cudaGetErrorString(e));
    return set_error(LEYLINE_ERR_CUDA, msg);
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int wait_pool(leyline_pool_t* p)
{
    if (p->has_work) {
        cudaError_t e = cudaEventSynchronize(p->done);
        if (e != cudaSuccess) return cuda_error(e, "waiting for the pool's work");
    }
    return LEYLINE_OK;
}

// Entry points whose work depends on host-side state at enqueue time (a plan made for the
// cache as it stands, ring positions, lengths) refuse a stream under graph capture: a replay
// would apply that state to a cache that has moved on.
int refuse_capture(cudaStream_t stream, const char* what)
{
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &st);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();  // not left for a later launch check to find
        if (e == cudaErrorStreamCaptureImplicit)  // the legacy stream while another stream captures
            return set_error(LEYLINE_ERR_INVALID_ARG, "the legacy default stream cannot be used while another "
                                                      "stream is being captured");
        return cuda_error(e, "querying the stream's capture status");
    }
    if (st != cudaStreamCaptureStatusNone) {
        char msg[160];
        snprintf(msg, sizeof msg, "%s cannot be captured in a CUDA graph: it is planned on the host for the cache as "
                 "it stands", what);
        return set_error(LEYLINE_ERR_INVALID_ARG, msg);
    }
    return LEYLINE_OK;
}

// Make `stream` wait for the pool's previous work when it came from another stream.
int order_after_previous(leyline_pool_t* p, cudaStream_t stream)
{
    if (p->has_work && p->last_stream != stream) {
        cudaError_t e = cudaStreamWaitEvent(stream, p->done, 0);
        if (e != cudaSuccess) return cuda_error(e, "ordering after the previous splice");
    }
    return LEYLINE_OK;
}

int mark_done(leyline_pool_t* p, cudaStream_t stream)
{
    cudaError_t e = cudaEventRecord(p->done, stream);
    if (e != cudaSuccess) return cuda_error(e, "recording completion event");
    p->has_work = true;
    p->last_stream = stream;
    return LEYLINE_OK;
}

}  // namespace

namespace leyline {

int resolve_access(const void* ptr, int device, const char* what, void** alias, bool* is_host)
{
    char msg[256];
    *alias = const_cast<void*>(ptr);
    *is_host = false;
    DeviceGuard guard(device);
    cudaPointerAttributes at{};
    cudaError_t e = cudaPointerGetAttributes(&at, ptr);
    if (e != cudaSuccess) {
        cudaGetLastError();
        snprintf(msg, sizeof msg, "%s: not a CUDA-visible pointer (%s)", what, cudaGetErrorString(e));
        return set_error(LEYLINE_ERR_INVALID_ARG, msg);
    }
    switch (at.type) {
    case cudaMemoryTypeDevice:
        if (at.device != device) {
            snprintf(msg, sizeof msg, "%s: memory of device %d, the pool is on device %d", what, at.device, device);
            return set_error(LEYLINE_ERR_INVALID_ARG, msg);
        }
        return LEYLINE_OK;
    case cudaMemoryTypeManaged:
        return LEYLINE_OK;
    case cudaMemoryTypeHost:
        if (!at.devicePointer) {
            snprintf(msg, sizeof msg, "%s: pinned host memory without a device mapping", what);
            return set_error(LEYLINE_ERR_INVALID_ARG, msg);
        }
        *alias = at.devicePointer;
        *is_host = true;
        return LEYLINE_OK;
    default:
        snprintf(msg, sizeof msg, "%s: pageable host memory; use device memory or pinned host memory", what);
        return set_error(LEYLINE_ERR_INVALID_ARG, msg);
    }
}

int resolve_repl_rows(const leyline_directive_t* dirs, int32_t n, int device, std::vector<leyline_directive_t>* work,
                      const leyline_directive_t** out, bool* host_rows)
{
    *out = dirs;
    *host_rows = false;
    for (int32_t k = 0; k < n; ++k) {
        if (dirs[k].n_repl <= 0 || !dirs[k].repl_rows) continue;  // the planner reports a missing pointer
        char what[64];
        snprintf(what, sizeof what, "directive %d: repl_rows", k);
        void* alias;
        bool host;
        int rc = resolve_access(dirs[k].repl_rows, device, what, &alias, &host);
        if (rc != LEYLINE_OK) return rc;
        *host_rows = *host_rows || host;
        if (alias != dirs[k].repl_rows) {
            if (work->empty()) work->assign(dirs, dirs + n);
            (*work)[k].repl_rows = alias;
            *out = work->data();
        }
    }
    return LEYLINE_OK;
}

}  // namespace leyline

extern "C" {

const char* leyline_last_error(void) { return last_error_cstr(); }

const char* leyline_version(void) { return "leyline-gb300 0.1.0 sm_103a"; }

int leyline_pool_create(const leyline_pool_desc_t* desc, void* kv_dev, leyline_pool_t** out)
{
    clear_error();
    if (!out) return set_error(LEYLINE_ERR_INVALID_ARG, "null output pointer");
    *out = nullptr;
    Geometry g;
    int rc = make_geometry(desc, &g);
    if (rc != LEYLINE_OK) return rc;
    if (!kv_dev || (reinterpret_cast<uintptr_t>(kv_dev) & 15) != 0)
        return set_error(LEYLINE_ERR_INVALID_ARG, "kv_dev must be a non-null 16-byte aligned device pointer");
    leyline_pool_t* p = new (std::nothrow) leyline_pool();
    if (!p) return set_error(LEYLINE_ERR_INVALID_ARG, "out of host memory");
    p->desc = *desc;
    p->g = g;
    p->kv = kv_dev;
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, p->device);
    if (e == cudaSuccess) e = (cudaError_t)move_rotate_blocks_per_sm(&p->move_blocks_per_sm);
    p->q_cap = 2 * g.num_pages;
    if (e == cudaSuccess) e = cudaMalloc(&p->d_queue, sizeof(int32_t) * (size_t)p->q_cap);
    if (e == cudaSuccess) e = cudaMalloc(&p->d_status, sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMemset(p->d_status, 0, sizeof(int32_t));
    // the plan slots are allocated now: cudaHostAlloc during a call would wait for the GPU
    for (int i = 0; i < leyline_pool::kPlanSlots && e == cudaSuccess; ++i) {
        e = cudaEventCreateWithFlags(&p->plan_uploaded[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaHostAlloc((void**)&p->h_plan[i], kPlanSlotBytes, cudaHostAllocDefault);
        if (e == cudaSuccess) p->h_plan_cap[i] = kPlanSlotBytes;
        if (e == cudaSuccess) e = cudaMalloc(&p->d_plan[i], kPlanSlotBytes);
        if (e == cudaSuccess) p->d_plan_cap[i] = kPlanSlotBytes;
    }
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->done, cudaEventDisableTiming);
    if (e == cudaSuccess && (g.flags & LEYLINE_POOL_LAZY)) {
        // every slot starts with nothing pending; readers take theta_j from a device table
        const size_t slots = (size_t)g.num_pages * (size_t)g.block_size;
        e = cudaMalloc(&p->d_pending, sizeof(int32_t) * slots);
        if (e == cudaSuccess) e = cudaMemset(p->d_pending, 0, sizeof(int32_t) * slots);
        // the readers' turn table: theta_j, then cos / sin of m theta_j and m kTurnSpan theta_j
        const int half = g.rope_dim / 2;
        std::vector<double> tt(turn_table_doubles(half), 0.0);
        double* lo = tt.data() + (half + 1) / 2 * 2;
        double* hi = lo + (size_t)2 * half * kTurnSpan;
        for (int j = 0; j < half; ++j) {
            const double th = std::pow(g.theta, -2.0 * j / g.rope_dim);
            tt[j] = th;
            for (int m = 0; m < kTurnSpan; ++m) {
                const double a = (double)m * th, b = (double)((int64_t)m * kTurnSpan) * th;
                lo[2 * ((size_t)j * kTurnSpan + m)] = std::cos(a);
                lo[2 * ((size_t)j * kTurnSpan + m) + 1] = std::sin(a);
                hi[2 * ((size_t)j * kTurnSpan + m)] = std::cos(b);
                hi[2 * ((size_t)j * kTurnSpan + m) + 1] = std::sin(b);
            }
        }
        if (e == cudaSuccess) e = cudaMalloc(&p->d_theta_j, sizeof(double) * tt.size());
        if (e == cudaSuccess)
            e = cudaMemcpy(p->d_theta_j, tt.data(), sizeof(double) * tt.size(), cudaMemcpyHostToDevice);
        // materialize's row lists: a launch lists rows of live requests, at most one per slot
        if (e == cudaSuccess && materialize_uses_list(g)) {
            e = cudaMalloc(&p->d_mat_slot, sizeof(long long) * slots);
            if (e == cudaSuccess) e = cudaMalloc(&p->d_mat_pend, sizeof(int32_t) * slots);
            if (e == cudaSuccess) e = cudaMalloc(&p->d_mat_n, 2 * sizeof(unsigned long long));
            if (e == cudaSuccess) e = cudaMemset(p->d_mat_n, 0, 2 * sizeof(unsigned long long));
        }
    }
    if (e == cudaSuccess) e = (cudaError_t)launch_init_queue(p->d_queue, g.num_pages, nullptr);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        int r = cuda_error(e, "creating the pool");
        leyline_pool_destroy(p);
        return r;
    }
    if (p->move_blocks_per_sm < 1) p->move_blocks_per_sm = 1;
    if ((cudaError_t)rotate_in_place_blocks_per_sm(&p->reindex_blocks_per_sm) != cudaSuccess ||
        p->reindex_blocks_per_sm < 1)
        p->reindex_blocks_per_sm = 1;
    {
        int err = bulk_prepare(g.row_vecs * 16, &p->bulk_blocks_per_sm);
        if (err != 0) {
            int r = cuda_error((cudaError_t)err, "preparing the bulk-copy kernel");
            leyline_pool_destroy(p);
            return r;
        }
        // The register-staged vector kernel is the default (measured faster on
        // GB300); LEYLINE_MOVE_KERNEL=bulk selects the bulk-load (TMA) kernel for
        // the MLA row shape (latent 512 + rope 64), for A/B measurements.
        const char* env = getenv("LEYLINE_MOVE_KERNEL");
        const bool want_bulk = env && strcmp(env, "bulk") == 0;
        const bool mla = g.latent_vecs == 64 && g.rope_vecs == 8 && !(g.flags & LEYLINE_POOL_SPLIT_ROPE);
        p->move_kernel = (want_bulk && mla && p->bulk_blocks_per_sm > 0) ? MOVE_BULK : MOVE_VECTOR;
    }
    p->q_head = 0;
    p->q_tail = g.num_pages;  // all pages free, ids 0..num_pages-1 in order
    *out = p;
    return LEYLINE_OK;
}

int leyline_pool_destroy(leyline_pool_t* p)
{
    if (!p) return set_error(LEYLINE_ERR_INVALID_ARG, "null pool");
    DeviceGuard guard(p->device);
    if (p->has_work) cudaEventSynchronize(p->done);
    for (auto& ev : p->tev) {
        cudaEventDestroy(ev.first);
        cudaEventDestroy(ev.second);
    }
    for (int i = 0; i < leyline_pool::kPlanSlots; ++i) {
        if (p->plan_uploaded[i]) cudaEventDestroy(p->plan_uploaded[i]);
        if (p->h_plan[i]) cudaFreeHost(p->h_plan[i]);
        if (p->d_plan[i]) cudaFree(p->d_plan[i]);
    }
    if (p->done) cudaEventDestroy(p->done);
    if (p->d_status) cudaFree(p->d_status);
    if (p->d_queue) cudaFree(p->d_queue);
    if (p->d_stage) cudaFree(p->d_stage);
    if (p->d_pending) cudaFree(p->d_pending);
    if (p->d_theta_j) cudaFree(p->d_theta_j);
    if (p->d_mat_slot) cudaFree(p->d_mat_slot);
    if (p->d_mat_pend) cudaFree(p->d_mat_pend);
    if (p->d_mat_n) cudaFree(p->d_mat_n);
    if (p->d_ckpt_queue) cudaFree(p->d_ckpt_queue);
    if (p->d_ckpt_pending) cudaFree(p->d_ckpt_pending);
    delete p;
    return LEYLINE_OK;
}

int64_t leyline_free_page_count(const leyline_pool_t* p)
{
    if (!p) return set_error(LEYLINE_ERR_INVALID_ARG, "null pool");
    return p->q_tail - p->q_head;
}

int leyline_alloc_pages(leyline_pool_t* p, int32_t n, int32_t* ids)
{
    clear_error();
    if (!p || n < 0 || (n > 0 && !ids)) return set_error(LEYLINE_ERR_INVALID_ARG, "bad arguments");
    p->window_open = false;  // other work on the pool ends the window of overlapping splices
    if (n > p->q_tail - p->q_head) return set_error(LEYLINE_ERR_NO_PAGES, "not enough free pages");
    if (n == 0) return LEYLINE_OK;
    DeviceGuard guard(p->device);
    int rc = wait_pool(p);
    if (rc != LEYLINE_OK) return rc;
    // the ring may wrap: at most two contiguous pieces
    int64_t done = 0;
    while (done < n) {
        const int64_t at = (p->q_head + done) % p->q_cap;
        const int64_t len = std::min<int64_t>(n - done, p->q_cap - at);
        cudaError_t e = cudaMemcpy(ids + done, p->d_queue + at, sizeof(int32_t) * (size_t)len, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_error(e, "reading the free-page ring");
        done += len;
    }
    p->q_head += n;
    return LEYLINE_OK;
}

int leyline_free_pages(leyline_pool_t* p, int32_t n, const int32_t* ids)
{
    clear_error();
    if (!p || n < 0 || (n > 0 && !ids)) return set_error(LEYLINE_ERR_INVALID_ARG, "bad arguments");
    p->window_open = false;  // other work on the pool ends the window of overlapping splices
    if (p->q_tail - p->q_head + n > p->g.num_pages)
        return set_error(LEYLINE_ERR_INVALID_ARG, "more pages returned than the pool holds");
    for (int32_t i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= p->g.num_pages) return set_error(LEYLINE_ERR_INVALID_ARG, "page id out of range");
    if (n == 0) return LEYLINE_OK;
    DeviceGuard guard(p->device);
    int rc = wait_pool(p);
    if (rc != LEYLINE_OK) return rc;
    int64_t done = 0;
    while (done < n) {
        const int64_t at = (p->q_tail + done) % p->q_cap;
        const int64_t len = std::min<int64_t>(n - done, p->q_cap - at);
        cudaError_t e = cudaMemcpy(p->d_queue + at, ids + done, sizeof(int32_t) * (size_t)len, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_error(e, "writing the free-page ring");
        if (p->d_pending) {  // a free page carries no pending turn: clear the returned pages' counts
            e = (cudaError_t)launch_clear_pending(p->d_pending, p->d_queue + at, len, p->g.block_size, nullptr);
            if (e == cudaSuccess) e = cudaStreamSynchronize(nullptr);
            if (e != cudaSuccess) return cuda_error(e, "clearing pending turns of returned pages");
        }
        done += len;
    }
    p->q_tail += n;
    return LEYLINE_OK;
}

int leyline_splice_plan(const leyline_pool_desc_t* desc, const int64_t* seq_lens_host, int32_t num_reqs,
                        int32_t max_blocks, const leyline_directive_t* dirs, int32_t n, int64_t free_pages,
                        leyline_stats_t* stats, int64_t* new_seq_lens)
{
    clear_error();
    Geometry g;
    int rc = make_geometry(desc, &g);
    if (rc != LEYLINE_OK) return rc;
    if (num_reqs > 0 && !seq_lens_host) return set_error(LEYLINE_ERR_INVALID_ARG, "null seq_lens_host");
    Plan plan;
    rc = build_plan(g, seq_lens_host, num_reqs, max_blocks, dirs, n, free_pages, &plan);
    if (rc != LEYLINE_OK) return rc;
    if (stats) *stats = plan.stats;
    if (new_seq_lens) {
        for (int32_t r = 0; r < num_reqs; ++r) new_seq_lens[r] = seq_lens_host[r];
        for (const ReqPlan& rp : plan.reqs) new_seq_lens[rp.req] = rp.new_len;
    }
    return LEYLINE_OK;
}

int leyline_splice(leyline_pool_t* p, leyline_block_table_t* bt, const leyline_directive_t* dirs, int32_t n,
                   void* stream_v)
{
    NvtxRange range("leyline_splice");
    clear_error();
    const HostClock t_enter = host_now();
    if (!p) return set_error(LEYLINE_ERR_INVALID_ARG, "null pool");
    {
        DeviceGuard capture_guard(p->device);
        int rc0 = refuse_capture((cudaStream_t)stream_v, "leyline_splice");
        if (rc0 != LEYLINE_OK) return rc0;
    }
    if (!bt || !bt->table || !bt->seq_lens_dev || !bt->seq_lens_host || bt->num_reqs < 0 || bt->max_blocks < 0)
        return set_error(LEYLINE_ERR_INVALID_ARG, "incomplete block table");
    for (int32_t r = 0; r < bt->num_reqs; ++r)
        if (bt->seq_lens_host[r] < 0 || bt->seq_lens_host[r] > (int64_t)bt->max_blocks * p->g.block_size)
            return set_error(LEYLINE_ERR_INVALID_ARG, "seq_lens_host entry outside [0, max_blocks * block_size]");
    std::vector<leyline_directive_t> resolved;
    const leyline_directive_t* use = dirs;
    bool host_rows = false;
    int rc = resolve_repl_rows(dirs, n, p->device, &resolved, &use, &host_rows);
    if (rc != LEYLINE_OK) return rc;
    const HostClock t_resolved = host_now();
    Plan plan;
    const int64_t free_now = p->q_tail - p->q_head;
    {
        NvtxRange plan_range("leyline_splice: plan");
        rc = build_plan(p->g, bt->seq_lens_host, bt->num_reqs, bt->max_blocks, use, n, free_now, &plan);
    }
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
    cudaStream_t stream = (cudaStream_t)stream_v;
    DeviceGuard guard(p->device);
    if (!guard.ok) return set_error(LEYLINE_ERR_CUDA, "cannot select the pool's device");

    SpliceArgs a{};
    a.kv = p->kv;
    a.table = bt->table;
    a.table_w = bt->table;
    a.seq_lens_dev = bt->seq_lens_dev;
    a.free_q = p->d_queue;
    a.q_cap = p->q_cap;
    a.pop_base = p->q_head;
    a.push_base = p->q_tail;
    a.status = p->d_status;
    a.total_tiles = plan.total_tiles;
    a.total_commit = plan.total_commit;
    a.n_reqs = (int32_t)plan.reqs.size();
    a.n_trig = plan.n_trig;
    a.max_blocks = bt->max_blocks;
    a.pending = p->d_pending;
    a.g = p->g;

    cudaError_t e;
    if (plan.reindex) {
        if ((size_t)plan.total_stage > p->d_stage_cap) {
            rc = wait_pool(p);
            if (rc != LEYLINE_OK) return rc;
            if (p->d_stage) cudaFree(p->d_stage);
            p->d_stage = nullptr;
            p->d_stage_cap = 0;
            const size_t cap = std::max<size_t>((size_t)plan.total_stage * 2, 1 << 14);
            e = cudaMalloc(&p->d_stage, sizeof(int32_t) * cap);
            if (e != cudaSuccess) return cuda_error(e, "allocating the staging buffer");
            p->d_stage_cap = cap;
        }
        a.stage = p->d_stage;
        a.total_prep = plan.total_prep;
        a.total_repl = plan.total_repl;
        a.total_fresh = plan.total_fresh;
        a.reindex = 1;
    }
    rc = order_after_previous(p, stream);
    if (rc != LEYLINE_OK) return rc;
    const bool in_params = plan_fits_params(plan);
    ParamPlan pp;
    if (in_params) {
        pack_param_plan(plan, &pp);
    } else {
        // Plan too large for a kernel parameter: upload it (reqs | segs | trig).
        const size_t off_segs = align_up(sizeof(ReqPlan) * plan.reqs.size(), 16);
        const size_t off_trig = align_up(off_segs + sizeof(Seg) * plan.segs.size(), 16);
        const size_t total = align_up(off_trig + sizeof(float) * plan.trig.size(), 256);
        const int slot = p->next_slot;
        if (total > p->d_plan_cap[slot]) {  // a larger device buffer: no kernel may still read it
            rc = wait_pool(p);
            if (rc != LEYLINE_OK) return rc;
            if (p->d_plan[slot]) cudaFree(p->d_plan[slot]);
            p->d_plan[slot] = nullptr;
            p->d_plan_cap[slot] = 0;
            const size_t cap = std::max<size_t>(total * 2, 1 << 16);
            e = cudaMalloc(&p->d_plan[slot], cap);
            if (e != cudaSuccess) return cuda_error(e, "allocating the plan buffer");
            p->d_plan_cap[slot] = cap;
        }
        p->next_slot = (slot + 1) % leyline_pool::kPlanSlots;
        if (p->slot_used[slot]) {  // the slot's last upload may still be in flight
            e = cudaEventSynchronize(p->plan_uploaded[slot]);
            if (e != cudaSuccess) return cuda_error(e, "waiting for an earlier plan upload");
        }
        if (total > p->h_plan_cap[slot]) {
            if (p->h_plan[slot]) cudaFreeHost(p->h_plan[slot]);
            p->h_plan[slot] = nullptr;
            p->h_plan_cap[slot] = 0;
            const size_t cap = std::max<size_t>(total * 2, 1 << 16);
            e = cudaHostAlloc((void**)&p->h_plan[slot], cap, cudaHostAllocDefault);
            if (e != cudaSuccess) return cuda_error(e, "allocating the pinned plan buffer");
            p->h_plan_cap[slot] = cap;
        }
        char* h = p->h_plan[slot];
        memcpy(h, plan.reqs.data(), sizeof(ReqPlan) * plan.reqs.size());
        memcpy(h + off_segs, plan.segs.data(), sizeof(Seg) * plan.segs.size());
        if (!plan.trig.empty()) memcpy(h + off_trig, plan.trig.data(), sizeof(float) * plan.trig.size());
        // copied by a kernel in the chain of dependent launches (see launch_upload_plan)
        e = (cudaError_t)launch_upload_plan(h, p->d_plan[slot], total, stream);
        if (e != cudaSuccess) return cuda_error(e, "uploading the plan");
        ++plan.stats.kernels_launched;
        e = cudaEventRecord(p->plan_uploaded[slot], stream);
        if (e != cudaSuccess) return cuda_error(e, "recording the plan upload");
        p->slot_used[slot] = true;
        a.reqs = reinterpret_cast<const ReqPlan*>(p->d_plan[slot]);
        a.segs = reinterpret_cast<const Seg*>(p->d_plan[slot] + off_segs);
        a.trig = reinterpret_cast<const float*>(p->d_plan[slot] + off_trig);
    }

    cudaEvent_t t0 = nullptr, t1 = nullptr;
    if (p->timing) {
        if (p->tev_used == p->tev.size()) {
            cudaEvent_t x, y;
            if (cudaEventCreate(&x) != cudaSuccess) return set_error(LEYLINE_ERR_CUDA, "creating timing events");
            if (cudaEventCreate(&y) != cudaSuccess) {
                cudaEventDestroy(x);
                return set_error(LEYLINE_ERR_CUDA, "creating timing events");
            }
            p->tev.emplace_back(x, y);
        }
        t0 = p->tev[p->tev_used].first;
        t1 = p->tev[p->tev_used].second;
        ++p->tev_used;
    }
    a.move_kernel = host_rows ? MOVE_VECTOR : p->move_kernel;  // rows of R in host memory: plain loads
    const int grid = p->sm_count * (plan.reindex                    ? p->reindex_blocks_per_sm
                                    : a.move_kernel == MOVE_BULK ? p->bulk_blocks_per_sm
                                                                 : p->move_blocks_per_sm);
    // Overlap with the calls before it.  A rewrite whose plan travels as a kernel parameter
    // and whose move runs in the MLA vector kernel may start before the calls still running
    // (the window) end, when on the same stream it rewrites no request they rewrite and
    // takes only pages that were on the free list before the window's first call returned
    // any: it then reads nothing they write and writes nothing they read.
    const bool mla = p->g.latent_vecs == 64 && p->g.rope_vecs == 8 && p->g.rope_heads == 1;
    const bool vector_mla = mla && !(a.move_kernel == MOVE_BULK && !(p->g.flags & LEYLINE_POOL_SPLIT_ROPE));
    const bool chainable = !plan.reindex && in_params && !p->timing && vector_mla && plan.total_tiles > 0 &&
                           plan.total_commit > 0;
    bool overlap = chainable && p->window_open && p->has_work && stream == p->last_stream &&
                   p->window_calls < leyline_pool::kOverlapWindow && p->q_head + plan.total_pop <= p->window_tail;
    for (size_t r = 0; overlap && r < plan.reqs.size(); ++r)
        if (std::find(p->window_reqs.begin(), p->window_reqs.end(), plan.reqs[r].req) != p->window_reqs.end())
            overlap = false;
    a.overlap_prev = overlap ? 1 : 0;
    int err = launch_splice(a, in_params ? &pp : nullptr, grid, stream, t0, t1);
    if (err != 0) {
        p->window_open = false;
        return cuda_error((cudaError_t)err, "launching the splice kernels");
    }
    rc = mark_done(p, stream);
    if (rc != LEYLINE_OK) return rc;
    if (plan.reindex && !p->d_pending) p->ckpt_turned = true;  // bands turned in place
    if (chainable) {
        if (!overlap) {  // this call waited for everything before it: a new window opens
            p->window_open = true;
            p->window_calls = 0;
            p->window_tail = p->q_tail;
            p->window_reqs.clear();
        }
        ++p->window_calls;
        for (const ReqPlan& rp : plan.reqs) p->window_reqs.push_back(rp.req);
    } else {
        p->window_open = false;
    }

    for (const ReqPlan& rp : plan.reqs) bt->seq_lens_host[rp.req] = rp.new_len;
    p->q_head += plan.total_pop;
    p->q_tail += plan.total_push;
    p->last_stats = plan.stats;
    p->last_stats.overlapped = overlap ? 1 : 0;
    set_host_times(&p->last_stats, t_enter, t_resolved, t_planned);
    return LEYLINE_OK;
}

int leyline_last_stats(const leyline_pool_t* p, leyline_stats_t* out)
{
    if (!p || !out) return set_error(LEYLINE_ERR_INVALID_ARG, "null argument");
    *out = p->last_stats;
    return LEYLINE_OK;
}

int leyline_gather(leyline_pool_t* p, const leyline_block_table_t* bt, int32_t req, int32_t layer, int64_t t0,
                   int64_t t1, void* out, void* stream_v)
{
    NvtxRange range("leyline_gather");
    clear_error();
    if (!p || !bt || !bt->table || !bt->seq_lens_host) return set_error(LEYLINE_ERR_INVALID_ARG, "null argument");
    p->window_open = false;  // other work on the pool ends the window of overlapping splices
    if (req < 0 || req >= bt->num_reqs) return set_error(LEYLINE_ERR_INVALID_ARG, "request out of range");
    if (layer < 0 || layer >= p->g.num_layers) return set_error(LEYLINE_ERR_INVALID_ARG, "layer out of range");
    if (t0 < 0 || t0 > t1 || t1 > bt->seq_lens_host[req] || t1 > (int64_t)bt->max_blocks * p->g.block_size)
        return set_error(LEYLINE_ERR_INVALID_ARG, "rows outside [0, seq_len]");
    if (t1 > t0 && (!out || (reinterpret_cast<uintptr_t>(out) & 15) != 0))
        return set_error(LEYLINE_ERR_INVALID_ARG, "out must be a 16-byte aligned pointer");
    if (t1 == t0) return LEYLINE_OK;
    bool out_host = false;
    int rc0 = resolve_access(out, p->device, "gather output", &out, &out_host);
    if (rc0 != LEYLINE_OK) return rc0;
    cudaStream_t stream = (cudaStream_t)stream_v;
    DeviceGuard guard(p->device);
    int rc = order_after_previous(p, stream);
    if (rc != LEYLINE_OK) return rc;
    const int32_t* row = bt->table + (int64_t)req * bt->max_blocks;
    int err = p->d_pending ? launch_gather_lazy(p->kv, row, p->g, layer, t0, t1, out, p->d_pending, p->d_theta_j,
                                                p->d_status, stream)
                           : launch_gather(p->kv, row, p->g, layer, t0, t1, out, p->d_status, stream);
    if (err != 0) return cuda_error((cudaError_t)err, "launching the gather kernel");
    return mark_done(p, stream);
}

int leyline_materialize_requests(leyline_pool_t* p, const leyline_block_table_t* bt, const int32_t* reqs, int32_t n,
                                 void* stream_v)
{
    NvtxRange range("leyline_materialize_requests");
    clear_error();
    if (!p || !bt || !bt->table || !bt->seq_lens_host || n < 0 || (n > 0 && !reqs))
        return set_error(LEYLINE_ERR_INVALID_ARG, "null argument");
    {
        DeviceGuard capture_guard(p->device);
        int rc0 = refuse_capture((cudaStream_t)stream_v, "leyline_materialize_requests");
        if (rc0 != LEYLINE_OK) return rc0;
    }
    p->window_open = false;  // other work on the pool ends the window of overlapping splices
    if (!p->d_pending) return set_error(LEYLINE_ERR_INVALID_ARG, "the pool was not created with LEYLINE_POOL_LAZY");
    std::vector<int32_t> seen(reqs, reqs + n);
    std::sort(seen.begin(), seen.end());
    for (int32_t k = 0; k < n; ++k) {
        if (seen[k] < 0 || seen[k] >= bt->num_reqs) return set_error(LEYLINE_ERR_INVALID_ARG, "request out of range");
        if (k > 0 && seen[k] == seen[k - 1])  // two warps would turn the same rows
            return set_error(LEYLINE_ERR_INVALID_ARG, "a request appears twice");
        const int64_t len = bt->seq_lens_host[seen[k]];
        if (len < 0 || len > (int64_t)bt->max_blocks * p->g.block_size)
            return set_error(LEYLINE_ERR_INVALID_ARG, "seq_len outside the block table");
    }
    cudaStream_t stream = (cudaStream_t)stream_v;
    DeviceGuard guard(p->device);

    int rc = order_after_previous(p, stream);
    if (rc != LEYLINE_OK) return rc;
    bool launched = false;
    for (int32_t k0 = 0; k0 < n; k0 += kMaterializeReqs) {  // up to kMaterializeReqs requests per launch
        MaterializeSet set{};
        int64_t rows = 0;
        for (int32_t k = k0; k < n && k < k0 + kMaterializeReqs; ++k) {
            const int64_t len = bt->seq_lens_host[reqs[k]];
            if (len == 0) continue;
            rows += len;
            set.req[set.n] = reqs[k];
            set.row_end[set.n] = rows;
            ++set.n;
        }
        if (set.n == 0) continue;
        const MaterializeScratch scratch{p->d_mat_slot, p->d_mat_pend, p->d_mat_n ? p->d_mat_n + p->mat_turn : nullptr,
                                         p->d_mat_n ? p->d_mat_n + (1 - p->mat_turn) : nullptr};
        int err = launch_materialize(p->kv, bt->table, bt->max_blocks, set, p->g, p->d_pending, p->d_theta_j,
                                     p->d_status, scratch, stream);
        if (err == 0 && materialize_uses_list(p->g)) p->mat_turn = 1 - p->mat_turn;
        if (err != 0) return cuda_error((cudaError_t)err, "launching the materialize kernel");
        launched = true;
        p->ckpt_turned = true;  // stored bands turned in place
    }
    return launched ? mark_done(p, stream) : LEYLINE_OK;
}

int leyline_materialize(leyline_pool_t* p, const leyline_block_table_t* bt, int32_t req, void* stream_v)
{
    return leyline_materialize_requests(p, bt, &req, 1, stream_v);
}

int32_t* leyline_pending_ptr(leyline_pool_t* p)
{
    clear_error();
    if (!p) {
        set_error(LEYLINE_ERR_INVALID_ARG, "null pool");
        return nullptr;
    }
    return p->d_pending;
}

int leyline_sync_status(leyline_pool_t* p)
{
    clear_error();
    if (!p) return set_error(LEYLINE_ERR_INVALID_ARG, "null pool");
    p->window_open = false;  // other work on the pool ends the window of overlapping splices
    DeviceGuard guard(p->device);
    int rc = wait_pool(p);
    if (rc != LEYLINE_OK) return rc;
    int32_t st = 0;
    cudaError_t e = cudaMemcpy(&st, p->d_status, sizeof st, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_error(e, "reading the status word");
    if (st != 0) {
        cudaMemset(p->d_status, 0, sizeof(int32_t));
        char msg[128];
        snprintf(msg, sizeof msg, "device check failed (status bits 0x%x)", st);
        return set_error(LEYLINE_ERR_DEVICE_CHECK, msg);
    }
    return LEYLINE_OK;
}

int leyline_pool_checkpoint(leyline_pool_t* p, void* stream_v)
{
    NvtxRange range("leyline_pool_checkpoint");
    clear_error();
    if (!p) return set_error(LEYLINE_ERR_INVALID_ARG, "null pool");
    p->window_open = false;  // other work on the pool ends the window of overlapping splices
    cudaStream_t stream = (cudaStream_t)stream_v;
    DeviceGuard guard(p->device);
    if (!guard.ok) return set_error(LEYLINE_ERR_CUDA, "cannot select the pool's device");
    int rc_cap = refuse_capture(stream, "leyline_pool_checkpoint");
    if (rc_cap != LEYLINE_OK) return rc_cap;
    const size_t slots = (size_t)p->g.num_pages * (size_t)p->g.block_size;
    cudaError_t e = cudaSuccess;
    if (!p->d_ckpt_queue) e = cudaMalloc(&p->d_ckpt_queue, sizeof(int32_t) * (size_t)p->q_cap);
    if (e == cudaSuccess && p->d_pending && !p->d_ckpt_pending)
        e = cudaMalloc(&p->d_ckpt_pending, sizeof(int32_t) * slots);
    if (e != cudaSuccess) return cuda_error(e, "allocating the checkpoint");
    int rc = order_after_previous(p, stream);
    if (rc != LEYLINE_OK) return rc;
    e = cudaMemcpyAsync(p->d_ckpt_queue, p->d_queue, sizeof(int32_t) * (size_t)p->q_cap, cudaMemcpyDeviceToDevice,
                        stream);
    if (e == cudaSuccess && p->d_pending)
        e = cudaMemcpyAsync(p->d_ckpt_pending, p->d_pending, sizeof(int32_t) * slots, cudaMemcpyDeviceToDevice,
                            stream);
    if (e != cudaSuccess) return cuda_error(e, "copying the page accounting");
    rc = mark_done(p, stream);
    if (rc != LEYLINE_OK) return rc;
    p->has_ckpt = true;
    p->ckpt_head = p->q_head;
    p->ckpt_tail = p->q_tail;
    p->ckpt_turned = false;
    return LEYLINE_OK;
}

int leyline_pool_rollback(leyline_pool_t* p, int32_t flags, void* stream_v)
{
    NvtxRange range("leyline_pool_rollback");
    clear_error();
    if (!p) return set_error(LEYLINE_ERR_INVALID_ARG, "null pool");
    p->window_open = false;  // other work on the pool ends the window of overlapping splices
    if ((flags & ~LEYLINE_ROLLBACK_ACCEPT_TURNED) != 0) return set_error(LEYLINE_ERR_INVALID_ARG, "unknown flags");
    if (!p->has_ckpt) return set_error(LEYLINE_ERR_INVALID_ARG, "the pool has no checkpoint");
    // Pages returned since the checkpoint sit at ring positions from ckpt_tail on: once the
    // head passed that point, one of them was taken again and may have been written.
    if (p->q_head > p->ckpt_tail)
        return set_error(LEYLINE_ERR_INVALID_ARG,
                         "pages returned since the checkpoint have been taken again: their rows may be overwritten");
    if (p->ckpt_turned && !(flags & LEYLINE_ROLLBACK_ACCEPT_TURNED))
        return set_error(LEYLINE_ERR_INVALID_ARG,
                         "stored rope bands were turned in place since the checkpoint (re-index splice of an eager "
                         "pool, or materialize); a rollback would not undo that");
    cudaStream_t stream = (cudaStream_t)stream_v;
    DeviceGuard guard(p->device);
    if (!guard.ok) return set_error(LEYLINE_ERR_CUDA, "cannot select the pool's device");
    int rc = refuse_capture(stream, "leyline_pool_rollback");
    if (rc != LEYLINE_OK) return rc;
    rc = order_after_previous(p, stream);
    if (rc != LEYLINE_OK) return rc;
    const size_t slots = (size_t)p->g.num_pages * (size_t)p->g.block_size;
    // Only the ring entries written since the checkpoint differ from its copy: returned pages
    // are written at positions [ckpt_tail, q_tail), while taking pages only moves the head.
    const int64_t pushed = p->q_tail - p->ckpt_tail;
    cudaError_t e = cudaSuccess;
    if (pushed >= p->q_cap) {
        e = cudaMemcpyAsync(p->d_queue, p->d_ckpt_queue, sizeof(int32_t) * (size_t)p->q_cap, cudaMemcpyDeviceToDevice,
                            stream);
    } else if (pushed > 0) {
        const int64_t at = p->ckpt_tail % p->q_cap;
        const int64_t first = std::min(pushed, p->q_cap - at);  // up to the ring's end, then from its start
        e = cudaMemcpyAsync(p->d_queue + at, p->d_ckpt_queue + at, sizeof(int32_t) * (size_t)first,
                            cudaMemcpyDeviceToDevice, stream);
        if (e == cudaSuccess && pushed > first)
            e = cudaMemcpyAsync(p->d_queue, p->d_ckpt_queue, sizeof(int32_t) * (size_t)(pushed - first),
                                cudaMemcpyDeviceToDevice, stream);
    }
    if (e == cudaSuccess && p->d_pending)
        e = cudaMemcpyAsync(p->d_pending, p->d_ckpt_pending, sizeof(int32_t) * slots, cudaMemcpyDeviceToDevice,
                            stream);
    if (e != cudaSuccess) return cuda_error(e, "restoring the page accounting");
    rc = mark_done(p, stream);
    if (rc != LEYLINE_OK) return rc;
    p->q_head = p->ckpt_head;
    p->q_tail = p->ckpt_tail;
    p->ckpt_turned = false;
    return LEYLINE_OK;
}

int leyline_kernel_timing_enable(leyline_pool_t* p, int32_t enable)
{
    if (!p) return set_error(LEYLINE_ERR_INVALID_ARG, "null pool");
    p->window_open = false;  // other work on the pool ends the window of overlapping splices
    p->timing = enable != 0;
    p->tev_used = 0;
    if (p->timing && p->tev.size() < kTimingEventsUpFront) {
        // created now, so that the timed calls themselves create no events
        DeviceGuard guard(p->device);
        while (p->tev.size() < kTimingEventsUpFront) {
            cudaEvent_t x, y;
            if (cudaEventCreate(&x) != cudaSuccess) return set_error(LEYLINE_ERR_CUDA, "creating timing events");
            if (cudaEventCreate(&y) != cudaSuccess) {
                cudaEventDestroy(x);
                return set_error(LEYLINE_ERR_CUDA, "creating timing events");
            }
            p->tev.emplace_back(x, y);
        }
    }
    return LEYLINE_OK;
}

int leyline_kernel_timing_read(leyline_pool_t* p, double* total_ms, int32_t* launches)
{
    if (!p || !total_ms || !launches) return set_error(LEYLINE_ERR_INVALID_ARG, "null argument");
    DeviceGuard guard(p->device);
    double sum = 0.0;
    for (size_t i = 0; i < p->tev_used; ++i) {
        cudaError_t e = cudaEventSynchronize(p->tev[i].second);
        if (e != cudaSuccess) return cuda_error(e, "waiting for timing events");
        float ms = 0.f;
        e = cudaEventElapsedTime(&ms, p->tev[i].first, p->tev[i].second);
        if (e != cudaSuccess) return cuda_error(e, "reading timing events");
        sum += ms;
    }
    *total_ms = sum;
    *launches = (int32_t)p->tev_used;
    p->tev_used = 0;
    return LEYLINE_OK;
}

}  // extern "C"
