/*
 * leyline.h -- C ABI of the GB300 Leyline AMORTIZE splice library (libleyline.so).
 *
 * The operation: "Leyline: KV Cache Directives for Agentic Inference"
 * (technical summary of arXiv 2606.01065).
 *   section 2.1  A directive D = (s_start, s_end, R, m) replaces the token span
 *                [s_start, s_end) of a sequence by the token sequence R.  Mode
 *                AMORTIZE splices in place: R is inserted, downstream positions
 *                are re-indexed, and the downstream tokens keep their position-
 *                free KV content (K_nope and V).  Mode FORGET routes the edit to
 *                a prefix-trimming re-prefill instead.
 *   section 2.2  With |S| = s_end - s_start, every downstream token moves by
 *                Delta = |R| - |S|, and its cached RoPE band is corrected in
 *                closed form: K_pe_new = R(Delta) K_pe.  Because R(a)R(b) =
 *                R(a+b), this equals encoding the token from scratch at its new
 *                position.  In MLA the key splits into K_nope (position-free, from
 *                the compressed latent) and K_pe (RoPE-rotated).
 *   section 2.3  Serving integration: match the prefix [0, s_start), prefill R
 *                into new slots, then a rotation kernel delta-rotates and
 *                re-indexes every downstream slot.  This library is that last
 *                step plus the slot writes; matching and prefill stay with the
 *                caller.
 *   section 3    The directive interface sits above block-level (paged) storage.
 *   section 4.3  bf16 storage makes delta-rotation drift; computing the rotation
 *                in fp32 mitigates it.  The library rotates in fp32 and stores bf16.
 *
 * Storage model.  A pool holds num_pages pages per layer.  One page stores
 * block_size consecutive token slots of one request.  A slot row is
 * latent_dim + rope_dim bf16 values: the compressed latent first (moved bit for
 * bit, never recomputed), the RoPE band k_pe last (rope_heads bands for GQA/MHA
 * rows).  The pool memory is laid out
 *     kv[layer][page][slot][latent_dim + rope_heads * rope_dim]      (bf16, row-major)
 * and one block table, shared by all layers, maps block b of request r to a page:
 *     table[r * max_blocks + b] = page id, for b < ceil(seq_len[r] / block_size).
 * A page belongs to one request: no two live table entries may name the same
 * page (a splice returns a request's old pages to the free list, and a lazy read
 * turns each listed row once).  The device checks that page ids are in range,
 * not that they are distinct.
 *
 * How a splice is carried out.  Every block from floor(s_min / block_size) on
 * (s_min = the smallest s_start of the request's directives) is rewritten into
 * fresh pages taken from the pool's free-page list; the request's old pages from
 * that block on go back onto the list when the rewrite is committed.  Source
 * rows are never written, so the call has no read/write hazard whatever the sign
 * of Delta, and a call that fails validation changes nothing.  The prefix rows
 * of the first rewritten block are copied unchanged.
 *
 * Conventions.  All functions return LEYLINE_OK (0) or a negative
 * LEYLINE_ERR_* code, and never throw or abort.  leyline_last_error() gives a
 * message for the calling thread.  Device pointers are CUDA global-memory
 * pointers on the device that was current at leyline_pool_create; every bf16
 * buffer must be 16-byte aligned.  "stream" is a cudaStream_t (NULL = legacy
 * default stream).  Work is enqueued asynchronously; host-side state (the
 * seq_lens_host mirror and the free-page count) is updated at enqueue time.
 * Calls on one pool must not run concurrently from several host threads.
 */
#ifndef LEYLINE_H
#define LEYLINE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ errors ---- */
#define LEYLINE_OK 0
#define LEYLINE_ERR_INVALID_ARG (-1)       /* null / misaligned pointer, bad size or descriptor */
#define LEYLINE_ERR_INVALID_DIRECTIVE (-2) /* s_start > s_end, s_end > seq_len, bad req, n_repl < 0 */
#define LEYLINE_ERR_OVERLAP (-3)           /* two spans of one request overlap or share s_start */
#define LEYLINE_ERR_NO_PAGES (-4)          /* not enough free pages for the rewritten blocks */
#define LEYLINE_ERR_UNSUPPORTED_MODE (-5)  /* FORGET (caller re-prefills) or unknown mode */
#define LEYLINE_ERR_CUDA (-6)              /* a CUDA runtime call failed */
#define LEYLINE_ERR_CAPACITY (-7)          /* new length exceeds max_blocks * block_size */
#define LEYLINE_ERR_DEVICE_CHECK (-8)      /* a device-side bounds check fired (leyline_sync_status) */
#define LEYLINE_ERR_SCRATCH (-9)           /* plan larger than the static scratch of leyline_splice_noalloc */

/* --------------------------------------------------------------- types ---- */
typedef struct leyline_pool leyline_pool_t; /* opaque, owned by the library */

/* RoPE pair layout of the rope band (the pages fix none; half-split is the
 * rotate_half convention, pair j = (j, j + rope_dim/2)). */
typedef enum { LEYLINE_PAIRS_HALF_SPLIT = 0, LEYLINE_PAIRS_INTERLEAVED = 1 } leyline_pair_layout_t;

/* Arithmetic of the delta-rotation.  FP32 is the product path (section 4.3).
 * BF16_NAIVE rounds cos, sin, each product and each sum to bf16; it exists only
 * as the comparison arm of drift studies. */
typedef enum { LEYLINE_ROTATE_FP32 = 0, LEYLINE_ROTATE_BF16_NAIVE = 1 } leyline_rotate_precision_t;

/* Pool flags.
 * LEYLINE_POOL_REINDEX: a splice keeps a surviving block in its page when all the
 *   block's rows come from one run of survivors shifted by a multiple of block_size
 *   (every survivor at block_size 1): only its block-table entry moves, and its rope
 *   bands are turned in place (256 bytes per slot and layer instead of 2304; the
 *   latent is not touched).  The other new blocks (rows of R, and survivors or prefix
 *   rows at run boundaries) get fresh pages, and old blocks not kept return to the
 *   free list.  A call whose fresh pages would take more survivor and prefix rows
 *   than its kept pages hold rewrites as without the flag (statistics: reindexed).
 *   The rotation happens in place before the commit, so a call that fails after
 *   validation leaves the pool inconsistent (as any LEYLINE_ERR_CUDA does).  Requires
 *   rope_dim <= 256 and rope_heads * rope_dim <= 512 (else pool creation fails
 *   with LEYLINE_ERR_INVALID_ARG). */
#define LEYLINE_POOL_REINDEX 1
/* LEYLINE_POOL_LAZY: a splice does not turn rope bands.  The pool keeps, per slot,
 * an int32 count of positions that the stored band still has to turn (the
 * "pending" turn); a splice moves a survivor's count with it and adds the turn
 * the eager splice would have applied, and rows of R start at 0.  Readers apply
 * R(pending) once: leyline_gather does, leyline_materialize applies it in place
 * and clears it, and attention kernels can read the counts through
 * leyline_pending_ptr.  A band is then rounded to bf16 once per read instead of
 * once per splice (section 4.3: the drift of repeated bf16 rotation), and with
 * LEYLINE_POOL_REINDEX a splice moves no cache bytes for survivors at all.
 * Readers form the cos and sin of pending * theta_j in fp64 and round them once
 * to the rotation's precision, as an eager splice does for its Delta: for
 * |pending| < 2^22 as the angle-addition product of cos/sin(hi * 2048 * theta_j)
 * and cos/sin(lo * theta_j) (pending = hi * 2048 + lo), else by fp64 sincos of
 * the angle.  An attention kernel that applies the counts itself matches
 * leyline_gather when it does the same. */
#define LEYLINE_POOL_LAZY 2
/* LEYLINE_POOL_SPLIT_ROPE: the pool buffer holds the latents and the rope bands in
 * two arrays instead of whole rows: bf16 latent[num_layers][num_pages][block_size]
 * [latent_dim], then bf16 rope[num_layers][num_pages][block_size][rope_heads *
 * rope_dim] (the layout of paged MLA attention kernels that take a latent cache and a
 * rope cache).  The buffer size is the same.  Rows of R, gather outputs and every
 * other interface keep whole rows [latent | rope bands].  A splice that turns bands
 * in place (LEYLINE_POOL_REINDEX, leyline_materialize) then streams contiguous bands
 * instead of 128 bytes out of every row. */
#define LEYLINE_POOL_SPLIT_ROPE 4

typedef struct {
    int32_t num_layers;       /* >= 1 */
    int32_t latent_dim;       /* multiple of 8 (512 for DeepSeek-V2/V3 MLA) */
    int32_t rope_dim;         /* multiple of 16 (64 for DeepSeek-V2/V3 MLA) */
    int32_t block_size;       /* tokens per page, >= 1 (16: vLLM-style blocks; 1: per-token) */
    int64_t num_pages;        /* pages per layer, 1 .. 2^31 - 1 */
    double rope_theta;        /* RoPE base, > 0 (10000) */
    int32_t pair_layout;      /* leyline_pair_layout_t */
    int32_t rotate_precision; /* leyline_rotate_precision_t */
    uint32_t flags;           /* LEYLINE_POOL_* bits */
    int32_t rope_heads;       /* RoPE bands per row, each rope_dim wide (0 or 1: one band, the MLA
                                 row).  > 1 for GQA/MHA caches (section 5: the directive
                                 abstraction extends to GQA/MHA): the row is then [V | keys of
                                 rope_heads heads], the keys fully RoPE'd, each head's band turned
                                 with the same theta_j */
} leyline_pool_desc_t;

/* Block tables of num_reqs requests.  Caller-owned; the library borrows them for
 * the duration of enqueued work.  table and seq_lens_dev are device int32 arrays
 * ([num_reqs][max_blocks] and [num_reqs]); seq_lens_host is the host mirror of
 * the lengths, read to validate directives and updated by leyline_splice when
 * the work is enqueued.  Unused table entries should hold -1. */
typedef struct {
    int32_t* table;
    int32_t* seq_lens_dev;
    int64_t* seq_lens_host;
    int32_t num_reqs;
    int32_t max_blocks;
} leyline_block_table_t;

/* Directive modes.  AMORTIZE and FORGET are the two modes of section 2.1.
 * EVICT is the compaction of the KV-streams page: the span is dropped (and R
 * inserted) but downstream tokens keep the positions they were encoded at, so
 * their rope bands are not turned.  In one call, a surviving run moves by the
 * summed Delta of every directive to its left and is turned by the summed Delta
 * of the AMORTIZE directives among them. */
typedef enum { LEYLINE_AMORTIZE = 0, LEYLINE_FORGET = 1, LEYLINE_EVICT = 2 } leyline_mode_t;

/* One directive D = (s_start, s_end, R, m) for request `req` (section 2.1).
 * [s_start, s_end) is half-open, in the request's coordinates before the call;
 * several directives of one request must not overlap and must have distinct
 * s_start.  repl_rows: bf16 [num_layers][n_repl][row] (row as in the pool) in
 * device memory of the pool's GPU or in pinned host memory (cudaHostAlloc or
 * cudaHostRegister; the kernel reads it in place over the host link), 16-byte
 * aligned; pageable memory is refused with INVALID_ARG.  These are
 * the rows of R already encoded at their final positions s_start + D_before + i
 * (D_before = the summed Delta of the request's directives left of this one),
 * as prefill writes them (section 2.3); they are copied bit for bit and must stay
 * live until the enqueued work has finished.  May be NULL when n_repl == 0. */
typedef struct {
    int32_t req;
    int32_t mode; /* leyline_mode_t */
    int64_t s_start;
    int64_t s_end;
    int32_t n_repl;
    int32_t reserved; /* must be 0 */
    const void* repl_rows;
} leyline_directive_t;

/* Work accounting of one splice call. */
typedef struct {
    int64_t downstream_slots;  /* surviving tokens at or after each request's first s_end, summed */
    int64_t repl_slots;        /* rows of R written */
    int64_t head_slots;        /* unchanged prefix rows copied into the first rewritten block */
    int64_t algorithmic_bytes; /* bytes that must move: 2 * row_bytes * num_layers * (downstream_slots +
                                  repl_slots); re-indexed requests count 2 * rope_bytes per turned
                                  downstream slot and nothing for unturned ones */
    int64_t moved_bytes;       /* algorithmic bytes plus the head rows' 2 * row_bytes * num_layers */
    int64_t pages_popped;      /* fresh pages taken for the rewritten blocks */
    int64_t pages_pushed;      /* old pages returned to the free-page list */
    int32_t requests_touched;
    int32_t kernels_launched;  /* kernels this call enqueued (leyline_splice_plan: without the copy
                                  kernel that leyline_splice adds for a plan it uploads) */
    int32_t reindexed;         /* 1: the call kept survivors in their pages (LEYLINE_POOL_REINDEX) */
    int32_t overlapped;        /* 1: the call's move kernel may start before the previous call's work
                                  on the stream ends (see leyline_splice) */
    /* Host time of the call (leyline_splice, leyline_splice_noalloc; 0 from the dry run),
     * in nanoseconds of the host's monotonic clock: */
    int64_t host_ns;           /* the whole call, from entry to return (kernels are enqueued, not waited for) */
    int64_t resolve_ns;        /* classifying the directives' pointers to rows of R */
    int64_t plan_ns;           /* the host planner */
    int64_t timed_kernel_bytes; /* algorithmic bytes of the kernel that kernel timing brackets: the
                                   move+rotate kernel (all of algorithmic_bytes) for a rewrite, the
                                   in-place rotation (2 * rope_bytes per turned slot and layer) for
                                   a re-index call that turns bands, else the launches before the
                                   commit (all of algorithmic_bytes) */
} leyline_stats_t;

/* -------------------------------------------------------------- pool ---- */

/* Create a pool over caller-owned device memory kv_dev (bf16
 * [num_layers][num_pages][block_size][row], row = latent_dim + rope_heads * rope_dim,
 * 16-byte aligned; with LEYLINE_POOL_SPLIT_ROPE the latent array then the rope array).
 * All pages start free.  The library allocates the free-page list (a ring of
 * 2 * num_pages ids) and small plan and staging buffers on the current device;
 * a LEYLINE_POOL_LAZY pool also its pending counts (4 bytes per slot), the
 * readers' turn table (32 * rope_dim KiB) and, when a row's rope bands span 128
 * bytes (rope_heads * rope_dim == 64), the lists materialize works from (12 bytes
 * per slot).  Synchronous.
 * Errors: INVALID_ARG (bad descriptor, null/misaligned kv_dev), CUDA. */
int leyline_pool_create(const leyline_pool_desc_t* desc, void* kv_dev, leyline_pool_t** out);

/* Wait for the pool's enqueued work and free what the library allocated (never kv_dev). */
int leyline_pool_destroy(leyline_pool_t* pool);

/* Take n pages off the free-page list, for the caller's initial fill or prefill.
 * Synchronous (waits for the pool's enqueued work).  page_ids_host receives n ids
 * (the k-th id taken first).  Errors: INVALID_ARG, NO_PAGES, CUDA. */
int leyline_alloc_pages(leyline_pool_t* pool, int32_t n, int32_t* page_ids_host);

/* Return n pages (ids from page_ids_host) to the free-page list.  Synchronous.
 * Errors: INVALID_ARG (id out of range, more pages than the pool holds), CUDA. */
int leyline_free_pages(leyline_pool_t* pool, int32_t n, const int32_t* page_ids_host);

/* Number of free pages as seen at enqueue time (negative code on a NULL pool). */
int64_t leyline_free_page_count(const leyline_pool_t* pool);

/* Checkpoint and rollback of the pool's page accounting.  A rewrite splice
 * (section 2.3's rotation kernel, run out of place) only reads its source pages
 * and hands them back to the free-page list, so until those pages are taken
 * again the cache before the splice still exists; these two calls get it back,
 * to repeat a splice on the same input (benchmark repeats: section 2.3 gives no
 * other way to run the same edit twice) or to drop a splice whose edit was
 * rejected.  The pages say nothing about undoing a splice.
 *
 * leyline_pool_checkpoint saves the free-page list, its positions and, in a
 * LEYLINE_POOL_LAZY pool, the pending counts, into device memory the pool
 * allocates on the first checkpoint (4 bytes per ring entry, 2 * num_pages, plus
 * 4 bytes per slot in lazy pools) and keeps until destroyed.  A later checkpoint
 * replaces it.  Enqueued on `stream` after the pool's earlier work.
 * Errors: INVALID_ARG (null pool), CUDA.
 *
 * leyline_pool_rollback puts the saved accounting back (enqueued on `stream`):
 * pages taken since the checkpoint are free again and pages returned since are
 * owned again.  It copies back only the free-list entries written since the
 * checkpoint (4 bytes per page returned since) and, in lazy pools, all pending
 * counts.  The block table and the lengths are the caller's: the caller
 * restores them too (table, seq_lens_dev and seq_lens_host as they were at the
 * checkpoint), after the pool's work on the stream.  Refused, with nothing
 * changed (INVALID_ARG), when
 *   - the pool has no checkpoint;
 *   - a page returned since the checkpoint has been taken again (its rows may
 *     have been overwritten): the splices since the checkpoint took more pages
 *     than were free at the checkpoint;
 *   - stored rope bands were turned in place since the checkpoint (a re-index
 *     splice of an eager pool, or leyline_materialize), unless flags holds
 *     LEYLINE_ROLLBACK_ACCEPT_TURNED: the accounting is then restored but those
 *     bands stay turned (benchmark repeats, where the work and not the values
 *     matters).
 * Both refuse a `stream` under graph capture (INVALID_ARG): the ring positions
 * they save and restore are host state at enqueue time.
 * Errors: INVALID_ARG, CUDA. */
#define LEYLINE_ROLLBACK_ACCEPT_TURNED 1
int leyline_pool_checkpoint(leyline_pool_t* pool, void* stream);
int leyline_pool_rollback(leyline_pool_t* pool, int32_t flags, void* stream);

/* -------------------------------------------------------------- splice ---- */

/* Apply n AMORTIZE directives (any mix of requests) as one composed pass per
 * request (section 2.2 / 2.3): for each request with at least one effective
 * directive, drop its spans, write the rows of R, move every downstream slot to
 * its new position (latent bit for bit) and rotate its rope band by the
 * accumulated Delta in fp32, storing bf16.  Directives with s_start == s_end and
 * n_repl == 0 are no-ops.  On return the work is enqueued on `stream`, the
 * seq_lens_host entries hold the new lengths and the pages are accounted; the
 * table and seq_lens_dev change when the enqueued work runs.  Enqueues two
 * kernels (move+rotate, then commit; a re-index call up to four).  The plan
 * travels as a kernel parameter when it has at most 8 requests, 24 segments and
 * 10 rotated segments; otherwise it is staged in one of 8 pinned host slots and
 * a first kernel copies it to the device (the call then waits on the host only
 * when all 8 slots are still in flight).
 * Calls enqueued back to back on one stream keep stream order for everything
 * the caller can observe, but the library may let a call's kernels start
 * before the previous calls' kernels end: only for a rewrite whose plan is a
 * kernel parameter, which shares no request with the calls that may still run
 * and takes no page they returned (stats: overlapped).  Any other work on the
 * stream between two calls, or a call on another stream, orders them fully.
 * Errors (nothing is enqueued or changed): INVALID_ARG, INVALID_DIRECTIVE,
 * OVERLAP, UNSUPPORTED_MODE (FORGET: the caller re-prefills, section 2.1),
 * CAPACITY, NO_PAGES.  INVALID_ARG also when `stream` is being captured into a
 * CUDA graph: the call is planned on the host for the cache as it stands, and a
 * replay would apply that plan to a cache that has moved on.  CUDA: a launch
 * failed after validation; the pool must then be considered inconsistent. */
int leyline_splice(leyline_pool_t* pool, leyline_block_table_t* bt, const leyline_directive_t* dirs,
                   int32_t n, void* stream);

/* The same splice as leyline_splice, for callers that must not allocate device
 * memory while they run: a serving framework that has reserved nearly all of the
 * GPU's memory in its own caching allocator (a cudaMalloc behind its back fails
 * or fragments what it manages), or a process whose device footprint must stay
 * fixed after start-up.  The paper has no counterpart; this is an interface
 * variant only.  It makes no device, pinned-host or torch allocation: its
 * scratch is a static 4 MiB device array that every GPU which loads the library
 * holds until the process exits, and the plan is staged through a static host
 * array (the host-side planning itself uses ordinary C++ containers).  The
 * array's device address is looked up on the first call on each device.  All
 * calls share the array:
 * calls that overlap on the GPU without ordering (different streams, different
 * pools) race on it.  Copying the plan from pageable memory may make the call
 * wait for earlier work on `stream`.  Same arguments, results and error codes
 * as leyline_splice, plus SCRATCH when the call's plan exceeds 4 MiB (with a
 * 64-wide rope band, about 12,000 directives that shift their downstream
 * rows): split the directives over several calls.  While kernel timing is on
 * (leyline_kernel_timing_enable), a call is timed with the events created when
 * timing was switched on; calls beyond those 256 are not timed. */
int leyline_splice_noalloc(leyline_pool_t* pool, leyline_block_table_t* bt, const leyline_directive_t* dirs,
                           int32_t n, void* stream);

/* Host-only dry run of leyline_splice: validates the directives against
 * seq_lens_host (length num_reqs) and the pool geometry in desc, and reports the
 * work and the page demand in *stats without touching any device.  If
 * new_seq_lens is not NULL it receives the length of every request after the
 * splice.  free_pages: pages available (pass a negative value to skip the page
 * check).  Returns the same error codes as leyline_splice. */
int leyline_splice_plan(const leyline_pool_desc_t* desc, const int64_t* seq_lens_host, int32_t num_reqs,
                        int32_t max_blocks, const leyline_directive_t* dirs, int32_t n, int64_t free_pages,
                        leyline_stats_t* stats, int64_t* new_seq_lens);

/* Statistics of the last successful leyline_splice on this pool. */
int leyline_last_stats(const leyline_pool_t* pool, leyline_stats_t* out);

/* -------------------------------------------------------------- gather ---- */

/* Copy the logical rows [t0, t1) of request `req`, layer `layer` into out_dev
 * (bf16 [t1 - t0][row], 16-byte aligned, in device memory of the pool's GPU or in
 * pinned host memory, which the kernel writes in place), reading
 * through the block table.  In a LEYLINE_POOL_LAZY pool each row's rope bands
 * are turned by the row's pending count on the way out.  Asynchronous on `stream`.
 * Errors: INVALID_ARG (range outside [0, seq_lens_host[req]], bad layer/req,
 * pageable or foreign-device output). */
int leyline_gather(leyline_pool_t* pool, const leyline_block_table_t* bt, int32_t req, int32_t layer,
                   int64_t t0, int64_t t1, void* out_dev, void* stream);

/* ---------------------------------------------------------- lazy mode ---- */

/* LEYLINE_POOL_LAZY pools: turn the stored rope bands of rows [0, seq_len) of
 * request `req` (all layers) by their pending counts, in fp32, storing bf16, and
 * set the counts to 0.  Asynchronous on `stream`.  Errors: INVALID_ARG (not a lazy
 * pool, bad request, `stream` under graph capture). */
int leyline_materialize(leyline_pool_t* pool, const leyline_block_table_t* bt, int32_t req, void* stream);

/* leyline_materialize for the n requests reqs[0..n) (host array, distinct ids), in one
 * launch per 64 requests: their rows form one list, so the launches are few and full.
 * Errors: INVALID_ARG (not a lazy pool, a request out of range or listed twice, or
 * `stream` under graph capture: the launches are sized from seq_lens_host as it
 * stands). */
int leyline_materialize_requests(leyline_pool_t* pool, const leyline_block_table_t* bt, const int32_t* reqs,
                                 int32_t n, void* stream);

/* LEYLINE_POOL_LAZY pools: device pointer to the pending counts, int32
 * [num_pages][block_size] (the count of the slot at position t of a request is
 * at page * block_size + t % block_size, page = table[t / block_size]).  Owned by
 * the pool; NULL for other pools. */
int32_t* leyline_pending_ptr(leyline_pool_t* pool);

/* ----------------------------------------------------------- checking ---- */

/* Wait for the pool's enqueued work and read its device status word.  Returns
 * LEYLINE_OK, LEYLINE_ERR_DEVICE_CHECK if a kernel met a page id or position
 * outside the pool or table (it then skipped that row; the status is cleared by
 * this call), or LEYLINE_ERR_CUDA. */
int leyline_sync_status(leyline_pool_t* pool);

/* Kernel timing for benchmarks.  While enabled, each splice records CUDA events
 * on its stream around its dominant kernel (stats: timed_kernel_bytes): the
 * move+rotate kernel, a re-index call's in-place rotation, or the launches before
 * a lazy re-index call's commit.  leyline_kernel_timing_read waits
 * for them and returns the summed kernel time (ms) and the number of timed
 * launches since the last enable, then keeps timing.  Enabling creates the events
 * of the first 256 timed calls at once, so that those calls create none. */
int leyline_kernel_timing_enable(leyline_pool_t* pool, int32_t enable);
int leyline_kernel_timing_read(leyline_pool_t* pool, double* total_ms, int32_t* launches);

/* Message of the last error on the calling thread ("" if none). */
const char* leyline_last_error(void);

/* Library version, e.g. "leyline-gb300 0.1.0 sm_103a". */
const char* leyline_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LEYLINE_H */
