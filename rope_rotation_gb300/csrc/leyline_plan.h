// leyline_plan.h -- the splice plan: what the host planner hands to the kernels.
//
// A splice of one request ("Leyline: KV Cache Directives for Agentic
// Inference", sections 2.1-2.3) is described in the request's NEW coordinates as
// a short list of segments that tile the rewritten range [b0 * B, new_len):
//   HEAD   prefix rows of the first rewritten block, copied unchanged (Delta 0)
//   REPL   rows of a directive's R, copied bit for bit
//   COPY   a surviving run whose accumulated Delta is 0, moved unchanged
//   ROT    a surviving run moved by Delta != 0; its rope band is turned by R(Delta)
//          (in a lazy pool such a run is a COPY segment whose turn is added to the
//          rows' pending counts instead)
// The kernels look up the segment of a destination row, read the source row
// through the old block table (or from R), and write it into a fresh page.
// A re-indexed request (block size 1, pool flag LEYLINE_POOL_REINDEX) keeps its
// surviving rows in their pages instead: a prep kernel stages the new table
// entries (the old page of each kept row, a fresh page for each row of R) and
// returns the pages of the dropped tokens (DROP segments) to the free ring; the
// move kernel turns the rope bands of ROT rows in place and copies R rows; the
// commit kernel installs the staged entries.
#pragma once

#include <cstdint>

namespace leyline {

constexpr int kTileRows = 16;  // destination rows per move+rotate tile

// Row segments (HEAD, REPL, COPY, ROT) cover a request's new rows [row0, new_len) in
// order.  Re-index mode adds two lists after them: DROP runs of old blocks returned to
// the free list, and FRESH runs of new rows written into fresh pages.
enum SegKind : int32_t { SEG_HEAD = 0, SEG_REPL = 1, SEG_COPY = 2, SEG_ROT = 3, SEG_DROP = 4, SEG_FRESH = 5 };

struct Geometry {
    int32_t num_layers;
    int32_t latent_dim;
    int32_t rope_dim;
    int32_t block_size;
    int32_t row_elems;    // latent_dim + rope_heads * rope_dim
    int32_t row_vecs;     // row_elems / 8 (16-byte vectors)
    int32_t latent_vecs;  // latent_dim / 8
    int32_t rope_vecs;    // rope_heads * rope_dim / 8 (all RoPE bands of a row)
    int32_t rope_heads;   // RoPE bands per row (1: MLA)
    int32_t head_vecs;    // rope_dim / 8 (one band)
    int64_t num_pages;
    int64_t layer_vecs;   // num_pages * block_size * row_vecs
    // Where the parts of the row of (layer, slot) live, in 16-byte vectors from the
    // pool base: the latent at lat_layer_vecs * layer + lat_row_vecs * slot, the rope
    // bands at rope_base_vecs + rope_layer_vecs * layer + rope_row_vecs * slot.  One
    // array of whole rows: the bands follow the latent in the row.  Split rope
    // (LEYLINE_POOL_SPLIT_ROPE): an array of latents followed by an array of bands.
    int64_t lat_layer_vecs;
    int64_t rope_layer_vecs;
    int64_t rope_base_vecs;
    int32_t lat_row_vecs;
    int32_t rope_row_vecs;
    double theta;
    int32_t pair_layout;
    int32_t precision;
    uint32_t flags;       // LEYLINE_POOL_* bits
    int32_t pad;
};

struct ReqPlan {
    int32_t req;           // table row
    int32_t b0;            // first rewritten block
    int32_t n_new;         // fresh pages: ceil(new_len / B) - b0
    int32_t n_old;         // pages returned: ceil(old_len / B) - b0
    int64_t row0;          // b0 * B, first rewritten destination row
    int64_t new_len;
    int64_t old_len;
    int64_t tile_begin;    // first flat move+rotate tile of this request
    int64_t commit_begin;  // first flat commit index of this request
    int32_t seg_begin;
    int32_t seg_count;
    int32_t pop_off;       // first fresh page of this request in the ring's pop region
    int32_t push_off;      // first returned page of this request in the ring's push region
    int64_t stage_begin;   // re-index: first staged table entry of this request
    int64_t prep_begin;    // re-index: first flat prep item of this request
    int64_t drop_count;    // re-index: old blocks returned to the free list
    int32_t drop_seg_begin;  // re-index: DROP runs (old blocks returned)
    int32_t drop_seg_count;
    int64_t repl_begin;    // re-index: first of this request's rows of R in the call's list of them
    int64_t fresh_begin;   // re-index: first of this request's other fresh rows in the call's list
    int32_t fresh_seg_begin;  // re-index: FRESH runs (survivor and prefix rows written into fresh pages)
    int32_t fresh_seg_count;
};

struct Seg {
    int64_t new_start;     // first destination row of the segment (not used by DROP)
    int64_t src_start;     // source position (HEAD/COPY/ROT/DROP) or row index in R (REPL)
    const void* repl;      // R rows [num_layers][n_repl][row] (REPL only)
    int32_t kind;          // SegKind
    int32_t trig;          // trig table entry (ROT only), else -1
    int32_t n_repl;        // rows of R per layer (REPL); dropped tokens (DROP)
    int32_t aux;           // re-index: R rows of the request before this segment (REPL),
                           // dropped tokens of the request before this segment (DROP)
    int32_t turn;          // positions the segment's rows turn (ROT; in lazy pools also COPY)
    int32_t tile_off;      // re-index: first rotate-kernel tile of this ROT segment's kept rows
                           // within its request, -1 for other segments
    int32_t kb0, kb1;      // re-index, COPY/ROT: new blocks [kb0, kb1) keep their old pages
                           // (block kb0 - shift / B ...), all rows of the segment; else kb0 = kb1
    int32_t kept_before;   // re-index: kept blocks of the request's earlier segments
    int32_t pad2;
};

static_assert(sizeof(ReqPlan) == 128, "ReqPlan layout");
static_assert(sizeof(Seg) == 64, "Seg layout");

}  // namespace leyline
