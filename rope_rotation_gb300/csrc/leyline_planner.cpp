// leyline_planner.cpp -- host-side validation and planning of a splice call.
//
// "Leyline: KV Cache Directives for Agentic Inference":
//   section 2.1  D = (s_start, s_end, R, m); AMORTIZE splices in place; FORGET is
//                routed to a re-prefill, which this library does not do.
//   section 2.2  Delta = |R| - |S| for every downstream token.
//   section 2.3  prefix [0, s_start) kept, R written to new slots, downstream
//                slots re-indexed and rotated.
//
// Several directives of one request are composed into one pass: with the spans
// sorted, directive k's rows of R start at s_k + D_{k-1} and the surviving run
// [e_k, s_{k+1}) moves by D_k, where D_k is the summed Delta of directives 1..k.
// This equals applying the directives one at a time, right to left.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>

#include "leyline_internal.h"

namespace leyline {

namespace {
thread_local std::string g_last_error;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Nearest bf16 value (ties to even) of a double, returned as the float it
// denotes: the significand is cut to 8 bits straight from the double's bit
// pattern, so the value is rounded once (not through float first).
float bf16_nearest(double x)
{
    uint64_t b;
    std::memcpy(&b, &x, sizeof b);
    const bool neg = (b >> 63) != 0;
    const int exp = (int)((b >> 52) & 0x7FF);
    if (exp == 0x7FF) return (float)x;
    if (exp == 0) return neg ? -0.0f : 0.0f;
    const int E = exp - 1023;  // |x| in [2^E, 2^(E+1))
    double r;
    if (E >= -126) {
        const uint64_t mant = (b & ((uint64_t(1) << 52) - 1)) | (uint64_t(1) << 52);
        uint64_t q = mant >> 45;
        const uint64_t rem = mant & ((uint64_t(1) << 45) - 1), half = uint64_t(1) << 44;
        if (rem > half || (rem == half && (q & 1))) ++q;
        r = std::ldexp((double)q, E - 7);
    } else {  // bf16 subnormal range: steps of 2^-133
        r = std::ldexp(std::nearbyint(std::ldexp(std::fabs(x), 133)), -133);
    }
    return neg ? -(float)r : (float)r;
}

// cos / sin of Delta * theta_j for every pair j of a rotated segment (theta_j given).  The angle is
// formed in fp64 (Delta * theta_0 reaches 1e5 rad, where an fp32 angle would be off
// by ~1e-2 rad, more than a bf16 step), the library's cos / sin reduce it exactly,
// and the result is rounded once to the arithmetic of the rotation.
void segment_trig(const Geometry& g, const double* theta_j, int64_t delta, float* out)
{
    const int half = g.rope_dim / 2;
    for (int j = 0; j < half; ++j) {
        const double phi = (double)delta * theta_j[j];
        double s, c;
        sincos(phi, &s, &c);
        if (g.precision == LEYLINE_ROTATE_BF16_NAIVE) {
            out[2 * j] = bf16_nearest(c);
            out[2 * j + 1] = bf16_nearest(s);
        } else {
            out[2 * j] = (float)c;
            out[2 * j + 1] = (float)s;
        }
    }
}
}  // namespace

int set_error(int code, const std::string& msg)
{
    g_last_error = msg;
    return code;
}

void clear_error() { g_last_error.clear(); }

const char* last_error_cstr() { return g_last_error.c_str(); }

int make_geometry(const leyline_pool_desc_t* d, Geometry* g)
{
    if (!d) return set_error(LEYLINE_ERR_INVALID_ARG, "null pool descriptor");
    if (d->num_layers < 1) return set_error(LEYLINE_ERR_INVALID_ARG, "num_layers must be >= 1");
    if (d->latent_dim < 0 || d->latent_dim % 8 != 0)
        return set_error(LEYLINE_ERR_INVALID_ARG, "latent_dim must be a non-negative multiple of 8");
    if (d->rope_dim < 16 || d->rope_dim % 16 != 0)
        return set_error(LEYLINE_ERR_INVALID_ARG, "rope_dim must be a positive multiple of 16");
    if (d->block_size < 1) return set_error(LEYLINE_ERR_INVALID_ARG, "block_size must be >= 1");
    if (d->num_pages < 1 || d->num_pages > INT32_MAX)
        return set_error(LEYLINE_ERR_INVALID_ARG, "num_pages must be in [1, 2^31 - 1]");
    if (!(d->rope_theta > 0.0)) return set_error(LEYLINE_ERR_INVALID_ARG, "rope_theta must be > 0");
    if (d->pair_layout != LEYLINE_PAIRS_HALF_SPLIT && d->pair_layout != LEYLINE_PAIRS_INTERLEAVED)
        return set_error(LEYLINE_ERR_INVALID_ARG, "unknown pair_layout");
    if (d->rotate_precision != LEYLINE_ROTATE_FP32 && d->rotate_precision != LEYLINE_ROTATE_BF16_NAIVE)
        return set_error(LEYLINE_ERR_INVALID_ARG, "unknown rotate_precision");
    if ((d->flags & ~(uint32_t)(LEYLINE_POOL_REINDEX | LEYLINE_POOL_LAZY | LEYLINE_POOL_SPLIT_ROPE)) != 0)
        return set_error(LEYLINE_ERR_INVALID_ARG, "unknown pool flags");
    if (d->rope_heads < 0 || d->rope_heads > 1024)
        return set_error(LEYLINE_ERR_INVALID_ARG, "rope_heads must be in [0, 1024]");
    if ((d->flags & LEYLINE_POOL_REINDEX) && (d->rope_dim > 256 || (int64_t)d->rope_dim * std::max(d->rope_heads, 1) > 512))
        return set_error(LEYLINE_ERR_INVALID_ARG,
                         "LEYLINE_POOL_REINDEX supports rope_dim <= 256 and rope_heads * rope_dim <= 512");
    g->num_layers = d->num_layers;
    g->latent_dim = d->latent_dim;
    g->rope_dim = d->rope_dim;
    g->block_size = d->block_size;
    const int heads = d->rope_heads > 1 ? d->rope_heads : 1;
    g->rope_heads = heads;
    g->row_elems = d->latent_dim + heads * d->rope_dim;
    g->row_vecs = g->row_elems / 8;
    g->latent_vecs = d->latent_dim / 8;
    g->head_vecs = d->rope_dim / 8;
    g->rope_vecs = heads * g->head_vecs;
    g->num_pages = d->num_pages;
    g->layer_vecs = d->num_pages * (int64_t)d->block_size * g->row_vecs;
    const int64_t slots = d->num_pages * (int64_t)d->block_size;
    if (d->flags & LEYLINE_POOL_SPLIT_ROPE) {
        g->lat_row_vecs = g->latent_vecs;
        g->rope_row_vecs = g->rope_vecs;
        g->lat_layer_vecs = slots * g->latent_vecs;
        g->rope_layer_vecs = slots * g->rope_vecs;
        g->rope_base_vecs = (int64_t)d->num_layers * g->lat_layer_vecs;
    } else {
        g->lat_row_vecs = g->rope_row_vecs = g->row_vecs;
        g->lat_layer_vecs = g->rope_layer_vecs = g->layer_vecs;
        g->rope_base_vecs = g->latent_vecs;
    }
    g->theta = d->rope_theta;
    g->pair_layout = d->pair_layout;
    g->precision = d->rotate_precision;
    g->flags = d->flags;
    g->pad = 0;
    return LEYLINE_OK;
}

namespace {

struct PlanCounts {
    int64_t kept_rows = 0;          // re-index: rows whose blocks keep their pages
    int64_t kept_turned_rows = 0;   // of which turned in place
    int64_t fresh_rows = 0;         // survivor and prefix rows written into fresh pages
    int64_t fresh_head_rows = 0;    // of which unchanged prefix rows of a boundary block
    int64_t fresh_repl_rows = 0;    // rows of R (written into fresh pages too)
};

// Segments, pages and work counts of every touched request, as a rewrite (reindex =
// false) or re-indexed (true).  Directives are validated and ordered by request and
// s_start (order).
int plan_requests(const Geometry& g, const int64_t* seq_lens_host, int32_t max_blocks,
                  const leyline_directive_t* dirs, int32_t n, const std::vector<int32_t>& order, bool reindex,
                  bool lazy, Plan* plan, PlanCounts* counts, char* msg, size_t msg_size)
{
    const int64_t B = g.block_size;
    plan->reindex = reindex;
    int64_t tiles = 0, commit = 0, pops = 0, pushes = 0;
    std::vector<double> theta_j(g.rope_dim / 2);  // theta^(-2j/d) in fp64
    for (int j = 0; j < g.rope_dim / 2; ++j) theta_j[j] = std::pow(g.theta, -2.0 * (double)j / (double)g.rope_dim);
    leyline_stats_t& st = plan->stats;
    for (int32_t i = 0; i < n;) {
        const int32_t req = dirs[order[i]].req;
        int32_t j = i;
        std::vector<const leyline_directive_t*> eff;
        for (; j < n && dirs[order[j]].req == req; ++j) {
            const leyline_directive_t* d = &dirs[order[j]];
            if (d->s_start == d->s_end && d->n_repl == 0) continue;  // no-op
            eff.push_back(d);
        }
        i = j;
        if (eff.empty()) continue;

        const int64_t L = seq_lens_host[req];
        if (L > (int64_t)max_blocks * B) {
            snprintf(msg, msg_size, "request %d: seq_len %lld exceeds the table capacity", req, (long long)L);
            return set_error(LEYLINE_ERR_INVALID_ARG, msg);
        }
        int64_t delta_total = 0;
        for (const auto* d : eff) delta_total += (int64_t)d->n_repl - (d->s_end - d->s_start);
        const int64_t Lp = L + delta_total;
        if (Lp > (int64_t)max_blocks * B || Lp > INT32_MAX) {
            snprintf(msg, msg_size, "request %d: new length %lld exceeds the table capacity %lld", req,
                     (long long)Lp, (long long)max_blocks * B);
            return set_error(LEYLINE_ERR_CAPACITY, msg);
        }
        ReqPlan rp{};
        rp.req = req;
        rp.b0 = (int32_t)(eff.front()->s_start / B);
        rp.row0 = (int64_t)rp.b0 * B;
        rp.old_len = L;
        rp.new_len = Lp;
        rp.seg_begin = (int32_t)plan->segs.size();
        rp.pop_off = (int32_t)pops;
        rp.push_off = (int32_t)pushes;
        rp.tile_begin = tiles;
        rp.commit_begin = commit;

        // row segments in new coordinates.  D: index shift left of the current position
        // (every directive); A: rotation (AMORTIZE directives only, section 2.1; EVICT
        // keeps positions).
        const int64_t s1 = eff.front()->s_start;
        if (rp.row0 < s1) {
            Seg s{rp.row0, rp.row0, nullptr, SEG_HEAD, -1, 0, 0, 0, 0};
            plan->segs.push_back(s);
            st.head_slots += s1 - rp.row0;
        }
        int64_t D = 0, A = 0;
        for (size_t k = 0; k < eff.size(); ++k) {
            const leyline_directive_t* d = eff[k];
            if (d->n_repl > 0) {
                Seg s{d->s_start + D, 0, d->repl_rows, SEG_REPL, -1, d->n_repl, 0, 0, 0};
                plan->segs.push_back(s);
                st.repl_slots += d->n_repl;
            }
            const int64_t dk = (int64_t)d->n_repl - (d->s_end - d->s_start);
            D += dk;
            if (d->mode == LEYLINE_AMORTIZE) A += dk;
            const int64_t run_end = (k + 1 < eff.size()) ? eff[k + 1]->s_start : L;
            if (run_end > d->s_end) {
                Seg s{d->s_end + D, d->s_end, nullptr, (A == 0 || lazy) ? SEG_COPY : SEG_ROT, -1, 0, 0, (int32_t)A,
                      0};
                if (A != 0 && !lazy) {
                    s.trig = plan->n_trig++;
                    plan->trig.resize((size_t)plan->n_trig * g.rope_dim);
                    segment_trig(g, theta_j.data(), A, plan->trig.data() + (size_t)s.trig * g.rope_dim);
                }
                plan->segs.push_back(s);
                st.downstream_slots += run_end - d->s_end;
            }
        }
        rp.seg_count = (int32_t)plan->segs.size() - rp.seg_begin;
        if (rp.seg_count == 0) {  // nothing left to write (pure truncation at a block boundary)
            Seg s{rp.row0, rp.row0, nullptr, SEG_HEAD, -1, 0, 0, 0, 0};
            plan->segs.push_back(s);
            rp.seg_count = 1;
        }
        const int64_t nb_new = ceil_div(Lp, B), nb_old = ceil_div(L, B);
        if (!reindex) {
            rp.n_new = (int32_t)(nb_new - rp.b0);
            rp.n_old = (int32_t)(nb_old - rp.b0);
            tiles += ceil_div(Lp - rp.row0, kTileRows);
            commit += std::max<int64_t>(1, std::max(rp.n_new, rp.n_old));
        } else {
            // Kept blocks: new block j keeps its old page when every row of it comes from one
            // COPY/ROT segment whose shift is a multiple of B (then old block j - shift / B
            // holds exactly those rows).  Every other new block gets a fresh page, written
            // row by row; every old block not kept returns to the free list.
            const int32_t last = rp.seg_begin + rp.seg_count;
            int64_t kept = 0, wt = 0;
            for (int32_t k = rp.seg_begin; k < last; ++k) {
                Seg& s = plan->segs[k];
                const int64_t end = k + 1 < last ? plan->segs[k + 1].new_start : Lp;
                s.kept_before = (int32_t)kept;
                s.kb0 = s.kb1 = 0;
                s.tile_off = -1;
                const int64_t shift = s.new_start - s.src_start;
                if ((s.kind == SEG_COPY || s.kind == SEG_ROT) && end > s.new_start && shift % B == 0) {
                    const int64_t k0 = ceil_div(s.new_start, B);
                    const int64_t k1 = end == Lp ? nb_new : end / B;  // a last partial block moves whole
                    if (k1 > k0) {
                        s.kb0 = (int32_t)k0;
                        s.kb1 = (int32_t)k1;
                        kept += k1 - k0;
                        const int64_t kr = std::min(k1 * B, end) - k0 * B;  // kept rows
                        counts->kept_rows += kr;
                        if (s.kind == SEG_ROT) {
                            s.tile_off = (int32_t)wt;
                            wt += ceil_div(kr, kTileRows);
                            counts->kept_turned_rows += kr;
                        } else if (lazy && s.turn != 0) {
                            counts->kept_turned_rows += kr;
                        }
                    }
                }
            }
            tiles += wt;
            rp.n_new = (int32_t)(nb_new - rp.b0 - kept);  // fresh pages
            rp.n_old = (int32_t)(nb_old - rp.b0 - kept);  // pages returned
            // Rows of the fresh blocks: rows of R (one list per call), and FRESH runs of the
            // other rows (survivors and prefix rows of segments outside their kept blocks)
            rp.repl_begin = plan->total_repl;
            rp.fresh_seg_begin = (int32_t)plan->segs.size();
            rp.fresh_begin = plan->total_fresh;
            int64_t fresh = 0;
            auto fresh_run = [&](int64_t r0, int64_t r1) {
                if (r1 <= r0) return;
                Seg f{r0, 0, nullptr, SEG_FRESH, -1, (int32_t)(r1 - r0), (int32_t)fresh, 0, 0};
                plan->segs.push_back(f);
                fresh += r1 - r0;
            };
            for (int32_t k = rp.seg_begin; k < last; ++k) {
                const Seg s = plan->segs[k];
                const int64_t end = k + 1 < last ? plan->segs[k + 1].new_start : Lp;
                if (s.kind == SEG_REPL) {
                    plan->total_repl += s.n_repl;
                    counts->fresh_repl_rows += s.n_repl;
                } else if (s.kb1 > s.kb0) {
                    fresh_run(s.new_start, (int64_t)s.kb0 * B);
                    fresh_run(std::min((int64_t)s.kb1 * B, end), end);
                } else {
                    fresh_run(s.new_start, end);
                }
            }
            rp.fresh_seg_count = (int32_t)plan->segs.size() - rp.fresh_seg_begin;
            plan->total_fresh += fresh;
            counts->fresh_rows += fresh;
            // rows of the first block before the first directive are unchanged prefix rows
            counts->fresh_head_rows += s1 - rp.row0;
            // DROP runs: old blocks [b0, nb_old) minus the kept ones, in order
            rp.drop_seg_begin = (int32_t)plan->segs.size();
            int64_t ob = rp.b0, pushed = 0;
            auto drop_run = [&](int64_t o0, int64_t o1) {
                if (o1 <= o0) return;
                Seg d{-1, o0, nullptr, SEG_DROP, -1, (int32_t)(o1 - o0), (int32_t)pushed, 0, 0};
                plan->segs.push_back(d);
                pushed += o1 - o0;
            };
            for (int32_t k = rp.seg_begin; k < last; ++k) {
                const Seg s = plan->segs[k];
                if (s.kb1 > s.kb0) {
                    const int64_t sb = (s.new_start - s.src_start) / B;  // block shift
                    drop_run(ob, s.kb0 - sb);
                    ob = s.kb1 - sb;
                }
            }
            drop_run(ob, nb_old);
            rp.drop_seg_count = (int32_t)plan->segs.size() - rp.drop_seg_begin;
            rp.drop_count = pushed;
            rp.stage_begin = plan->total_stage;
            rp.prep_begin = plan->total_prep;
            const int64_t new_blocks = nb_new - rp.b0;
            plan->total_stage += new_blocks;
            plan->total_prep += new_blocks + pushed;
            const int64_t tail = std::max<int64_t>(0, nb_old - nb_new);  // entries past the new end
            // lazy pools clear the counts of returned pages: at prep, or at commit when the
            // fresh-rows kernel still reads survivors from them (the request has FRESH runs)
            const int64_t clears = (lazy && rp.fresh_seg_count > 0) ? pushed : 0;
            commit += std::max<int64_t>(1, new_blocks + tail + clears);
        }
        pops += rp.n_new;
        pushes += rp.n_old;
        plan->reqs.push_back(rp);
    }
    plan->total_tiles = tiles;
    plan->total_commit = commit;
    plan->total_pop = pops;
    plan->total_push = pushes;
    return LEYLINE_OK;
}

}  // namespace

int build_plan(const Geometry& g, const int64_t* seq_lens_host, int32_t num_reqs, int32_t max_blocks,
               const leyline_directive_t* dirs, int32_t n, int64_t free_pages, Plan* plan)
{
    char msg[256];
    *plan = Plan{};
    if (n < 0) return set_error(LEYLINE_ERR_INVALID_ARG, "negative directive count");
    if (n > 0 && !dirs) return set_error(LEYLINE_ERR_INVALID_ARG, "null directive array");
    if (num_reqs < 0 || max_blocks < 0) return set_error(LEYLINE_ERR_INVALID_ARG, "negative table size");
    if (n > 0 && !seq_lens_host) return set_error(LEYLINE_ERR_INVALID_ARG, "null seq_lens_host");
    const int64_t B = g.block_size;

    // 1. each directive on its own
    for (int32_t k = 0; k < n; ++k) {
        const leyline_directive_t& d = dirs[k];
        if (d.req < 0 || d.req >= num_reqs) {
            snprintf(msg, sizeof msg, "directive %d: request %d out of range [0, %d)", k, d.req, num_reqs);
            return set_error(LEYLINE_ERR_INVALID_DIRECTIVE, msg);
        }
        if (d.mode == LEYLINE_FORGET) {
            snprintf(msg, sizeof msg, "directive %d: FORGET is served by a re-prefill, not by the splice", k);
            return set_error(LEYLINE_ERR_UNSUPPORTED_MODE, msg);
        }
        if (d.mode != LEYLINE_AMORTIZE && d.mode != LEYLINE_EVICT) {
            snprintf(msg, sizeof msg, "directive %d: unknown mode %d", k, d.mode);
            return set_error(LEYLINE_ERR_UNSUPPORTED_MODE, msg);
        }
        if (d.reserved != 0) {
            snprintf(msg, sizeof msg, "directive %d: reserved field must be 0", k);
            return set_error(LEYLINE_ERR_INVALID_ARG, msg);
        }
        const int64_t L = seq_lens_host[d.req];
        if (d.s_start < 0 || d.s_start > d.s_end || d.s_end > L) {
            snprintf(msg, sizeof msg, "directive %d: need 0 <= s_start <= s_end <= seq_len, got [%lld, %lld) of %lld",
                     k, (long long)d.s_start, (long long)d.s_end, (long long)L);
            return set_error(LEYLINE_ERR_INVALID_DIRECTIVE, msg);
        }
        if (d.n_repl < 0) {
            snprintf(msg, sizeof msg, "directive %d: n_repl < 0", k);
            return set_error(LEYLINE_ERR_INVALID_DIRECTIVE, msg);
        }
        if (d.n_repl > 0 && (!d.repl_rows || (reinterpret_cast<uintptr_t>(d.repl_rows) & 15) != 0)) {
            snprintf(msg, sizeof msg, "directive %d: repl_rows must be a non-null 16-byte aligned pointer", k);
            return set_error(LEYLINE_ERR_INVALID_ARG, msg);
        }
    }

    // 2. group by request, sort by s_start, check non-overlap
    std::vector<int32_t> order(n);
    for (int32_t k = 0; k < n; ++k) order[k] = k;
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
        if (dirs[a].req != dirs[b].req) return dirs[a].req < dirs[b].req;
        return dirs[a].s_start < dirs[b].s_start;
    });
    for (int32_t i = 0; i + 1 < n; ++i) {
        const leyline_directive_t& a = dirs[order[i]];
        const leyline_directive_t& b = dirs[order[i + 1]];
        if (a.req != b.req) continue;
        if (a.s_start == b.s_start || a.s_end > b.s_start) {
            snprintf(msg, sizeof msg, "request %d: spans [%lld, %lld) and [%lld, %lld) overlap or share s_start",
                     a.req, (long long)a.s_start, (long long)a.s_end, (long long)b.s_start, (long long)b.s_end);
            return set_error(LEYLINE_ERR_OVERLAP, msg);
        }
    }

    // 3. plan each touched request.  Re-index pools keep the pages of surviving blocks
    // whose rows all shift by a multiple of the block size and write the other blocks'
    // rows into fresh pages.  With pages of several slots, a call whose fresh pages take
    // more survivor and prefix rows than the kept pages hold is planned as a rewrite: the
    // rewrite kernel moves whole rows faster than the fresh-rows kernel.  (Rows of R are
    // written by their own kernel in either plan.)
    const bool lazy = (g.flags & LEYLINE_POOL_LAZY) != 0;
    PlanCounts counts;
    int rc = plan_requests(g, seq_lens_host, max_blocks, dirs, n, order, (g.flags & LEYLINE_POOL_REINDEX) != 0, lazy,
                           plan, &counts, msg, sizeof msg);
    if (rc != LEYLINE_OK) return rc;
    if (plan->reindex && B > 1 && counts.kept_rows < counts.fresh_rows) {
        *plan = Plan{};
        counts = PlanCounts{};
        rc = plan_requests(g, seq_lens_host, max_blocks, dirs, n, order, false, lazy, plan, &counts, msg, sizeof msg);
        if (rc != LEYLINE_OK) return rc;
    }
    const bool reindex = plan->reindex;

    if (free_pages >= 0 && plan->total_pop > free_pages) {
        snprintf(msg, sizeof msg, "splice needs %lld fresh pages, %lld free", (long long)plan->total_pop,
                 (long long)free_pages);
        return set_error(LEYLINE_ERR_NO_PAGES, msg);
    }
    const int64_t row_bytes = (int64_t)g.row_elems * 2;
    const int64_t rope_bytes = (int64_t)g.rope_vecs * 16;  // every RoPE band of a row
    leyline_stats_t& st = plan->stats;
    const int64_t L2 = 2 * (int64_t)g.num_layers;
    if (reindex) {
        // kept rows: turned bands in place (lazy: the 4-byte count read and written);
        // fresh rows: whole rows of R and of boundary survivors, head rows as overhead
        const int64_t fresh_alg = plan->total_repl + plan->total_fresh - counts.fresh_head_rows;
        st.algorithmic_bytes = lazy ? L2 * row_bytes * fresh_alg + 8 * (counts.kept_turned_rows + fresh_alg)
                                    : L2 * (rope_bytes * counts.kept_turned_rows + row_bytes * fresh_alg);
        st.moved_bytes = st.algorithmic_bytes + L2 * row_bytes * counts.fresh_head_rows;
        st.timed_kernel_bytes =
            plan->total_tiles > 0 ? L2 * rope_bytes * counts.kept_turned_rows : st.algorithmic_bytes;
    } else {
        st.algorithmic_bytes = L2 * row_bytes * (st.downstream_slots + st.repl_slots);
        st.moved_bytes = L2 * row_bytes * (st.downstream_slots + st.repl_slots + st.head_slots);
        st.timed_kernel_bytes = st.algorithmic_bytes;
    }
    st.pages_popped = plan->total_pop;
    st.pages_pushed = plan->total_push;
    st.requests_touched = (int32_t)plan->reqs.size();
    // rewrite: move+rotate and commit; re-index: prep with the rows of R (one launch), other
    // fresh rows, the in-place rotation, commit (each if any).  A plan that leyline_splice
    // uploads adds its copy kernel (counted there).
    st.kernels_launched = plan->reqs.empty() ? 0
                          : reindex ? (plan->total_prep + plan->total_repl > 0) + (plan->total_fresh > 0) +
                                          (plan->total_tiles > 0) + (plan->total_commit > 0)
                                    : (plan->total_tiles > 0) + (plan->total_commit > 0);
    st.reindexed = (!plan->reqs.empty() && reindex) ? 1 : 0;
    return LEYLINE_OK;
}

bool plan_fits_params(const Plan& plan)
{
    return plan.reqs.size() <= (size_t)kParamReqs && plan.segs.size() <= (size_t)kParamSegs &&
           plan.trig.size() <= (size_t)kParamTrigFloats;
}

void pack_param_plan(const Plan& plan, ParamPlan* pp)
{
    std::memset(pp, 0, sizeof *pp);
    std::copy(plan.reqs.begin(), plan.reqs.end(), pp->reqs);
    std::copy(plan.segs.begin(), plan.segs.end(), pp->segs);
    std::copy(plan.trig.begin(), plan.trig.end(), pp->trig);
}

}  // namespace leyline
