// planner_sanitize.cpp -- a fuzz driver for the host planner (leyline_planner.cpp), built by
// tests/test_planner_sanitizers.py with AddressSanitizer and UndefinedBehaviorSanitizer.
//
// The planner reads caller-supplied directives, lengths and pool descriptors.  This driver
// feeds it seeded random ones, valid and invalid (negative and out-of-range spans,
// overlapping spans, unknown modes and flags, lengths past the table's capacity, a pool with
// few free pages), and on every accepted call checks what the plan promises:
//   - each touched request's new length is its old length plus the summed |R| - |S| of its
//     effective directives ("Leyline: KV Cache Directives for Agentic Inference", section 2.2);
//   - its segments and their index ranges lie inside the plan's arrays;
//   - a rewrite takes one fresh page per block from the first rewritten one on, and returns
//     the old ones; no plan takes more pages than are free;
//   - a plan small enough for a kernel parameter packs without overrunning it.
// The sanitizers turn any out-of-bounds access, overflow or misaligned read into a failure.
// Exit code 0: every check held.  Usage: planner_sanitize <iterations> <seed>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "leyline_internal.h"

using namespace leyline;

namespace {

uint64_t g_state = 0;

uint64_t next_u64()
{
    uint64_t z = (g_state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

int64_t uniform(int64_t lo, int64_t hi)  // inclusive
{
    return lo + (int64_t)(next_u64() % (uint64_t)(hi - lo + 1));
}

bool chance(int percent) { return uniform(0, 99) < percent; }

int failures = 0;

void fail(long iter, const char* what)
{
    std::fprintf(stderr, "iteration %ld: %s\n", iter, what);
    ++failures;
}

}  // namespace

int main(int argc, char** argv)
{
    const long iters = argc > 1 ? std::atol(argv[1]) : 20000;
    g_state = argc > 2 ? (uint64_t)std::atoll(argv[2]) : 1;
    long accepted = 0, refused = 0;
    static const int32_t kLatent[] = {0, 64, 128, 512};
    static const int32_t kRope[] = {16, 32, 64, 128};
    static const int32_t kBlock[] = {1, 2, 4, 16};
    // a 16-byte aligned stand-in for rows of R: the planner stores it and never reads it
    alignas(16) static unsigned char fake_rows[16];
    for (long it = 0; it < iters; ++it) {
        leyline_pool_desc_t d{};
        d.num_layers = (int32_t)uniform(chance(2) ? -1 : 1, 4);
        d.latent_dim = kLatent[uniform(0, 3)] + (chance(2) ? 4 : 0);
        d.rope_dim = kRope[uniform(0, 3)] + (chance(2) ? 8 : 0);
        d.block_size = kBlock[uniform(0, 3)] * (chance(2) ? 0 : 1);
        d.num_pages = chance(2) ? 0 : uniform(1, 1 << 20);
        d.rope_theta = chance(2) ? -1.0 : 10000.0;
        d.pair_layout = (int32_t)uniform(0, chance(3) ? 2 : 1);
        d.rotate_precision = (int32_t)uniform(0, chance(3) ? 2 : 1);
        d.flags = (uint32_t)uniform(0, chance(3) ? 15 : 7);
        d.rope_heads = (int32_t)uniform(0, chance(3) ? 2000 : 4);
        Geometry g{};
        if (make_geometry(&d, &g) != LEYLINE_OK) {
            ++refused;
            continue;
        }
        const int32_t B = g.block_size;
        const int32_t num_reqs = (int32_t)uniform(0, 4);
        std::vector<int64_t> lens(num_reqs > 0 ? num_reqs : 1);
        int64_t longest = 0;
        for (int32_t r = 0; r < num_reqs; ++r) {
            lens[r] = uniform(0, 300);
            longest = lens[r] > longest ? lens[r] : longest;
        }
        int32_t max_blocks = (int32_t)((longest + 200 + B - 1) / B);
        if (chance(10)) max_blocks = (int32_t)((longest + B - 1) / B);  // no room to grow
        const int32_t n = (int32_t)uniform(0, 6);
        std::vector<leyline_directive_t> dirs(n > 0 ? n : 1);
        for (int32_t k = 0; k < n; ++k) {
            leyline_directive_t& x = dirs[k];
            x.req = (int32_t)uniform(chance(3) ? -1 : 0, num_reqs > 0 ? num_reqs - (chance(3) ? 0 : 1) : 0);
            const int64_t L = (x.req >= 0 && x.req < num_reqs) ? lens[x.req] : 10;
            x.mode = chance(5) ? (int32_t)uniform(1, 9) : (chance(20) ? LEYLINE_EVICT : LEYLINE_AMORTIZE);
            x.s_start = uniform(chance(3) ? -5 : 0, L + (chance(3) ? 5 : 0));
            x.s_end = x.s_start + uniform(chance(3) ? -3 : 0, 80);
            x.n_repl = (int32_t)uniform(chance(3) ? -2 : 0, 40);
            x.reserved = chance(2) ? 1 : 0;
            x.repl_rows = chance(3) ? nullptr : fake_rows;
        }
        const int64_t free_pages = chance(20) ? uniform(0, 40) : -1;
        Plan plan;
        const int rc = build_plan(g, lens.data(), num_reqs, max_blocks, dirs.data(), n, free_pages, &plan);
        if (rc != LEYLINE_OK) {
            ++refused;
            continue;
        }
        ++accepted;
        // new lengths: old length plus the summed Delta of the request's effective directives
        std::vector<int64_t> want(lens.begin(), lens.begin() + (num_reqs > 0 ? num_reqs : 0));
        for (int32_t k = 0; k < n; ++k)
            want[dirs[k].req] += dirs[k].n_repl - (dirs[k].s_end - dirs[k].s_start);
        int64_t pops = 0, pushes = 0;
        for (const ReqPlan& rp : plan.reqs) {
            if (rp.req < 0 || rp.req >= num_reqs) {
                fail(it, "plan names a request outside the table");
                continue;
            }
            if (rp.old_len != lens[rp.req] || rp.new_len != want[rp.req]) fail(it, "wrong lengths");
            if (rp.new_len > (int64_t)max_blocks * B) fail(it, "new length past the table's capacity");
            if (rp.seg_begin < 0 || rp.seg_count < 0 || (size_t)rp.seg_begin + (size_t)rp.seg_count > plan.segs.size())
                fail(it, "segments outside the plan");
            if (rp.b0 < 0 || (int64_t)rp.b0 * B > rp.old_len) fail(it, "first rewritten block past the old end");
            if (rp.n_new < 0 || rp.n_old < 0) fail(it, "negative page counts");
            if (!plan.reindex) {  // a rewrite takes a fresh page for every block from b0 on
                if (rp.n_new != (rp.new_len + B - 1) / B - rp.b0 || rp.n_old != (rp.old_len + B - 1) / B - rp.b0)
                    fail(it, "rewritten block counts");
                pops += rp.n_new;
                pushes += rp.n_old;
            }
            for (int32_t q = 0; q < rp.seg_count && (size_t)(rp.seg_begin + q) < plan.segs.size(); ++q) {
                const Seg& s = plan.segs[rp.seg_begin + q];
                if (s.kind == SEG_ROT && (s.trig < 0 || s.trig >= plan.n_trig)) fail(it, "rotated segment without trig");
                if (s.kind == SEG_REPL && (s.n_repl <= 0 || !s.repl)) fail(it, "empty or rowless R segment");
            }
        }
        if (!plan.reindex && (plan.total_pop != pops || plan.total_push != pushes)) fail(it, "page totals");
        if ((int64_t)plan.trig.size() != (int64_t)plan.n_trig * g.rope_dim) fail(it, "trig table size");
        if (plan.total_pop < 0 || plan.total_push < 0) fail(it, "negative page totals");
        if (free_pages >= 0 && plan.total_pop > free_pages) fail(it, "takes more pages than are free");
        if (plan.stats.algorithmic_bytes < 0 || plan.stats.timed_kernel_bytes < 0 ||
            plan.stats.timed_kernel_bytes > plan.stats.algorithmic_bytes)
            fail(it, "byte accounting");
        if (plan_fits_params(plan)) {
            ParamPlan* pp = new ParamPlan;
            pack_param_plan(plan, pp);
            delete pp;
        }
    }
    std::printf("%ld calls planned, %ld refused, %d failed checks\n", accepted, refused, failures);
    return failures == 0 ? 0 : 1;
}
