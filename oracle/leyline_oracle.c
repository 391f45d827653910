/*
 * leyline_oracle.c -- plain fp64 CPU statement of the Leyline AMORTIZE splice.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file.  It shares no code, header, table or constant
 * with the GPU library, and the GPU library never calls it.
 *
 * Source: "Leyline: KV Cache Directives for Agentic Inference" (technical
 * summary of arXiv 2606.01065):
 *   - section 2.1 (directive abstraction): D = (s_start, s_end, R, m); the span
 *     [s_start, s_end) is replaced by the token sequence R; mode AMORTIZE splices
 *     in place, re-indexes downstream positions and keeps K_nope and V.
 *   - section 2.2 (delta-rotation): Delta = |R| - |S|; every downstream slot gets
 *     K_pe_new = R(Delta) K_pe; by R(a)R(b) = R(a+b) this equals encoding the
 *     token from scratch at position i + Delta.
 *   - section 2.3 (serving-stack integration): the prefix [0, s_start) is kept,
 *     R is prefilled into new slots, the rotation kernel re-indexes and rotates
 *     every downstream slot.
 *
 * What this oracle computes is the plain definition that the delta-rotation
 * reaches exactly (section 2.2): the new logical cache is
 *     old[0:s_start] ++ R ++ old[s_end:L]
 * with every surviving token re-encoded from scratch at its new position p: its
 * stored bf16 k_pe is taken to fp64, rotated back by R(-t) from its old position
 * t and forward by R(p), then rounded once to bf16 (round to nearest even).
 * Latents, prefix rows and the rows of R are copied bit for bit.
 *
 * Readings where the pages are silent (each is stated again where it is used):
 *   - RoPE pairs: half-split (j, j + d/2) by default, interleaved (2j, 2j+1)
 *     optionally; theta_j = theta^(-2j/d); R(p) turns pair j by +p*theta_j with
 *     x' = x cos - y sin, y' = x sin + y cos.
 *   - Several directives of one request are non-overlapping spans in the
 *     pre-call coordinates with distinct s_start; they are applied one at a
 *     time, right to left, so that earlier coordinates stay valid.
 *   - Rows of R arrive already encoded at their final positions (prefill,
 *     section 2.3) and are copied as they are.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 ---- */

/* bf16 bits -> value.  bf16 is the upper half of an IEEE binary32. */
double lo_bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (ties to even).  bf16 keeps 8 significant
 * bits and the binary32 exponent range; below 2^-126 the spacing is 2^-133.
 * The rounding decision is taken in fp64 by nearbyint (default mode: nearest,
 * ties to even); the rounded value has at most 8 significant bits, so the final
 * conversion to float is exact and only serves to read off the bit pattern. */
uint16_t lo_bf16_round(double x)
{
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (ax == 0.0) return sign;
    if (isinf(ax)) return (uint16_t)(sign | 0x7F80);
    double r;
    if (ax >= ldexp(1.0, -126)) {
        int e;
        double m = frexp(ax, &e);                 /* ax = m * 2^e, 0.5 <= m < 1 */
        r = ldexp(nearbyint(ldexp(m, 8)), e - 8); /* 8 significant bits */
    } else {
        r = ldexp(nearbyint(ldexp(ax, 133)), -133);
    }
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80); /* overflow -> inf */
    float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

void lo_bf16_round_array(const double* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = lo_bf16_round(x[i]);
}

void lo_bf16_value_array(const uint16_t* h, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = lo_bf16_value(h[i]);
}

/* ---------------------------------------------------------------- RoPE ---- */

/* Pair index pair (ix, iy) of pair j in a rope band of width d. */
static void lo_pair(int layout, int d, int j, int* ix, int* iy)
{
    if (layout == 0) { *ix = j; *iy = j + d / 2; }  /* half-split */
    else             { *ix = 2 * j; *iy = 2 * j + 1; } /* interleaved */
}

/* theta_j = theta^(-2j/d). */
double lo_theta_j(int j, int d, double theta)
{
    return pow(theta, -2.0 * (double)j / (double)d);
}

/* out = R(pos) in: turn each pair j by the angle pos * theta_j (section 2.2:
 * RoPE is a unitary rotation with R(a)R(b) = R(a+b)).  fp64 throughout. */
void lo_rope(const double* in, int d, double pos, double theta, int layout, double* out)
{
    for (int j = 0; j < d / 2; ++j) {
        int ix, iy;
        lo_pair(layout, d, j, &ix, &iy);
        double a = pos * lo_theta_j(j, d, theta);
        double c = cos(a), s = sin(a);
        double x = in[ix], y = in[iy];
        out[ix] = x * c - y * s;
        out[iy] = x * s + y * c;
    }
}

/* Re-encode one stored bf16 k_pe band from position `from` to position `to`:
 * bf16 -> fp64, R(-from), R(to), round once to bf16.  n_rows bands of width d,
 * contiguous.  Section 2.2: applying R(Delta) to R(i) x equals R(i + Delta) x. */
void lo_rerotate(const uint16_t* kpe_in, int64_t n_rows, int d, const int64_t* from, const int64_t* to,
                 double theta, int layout, uint16_t* kpe_out)
{
    double* v = (double*)malloc(sizeof(double) * 3 * (size_t)d);
    double* u = v + d;
    double* w = u + d;
    for (int64_t r = 0; r < n_rows; ++r) {
        const uint16_t* in = kpe_in + r * d;
        uint16_t* out = kpe_out + r * d;
        if (from[r] == to[r]) { memcpy(out, in, sizeof(uint16_t) * (size_t)d); continue; }
        for (int i = 0; i < d; ++i) v[i] = lo_bf16_value(in[i]);
        lo_rope(v, d, -(double)from[r], theta, layout, u);
        lo_rope(u, d, (double)to[r], theta, layout, w);
        for (int i = 0; i < d; ++i) out[i] = lo_bf16_round(w[i]);
    }
    free(v);
}

/* The naive bf16-only delta-rotation, the comparison arm of the drift study
 * (section 4.3: the drift of delta-rotation in bf16, which computing the
 * rotation in fp32 mitigates).  Reading: cos and sin of delta*theta_j are rounded
 * to bf16, each product is rounded to bf16, and the difference / sum of the two
 * rounded products is rounded to bf16. */
void lo_rotate_bf16only(const uint16_t* kpe_in, int64_t n_rows, int d, const int64_t* delta,
                        double theta, int layout, uint16_t* kpe_out)
{
    for (int64_t r = 0; r < n_rows; ++r) {
        const uint16_t* in = kpe_in + r * d;
        uint16_t* out = kpe_out + r * d;
        for (int j = 0; j < d / 2; ++j) {
            int ix, iy;
            lo_pair(layout, d, j, &ix, &iy);
            double a = (double)delta[r] * lo_theta_j(j, d, theta);
            double c = lo_bf16_value(lo_bf16_round(cos(a)));
            double s = lo_bf16_value(lo_bf16_round(sin(a)));
            double x = lo_bf16_value(in[ix]), y = lo_bf16_value(in[iy]);
            double xc = lo_bf16_value(lo_bf16_round(x * c));
            double ys = lo_bf16_value(lo_bf16_round(y * s));
            double xs = lo_bf16_value(lo_bf16_round(x * s));
            double yc = lo_bf16_value(lo_bf16_round(y * c));
            out[ix] = lo_bf16_round(xc - ys);
            out[iy] = lo_bf16_round(xs + yc);
        }
    }
}

/* ------------------------------------------------------------- splice ---- */

/* Logical splice of one request of length L (section 2.1, AMORTIZE): the new
 * token list is built by applying the n directives right to left, each as
 * list = list[0:s] ++ R ++ list[e:].  Entry p of the result says where new
 * position p comes from: kind 0 = original token idx[p]; kind 1 = row idx[p] of
 * the replacement rows of directive which[p].
 * Returns the new length, or -1 if a directive is out of range, the spans overlap
 * or share an s_start, or the result does not fit in `cap`. */
int64_t lo_splice_map(int64_t L, int32_t n, const int64_t* s_start, const int64_t* s_end,
                      const int32_t* n_repl, int64_t cap, int32_t* kind, int64_t* idx, int32_t* which)
{
    if (L < 0 || n < 0) return -1;
    int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    for (int32_t k = 0; k < n; ++k) {
        if (s_start[k] < 0 || s_start[k] > s_end[k] || s_end[k] > L || n_repl[k] < 0) { free(order); return -1; }
        order[k] = k;
    }
    /* insertion sort by s_start */
    for (int32_t a = 1; a < n; ++a) {
        int32_t v = order[a], b = a - 1;
        while (b >= 0 && s_start[order[b]] > s_start[v]) { order[b + 1] = order[b]; --b; }
        order[b + 1] = v;
    }
    for (int32_t a = 0; a + 1 < n; ++a) {
        if (s_start[order[a + 1]] == s_start[order[a]] || s_end[order[a]] > s_start[order[a + 1]]) {
            free(order);
            return -1;
        }
    }
    if (L > cap) { free(order); return -1; }
    int64_t len = L;
    for (int64_t t = 0; t < L; ++t) { kind[t] = 0; idx[t] = t; which[t] = -1; }
    for (int32_t a = n - 1; a >= 0; --a) {
        int32_t k = order[a];
        int64_t s = s_start[k], e = s_end[k], r = n_repl[k];
        int64_t newlen = len - (e - s) + r;
        if (newlen > cap) { free(order); return -1; }
        /* move the tail list[e:len] to start at s + r */
        memmove(kind + s + r, kind + e, sizeof(int32_t) * (size_t)(len - e));
        memmove(idx + s + r, idx + e, sizeof(int64_t) * (size_t)(len - e));
        memmove(which + s + r, which + e, sizeof(int32_t) * (size_t)(len - e));
        for (int64_t i = 0; i < r; ++i) { kind[s + i] = 1; idx[s + i] = i; which[s + i] = k; }
        len = newlen;
    }
    free(order);
    return len;
}

/* Rotation of a surviving token t: the summed Delta of the directives left of it
 * (s_end <= t) whose mode turns positions.  Mode 0 (AMORTIZE, "Leyline: KV Cache
 * Directives for Agentic Inference" section 2.1) re-indexes and re-encodes the
 * downstream tokens; mode 2 (EVICT, the KV-streams page: evict without resetting
 * positions) re-indexes them but keeps the positions they were encoded at.
 * modes == NULL means every directive is AMORTIZE. */
static int64_t lo_turn_of(int64_t t, int32_t n, const int64_t* s_start, const int64_t* s_end,
                          const int32_t* n_repl, const int32_t* modes)
{
    int64_t a = 0;
    for (int32_t k = 0; k < n; ++k)
        if (s_end[k] <= t && (!modes || modes[k] == 0))
            a += (int64_t)n_repl[k] - (s_end[k] - s_start[k]);
    return a;
}

/* Splice the whole logical cache of one request.
 *   cache_in  : bf16 [num_layers][L][row], row = latent_dim + rope_dim, k_pe last
 *   repl[k]   : bf16 [num_layers][n_repl[k]][row], rows of R for directive k
 *   cache_out : bf16 [num_layers][cap][row]
 * Latents, prefix rows and R rows are copied bit for bit; k_pe of a surviving
 * token moved from t to p is re-encoded from scratch (lo_rerotate).  Returns the
 * new length or -1 (as lo_splice_map). */
int64_t lo_splice_request_heads(int num_layers, int latent_dim, int rope_dim, int rope_heads, double theta,
                                int layout, const uint16_t* cache_in, int64_t L, int32_t n,
                                const int64_t* s_start, const int64_t* s_end, const int32_t* n_repl,
                                const int32_t* modes, const uint16_t* const* repl, uint16_t* cache_out,
                                int64_t cap);

int64_t lo_splice_request_modes(int num_layers, int latent_dim, int rope_dim, double theta, int layout,
                                const uint16_t* cache_in, int64_t L, int32_t n, const int64_t* s_start,
                                const int64_t* s_end, const int32_t* n_repl, const int32_t* modes,
                                const uint16_t* const* repl, uint16_t* cache_out, int64_t cap)
{
    return lo_splice_request_heads(num_layers, latent_dim, rope_dim, 1, theta, layout, cache_in, L, n, s_start,
                                   s_end, n_repl, modes, repl, cache_out, cap);
}

int64_t lo_splice_request(int num_layers, int latent_dim, int rope_dim, double theta, int layout,
                          const uint16_t* cache_in, int64_t L, int32_t n, const int64_t* s_start,
                          const int64_t* s_end, const int32_t* n_repl, const uint16_t* const* repl,
                          uint16_t* cache_out, int64_t cap)
{
    return lo_splice_request_modes(num_layers, latent_dim, rope_dim, theta, layout, cache_in, L, n, s_start, s_end,
                                   n_repl, NULL, repl, cache_out, cap);
}

/* As lo_splice_request, with a mode per directive (see lo_turn_of): a surviving
 * token t is re-encoded from position t to position t + turn(t).  The row ends
 * in rope_heads RoPE bands of width rope_dim (the keys of rope_heads attention
 * heads, the GQA/MHA extension named in section 5 of the Leyline page); each band
 * is re-encoded on its own.  rope_heads = 1 is the MLA row (latent, then k_pe). */
int64_t lo_splice_request_heads(int num_layers, int latent_dim, int rope_dim, int rope_heads, double theta,
                                int layout, const uint16_t* cache_in, int64_t L, int32_t n,
                                const int64_t* s_start, const int64_t* s_end, const int32_t* n_repl,
                                const int32_t* modes, const uint16_t* const* repl, uint16_t* cache_out,
                                int64_t cap)
{
    const int row = latent_dim + rope_heads * rope_dim;
    int32_t* kind = (int32_t*)malloc(sizeof(int32_t) * (size_t)(cap > 0 ? cap : 1));
    int64_t* idx = (int64_t*)malloc(sizeof(int64_t) * (size_t)(cap > 0 ? cap : 1));
    int32_t* which = (int32_t*)malloc(sizeof(int32_t) * (size_t)(cap > 0 ? cap : 1));
    int64_t newlen = lo_splice_map(L, n, s_start, s_end, n_repl, cap, kind, idx, which);
    if (newlen >= 0) {
        for (int l = 0; l < num_layers; ++l) {
            for (int64_t p = 0; p < newlen; ++p) {
                uint16_t* dst = cache_out + ((int64_t)l * cap + p) * row;
                if (kind[p] == 1) {
                    int32_t k = which[p];
                    const uint16_t* src = repl[k] + ((int64_t)l * n_repl[k] + idx[p]) * row;
                    memcpy(dst, src, sizeof(uint16_t) * (size_t)row);
                } else {
                    int64_t t = idx[p];
                    int64_t to = t + lo_turn_of(t, n, s_start, s_end, n_repl, modes);
                    const uint16_t* src = cache_in + ((int64_t)l * L + t) * row;
                    memcpy(dst, src, sizeof(uint16_t) * (size_t)latent_dim);
                    for (int h = 0; h < rope_heads; ++h)
                        lo_rerotate(src + latent_dim + h * rope_dim, 1, rope_dim, &t, &to, theta, layout,
                                    dst + latent_dim + h * rope_dim);
                }
            }
        }
    }
    free(kind);
    free(idx);
    free(which);
    return newlen;
}
