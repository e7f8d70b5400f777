/*
 * kvi_oracle.c -- plain, slow, single-threaded float64 CPU oracle for the
 * retrieve-and-inject path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) includes, links or calls this file; only the tests,
 * the smoke check and the benchmark's CPU-baseline leg do.  It shares no code,
 * header, table or constant with the CUDA path.
 *
 * What it follows (page: "InferScale: GPU-Native KV Injection for
 * Personalized LLM Serving", the pith.science review of arXiv 2607.27090):
 *   - Figure 2 caption: each fact has a retrieval embedding and a pre-RoPE K/V
 *     tensor under one fact_id; at serving time the top-k retrieved facts are
 *     resolved to their KV and positioned by Chunked RoPE.
 *   - Section 5.1 / Theorem 6 (Chunked RoPE): keys are stored before rotary
 *     encoding and rotated to their serving positions on injection; exact
 *     relocation follows from R_a^T R_b = R_{b-a}.
 *   - Section 3.4 (KV-connector premise): K/V are scatter-copied into the
 *     engine's paged blocks (vLLM PagedAttention layout) before the forward
 *     pass.
 *
 * Readings where the page is silent (each one is listed with its reason in the
 * design notes):
 *   - similarity is the plain dot product (equal to cosine for the unit-norm
 *     embeddings used), computed exactly up to float64 rounding; the exact
 *     scan stands in for the paper's approximate GPU index;
 *   - top-k order is the total order (score descending, fact id ascending);
 *   - rotary pairing is rotate-half: element i pairs with i + D/2, with
 *     frequency omega_i = theta^(-2i/D) (RoFormer frequencies, no scaling);
 *     the variants below (interleaved pairing, Llama 3.1 frequency scaling,
 *     a caller's cos/sin table) are the other conventions an engine may use;
 *   - facts are placed contiguously in rank order from a start position.
 *
 * Every function below is pinned by the CPU tests against closed forms,
 * invariants or brute force; none is checked only against itself.
 *
 * Build: plain C11, -ffp-contract=off so that no multiply-add is fused and
 * the results are the same on x86-64 and aarch64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status codes returned by the oracle (independent of the library's own). */
enum { KVO_OK = 0, KVO_BAD_ARG = 1, KVO_OUT_OF_RANGE = 2, KVO_CAPACITY = 3 };
/* Rotary pairings (see kvo_pair). */
enum { KVO_PAIR_HALF = 0, KVO_PAIR_INTERLEAVED = 1 };

/* bf16 -> double: a bf16 value is the upper 16 bits of an IEEE binary32. */
double kvo_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Step 1, scores.  s_i = sum_j q_j * e_ij, summed left to right in float64,
 * for every fact i < n.  The embeddings are the "retrieval space" of the
 * Figure 2 caption; the dot product is the similarity (reading above). */
void kvo_scores(const float *q, const float *emb, int64_t n, int64_t e,
                double *out)
{
    for (int64_t i = 0; i < n; ++i) {
        const float *row = emb + i * e;
        double s = 0.0;
        for (int64_t j = 0; j < e; ++j)
            s += (double)q[j] * (double)row[j];
        out[i] = s;
    }
}

typedef struct { double s; int32_t id; } kvo_key;

/* (score descending, id ascending): a total order over distinct ids. */
static int kvo_key_cmp(const void *a, const void *b)
{
    const kvo_key *x = (const kvo_key *)a, *y = (const kvo_key *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->id > y->id) - (x->id < y->id);
}

/* Step 2, select.  Sort all ids by (score descending, id ascending) and keep
 * the first k; sel[] receives them in rank order.  "Top-k retrieved facts"
 * of the Figure 2 caption, taken exactly.  Returns KVO_BAD_ARG for k <= 0 or
 * k > n. */
int kvo_topk(const double *s, int64_t n, int32_t k, int32_t *sel)
{
    if (k <= 0 || (int64_t)k > n) return KVO_BAD_ARG;
    kvo_key *keys = (kvo_key *)malloc((size_t)n * sizeof *keys);
    if (!keys) return KVO_BAD_ARG;
    for (int64_t i = 0; i < n; ++i) { keys[i].s = s[i]; keys[i].id = (int32_t)i; }
    qsort(keys, (size_t)n, sizeof *keys, kvo_key_cmp);
    for (int32_t j = 0; j < k; ++j) sel[j] = keys[j].id;
    free(keys);
    return KVO_OK;
}

/* Step 3, place.  pos_0 = start, pos_{j+1} = pos_j + len[sel_j]: the facts
 * sit back to back in rank order from `start` (reading of the truncated
 * Figure 2 caption, "positioned by chunked RoPE").  Writes pos[0..k) and
 * returns the total number of tokens placed, or -1 if an id is out of range
 * or a length is negative. */
int64_t kvo_place(const int32_t *sel, int32_t k, const int32_t *fact_len,
                  int64_t n_facts, int64_t start, int64_t *pos)
{
    int64_t p = start;
    for (int32_t j = 0; j < k; ++j) {
        if (sel[j] < 0 || (int64_t)sel[j] >= n_facts) return -1;
        if (fact_len[sel[j]] < 0) return -1;
        pos[j] = p;
        p += fact_len[sel[j]];
    }
    return p - start;
}

/* Step 4, frequencies.  omega_i = theta^(-2i/D) for i < D/2. */
void kvo_rope_omega(double theta, int32_t d, double *omega)
{
    for (int32_t i = 0; i < d / 2; ++i)
        omega[i] = pow(theta, -2.0 * (double)i / (double)d);
}

/* Step 5, rotate one head vector x[D] to position p (Section 5.1, Chunked
 * RoPE; rotate-half pairing).  For each i < D/2, with a = p * omega_i:
 *   y_i       = x_i cos a - x_{i+D/2} sin a
 *   y_{i+D/2} = x_{i+D/2} cos a + x_i sin a
 * p is a double so that the relocation identity can be checked at any real
 * offset; the path itself uses integer positions. */
void kvo_rotate(const double *x, int32_t d, double theta, double p, double *y)
{
    const int32_t half = d / 2;
    for (int32_t i = 0; i < half; ++i) {
        const double w = pow(theta, -2.0 * (double)i / (double)d);
        const double a = p * w;
        const double c = cos(a), s = sin(a);
        const double x0 = x[i], x1 = x[i + half];
        y[i] = x0 * c - x1 * s;
        y[i + half] = x1 * c + x0 * s;
    }
}

/* Variants of step 4-5.  The pairing maps pair i to its two elements:
 *   KVO_PAIR_HALF        (i, i + D/2)   -- rotate-half, as kvo_rotate;
 *   KVO_PAIR_INTERLEAVED (2i, 2i + 1)   -- GPT-J / RoFormer's original form.
 * Element a of pair i is the one multiplied by cos in its own output:
 *   y_a = x_a cos - x_b sin,   y_b = x_b cos + x_a sin. */
static void kvo_pair(int32_t pairing, int32_t d, int32_t i, int32_t *a, int32_t *b)
{
    if (pairing == KVO_PAIR_INTERLEAVED) {
        *a = 2 * i;
        *b = 2 * i + 1;
    } else {
        *a = i;
        *b = i + d / 2;
    }
}

/* Rotate x[D] to position p with explicit per-pair frequencies omega[D/2]. */
void kvo_rotate_pairs(const double *x, int32_t d, const double *omega, int32_t pairing,
                      double p, double *y)
{
    for (int32_t i = 0; i < d / 2; ++i) {
        int32_t ia, ib;
        kvo_pair(pairing, d, i, &ia, &ib);
        const double ang = p * omega[i];
        const double c = cos(ang), sn = sin(ang);
        y[ia] = x[ia] * c - x[ib] * sn;
        y[ib] = x[ib] * c + x[ia] * sn;
    }
}

/* Rotate x[D] by given cos/sin values of each pair (a caller's table row):
 * the exact rotation with those coefficients. */
void kvo_rotate_cs(const double *x, int32_t d, const double *c, const double *sn,
                   int32_t pairing, double *y)
{
    for (int32_t i = 0; i < d / 2; ++i) {
        int32_t ia, ib;
        kvo_pair(pairing, d, i, &ia, &ib);
        y[ia] = x[ia] * c[i] - x[ib] * sn[i];
        y[ib] = x[ib] * c[i] + x[ia] * sn[i];
    }
}

/* Llama 3.1 frequency scaling of omega_i = theta^(-2i/D) (the published
 * "llama3" rope scaling, restated): with wavelength lambda = 2 pi / omega,
 * a component whose wavelength is shorter than orig / high keeps omega, one
 * longer than orig / low is slowed down to omega / factor, and in between
 * the two are blended with weight g = (orig / lambda - low) / (high - low):
 *   omega' = (1 - g) omega / factor + g omega. */
void kvo_rope_omega_llama3(double theta, int32_t d, double factor, double low,
                           double high, double orig, double *omega)
{
    const double two_pi = 2.0 * acos(-1.0);
    kvo_rope_omega(theta, d, omega);
    for (int32_t i = 0; i < d / 2; ++i) {
        const double w = omega[i];
        const double lambda = two_pi / w;
        if (lambda < orig / high) {
            omega[i] = w;
        } else if (lambda > orig / low) {
            omega[i] = w / factor;
        } else {
            const double g = (orig / lambda - low) / (high - low);
            omega[i] = (1.0 - g) * w / factor + g * w;
        }
    }
}

/* Paged slot of token position p: block table entry p div B, offset p mod B
 * (vLLM PagedAttention layout behind the Section 3.4 scatter-copy).  Returns
 * KVO_OUT_OF_RANGE if p lies beyond the table or the entry is not a block of
 * the pool. */
int kvo_slot(int64_t p, const int32_t *block_table, int32_t table_len,
             int32_t block_size, int32_t num_blocks, int32_t *blk, int32_t *off)
{
    if (p < 0 || block_size <= 0) return KVO_OUT_OF_RANGE;
    const int64_t e = p / block_size;
    if (e >= table_len) return KVO_OUT_OF_RANGE;
    const int32_t b = block_table[e];
    if (b < 0 || b >= num_blocks) return KVO_OUT_OF_RANGE;
    *blk = b;
    *off = (int32_t)(p % block_size);
    return KVO_OK;
}

/* Expected rows of one injected token: store row `row`, at position p.
 * Store layout kv[L][2][n_tokens][H][D] (bf16 bits).
 *   k_out[L][H][D]: float64 rotated K (unrounded),
 *   v_out[L][H][D]: V bits, copied unchanged.
 * The rotation: with cos_tab/sin_tab (float32 [tab_positions][D/2]) the
 * table row p; otherwise the frequencies omega[D/2]; pairs per `pairing`.
 * Returns KVO_OUT_OF_RANGE if the row lies outside the store or p outside
 * the table. */
int kvo_token_rows_ex(const uint16_t *kv, int32_t L, int32_t H, int32_t D,
                      int64_t n_tokens, int64_t row, const double *omega,
                      int32_t pairing, const float *cos_tab, const float *sin_tab,
                      int64_t tab_positions, int64_t p, double *k_out, uint16_t *v_out)
{
    if (row < 0 || row >= n_tokens) return KVO_OUT_OF_RANGE;
    if (cos_tab && (p < 0 || p >= tab_positions)) return KVO_OUT_OF_RANGE;
    double *x = (double *)malloc((size_t)D * sizeof *x);
    double *c = (double *)malloc((size_t)D * sizeof *c);
    double *sn = (double *)malloc((size_t)D * sizeof *sn);
    if (!x || !c || !sn) { free(x); free(c); free(sn); return KVO_BAD_ARG; }
    if (cos_tab) {
        for (int32_t i = 0; i < D / 2; ++i) {
            c[i] = (double)cos_tab[p * (D / 2) + i];
            sn[i] = (double)sin_tab[p * (D / 2) + i];
        }
    }
    const int64_t hd = (int64_t)H * D;
    for (int32_t l = 0; l < L; ++l) {
        const uint16_t *krow = kv + (((int64_t)l * 2 + 0) * n_tokens + row) * hd;
        const uint16_t *vrow = kv + (((int64_t)l * 2 + 1) * n_tokens + row) * hd;
        for (int32_t h = 0; h < H; ++h) {
            for (int32_t i = 0; i < D; ++i)
                x[i] = kvo_bf16_to_double(krow[(int64_t)h * D + i]);
            double *y = k_out + ((int64_t)l * H + h) * D;
            if (cos_tab) kvo_rotate_cs(x, D, c, sn, pairing, y);
            else kvo_rotate_pairs(x, D, omega, pairing, (double)p, y);
            for (int32_t i = 0; i < D; ++i)
                v_out[((int64_t)l * H + h) * D + i] = vrow[(int64_t)h * D + i];
        }
    }
    free(x);
    free(c);
    free(sn);
    return KVO_OK;
}

/* The plain reading: rotate-half with omega_i = theta^(-2i/D). */
int kvo_token_rows(const uint16_t *kv, int32_t L, int32_t H, int32_t D,
                   int64_t n_tokens, int64_t row, double theta, int64_t p,
                   double *k_out, uint16_t *v_out)
{
    double *omega = (double *)malloc((size_t)(D / 2 + 1) * sizeof *omega);
    if (!omega) return KVO_BAD_ARG;
    kvo_rope_omega(theta, D, omega);
    const int rc = kvo_token_rows_ex(kv, L, H, D, n_tokens, row, omega, KVO_PAIR_HALF,
                                     NULL, NULL, 0, p, k_out, v_out);
    free(omega);
    return rc;
}

/* Step 6, expected cache for one request (Section 3.4 scatter-copy).
 *
 * Inputs: store kv bits [L][2][n_tokens][H][D]; per fact start row and length;
 * the injected facts `ids[n]` with their start positions `starts[n]`; the
 * request's block table; the pool geometry (num_blocks, block_size).
 *
 * Outputs, both laid out like the pool [L][2][num_blocks][B][H][D]:
 *   expect[]  float64 expected value of every written element,
 *   written[] 1 for every element the injection writes, 0 elsewhere (those
 *             elements must keep their pre-call contents).
 * A K element is the rotated pre-RoPE key at the token's position; a V
 * element is the stored bits read as a number.
 *
 * Returns KVO_OK, KVO_OUT_OF_RANGE (id, store row or slot out of range) or
 * KVO_CAPACITY (a slot written twice: overlapping positions). */
int kvo_inject_expected_ex(const uint16_t *kv, int32_t L, int32_t H, int32_t D,
                           int64_t n_tokens, const int64_t *fact_start,
                           const int32_t *fact_len, int64_t n_facts,
                           const int32_t *ids, const int64_t *starts, int32_t n,
                           const int32_t *block_table, int32_t table_len,
                           int32_t num_blocks, int32_t block_size, const double *omega,
                           int32_t pairing, const float *cos_tab, const float *sin_tab,
                           int64_t tab_positions, double *expect, uint8_t *written)
{
    const int64_t hd = (int64_t)H * D;
    const int64_t tok_per_kv = (int64_t)num_blocks * block_size;
    const int64_t n_el = (int64_t)L * 2 * tok_per_kv * hd;
    memset(written, 0, (size_t)n_el);
    for (int64_t e = 0; e < n_el; ++e) expect[e] = 0.0;

    double *kr = (double *)malloc((size_t)(L * hd) * sizeof *kr);
    uint16_t *vr = (uint16_t *)malloc((size_t)(L * hd) * sizeof *vr);
    if (!kr || !vr) { free(kr); free(vr); return KVO_BAD_ARG; }
    int rc = KVO_OK;
    for (int32_t j = 0; j < n && rc == KVO_OK; ++j) {
        const int32_t f = ids[j];
        if (f < 0 || (int64_t)f >= n_facts) { rc = KVO_OUT_OF_RANGE; break; }
        for (int32_t t = 0; t < fact_len[f]; ++t) {
            const int64_t p = starts[j] + t;
            int32_t blk, off;
            if (kvo_slot(p, block_table, table_len, block_size, num_blocks,
                         &blk, &off) != KVO_OK) { rc = KVO_OUT_OF_RANGE; break; }
            if (kvo_token_rows_ex(kv, L, H, D, n_tokens, fact_start[f] + t, omega, pairing,
                                  cos_tab, sin_tab, tab_positions, p, kr, vr) != KVO_OK) {
                rc = KVO_OUT_OF_RANGE;
                break;
            }
            for (int32_t l = 0; l < L; ++l) {
                for (int32_t c = 0; c < 2; ++c) {
                    const int64_t base =
                        ((((int64_t)l * 2 + c) * num_blocks + blk) * block_size + off) * hd;
                    if (written[base]) { rc = KVO_CAPACITY; break; }
                    for (int64_t x = 0; x < hd; ++x) {
                        written[base + x] = 1;
                        expect[base + x] = c == 0 ? kr[l * hd + x]
                                                  : kvo_bf16_to_double(vr[l * hd + x]);
                    }
                }
                if (rc != KVO_OK) break;
            }
            if (rc != KVO_OK) break;
        }
    }
    free(kr);
    free(vr);
    return rc;
}

/* The plain reading of kvo_inject_expected_ex: rotate-half, theta. */
int kvo_inject_expected(const uint16_t *kv, int32_t L, int32_t H, int32_t D,
                        int64_t n_tokens, const int64_t *fact_start,
                        const int32_t *fact_len, int64_t n_facts,
                        const int32_t *ids, const int64_t *starts, int32_t n,
                        const int32_t *block_table, int32_t table_len,
                        int32_t num_blocks, int32_t block_size, double theta,
                        double *expect, uint8_t *written)
{
    double *omega = (double *)malloc((size_t)(D / 2 + 1) * sizeof *omega);
    if (!omega) return KVO_BAD_ARG;
    kvo_rope_omega(theta, D, omega);
    const int rc = kvo_inject_expected_ex(kv, L, H, D, n_tokens, fact_start, fact_len,
                                          n_facts, ids, starts, n, block_table, table_len,
                                          num_blocks, block_size, omega, KVO_PAIR_HALF, NULL,
                                          NULL, 0, expect, written);
    free(omega);
    return rc;
}

/* The whole request as one call (steps 1-6), used to time the oracle as a
 * CPU baseline: score all facts, select the top k, place them from `start`,
 * and produce every injected token's rows.  k_out must hold
 * (sum of selected lengths) * L * H * D doubles and v_out as many uint16.
 * Returns the number of tokens produced, or -1 on error. */
int64_t kvo_request(const float *q, const float *emb, int64_t n_facts, int64_t e,
                    int32_t k, const uint16_t *kv, int32_t L, int32_t H, int32_t D,
                    int64_t n_tokens, const int64_t *fact_start,
                    const int32_t *fact_len, int64_t start, double theta,
                    int32_t *sel, int64_t *pos, double *k_out, uint16_t *v_out,
                    int64_t max_tokens)
{
    double *s = (double *)malloc((size_t)n_facts * sizeof *s);
    if (!s) return -1;
    kvo_scores(q, emb, n_facts, e, s);
    const int rc = kvo_topk(s, n_facts, k, sel);
    free(s);
    if (rc != KVO_OK) return -1;
    const int64_t T = kvo_place(sel, k, fact_len, n_facts, start, pos);
    if (T < 0 || T > max_tokens) return -1;
    const int64_t per_tok = (int64_t)L * H * D;
    int64_t tok = 0;
    for (int32_t j = 0; j < k; ++j) {
        for (int32_t t = 0; t < fact_len[sel[j]]; ++t, ++tok) {
            if (kvo_token_rows(kv, L, H, D, n_tokens, fact_start[sel[j]] + t,
                               theta, pos[j] + t, k_out + tok * per_tok,
                               v_out + tok * per_tok) != KVO_OK)
                return -1;
        }
    }
    return tok;
}

/* kvo_slot over n positions (for checking large pools): blk[i], off[i] of
 * position p[i], or -1/-1 when it is out of range. */
void kvo_slots(const int64_t *p, int64_t n, const int32_t *block_table,
               int32_t table_len, int32_t block_size, int32_t num_blocks,
               int32_t *blk, int32_t *off)
{
    for (int64_t i = 0; i < n; ++i) {
        if (kvo_slot(p[i], block_table, table_len, block_size, num_blocks,
                     &blk[i], &off[i]) != KVO_OK) {
            blk[i] = -1;
            off[i] = -1;
        }
    }
}

/* Parity check of many injected tokens at once (for pools too large for
 * kvo_inject_expected; test infrastructure like the rest of this file).
 *
 * src and got hold T tokens' rows in the store's layout [L][2][T][H][D]
 * (bf16 bits): src[.][.][t] the store rows token t was injected from, got
 * the pool rows the path under test wrote for it; pos[t] its position.
 * Only tokens t0 <= t < t1 are checked (callers split T over threads).
 *
 * Expected values are those of kvo_token_rows_ex: K is src's K rotated to
 * pos[t] (Section 5.1, Chunked RoPE) -- with the cos and sin of
 * pos[t] * omega_i, which depend on the position only and are therefore
 * computed once per token for all of its L * H rows, or with the caller's
 * table row pos[t] -- and V is src's V bits unchanged.  A K element counts
 * as bad when |got - y| > k_rel |y| + k_abs (y the float64 expected value);
 * a V element when its bits differ.  Outputs: bad_k, bad_v, and first_bad =
 * the flat index into [L][2][T][H][D] of the first bad element met, or -1.
 * Returns KVO_OK, KVO_OUT_OF_RANGE (a position outside the table) or
 * KVO_BAD_ARG. */
int kvo_check_rows(const uint16_t *src, const uint16_t *got, int32_t L, int32_t H,
                   int32_t D, int64_t T, int64_t t0, int64_t t1, const int64_t *pos,
                   const double *omega, int32_t pairing, const float *cos_tab,
                   const float *sin_tab, int64_t tab_positions, double k_rel,
                   double k_abs, int64_t *bad_k, int64_t *bad_v, int64_t *first_bad)
{
    *bad_k = 0;
    *bad_v = 0;
    *first_bad = -1;
    if (t0 < 0 || t1 > T || t0 > t1 || D < 2 || D % 2) return KVO_BAD_ARG;
    const int32_t half = D / 2;
    double *c = (double *)malloc((size_t)half * sizeof *c);
    double *sn = (double *)malloc((size_t)half * sizeof *sn);
    double *x = (double *)malloc((size_t)D * sizeof *x);
    double *y = (double *)malloc((size_t)D * sizeof *y);
    if (!c || !sn || !x || !y) { free(c); free(sn); free(x); free(y); return KVO_BAD_ARG; }
    int rc = KVO_OK;
    const int64_t hd = (int64_t)H * D;
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t p = pos[t];
        if (cos_tab) {
            if (p < 0 || p >= tab_positions) { rc = KVO_OUT_OF_RANGE; break; }
            for (int32_t i = 0; i < half; ++i) {
                c[i] = (double)cos_tab[p * half + i];
                sn[i] = (double)sin_tab[p * half + i];
            }
        } else {
            for (int32_t i = 0; i < half; ++i) {
                const double ang = (double)p * omega[i];
                c[i] = cos(ang);
                sn[i] = sin(ang);
            }
        }
        for (int32_t l = 0; l < L; ++l) {
            const int64_t kbase = (((int64_t)l * 2 + 0) * T + t) * hd;
            const int64_t vbase = (((int64_t)l * 2 + 1) * T + t) * hd;
            for (int32_t h = 0; h < H; ++h) {
                const int64_t at = kbase + (int64_t)h * D;
                for (int32_t i = 0; i < D; ++i) x[i] = kvo_bf16_to_double(src[at + i]);
                kvo_rotate_cs(x, D, c, sn, pairing, y);
                for (int32_t i = 0; i < D; ++i) {
                    const double g = kvo_bf16_to_double(got[at + i]);
                    if (!(fabs(g - y[i]) <= k_rel * fabs(y[i]) + k_abs)) {
                        if (*first_bad < 0) *first_bad = at + i;
                        ++*bad_k;
                    }
                }
            }
            for (int64_t e = 0; e < hd; ++e) {
                if (got[vbase + e] != src[vbase + e]) {
                    if (*first_bad < 0) *first_bad = vbase + e;
                    ++*bad_v;
                }
            }
        }
    }
    free(c);
    free(sn);
    free(x);
    free(y);
    return rc;
}

/* ------------------------------------------------------------------------
 * Graph index.  The review's Summary retrieves facts through a GPU ANN index
 * (Jasper) instead of a scan, and its Axiom & Free-Parameter Ledger fixes
 * the index at 64 graph neighbours and beam width 64; the reference list
 * cites CAGRA, a GPU graph index searched best-first from a candidate
 * buffer.  Readings (the pages give nothing more):
 *   - the graph links each fact to its `d` most similar other facts, exact,
 *     under the same (score descending, id ascending) order as the top-k;
 *   - the search keeps the best `beam` scored facts, expands the best
 *     `width` not yet expanded per iteration, scores every neighbour at most
 *     once (visited set) and starts from caller-given seed facts.
 * ---------------------------------------------------------------------- */

/* Graph build.  nbr[i][0..d) = the d facts j != i with the largest
 * s_ij = <e_i, e_j> (float64, summed left to right), in (score descending,
 * id ascending) order.  Requires 1 <= d < n. */
int kvo_graph_build(const float *emb, int64_t n, int64_t e, int32_t d, int32_t *nbr)
{
    if (n < 2 || d < 1 || (int64_t)d >= n) return KVO_BAD_ARG;
    double *s = (double *)malloc((size_t)n * sizeof *s);
    kvo_key *keys = (kvo_key *)malloc((size_t)n * sizeof *keys);
    if (!s || !keys) { free(s); free(keys); return KVO_BAD_ARG; }
    for (int64_t i = 0; i < n; ++i) {
        kvo_scores(emb + i * e, emb, n, e, s);
        int64_t m = 0;
        for (int64_t j = 0; j < n; ++j) {
            if (j == i) continue;
            keys[m].s = s[j];
            keys[m].id = (int32_t)j;
            ++m;
        }
        qsort(keys, (size_t)m, sizeof *keys, kvo_key_cmp);
        for (int32_t r = 0; r < d; ++r) nbr[i * d + r] = keys[r].id;
    }
    free(s);
    free(keys);
    return KVO_OK;
}

typedef struct { kvo_key key; int expanded; } kvo_cand;

static int kvo_cand_cmp(const void *a, const void *b)
{
    return kvo_key_cmp(&((const kvo_cand *)a)->key, &((const kvo_cand *)b)->key);
}

static double kvo_dot(const float *q, const float *row, int64_t e)
{
    double s = 0.0;
    for (int64_t j = 0; j < e; ++j)
        s += (double)q[j] * (double)row[j];
    return s;
}

/* Graph search for one query q over the graph nbr[n][d].
 *   1. Each seed not seen before is scored; the beam C is the best `beam`
 *      of them in (score descending, id ascending) order, all unexpanded.
 *   2. At most max_iters times: the first `width` unexpanded entries of C
 *      are the parents (if there are none, stop) and are marked expanded;
 *      every neighbour of the parents (parents in C order, neighbours in
 *      list order) not seen before is scored; C becomes the best `beam` of
 *      C and the new facts.
 *   3. The result is the first k entries of C.
 * Every fact is scored at most once, so C never holds an id twice.  Writes
 * sel[0..k) and score[0..k) (-1 and 0 past the end of a short C) and
 * stats[0] = iterations run, stats[1] = facts scored.  Returns the number of
 * results, or -1 for bad arguments (k < 1 or > beam, width outside [1, 1024],
 * max_iters < 0, a seed or neighbour id outside [0, n)). */
int32_t kvo_graph_search(const float *q, const float *emb, int64_t n, int64_t e,
                         const int32_t *nbr, int32_t d, const int32_t *seeds,
                         int32_t n_seeds, int32_t beam, int32_t width, int32_t max_iters,
                         int32_t k, int32_t *sel, double *score, int64_t *stats)
{
    if (k < 1 || beam < k || width < 1 || width > 1024 || max_iters < 0 || d < 1 || n_seeds < 1 ||
        n < 1)
        return -1;
    unsigned char *seen = (unsigned char *)calloc((size_t)n, 1);
    const int64_t cap = (int64_t)beam + (int64_t)n_seeds + (int64_t)width * d;
    kvo_cand *c = (kvo_cand *)malloc((size_t)cap * sizeof *c);
    if (!seen || !c) { free(seen); free(c); return -1; }
    int64_t nc = 0, scored = 0, iters = 0;
    int32_t result = -1;
    for (int32_t i = 0; i < n_seeds; ++i) {
        const int32_t f = seeds[i];
        if (f < 0 || (int64_t)f >= n) goto done;
        if (seen[f]) continue;
        seen[f] = 1;
        c[nc].key.s = kvo_dot(q, emb + (int64_t)f * e, e);
        c[nc].key.id = f;
        c[nc].expanded = 0;
        ++nc;
        ++scored;
    }
    qsort(c, (size_t)nc, sizeof *c, kvo_cand_cmp);
    if (nc > beam) nc = beam;
    while (iters < max_iters) {
        int32_t parents[1024];
        int32_t np = 0;
        for (int64_t i = 0; i < nc && np < width && np < 1024; ++i) {
            if (!c[i].expanded) {
                c[i].expanded = 1;
                parents[np++] = c[i].key.id;
            }
        }
        if (np == 0) break;
        ++iters;
        int64_t m = nc;
        for (int32_t pi = 0; pi < np; ++pi) {
            for (int32_t r = 0; r < d; ++r) {
                const int32_t f = nbr[(int64_t)parents[pi] * d + r];
                if (f < 0 || (int64_t)f >= n) goto done;
                if (seen[f]) continue;
                seen[f] = 1;
                c[m].key.s = kvo_dot(q, emb + (int64_t)f * e, e);
                c[m].key.id = f;
                c[m].expanded = 0;
                ++m;
                ++scored;
            }
        }
        qsort(c, (size_t)m, sizeof *c, kvo_cand_cmp);
        nc = m < beam ? m : beam;
    }
    result = (int32_t)(nc < k ? nc : k);
    for (int32_t j = 0; j < k; ++j) {
        sel[j] = j < result ? c[j].key.id : -1;
        score[j] = j < result ? c[j].key.s : 0.0;
    }
    stats[0] = iters;
    stats[1] = scored;
done:
    free(seen);
    free(c);
    return result;
}
