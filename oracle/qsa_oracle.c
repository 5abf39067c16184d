/*
 * qsa_oracle.c -- plain, slow, fp64 CPU oracle for QSA two-stage sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this
 * file: only the test suite, the smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Every function restates one step of the method as the source pages describe it
 * (Qiita, ariera, "EVO-X2 ... llama.cpp" part 10, section "QSA and the QSA indexer";
 * devotd.net, "llama.cpp CDNA sparse attention", sections 2-3), in the pages' order:
 *   4-token block -> average pooling -> RMS norm -> RoPE -> score against the query
 *   -> top-k over blocks -> expand selected blocks to cells, append the open tail
 *   -> attention over the selected cells only.
 * All arithmetic is fp64; only the pooled-key cache is rounded on store, to fp32 or
 * to bf16 (the storage type of the cache tensor), and the tensor-core scoring mirror
 * rounds its two operands to bf16 when asked.
 *
 * Readings where the pages are silent (each one is listed with its reason in the
 * design notes): partial block divided by the number of present tokens; RMS norm per
 * indexer head over d with eps inside the square root and one weight vector w[d];
 * NeoX half-split RoPE over the full head dim at the block start position 4b with
 * theta_i = base^(-2i/d); score = scale * sum_h q_h . z_h; ties at the top-k boundary
 * go to the lower block index and NaN scores rank as -inf; the open partial block is
 * always appended as the tail and never competes; GQA head h uses KV head
 * floor(h * H_kv / H_q).
 *
 * Parity pins: every exported function is pinned by tests/test_oracle_*.py against
 * closed forms, textbook special cases, library routines or brute force.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

/* ------------------------------------------------------------------ element access */

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Value of element `idx` of an array stored as fp32 (dtype 0) or bf16 bits (dtype 1). */
static double elem(const void *base, int dtype, int64_t idx)
{
    if (dtype == ORC_BF16)
        return bf16_bits_to_double(((const uint16_t *)base)[idx]);
    return (double)((const float *)base)[idx];
}

/* Round an fp32 value to the nearest bf16 value, ties to even (what a tensor-core
 * operand holds when the scoring contraction runs in bf16). */
static float round_to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) { /* inf or NaN: keep, quiet the NaN */
        if (u & 0x007fffffu) u |= 0x00400000u;
        u &= 0xffff0000u;
    } else {
        uint32_t lsb = (u >> 16) & 1u;
        u = (u + 0x7fffu + lsb) & 0xffff0000u;
    }
    float r;
    memcpy(&r, &u, sizeof r);
    return r;
}

float oracle_round_bf16(float x) { return round_to_bf16(x); }

/*
 * Round an fp64 value to the nearest bf16 value, ties to even, in one step (not through
 * fp32: a value just above a bf16 midpoint must not first land on the midpoint).
 * bf16 keeps 8 significant bits, exponents down to 2^-126 and subnormals spaced 2^-133;
 * values at or beyond the midpoint above the largest finite bf16, (2 - 2^-7) * 2^127,
 * become infinite.  Returns the bit pattern.
 */
uint16_t oracle_bf16_bits_from_f64(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return 0x7fc0u;
    if (isinf(x)) return (uint16_t)(sign | 0x7f80u);
    double ax = fabs(x);
    if (ax == 0.0) return sign;
    int ex;
    frexp(ax, &ex);             /* ax = m * 2^ex with 0.5 <= m < 1 */
    int e_unit = ex - 8;        /* value of the last of the 8 significant bits */
    if (e_unit < -133) e_unit = -133;
    double r = nearbyint(ldexp(ax, -e_unit)); /* default rounding mode: ties to even */
    double v = ldexp(r, e_unit);
    if (v > 3.3895313892515355e38) return (uint16_t)(sign | 0x7f80u);
    float f = (float)v;         /* exact: v has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/* ------------------------------------------------------------------ step 1: pool */

/*
 * Average pooling of one 4-token micro-block (p1, "QSA indexer": the indexer keys of
 * 4 tokens are average-pooled into one representative vector per block).
 * Block b covers tokens 4b .. min(4b+3, n_ctx-1); the mean is over the tokens present.
 * raw: [n_ctx][H][d].  p: [H*d] (fp64).  Returns the number of tokens averaged.
 */
int oracle_pool_mean(const void *raw, int dtype, int64_t n_ctx, int H, int d,
                     int64_t b, double *p)
{
    int64_t t0 = 4 * b;
    int64_t t1 = t0 + 4 < n_ctx ? t0 + 4 : n_ctx;
    int c = (int)(t1 - t0);
    int64_t hd = (int64_t)H * d;
    for (int64_t e = 0; e < hd; ++e) {
        double s = 0.0;
        for (int64_t t = t0; t < t1; ++t)
            s += elem(raw, dtype, t * hd + e);
        p[e] = c > 0 ? s / (double)c : 0.0;
    }
    return c;
}

/*
 * RMS normalisation of one indexer head's pooled vector (p1, "QSA indexer": RMS norm
 * of the pooled summary): y_j = p_j / sqrt(mean_j p_j^2 + eps) * w_j.
 */
void oracle_rmsnorm(const double *p, int d, const float *w, double eps, double *y)
{
    double ss = 0.0;
    for (int j = 0; j < d; ++j)
        ss += p[j] * p[j];
    double inv = 1.0 / sqrt(ss / (double)d + eps);
    for (int j = 0; j < d; ++j)
        y[j] = p[j] * inv * (double)w[j];
}

/*
 * Rotary position embedding of one head vector in place (p1, "QSA indexer": RoPE adds
 * the position to the pooled summary).  NeoX half-split pairing: dimension i rotates
 * with dimension i + d/2 by angle pos * theta_i, theta_i = base^(-2i/d), i < d/2.
 */
void oracle_rope(double *y, int d, double pos, double base)
{
    int half = d / 2;
    for (int i = 0; i < half; ++i) {
        double theta = pow(base, -2.0 * (double)i / (double)d);
        double phi = pos * theta;
        double c = cos(phi), s = sin(phi);
        double a = y[i], b = y[i + half];
        y[i] = a * c - b * s;
        y[i + half] = a * s + b * c;
    }
}

/*
 * One pooled-key cache row: pool -> RMS norm (per head) -> RoPE at the block start
 * position 4b (per head), in fp64.  z: [H*d] fp64, not rounded.
 */
void oracle_pool_row_f64(const void *raw, int dtype, int64_t n_ctx, int H, int d,
                         const float *w, double eps, double base, int64_t b, double *z)
{
    int64_t hd = (int64_t)H * d;
    double *p = (double *)malloc(sizeof(double) * (size_t)hd);
    oracle_pool_mean(raw, dtype, n_ctx, H, d, b, p);
    for (int h = 0; h < H; ++h) {
        oracle_rmsnorm(p + (int64_t)h * d, d, w, eps, z + (int64_t)h * d);
        oracle_rope(z + (int64_t)h * d, d, 4.0 * (double)b, base);
    }
    free(p);
}

/*
 * The incremental pooled-key cache update (p1, "incremental pooled-key cache
 * (COMMON-004)": only newly completed or invalidated blocks are recomputed; the open
 * partial block is recomputed every step).  Writes rows [row_begin, row_end) of
 * `pooled` ([rows][H*d]) and leaves every other row untouched.  store_dtype: the cache
 * holds fp32 (ORC_F32, each value rounded to nearest fp32) or bf16 bits (ORC_BF16, each
 * value rounded to nearest bf16 directly from fp64).
 */
void oracle_pool_rows(const void *raw, int dtype, int64_t n_ctx, int H, int d,
                      const float *w, double eps, double base, int64_t row_begin,
                      int64_t row_end, int store_dtype, void *pooled)
{
    int64_t hd = (int64_t)H * d;
    double *z = (double *)malloc(sizeof(double) * (size_t)hd);
    for (int64_t b = row_begin; b < row_end; ++b) {
        oracle_pool_row_f64(raw, dtype, n_ctx, H, d, w, eps, base, b, z);
        for (int64_t e = 0; e < hd; ++e) {
            if (store_dtype == ORC_BF16)
                ((uint16_t *)pooled)[b * hd + e] = oracle_bf16_bits_from_f64(z[e]);
            else
                ((float *)pooled)[b * hd + e] = (float)z[e];
        }
    }
    free(z);
}

/* ------------------------------------------------------------------ step 2: score */

/*
 * Index scores (p1, "QSA indexer": score every pooled block against the query):
 *   s[i][b] = scale * sum_{h,j} q[i][h*d+j] * z[b][h*d+j]
 * q: [n_q][H*d] fp32; pooled: [n_rows][H*d] fp32 or bf16 bits (pooled_dtype);
 * scores: [n_q][n_rows] fp64.
 * q_pos (nullable): position of query i; row b is visible to query i only when the
 * block is complete at that position (4b+3 <= q_pos[i]); other rows get -inf.
 * round_bf16 != 0: both operands are first rounded to bf16 (tensor-core mirror).
 */
void oracle_scores(const float *q, int64_t n_q, const void *pooled, int pooled_dtype,
                   int64_t n_rows, int H, int d, double scale, const int32_t *q_pos,
                   int round_bf16, double *scores)
{
    int64_t hd = (int64_t)H * d;
    for (int64_t i = 0; i < n_q; ++i) {
        for (int64_t b = 0; b < n_rows; ++b) {
            if (q_pos && 4 * b + 3 > (int64_t)q_pos[i]) {
                scores[i * n_rows + b] = -INFINITY;
                continue;
            }
            double s = 0.0;
            for (int64_t e = 0; e < hd; ++e) {
                float qa = q[i * hd + e], zb = (float)elem(pooled, pooled_dtype, b * hd + e);
                if (round_bf16) {
                    qa = round_to_bf16(qa);
                    zb = round_to_bf16(zb);
                }
                s += (double)qa * (double)zb;
            }
            scores[i * n_rows + b] = scale * s;
        }
    }
}

/* ------------------------------------------------------------------ step 3: top-k */

typedef struct {
    double s;
    int64_t idx;
} scored_t;

/* Order: higher score first; equal scores -> lower index first; NaN ranks as -inf. */
static int cmp_desc(const void *pa, const void *pb)
{
    const scored_t *a = (const scored_t *)pa, *b = (const scored_t *)pb;
    double sa = isnan(a->s) ? -INFINITY : a->s;
    double sb = isnan(b->s) ? -INFINITY : b->s;
    if (sa > sb) return -1;
    if (sa < sb) return 1;
    return (a->idx > b->idx) - (a->idx < b->idx);
}

static int cmp_i32(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/*
 * Block-domain top-k (p1, "block-domain top-k (COMMON-006)": top-k is taken over the
 * block scores, not over cells).  Only full blocks b < n_full compete.  A full sort
 * by (score desc, index asc); the first min(k_blk, n_full) are returned in ascending
 * block order.  Returns the count.
 */
int64_t oracle_topk(const double *scores, int64_t n_full, int64_t k_blk, int32_t *blocks)
{
    if (n_full <= 0 || k_blk <= 0) return 0;
    scored_t *v = (scored_t *)malloc(sizeof(scored_t) * (size_t)n_full);
    for (int64_t b = 0; b < n_full; ++b) {
        v[b].s = scores[b];
        v[b].idx = b;
    }
    qsort(v, (size_t)n_full, sizeof(scored_t), cmp_desc);
    int64_t k = k_blk < n_full ? k_blk : n_full;
    for (int64_t j = 0; j < k; ++j)
        blocks[j] = (int32_t)v[j].idx;
    free(v);
    qsort(blocks, (size_t)k, sizeof(int32_t), cmp_i32);
    return k;
}

/*
 * The pages' earlier selection path, kept for A/B measurement (p1, "block-domain top-k
 * (COMMON-006)": before it, each block's score was copied to its 4 cells and the top-k
 * ran over cells).  cells[c] = scores[floor(c/4)] for c < 4*n_full.
 */
void oracle_expand_block_scores(const double *scores, int64_t n_full, double *cells)
{
    for (int64_t b = 0; b < n_full; ++b)
        for (int t = 0; t < 4; ++t)
            cells[4 * b + t] = scores[b];
}

/* ------------------------------------------------------------------ step 4: cells */

/*
 * Expand the selected blocks to KV cells and append the open tail (p1, "block-domain
 * top-k": expand only the selected pools to cell indices, then append the tail
 * indices; "why FA scaled": 2048 + 4 - 1 = 2051 cells at most).
 * p = position of the query (decode: n_ctx - 1).  Full blocks at p: n_full =
 * floor((p+1)/4); tail = 4*n_full .. p.  Returns n_cells.
 */
int64_t oracle_cells(const int32_t *blocks, int64_t count, int64_t p, int32_t *cells)
{
    int64_t n = 0;
    for (int64_t j = 0; j < count; ++j)
        for (int t = 0; t < 4; ++t)
            cells[n++] = 4 * blocks[j] + t;
    int64_t n_full = (p + 1) / 4;
    for (int64_t t = 4 * n_full; t <= p; ++t)
        cells[n++] = (int32_t)t;
    return n;
}

/* Row copy of the selected cells (p1, "selected K/V gather (COMMON-005)": get_rows). */
void oracle_get_rows(const void *src, int elem_bytes, int64_t row_elems, int64_t ld,
                     const int32_t *cells, int64_t n_cells, void *dst)
{
    for (int64_t j = 0; j < n_cells; ++j)
        memcpy((char *)dst + (size_t)(j * row_elems * elem_bytes),
               (const char *)src + (size_t)((int64_t)cells[j] * ld * elem_bytes),
               (size_t)(row_elems * elem_bytes));
}

/* ------------------------------------------------------------------ step 5: attention */

/*
 * Attention of one query token over a list of cells only (p1, "selected K/V gather":
 * attention runs over the compact ~2051 rows; devotd, section 2: only listed key
 * positions are processed).
 * q: [H_q][d_k] fp32.  K element (cell c, kv head g, j) = K[c*ld_k + g*d_k + j];
 * V element (c, g, j) = V[c*ld_v + g*d_v + j]; K and V are fp32 or bf16 (dtype).
 * Head h uses kv head g = floor(h*H_kv/H_q).  Logits = scale * q.k; softmax with the
 * maximum subtracted; out[h][:] = sum_j softmax_j * V[cell_j, g]; lse[h] = natural
 * log of sum_j exp(logit_j).  An empty list gives out = 0 and lse = -inf.
 */
void oracle_attention(const float *q, int H_q, int H_kv, int d_k, int d_v,
                      const void *K, const void *V, int dtype, int64_t ld_k, int64_t ld_v,
                      const int32_t *cells, int64_t n_cells, double scale, double *out,
                      double *lse)
{
    double *logit = (double *)malloc(sizeof(double) * (size_t)(n_cells > 0 ? n_cells : 1));
    for (int h = 0; h < H_q; ++h) {
        int g = (int)(((int64_t)h * H_kv) / H_q);
        double *o = out + (int64_t)h * d_v;
        for (int j = 0; j < d_v; ++j) o[j] = 0.0;
        if (n_cells <= 0) {
            if (lse) lse[h] = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (int64_t c = 0; c < n_cells; ++c) {
            int64_t row = (int64_t)cells[c] * ld_k + (int64_t)g * d_k;
            double s = 0.0;
            for (int j = 0; j < d_k; ++j)
                s += (double)q[(int64_t)h * d_k + j] * elem(K, dtype, row + j);
            logit[c] = scale * s;
            if (logit[c] > m) m = logit[c];
        }
        double z = 0.0;
        for (int64_t c = 0; c < n_cells; ++c) {
            double wgt = exp(logit[c] - m);
            z += wgt;
            int64_t row = (int64_t)cells[c] * ld_v + (int64_t)g * d_v;
            for (int j = 0; j < d_v; ++j)
                o[j] += wgt * elem(V, dtype, row + j);
        }
        for (int j = 0; j < d_v; ++j) o[j] /= z;
        if (lse) lse[h] = m + log(z);
    }
    free(logit);
}

/* ------------------------------------------------------------------ step 6: mask list */

/*
 * Mask -> key-position list (devotd, section 2: attendable key positions are gathered
 * from the mask into a list; the per-lane selection is kept as 64-bit words, one bit per
 * position, and the count uses the same words).
 * bits[w] bit t = (mask[64w + t] != 0), least significant bit first; positions are
 * written in ascending order, at most max_list of them; the return value is the true
 * count even when it exceeds max_list.
 */
int64_t oracle_mask_to_list(const uint8_t *mask, int64_t n_kv, int64_t max_list,
                            int32_t *pos, uint64_t *bits)
{
    int64_t n_words = (n_kv + 63) / 64;
    if (bits)
        for (int64_t w = 0; w < n_words; ++w) bits[w] = 0;
    int64_t count = 0;
    for (int64_t j = 0; j < n_kv; ++j) {
        if (mask[j] != 0) {
            if (bits) bits[j / 64] |= (uint64_t)1 << (j % 64);
            if (count < max_list) pos[count] = (int32_t)j;
            ++count;
        }
    }
    return count;
}
