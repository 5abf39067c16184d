// pool_update.cu -- incremental pooled-key cache update (4-token average pooling ->
// per-head RMS norm -> RoPE at the block start position), one CTA per recomputed row.
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, sections
// "QSA and the QSA indexer" (pooling, RMS norm, RoPE of the pooled summary) and
// "incremental pooled-key cache (COMMON-004)" (only new or invalidated rows and the open
// block are recomputed each step; completed rows are reused).
//
// The cache stores fp32, or bf16 rounded to nearest even (half the bytes of the scan that
// reads it back every step).
// In decode this touches one or two rows (<= 4 raw rows read, 8 KB written), so it is
// latency-bound: every thread issues all of its raw-key loads before using any, and the
// rotation angles avoid device fp64 transcendentals (slow on this part): the inverse
// frequencies base^(-2i/d) come from the host in fp64, the angle 4b * theta_i is formed
// and reduced modulo 2*pi in fp64 (exact to ~1e-11 rad at a million tokens), and only
// the reduced angle, |r| <= pi, goes through fp32 sincosf.
#include <math.h>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kPoolThreads = 512;

template <typename T, typename TP>
__global__ void __launch_bounds__(kPoolThreads)
pool_update_kernel(const T *__restrict__ raw, int64_t n_ctx, int H, int d,
                   const float *__restrict__ w, float eps, const RopeTable tab,
                   TP *__restrict__ pooled, int64_t row0, int64_t row1,
                   uint32_t *__restrict__ zero_hist)
{
    extern __shared__ float smem[];
    const int hd = H * d;
    const int half = d / 2;
    float *p_s = smem;            // [H*d] pooled means
    float *cos_s = smem + hd;     // [d/2]
    float *sin_s = cos_s + half;  // [d/2]

    pdl_wait();
    QSA_AFTER_WAIT(raw);
    QSA_AFTER_WAIT(w);
    pdl_trigger();
    if (zero_hist && blockIdx.x == 0)
        for (int i = threadIdx.x; i < (1 << kTopkHistBits); i += kPoolThreads) zero_hist[i] = 0u;

    const int64_t b = row0 + blockIdx.x;
    if (b >= row1) return;
    pool_row(raw, n_ctx, H, d, w, eps, tab, b, p_s, cos_s, sin_s,
             pooled + b * (int64_t)(H * d));
}

// Many rows (a rebuild, a prefill chunk's new rows): one warp per row, the row's H*D values
// in registers -- value e (of the row's H*D) on lane e % 32 as value e / 32 -- so no shared
// memory or block barrier is needed and a CTA's eight rows are in flight together.  Every
// value is formed as in pool_row, in the same order (the 4-token mean; per head the sum of
// squares over values lane, lane + 32, ... then the warp reduction; the rotation of the
// pair (i, i + D/2), both on one lane), so the two forms write the same bits.
constexpr int kWarpRowThreads = 256;

template <typename T, typename TP, int D, int NH>
__global__ void __launch_bounds__(kWarpRowThreads)
pool_rows_warp_kernel(const T *__restrict__ raw, int64_t n_ctx, const float *__restrict__ w,
                      float eps, const RopeTable tab, TP *__restrict__ pooled, int64_t row0,
                      int64_t row1, uint32_t *__restrict__ zero_hist)
{
    constexpr int HD = NH * D, PER = HD / 32, PH = D / 32, HALF = D / 2, MH = HALF / 32;
    static_assert(D % 64 == 0 && PER <= 64, "two rotation partners per lane, <= 64 values");
    pdl_wait();
    QSA_AFTER_WAIT(raw);
    QSA_AFTER_WAIT(w);
    pdl_trigger();
    if (zero_hist && blockIdx.x == 0)
        for (int i = threadIdx.x; i < (1 << kTopkHistBits); i += kWarpRowThreads) zero_hist[i] = 0u;
    const int lane = threadIdx.x & 31;
    const int64_t b = row0 + (int64_t)blockIdx.x * (kWarpRowThreads / 32) + (threadIdx.x >> 5);
    if (b >= row1) return;
    const int64_t t0 = 4 * b;
    const int c = (int)min((int64_t)4, n_ctx - t0);  // tokens present in this block (1..4)
    const float inv_c = 1.0f / (float)c;
    const T *rb = raw + t0 * HD;
    float p[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int e = lane + 32 * k;
        float v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) v[t] = t < c ? to_f32(rb[(int64_t)t * HD + e]) : 0.0f;
        p[k] = ((v[0] + v[1]) + (v[2] + v[3])) * inv_c;
    }
    float cs[MH], sn[MH], wa[MH], wb[MH];
#pragma unroll
    for (int m = 0; m < MH; ++m) {
        const int i = lane + 32 * m;
        // the angle 4b * theta_i, formed and reduced modulo 2 pi in fp64; fp32 sincos of
        // the reduced angle (|r| <= pi)
        const double phi = (4.0 * (double)b) * tab.theta[i];
        const double k = rint(phi * kInvTwoPi);
        const float r = (float)fma(-k, kTwoPi, phi);
        sincosf(r, &sn[m], &cs[m]);
        wa[m] = w[i];
        wb[m] = w[i + HALF];
    }
    TP *out_row = pooled + b * (int64_t)HD;
#pragma unroll
    for (int h = 0; h < NH; ++h) {
        float ss = 0.0f;
#pragma unroll
        for (int j = 0; j < PH; ++j) ss = fmaf(p[h * PH + j], p[h * PH + j], ss);
        ss = warp_sum(ss);
        const float inv = 1.0f / sqrtf(ss / (float)D + eps);
        TP *o = out_row + (int64_t)h * D;
#pragma unroll
        for (int m = 0; m < MH; ++m) {
            const int i = lane + 32 * m;
            const float ya = p[h * PH + m] * inv * wa[m];
            const float yb = p[h * PH + m + MH] * inv * wb[m];
            const float za = ya * cs[m] - yb * sn[m];
            const float zb = ya * sn[m] + yb * cs[m];
            store_pooled(o + i, za);
            store_pooled(o + i + HALF, zb);
        }
    }
}

}  // namespace

void make_rope_table(RopeTable *tab, int d, double base)
{
    for (int i = 0; i < d / 2 && i < kRopeMaxHalf; ++i)
        tab->theta[i] = pow(base, -2.0 * (double)i / (double)d);
}

template <typename T, typename TP>
cudaError_t launch_pool_typed(const void *raw_k, int64_t n_ctx, int H, int d,
                              const float *norm_w, float eps, const RopeTable &tab, void *pooled,
                              int64_t row0, int64_t row1, uint32_t *zero_hist, int64_t n,
                              cudaStream_t st)
{
    // enough rows of the indexer's shape to fill the GPU (16 rows in flight per SM): one warp
    // per row; fewer rows finish sooner as one CTA each, whose 512 threads shorten a row's
    // chain of loads
    if (n >= 2048 && d == 128 && H == 16) {
        const unsigned grid = (unsigned)((n + kWarpRowThreads / 32 - 1) / (kWarpRowThreads / 32));
        return launch(pool_rows_warp_kernel<T, TP, 128, 16>, dim3(grid), dim3(kWarpRowThreads), 0,
                      st, 1, (const T *)raw_k, n_ctx, norm_w, eps, tab, (TP *)pooled, row0, row1,
                      zero_hist);
    }
    const size_t smem = sizeof(float) * ((size_t)H * d + (size_t)d);
    auto k = pool_update_kernel<T, TP>;
    const cudaError_t e = ensure_kernel_attrs<pool_update_kernel<T, TP>>(smem);
    if (e != cudaSuccess) return e;
    return launch(k, dim3((unsigned)n), dim3(kPoolThreads), smem, st, 1, (const T *)raw_k, n_ctx,
                  H, d, norm_w, eps, tab, (TP *)pooled, row0, row1, zero_hist);
}

cudaError_t launch_pool_update(const void *raw_k, qsa_dtype dt, int64_t n_ctx, int H, int d,
                               const float *norm_w, float eps, double rope_base,
                               void *pooled, qsa_dtype pdt, int64_t row0, int64_t row1,
                               uint32_t *zero_hist, cudaStream_t st)
{
    int64_t n = row1 - row0;
    if (n <= 0) {
        if (!zero_hist) return cudaSuccess;
        n = 1;  // one CTA clears the histogram
    }
    // the table depends on (d, base) only: rebuild it when they change
    thread_local RopeTable tab;
    thread_local int tab_d = -1;
    thread_local double tab_base = 0.0;
    if (tab_d != d || tab_base != rope_base) {
        make_rope_table(&tab, d, rope_base);
        tab_d = d;
        tab_base = rope_base;
    }
    using bf = __nv_bfloat16;
    if (dt == QSA_BF16)
        return pdt == QSA_BF16
                   ? launch_pool_typed<bf, bf>(raw_k, n_ctx, H, d, norm_w, eps, tab, pooled, row0,
                                               row1, zero_hist, n, st)
                   : launch_pool_typed<bf, float>(raw_k, n_ctx, H, d, norm_w, eps, tab, pooled,
                                                  row0, row1, zero_hist, n, st);
    return pdt == QSA_BF16
               ? launch_pool_typed<float, bf>(raw_k, n_ctx, H, d, norm_w, eps, tab, pooled, row0,
                                              row1, zero_hist, n, st)
               : launch_pool_typed<float, float>(raw_k, n_ctx, H, d, norm_w, eps, tab, pooled,
                                                 row0, row1, zero_hist, n, st);
}

}  // namespace qsa
