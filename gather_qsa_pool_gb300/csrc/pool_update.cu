// pool_update.cu -- incremental pooled-key cache update (4-token average pooling ->
// per-head RMS norm -> RoPE at the block start position), one CTA per recomputed row.
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, sections
// "QSA and the QSA indexer" (pooling, RMS norm, RoPE of the pooled summary) and
// "incremental pooled-key cache (COMMON-004)" (only new or invalidated rows and the open
// block are recomputed each step; completed rows are reused).
//
// In decode this touches one or two rows (<= 4 raw rows read, 8 KB written), so it is
// latency-bound; a full rebuild (n_valid_full = 0) streams the raw indexer keys once.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

template <typename T>
__global__ void __launch_bounds__(512)
pool_update_kernel(const T *__restrict__ raw, int64_t n_ctx, int H, int d,
                   const float *__restrict__ w, float eps, double base,
                   float *__restrict__ pooled, int64_t row0)
{
    extern __shared__ float smem[];
    const int hd = H * d;
    const int half = d / 2;
    float *p_s = smem;            // [H*d] pooled means
    float *cos_s = smem + hd;     // [d/2]
    float *sin_s = cos_s + half;  // [d/2]

    pdl_wait();
    pdl_trigger();

    const int64_t b = row0 + blockIdx.x;
    const int64_t t0 = 4 * b;
    const int c = (int)min((int64_t)4, n_ctx - t0);  // tokens present in this block (1..4)
    const float inv_c = 1.0f / (float)c;

    for (int e = threadIdx.x; e < hd; e += blockDim.x) {
        float s = 0.0f;
        for (int t = 0; t < c; ++t) s += to_f32(raw[(t0 + t) * hd + e]);
        p_s[e] = s * inv_c;
    }
    // Rotation angles depend on (b, i) only: form them once per row, in fp64, so that
    // positions up to millions keep full angle accuracy.
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        const double theta = pow(base, -2.0 * (double)i / (double)d);
        const double phi = (4.0 * (double)b) * theta;
        double sv, cv;
        sincos(phi, &sv, &cv);
        cos_s[i] = (float)cv;
        sin_s[i] = (float)sv;
    }
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    for (int h = warp; h < H; h += nwarps) {
        const float *ph = p_s + h * d;
        float ss = 0.0f;
        for (int j = lane; j < d; j += 32) ss = fmaf(ph[j], ph[j], ss);
        ss = warp_sum(ss);
        const float inv = 1.0f / sqrtf(ss / (float)d + eps);
        float *out = pooled + b * (int64_t)hd + (int64_t)h * d;
        for (int i = lane; i < half; i += 32) {
            const float ya = ph[i] * inv * w[i];
            const float yb = ph[i + half] * inv * w[i + half];
            out[i] = ya * cos_s[i] - yb * sin_s[i];
            out[i + half] = ya * sin_s[i] + yb * cos_s[i];
        }
    }
}

}  // namespace

cudaError_t launch_pool_update(const void *raw_k, qsa_dtype dt, int64_t n_ctx, int H, int d,
                               const float *norm_w, float eps, double rope_base,
                               float *pooled, int64_t row0, int64_t row1, cudaStream_t st)
{
    const int64_t n = row1 - row0;
    if (n <= 0) return cudaSuccess;
    const int warps = H < 16 ? H : 16;
    const dim3 block(32 * warps);
    const size_t smem = sizeof(float) * ((size_t)H * d + (size_t)d);
    static bool attr_set[2] = {false, false};
    if (dt == QSA_BF16) {
        auto k = pool_update_kernel<__nv_bfloat16>;
        if (smem > 48 * 1024 && !attr_set[1]) {
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
            attr_set[1] = true;
        }
        return launch(k, dim3((unsigned)n), block, smem, st, 1,
                      (const __nv_bfloat16 *)raw_k, n_ctx, H, d, norm_w, eps, rope_base, pooled,
                      row0);
    }
    auto k = pool_update_kernel<float>;
    if (smem > 48 * 1024 && !attr_set[0]) {
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        attr_set[0] = true;
    }
    return launch(k, dim3((unsigned)n), block, smem, st, 1, (const float *)raw_k, n_ctx, H, d,
                  norm_w, eps, rope_base, pooled, row0);
}

}  // namespace qsa
