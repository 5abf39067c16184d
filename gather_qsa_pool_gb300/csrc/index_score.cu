// index_score.cu -- indexer scores of pooled rows against the query (CUDA-core fp32).
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "QSA and the QSA indexer" (the query is scored against every pooled block summary)
// and section "incremental pooled-key cache (COMMON-004)" (after the cache fix, this
// scan is the one step left whose cost grows with context).
//
// Decode (one query): a pure HBM stream of the fp32 pooled cache, H*d*4 bytes per row
// (8 KB at 16 heads x 128).  A persistent grid of warps walks the rows; each lane issues
// all of its 16-byte streaming loads for a row (and the next) before reducing, so that
// every SM keeps ~100 KB in flight; the query sits in shared memory.
// Several queries (a prefill chunk in fp32): a register-tiled fp32 GEMM with the causal
// block visibility rule applied in the epilogue.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kScoreThreads = 256;

// One query, H*d = NV*128 floats per row.  Warps gw, gw + nw, ... of the grid walk the
// rows [0, n_rows); R rows are loaded before any is reduced.
template <int NV, int R>
__device__ __forceinline__ void score_rows_loop(const float4 *q_s, const float *__restrict__ pooled,
                                                int64_t n_rows, int64_t gw, int64_t nw,
                                                float scale, float *__restrict__ scores,
                                                uint32_t *__restrict__ hist, int64_t n_hist)
{
    const int lane = threadIdx.x & 31;
    for (int64_t r0 = gw; r0 < n_rows; r0 += nw * R) {
        float4 v[R][NV];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = r0 + (int64_t)r * nw;
            if (row < n_rows) {
                const float4 *rp = reinterpret_cast<const float4 *>(pooled + row * (NV * 128)) + lane;
#pragma unroll
                for (int j = 0; j < NV; ++j) v[r][j] = ld_stream_f4(rp + 32 * j);
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = r0 + (int64_t)r * nw;
            if (row < n_rows) {
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                for (int j = 0; j < NV; ++j) {
                    const float4 qq = q_s[lane + 32 * j];
                    a0 = fmaf(v[r][j].x, qq.x, a0);
                    a1 = fmaf(v[r][j].y, qq.y, a1);
                    a2 = fmaf(v[r][j].z, qq.z, a2);
                    a3 = fmaf(v[r][j].w, qq.w, a3);
                }
                const float acc = warp_sum((a0 + a1) + (a2 + a3));
                if (lane == 0) {
                    const float sc = acc * scale;
                    scores[row] = sc;
                    if (hist && row < n_hist) atomicAdd(&hist[score_key(sc) >> (32 - kTopkHistBits)], 1u);
                }
            }
        }
    }
}

// The score of one row already in shared memory, with exactly the summation order of
// score_rows_loop (called by one warp).
template <int NV>
__device__ __forceinline__ float score_row_smem(const float4 *q_s, const float *row_s)
{
    const int lane = threadIdx.x & 31;
    const float4 *rp = reinterpret_cast<const float4 *>(row_s) + lane;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const float4 v = rp[32 * j];
        const float4 qq = q_s[lane + 32 * j];
        a0 = fmaf(v.x, qq.x, a0);
        a1 = fmaf(v.y, qq.y, a1);
        a2 = fmaf(v.z, qq.z, a2);
        a3 = fmaf(v.w, qq.w, a3);
    }
    return warp_sum((a0 + a1) + (a2 + a3));
}

template <int NV, int R>
__global__ void __launch_bounds__(kScoreThreads)
score_rows_kernel(const float *__restrict__ q, const float *__restrict__ pooled,
                  int64_t n_rows, float scale, float *__restrict__ scores,
                  uint32_t *__restrict__ hist, int64_t n_hist, uint32_t *__restrict__ ticket)
{
    __shared__ float4 q_s[NV * 32];
    pdl_wait();
    QSA_AFTER_WAIT(q);
    QSA_AFTER_WAIT(pooled);
    pdl_trigger();
    if (ticket && blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0u;
    for (int i = threadIdx.x; i < NV * 32; i += blockDim.x)
        q_s[i] = reinterpret_cast<const float4 *>(q)[i];
    __syncthreads();
    const int64_t nw = (int64_t)gridDim.x * (kScoreThreads / 32);
    const int64_t gw = (int64_t)blockIdx.x * (kScoreThreads / 32) + (threadIdx.x >> 5);
    score_rows_loop<NV, R>(q_s, pooled, n_rows, gw, nw, scale, scores, hist, n_hist);
}

// Decode step with the pooled-row update folded in: CTA i < n_pool recomputes row
// row0 + i (pool -> RMS norm -> rotation), stores it and scores it from shared memory;
// the other CTAs stream the rows [0, row0) that were already valid.
template <int NV, typename T>
__global__ void __launch_bounds__(kScoreThreads)
score_pool_kernel(const float *__restrict__ q, float *__restrict__ pooled, float scale,
                  float *__restrict__ scores, uint32_t *__restrict__ hist, int64_t n_hist,
                  uint32_t *__restrict__ ticket, const T *__restrict__ raw, int64_t n_ctx, int H, int d,
                  const float *__restrict__ w, float eps, int64_t row0, int n_pool,
                  const RopeTable tab)
{
    __shared__ float4 q_s[NV * 32];
    __shared__ __align__(16) float p_s[NV * 128];
    __shared__ float cs[kRopeMaxHalf], sn[kRopeMaxHalf];
    pdl_wait();
    QSA_AFTER_WAIT(q);
    QSA_AFTER_WAIT(pooled);
    QSA_AFTER_WAIT(raw);
    QSA_AFTER_WAIT(w);
    pdl_trigger();
    if (ticket && blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0u;
    for (int i = threadIdx.x; i < NV * 32; i += blockDim.x)
        q_s[i] = reinterpret_cast<const float4 *>(q)[i];
    __syncthreads();
    if ((int)blockIdx.x < n_pool) {
        const int64_t b = row0 + blockIdx.x;
        pool_row(raw, n_ctx, H, d, w, eps, tab, b, p_s, cs, sn, pooled + b * (int64_t)(NV * 128));
        if (threadIdx.x < 32) {
            const float acc = score_row_smem<NV>(q_s, p_s);
            if (threadIdx.x == 0) {
                const float sc = acc * scale;
                scores[b] = sc;
                if (hist && b < n_hist) atomicAdd(&hist[score_key(sc) >> (32 - kTopkHistBits)], 1u);
            }
        }
        return;
    }
    const int64_t nw = (int64_t)(gridDim.x - n_pool) * (kScoreThreads / 32);
    const int64_t gw = (int64_t)(blockIdx.x - n_pool) * (kScoreThreads / 32) + (threadIdx.x >> 5);
    score_rows_loop<NV, (NV <= 8 ? 2 : 1)>(q_s, pooled, row0, gw, nw, scale, scores, hist, n_hist);
}

// General case: scores[i][b] = scale * <q_i, pooled_b>, 64 queries x 64 rows per CTA,
// k-chunks of 16 staged in shared memory, 4x4 outputs per thread.
constexpr int kBM = 64, kBN = 64, kBK = 16;

__global__ void __launch_bounds__(256)
score_tiled_kernel(const float *__restrict__ q, int64_t n_q, int64_t ld_q,
                   const int32_t *__restrict__ q_pos, const float *__restrict__ pooled,
                   int64_t n_rows, int hd, float scale, float *__restrict__ scores,
                   int64_t ld_scores, uint32_t *__restrict__ hist, int64_t n_hist,
                   uint32_t *__restrict__ ticket)
{
    __shared__ float a_s[kBK][kBM + 4];
    __shared__ float b_s[kBK][kBN + 4];
    pdl_wait();
    QSA_AFTER_WAIT(q);
    QSA_AFTER_WAIT(q_pos);
    QSA_AFTER_WAIT(pooled);
    pdl_trigger();
    if (ticket && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *ticket = 0u;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int64_t m0 = (int64_t)blockIdx.y * kBM;
    const int64_t n0 = (int64_t)blockIdx.x * kBN;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < hd; k0 += kBK) {
        for (int e = threadIdx.x; e < kBK * kBM; e += 256) {
            const int kk = e % kBK, mm = e / kBK;
            const int64_t gm = m0 + mm;
            a_s[kk][mm] = (gm < n_q && k0 + kk < hd) ? q[gm * ld_q + k0 + kk] : 0.f;
            const int64_t gn = n0 + mm;
            b_s[kk][mm] = (gn < n_rows && k0 + kk < hd) ? pooled[gn * hd + k0 + kk] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kBK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = a_s[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = b_s[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t gm = m0 + ty * 4 + i;
        if (gm >= n_q) continue;
        const int64_t p = q_pos ? (int64_t)q_pos[gm] : INT64_MAX;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t gn = n0 + tx * 4 + j;
            if (gn >= n_rows) continue;
            const bool visible = q_pos == nullptr || 4 * gn + 3 <= p;
            const float sc = visible ? acc[i][j] * scale : -INFINITY;
            scores[gm * ld_scores + gn] = sc;
            if (hist && visible && gn < n_hist)
                atomicAdd(&hist[gm * (1 << kTopkHistBits) + (score_key(sc) >> (32 - kTopkHistBits))], 1u);
        }
    }
}

template <int NV, int R>
cudaError_t launch_rows(const float *q, const float *pooled, int64_t n_rows, float scale,
                        float *scores, uint32_t *hist, int64_t n_hist, uint32_t *ticket,
                        cudaStream_t st)
{
    static int blocks_per_sm = 0;
    auto k = score_rows_kernel<NV, R>;
    if (blocks_per_sm == 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, k,
                                                                      kScoreThreads, 0);
        if (e != cudaSuccess) return e;
        if (blocks_per_sm < 1) blocks_per_sm = 1;
    }
    const int64_t warps_needed = (n_rows + R - 1) / R;
    int64_t grid = (int64_t)device_sm_count() * blocks_per_sm;
    const int64_t grid_needed = (warps_needed + kScoreThreads / 32 - 1) / (kScoreThreads / 32);
    if (grid > grid_needed) grid = grid_needed;
    if (grid < 1) grid = 1;
    return launch(k, dim3((unsigned)grid), dim3(kScoreThreads), 0, st, 1, q, pooled, n_rows,
                  scale, scores, hist, n_hist, ticket);
}

template <int NV, typename T>
cudaError_t launch_fused(const float *q, const float *pooled, int64_t n_rows, int H, int d,
                         float scale, float *scores, uint32_t *hist, int64_t n_hist,
                         uint32_t *ticket,
                         const PoolFuse &pf, double rope_base, cudaStream_t st)
{
    static int blocks_per_sm = 0;
    auto k = score_pool_kernel<NV, T>;
    if (blocks_per_sm == 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, k,
                                                                      kScoreThreads, 0);
        if (e != cudaSuccess) return e;
        if (blocks_per_sm < 1) blocks_per_sm = 1;
    }
    thread_local RopeTable tab;
    thread_local int tab_d = -1;
    thread_local double tab_base = 0.0;
    if (tab_d != d || tab_base != rope_base) {
        make_rope_table(&tab, d, rope_base);
        tab_d = d;
        tab_base = rope_base;
    }
    const int n_pool = (int)(pf.row1 - pf.row0);
    int64_t grid = (int64_t)device_sm_count() * blocks_per_sm;
    const int64_t warps_needed = pf.row0;
    const int64_t grid_needed = n_pool + (warps_needed + kScoreThreads / 32 - 1) / (kScoreThreads / 32);
    if (grid > grid_needed) grid = grid_needed;
    if (grid < n_pool + 1) grid = n_pool + 1;
    (void)n_rows;
    return launch(k, dim3((unsigned)grid), dim3(kScoreThreads), 0, st, 1, q, (float *)pooled,
                  scale, scores, hist, n_hist, ticket, (const T *)pf.raw, pf.n_ctx, H, d, pf.w, pf.eps,
                  pf.row0, n_pool, tab);
}

}  // namespace

cudaError_t launch_score_pool_fused(const float *q, const float *pooled, int64_t n_rows, int H,
                                    int d, float scale, float *scores, uint32_t *hist,
                                    int64_t n_hist, uint32_t *ticket, const PoolFuse &pf,
                                    double rope_base,
                                    cudaStream_t st)
{
    const int hd = H * d;
    const int64_t n_pool = pf.row1 - pf.row0;
    const bool aligned = (reinterpret_cast<uintptr_t>(q) % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(pooled) % 16 == 0);
    if (!aligned || hd != 2048 || d / 2 > kRopeMaxHalf || n_pool < 0 || n_pool > kMaxFusedPoolRows ||
        pf.row1 != n_rows)
        return cudaErrorNotSupported;
    if (pf.dt == QSA_BF16)
        return launch_fused<16, __nv_bfloat16>(q, pooled, n_rows, H, d, scale, scores, hist,
                                               n_hist, ticket, pf, rope_base, st);
    return launch_fused<16, float>(q, pooled, n_rows, H, d, scale, scores, hist, n_hist, ticket, pf,
                                   rope_base, st);
}

cudaError_t launch_index_score(const float *q, int64_t n_q, int64_t ld_q, const int32_t *q_pos,
                               const float *pooled, int64_t n_rows, int H, int d, float scale,
                               float *scores, int64_t ld_scores, uint32_t *hist, int64_t n_hist,
                               uint32_t *ticket, cudaStream_t st)
{
    if (n_q == 0 || n_rows == 0) return cudaSuccess;
    const int hd = H * d;
    const bool aligned = (reinterpret_cast<uintptr_t>(q) % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(pooled) % 16 == 0);
    if (n_q == 1 && q_pos == nullptr && aligned && hd % 128 == 0) {
        switch (hd / 128) {
            case 1: return launch_rows<1, 4>(q, pooled, n_rows, scale, scores, hist, n_hist, ticket, st);
            case 2: return launch_rows<2, 4>(q, pooled, n_rows, scale, scores, hist, n_hist, ticket, st);
            case 4: return launch_rows<4, 2>(q, pooled, n_rows, scale, scores, hist, n_hist, ticket, st);
            case 8: return launch_rows<8, 2>(q, pooled, n_rows, scale, scores, hist, n_hist, ticket, st);
            case 16: return launch_rows<16, 1>(q, pooled, n_rows, scale, scores, hist, n_hist, ticket, st);
            default: break;
        }
    }
    const dim3 grid((unsigned)((n_rows + kBN - 1) / kBN), (unsigned)((n_q + kBM - 1) / kBM));
    return launch(score_tiled_kernel, grid, dim3(256), 0, st, 1, q, n_q, ld_q, q_pos, pooled,
                  n_rows, hd, scale, scores, ld_scores, hist, n_hist, ticket);
}

}  // namespace qsa
