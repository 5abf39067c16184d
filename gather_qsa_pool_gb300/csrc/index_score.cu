// index_score.cu -- indexer scores of pooled rows against the queries (CUDA-core fp32).
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "QSA and the QSA indexer" (the query is scored against every pooled block summary)
// and section "incremental pooled-key cache (COMMON-004)" (after the cache fix, this
// scan is the one step left whose cost grows with context).
//
// Up to four queries (a decode step, or a token and its drafts): a pure HBM stream of the
// pooled cache, H*d*4 bytes per row (8 KB at 16 heads x 128; half that with bf16
// storage), every row read once for all the queries (score_stream.cuh).  A persistent
// grid of warps walks the rows; each lane issues all of its 16-byte streaming loads for
// a row (and the next) before reducing, so that every SM keeps ~100 KB in flight; the
// queries sit in shared memory.
// More queries (a prefill chunk in fp32): a register-tiled fp32 GEMM with the causal
// block visibility rule applied in the epilogue.
#include "score_stream.cuh"

namespace qsa {
namespace {

constexpr int kScoreThreads = 256;

template <typename TP, int CH, int NQ, int R>
__global__ void __launch_bounds__(kScoreThreads)
score_stream_kernel(const float *__restrict__ q, int64_t ld_q, const int32_t *__restrict__ q_pos,
                    const TP *__restrict__ pooled, int64_t n_rows, float scale,
                    float *__restrict__ scores, int64_t ld_s, const ScoreSide side)
{
    constexpr int kHd = CH * 32 * (16 / (int)sizeof(TP));
    __shared__ float4 q_s[NQ * (kHd / 4)];
    pdl_wait();
    QSA_AFTER_WAIT(q);
    QSA_AFTER_WAIT(q_pos);
    QSA_AFTER_WAIT(pooled);
    pdl_trigger();
    if (side.ticket && blockIdx.x == 0 && threadIdx.x < NQ)
        side.ticket[threadIdx.x * side.ticket_stride] = 0u;
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) stage_query<TP>(q + qi * ld_q, kHd, q_s + qi * (kHd / 4));
    int64_t lim[NQ];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi)
        lim[qi] = q_pos ? ((int64_t)q_pos[qi] + 1) / 4 : INT64_MAX;  // 4b + 3 <= p  <=>  b < lim
    __syncthreads();
    const int64_t nw = (int64_t)gridDim.x * (kScoreThreads / 32);
    const int64_t gw = (int64_t)blockIdx.x * (kScoreThreads / 32) + (threadIdx.x >> 5);
    score_stream<TP, CH, NQ, R>(q_s, pooled, n_rows, gw, nw, scale, scores, ld_s, lim, side);
}

// General case: scores[i][b] = scale * <q_i, pooled_b>, 64 queries x 64 rows per CTA,
// k-chunks of 16 staged in shared memory, 4x4 outputs per thread.
constexpr int kBM = 64, kBN = 64, kBK = 16;

template <typename TP>
__global__ void __launch_bounds__(256)
score_tiled_kernel(const float *__restrict__ q, int64_t n_q, int64_t ld_q,
                   const int32_t *__restrict__ q_pos, const TP *__restrict__ pooled,
                   int64_t n_rows, int hd, float scale, float *__restrict__ scores,
                   int64_t ld_scores, const ScoreSide side)
{
    __shared__ float a_s[kBK][kBM + 4];
    __shared__ float b_s[kBK][kBN + 4];
    pdl_wait();
    QSA_AFTER_WAIT(q);
    QSA_AFTER_WAIT(q_pos);
    QSA_AFTER_WAIT(pooled);
    pdl_trigger();
    if (side.ticket && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < n_q &&
        threadIdx.x < kMaxStreamQueries)
        side.ticket[threadIdx.x * side.ticket_stride] = 0u;
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
            b_s[kk][mm] = (gn < n_rows && k0 + kk < hd) ? to_f32(pooled[gn * hd + k0 + kk]) : 0.f;
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
            if (side.hist && gm < kMaxStreamQueries)
                put_score(sc, (int)gm, gn, scores, ld_scores, side);
            else
                scores[gm * ld_scores + gn] = sc;
        }
    }
}

template <typename TP, int CH, int NQ, int R>
cudaError_t launch_stream(const float *q, int64_t ld_q, const int32_t *q_pos, const void *pooled,
                          int64_t n_rows, float scale, float *scores, int64_t ld_s,
                          const ScoreSide &side, cudaStream_t st)
{
    auto k = score_stream_kernel<TP, CH, NQ, R>;
    const int blocks_per_sm = occupancy_blocks<score_stream_kernel<TP, CH, NQ, R>>(kScoreThreads, 0);
    const int64_t warps_needed = (n_rows + R - 1) / R;
    int64_t grid = (int64_t)device_sm_count() * blocks_per_sm;
    const int64_t grid_needed = (warps_needed + kScoreThreads / 32 - 1) / (kScoreThreads / 32);
    if (grid > grid_needed) grid = grid_needed;
    if (grid < 1) grid = 1;
    return launch(k, dim3((unsigned)grid), dim3(kScoreThreads), 0, st, 1, q, ld_q, q_pos,
                  (const TP *)pooled, n_rows, scale, scores, ld_s, side);
}

// The streaming form for this shape, or cudaErrorNotSupported when it has none.
cudaError_t dispatch_stream(const float *q, int64_t n_q, int64_t ld_q, const int32_t *q_pos,
                            const void *pooled, qsa_dtype pdt, int64_t n_rows, int hd,
                            float scale, float *scores, int64_t ld_s, const ScoreSide &side,
                            cudaStream_t st)
{
    using bf = __nv_bfloat16;
#define QSA_STREAM(TP, CH, NQ, R) \
    return launch_stream<TP, CH, NQ, R>(q, ld_q, q_pos, pooled, n_rows, scale, scores, ld_s, side, st)
    if (pdt == QSA_F32) {
        if (n_q == 1) {
            switch (hd) {
                case 128: QSA_STREAM(float, 1, 1, 4);
                case 256: QSA_STREAM(float, 2, 1, 4);
                case 512: QSA_STREAM(float, 4, 1, 2);
                case 1024: QSA_STREAM(float, 8, 1, 2);
                case 2048: QSA_STREAM(float, 16, 1, (stream_rows<float, 1>()));
                default: break;
            }
        } else if (hd == 2048) {
            switch (n_q) {
                case 2: QSA_STREAM(float, 16, 2, (stream_rows<float, 2>()));
                case 3: QSA_STREAM(float, 16, 3, (stream_rows<float, 3>()));
                case 4: QSA_STREAM(float, 16, 4, (stream_rows<float, 4>()));
                default: break;
            }
        }
    } else if (hd == 2048) {
        switch (n_q) {
            case 1: QSA_STREAM(bf, 8, 1, (stream_rows<bf, 1>()));
            case 2: QSA_STREAM(bf, 8, 2, (stream_rows<bf, 2>()));
            case 3: QSA_STREAM(bf, 8, 3, (stream_rows<bf, 3>()));
            case 4: QSA_STREAM(bf, 8, 4, (stream_rows<bf, 4>()));
            default: break;
        }
    } else if (hd == 256 && n_q == 1) {
        QSA_STREAM(bf, 1, 1, 4);
    }
#undef QSA_STREAM
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_index_score(const float *q, int64_t n_q, int64_t ld_q, const int32_t *q_pos,
                               const void *pooled, qsa_dtype pdt, int64_t n_rows, int H, int d,
                               float scale, float *scores, int64_t ld_scores,
                               const ScoreSide &side, cudaStream_t st)
{
    if (n_q == 0 || n_rows == 0) return cudaSuccess;
    const int hd = H * d;
    const bool aligned = (reinterpret_cast<uintptr_t>(q) % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(pooled) % 16 == 0) && ld_q % 4 == 0;
    if (n_q <= kMaxStreamQueries && aligned) {
        const cudaError_t e = dispatch_stream(q, n_q, ld_q, q_pos, pooled, pdt, n_rows, hd, scale,
                                              scores, ld_scores, side, st);
        if (e != cudaErrorNotSupported) return e;
    }
    const dim3 grid((unsigned)((n_rows + kBN - 1) / kBN), (unsigned)((n_q + kBM - 1) / kBM));
    if (pdt == QSA_BF16)
        return launch(score_tiled_kernel<__nv_bfloat16>, grid, dim3(256), 0, st, 1, q, n_q, ld_q,
                      q_pos, (const __nv_bfloat16 *)pooled, n_rows, hd, scale, scores, ld_scores,
                      side);
    return launch(score_tiled_kernel<float>, grid, dim3(256), 0, st, 1, q, n_q, ld_q, q_pos,
                  (const float *)pooled, n_rows, hd, scale, scores, ld_scores, side);
}

}  // namespace qsa
