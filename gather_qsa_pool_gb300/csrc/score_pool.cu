// score_pool.cu -- the decode step's score kernel with the pooled-cache update folded in.
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, sections
// "incremental pooled-key cache (COMMON-004)" (each step recomputes only the open block
// and any newly completed one; completed rows are reused) and "QSA and the QSA indexer"
// (every pooled row is scored against the query).
//
// A decode step (one query, or a token with up to three draft tokens) recomputes at most
// a few pooled rows and then scans all of them.  One launch does both: CTA i < n_pool
// recomputes row row0 + i (pool -> RMS norm -> rotation), stores it and scores it for
// every query from shared memory; the other CTAs stream the rows [0, row0) that were
// already valid (score_stream.cuh), so the recomputation hides under the scan.
#include "score_stream.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 256;
constexpr int kHd = 2048;  // 16 heads x 128, the indexer shape of the pages' model

template <typename T, typename TP, int NQ>
__global__ void __launch_bounds__(kThreads)
score_pool_kernel(const float *__restrict__ q, TP *__restrict__ pooled, float scale,
                  float *__restrict__ scores, int64_t ld_s, const ScoreSide side,
                  const T *__restrict__ raw, int64_t n_ctx, int H, int d,
                  const float *__restrict__ w, float eps, int64_t row0, int n_pool,
                  const RopeTable tab)
{
    constexpr int CH = kHd * (int)sizeof(TP) / (16 * 32);  // 16-byte chunks per lane per row
    constexpr int R = stream_rows<TP, NQ>();
    __shared__ float4 q_s[NQ * (kHd / 4)];
    __shared__ __align__(16) float p_s[kHd];
    __shared__ float cs[kRopeMaxHalf], sn[kRopeMaxHalf];
    pdl_wait();
    QSA_AFTER_WAIT(q);
    QSA_AFTER_WAIT(pooled);
    QSA_AFTER_WAIT(raw);
    QSA_AFTER_WAIT(w);
    pdl_trigger();
    if (side.ticket && blockIdx.x == 0 && threadIdx.x < NQ)
        side.ticket[threadIdx.x * side.ticket_stride] = 0u;
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) stage_query<TP>(q + qi * kHd, kHd, q_s + qi * (kHd / 4));
    __syncthreads();
    if ((int)blockIdx.x < n_pool) {
        const int64_t b = row0 + blockIdx.x;
        pool_row(raw, n_ctx, H, d, w, eps, tab, b, p_s, cs, sn, pooled + b * (int64_t)kHd);
        if (threadIdx.x < 32) {
            float acc[NQ];
            score_row_smem<TP, CH, NQ>(q_s, p_s, acc);
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi)
                if ((int)threadIdx.x == qi) put_score(acc[qi] * scale, qi, b, scores, ld_s, side);
        }
        return;
    }
    int64_t lim[NQ];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) lim[qi] = INT64_MAX;
    const int64_t nw = (int64_t)(gridDim.x - n_pool) * (kThreads / 32);
    const int64_t gw = (int64_t)(blockIdx.x - n_pool) * (kThreads / 32) + (threadIdx.x >> 5);
    score_stream<TP, CH, NQ, R>(q_s, pooled, row0, gw, nw, scale, scores, ld_s, lim, side);
}

template <typename T, typename TP, int NQ>
cudaError_t launch_fused(const float *q, void *pooled, int H, int d, float scale, float *scores,
                         int64_t ld_s, const ScoreSide &side, const PoolFuse &pf,
                         const RopeTable &tab, cudaStream_t st)
{
    constexpr int R = stream_rows<TP, NQ>();
    auto k = score_pool_kernel<T, TP, NQ>;
    const int blocks_per_sm = occupancy_blocks<score_pool_kernel<T, TP, NQ>>(kThreads, 0);
    const int n_pool = (int)(pf.row1 - pf.row0);
    int64_t grid = (int64_t)device_sm_count() * blocks_per_sm;
    const int64_t warps_needed = (pf.row0 + R - 1) / R;
    const int64_t grid_needed = n_pool + (warps_needed + kThreads / 32 - 1) / (kThreads / 32);
    if (grid > grid_needed) grid = grid_needed;
    if (grid < n_pool + 1) grid = n_pool + 1;
    return launch(k, dim3((unsigned)grid), dim3(kThreads), 0, st, 1, q, (TP *)pooled, scale, scores,
                  ld_s, side, (const T *)pf.raw, pf.n_ctx, H, d, pf.w, pf.eps, pf.row0, n_pool, tab);
}

template <typename T, typename TP>
cudaError_t launch_fused_nq(int n_q, const float *q, void *pooled, int H, int d, float scale,
                            float *scores, int64_t ld_s, const ScoreSide &side,
                            const PoolFuse &pf, const RopeTable &tab, cudaStream_t st)
{
    switch (n_q) {
        case 1: return launch_fused<T, TP, 1>(q, pooled, H, d, scale, scores, ld_s, side, pf, tab, st);
        case 2: return launch_fused<T, TP, 2>(q, pooled, H, d, scale, scores, ld_s, side, pf, tab, st);
        case 3: return launch_fused<T, TP, 3>(q, pooled, H, d, scale, scores, ld_s, side, pf, tab, st);
        case 4: return launch_fused<T, TP, 4>(q, pooled, H, d, scale, scores, ld_s, side, pf, tab, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

cudaError_t launch_score_pool_fused(const float *q, int n_q, void *pooled, qsa_dtype pdt,
                                    int64_t n_rows, int H, int d, float scale, float *scores,
                                    int64_t ld_scores, const ScoreSide &side, const PoolFuse &pf,
                                    double rope_base, cudaStream_t st)
{
    const int64_t n_pool = pf.row1 - pf.row0;
    const bool aligned = (reinterpret_cast<uintptr_t>(q) % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(pooled) % 16 == 0);
    if (!aligned || H * d != kHd || d / 2 > kRopeMaxHalf || n_pool < 0 ||
        n_pool > kMaxFusedPoolRows || pf.row1 != n_rows || n_q < 1 || n_q > kMaxStreamQueries)
        return cudaErrorNotSupported;
    thread_local RopeTable tab;
    thread_local int tab_d = -1;
    thread_local double tab_base = 0.0;
    if (tab_d != d || tab_base != rope_base) {
        make_rope_table(&tab, d, rope_base);
        tab_d = d;
        tab_base = rope_base;
    }
    using bf = __nv_bfloat16;
    if (pf.dt == QSA_BF16)
        return pdt == QSA_BF16
                   ? launch_fused_nq<bf, bf>(n_q, q, pooled, H, d, scale, scores, ld_scores, side,
                                             pf, tab, st)
                   : launch_fused_nq<bf, float>(n_q, q, pooled, H, d, scale, scores, ld_scores,
                                                side, pf, tab, st);
    return pdt == QSA_BF16
               ? launch_fused_nq<float, bf>(n_q, q, pooled, H, d, scale, scores, ld_scores, side,
                                            pf, tab, st)
               : launch_fused_nq<float, float>(n_q, q, pooled, H, d, scale, scores, ld_scores,
                                               side, pf, tab, st);
}

}  // namespace qsa
