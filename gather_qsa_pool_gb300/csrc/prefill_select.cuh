// prefill_select.cuh -- the prefill selection with group maxima: the tensor-core score kernel
// also writes, per query, the largest score of every 32 consecutive pooled rows, and the
// top-k reads only the groups that can hold a winner (index_score_tc.cu, topk_maxima.cu,
// topk.cu; entry points in capi.cu).
#pragma once

#include "qsa_internal.cuh"

namespace qsa {

// launch_index_score_tc, plus maxima[i][g] = the largest visible score of rows 32g ..
// min(32g + 32, n_rows) - 1 of query i (-inf when none is visible; NaN scores ignored),
// g < ceil(n_rows / 32), row stride ld_maxima (each epilogue thread stores a tile's eight
// groups together).
qsa_status launch_index_score_tc_maxima(const float *q, int64_t n_q, int64_t ld_q,
                                        const int32_t *q_pos, const void *pooled,
                                        qsa_dtype pdt, int64_t n_rows, int H, int d, float scale,
                                        float *scores, int64_t ld_scores, float *maxima,
                                        int64_t ld_maxima, void *workspace, size_t ws_bytes,
                                        cudaStream_t st);

// launch_topk (no cell lists, queries at q_pos or all at the end) given those maxima: the
// maxima kernel (topk_maxima.cu), then the general kernel for the queries it handed back.
// workspace: topk_maxima_workspace_bytes(n_q) bytes, 256-byte aligned (a counter and the
// list of handed-back queries).
size_t topk_maxima_workspace_bytes(int64_t n_q);
cudaError_t launch_topk_maxima(const float *scores, int64_t n_q, int64_t ld, const int32_t *q_pos,
                               int64_t n_full, int64_t k_blk, const float *maxima,
                               int64_t ld_maxima, int32_t *blocks_out, int32_t *counts_out,
                               void *workspace, cudaStream_t st);

// The general top-k (topk.cu) for the queries list[0 .. *count) only, on a persistent grid.
cudaError_t launch_topk_listed(const float *scores, int64_t n_q, int64_t ld, const int32_t *q_pos,
                               int64_t n_full, int64_t k_blk, int32_t *blocks_out,
                               int32_t *counts_out, const uint32_t *count, const int32_t *list,
                               cudaStream_t st);

}  // namespace qsa
