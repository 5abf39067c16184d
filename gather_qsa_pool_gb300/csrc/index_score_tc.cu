// index_score_tc.cu -- multi-query index scores on the tcgen05 tensor cores (bf16
// operands, fp32 accumulation in tensor memory).
#include "qsa_internal.cuh"

namespace qsa {

size_t index_score_tc_workspace(int64_t n_q, int64_t n_rows, int H, int d)
{
    (void)n_q; (void)n_rows; (void)H; (void)d;
    return 0;
}

qsa_status launch_index_score_tc(const float *q, int64_t n_q, int64_t ld_q,
                                 const int32_t *q_pos, const float *pooled, int64_t n_rows,
                                 int H, int d, float scale, float *scores, int64_t ld_scores,
                                 void *workspace, size_t ws_bytes, cudaStream_t st)
{
    (void)q; (void)n_q; (void)ld_q; (void)q_pos; (void)pooled; (void)n_rows; (void)H; (void)d;
    (void)scale; (void)scores; (void)ld_scores; (void)workspace; (void)ws_bytes; (void)st;
    return QSA_ERR_UNSUPPORTED;
}

}  // namespace qsa
