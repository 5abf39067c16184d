// capi.cu -- the extern "C" entry points: argument validation on the host, then one
// launcher call per operation.  No entry point allocates device memory, synchronises or
// keeps state beyond cached kernel attributes; decode plans are host objects the caller
// creates and destroys.
#include <math.h>
#include <stdlib.h>

#include <atomic>

#include "attn_union.cuh"
#include "prefill_select.cuh"
#include "qsa_internal.cuh"

namespace qsa {

int device_sm_count()
{
    constexpr int kMaxDevices = 64;
    static std::atomic<int> sms_of[kMaxDevices];  // 0: not yet asked (static: zero at start)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return kTargetSMs;
    }
    int sms = sms_of[dev].load();
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms <= 0) {
            (void)cudaGetLastError();
            sms = kTargetSMs;
        }
        sms_of[dev].store(sms);
    }
    return sms;
}

namespace {
thread_local WaitCtl t_wait_ctl = {nullptr, kWaitLimitNs};
}  // namespace

WaitCtl current_wait_ctl() { return t_wait_ctl; }

}  // namespace qsa

using namespace qsa;

namespace {

constexpr size_t kMaxSmem = 227 * 1024;

inline qsa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA; }
inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline bool valid_dtype(qsa_dtype d) { return d == QSA_F32 || d == QSA_BF16; }
inline int esize_of(qsa_dtype d) { return d == QSA_BF16 ? 2 : 4; }

}  // namespace

extern "C" {

const char *qsa_status_str(qsa_status s)
{
    switch (s) {
        case QSA_OK: return "QSA_OK";
        case QSA_ERR_INVALID_ARG: return "QSA_ERR_INVALID_ARG";
        case QSA_ERR_UNSUPPORTED: return "QSA_ERR_UNSUPPORTED";
        case QSA_ERR_CUDA: return "QSA_ERR_CUDA";
        case QSA_ERR_TIMEOUT: return "QSA_ERR_TIMEOUT";
    }
    return "QSA_ERR_UNKNOWN";
}

int qsa_version(void) { return (2 << 16) | 4; }

void qsa_set_wait_options(int32_t *status_out, uint64_t pipeline_limit_ns)
{
    t_wait_ctl.status = status_out;
    t_wait_ctl.limit_ns = pipeline_limit_ns;
}

static qsa_status check_pool_update(const void *raw_k, qsa_dtype raw_dtype, int64_t n_ctx, int H,
                                    int d, const float *norm_w, float eps, double rope_base,
                                    const void *pooled, qsa_dtype pooled_dtype, int64_t cap_rows,
                                    int64_t n_valid_full)
{
    if (!raw_k || !norm_w || !pooled) return QSA_ERR_INVALID_ARG;
    if (!valid_dtype(raw_dtype) || !valid_dtype(pooled_dtype) || n_ctx < 0 || H < 1 || d < 2 ||
        (d & 1) || n_valid_full < 0 || cap_rows < 0 || !(eps >= 0.0f) || !(rope_base > 0.0))
        return QSA_ERR_INVALID_ARG;
    if (!aligned(raw_k, esize_of(raw_dtype)) || !aligned(norm_w, 4) ||
        !aligned(pooled, esize_of(pooled_dtype)))
        return QSA_ERR_INVALID_ARG;
    const int64_t n_rows = (n_ctx + 3) / 4;
    const int64_t n_full = n_ctx / 4;
    if (n_rows > cap_rows) return QSA_ERR_INVALID_ARG;
    if ((int64_t)H * d > 48 * 1024) return QSA_ERR_UNSUPPORTED;  // row staged in shared memory
    if (d / 2 > kRopeMaxHalf) return QSA_ERR_UNSUPPORTED;
    const int64_t row0 = n_valid_full < n_full ? n_valid_full : n_full;
    if (n_rows - row0 > 0x7fffffffLL) return QSA_ERR_UNSUPPORTED;
    return QSA_OK;
}

static cudaError_t run_pool_update(const void *raw_k, qsa_dtype raw_dtype, int64_t n_ctx, int H,
                                   int d, const float *norm_w, float eps, double rope_base,
                                   void *pooled, qsa_dtype pooled_dtype, int64_t n_valid_full,
                                   uint32_t *zero_hist, cudaStream_t st)
{
    const int64_t n_rows = (n_ctx + 3) / 4;
    const int64_t n_full = n_ctx / 4;
    const int64_t row0 = n_valid_full < n_full ? n_valid_full : n_full;
    return launch_pool_update(raw_k, raw_dtype, n_ctx, H, d, norm_w, eps, rope_base, pooled,
                              pooled_dtype, row0, n_rows, zero_hist, st);
}

qsa_status qsa_pool_update(const void *raw_k, qsa_dtype raw_dtype, int64_t n_ctx, int H, int d,
                           const float *norm_w, float eps, double rope_base, void *pooled,
                           qsa_dtype pooled_dtype, int64_t cap_rows, int64_t n_valid_full,
                           qsa_stream_t stream)
{
    const qsa_status v = check_pool_update(raw_k, raw_dtype, n_ctx, H, d, norm_w, eps, rope_base,
                                           pooled, pooled_dtype, cap_rows, n_valid_full);
    if (v != QSA_OK) return v;
    return from_cuda(run_pool_update(raw_k, raw_dtype, n_ctx, H, d, norm_w, eps, rope_base, pooled,
                                     pooled_dtype, n_valid_full, nullptr, (cudaStream_t)stream));
}

size_t qsa_index_score_workspace_size(int64_t n_q, int64_t n_rows, int H, int d,
                                      qsa_dtype pooled_dtype, qsa_precision precision)
{
    if (precision != QSA_PREC_BF16_TC || n_q <= 0 || n_rows <= 0 || H < 1 || d < 1 ||
        !valid_dtype(pooled_dtype))
        return 0;
    return index_score_tc_workspace(n_q, n_rows, H, d, pooled_dtype);
}

static qsa_status check_index_score(const float *q, int64_t n_q, int64_t ld_q, const void *pooled,
                                    qsa_dtype pooled_dtype, int64_t n_rows, int H, int d,
                                    float *scores, int64_t ld_scores)
{
    if (!q || !pooled || !scores) return QSA_ERR_INVALID_ARG;
    if (n_q < 0 || n_rows < 0 || H < 1 || d < 1 || ld_q < (int64_t)H * d || ld_scores < n_rows ||
        !valid_dtype(pooled_dtype))
        return QSA_ERR_INVALID_ARG;
    if (!aligned(q, 4) || !aligned(pooled, esize_of(pooled_dtype)) || !aligned(scores, 4))
        return QSA_ERR_INVALID_ARG;
    if ((n_q + 63) / 64 > 65535) return QSA_ERR_UNSUPPORTED;
    return QSA_OK;
}

qsa_status qsa_index_score(const float *q, int64_t n_q, int64_t ld_q, const int32_t *q_pos,
                           const void *pooled, qsa_dtype pooled_dtype, int64_t n_rows, int H,
                           int d, float scale, float *scores, int64_t ld_scores,
                           qsa_precision precision, void *workspace, size_t workspace_bytes,
                           qsa_stream_t stream)
{
    const qsa_status v = check_index_score(q, n_q, ld_q, pooled, pooled_dtype, n_rows, H, d,
                                           scores, ld_scores);
    if (v != QSA_OK) return v;
    if (precision == QSA_PREC_F32) {
        return from_cuda(launch_index_score(q, n_q, ld_q, q_pos, pooled, pooled_dtype, n_rows, H,
                                            d, scale, scores, ld_scores, ScoreSide{},
                                            (cudaStream_t)stream));
    }
    if (precision == QSA_PREC_BF16_TC) {
        const size_t need =
            qsa_index_score_workspace_size(n_q, n_rows, H, d, pooled_dtype, precision);
        if (workspace_bytes < need || (need > 0 && !workspace)) return QSA_ERR_INVALID_ARG;
        return launch_index_score_tc(q, n_q, ld_q, q_pos, pooled, pooled_dtype, n_rows, H, d,
                                     scale, scores, ld_scores, workspace, workspace_bytes,
                                     (cudaStream_t)stream);
    }
    return QSA_ERR_INVALID_ARG;
}

int64_t qsa_topk_max_candidates(void) { return topk_max_candidates(); }

static qsa_status check_topk(const float *scores, int64_t n_q, int64_t ld_scores, int64_t n_full,
                             int64_t k_blk, int32_t *blocks_out, int32_t *counts_out)
{
    if (!scores || !blocks_out || !counts_out) return QSA_ERR_INVALID_ARG;
    if (n_q < 0 || k_blk < 1 || n_full < 0 || ld_scores < n_full) return QSA_ERR_INVALID_ARG;
    if (k_blk > 0x7fffffffLL) return QSA_ERR_UNSUPPORTED;
    if (n_full > topk_max_candidates()) return QSA_ERR_UNSUPPORTED;
    if (n_q > 0x7fffffffLL) return QSA_ERR_UNSUPPORTED;
    return QSA_OK;
}

qsa_status qsa_topk_blocks(const float *scores, int64_t n_q, int64_t ld_scores,
                           const int32_t *q_pos, int64_t n_full, int64_t k_blk,
                           int32_t *blocks_out, int32_t *counts_out, qsa_stream_t stream)
{
    const qsa_status v = check_topk(scores, n_q, ld_scores, n_full, k_blk, blocks_out, counts_out);
    if (v != QSA_OK) return v;
    return from_cuda(launch_topk(scores, n_q, ld_scores, q_pos, n_full, k_blk, blocks_out,
                                 counts_out, 0, nullptr, nullptr, 0, nullptr, (cudaStream_t)stream));
}

qsa_status qsa_index_score_maxima(const float *q, int64_t n_q, int64_t ld_q,
                                  const int32_t *q_pos, const void *pooled,
                                  qsa_dtype pooled_dtype, int64_t n_rows, int H, int d,
                                  float scale, float *scores, int64_t ld_scores, float *maxima,
                                  int64_t ld_maxima, void *workspace, size_t workspace_bytes,
                                  qsa_stream_t stream)
{
    const qsa_status v = check_index_score(q, n_q, ld_q, pooled, pooled_dtype, n_rows, H, d,
                                           scores, ld_scores);
    if (v != QSA_OK) return v;
    if (!maxima || !aligned(maxima, 4) || ld_maxima < (n_rows + 31) / 32)
        return QSA_ERR_INVALID_ARG;
    const size_t need =
        qsa_index_score_workspace_size(n_q, n_rows, H, d, pooled_dtype, QSA_PREC_BF16_TC);
    if (workspace_bytes < need || (need > 0 && !workspace)) return QSA_ERR_INVALID_ARG;
    return launch_index_score_tc_maxima(q, n_q, ld_q, q_pos, pooled, pooled_dtype, n_rows, H, d,
                                        scale, scores, ld_scores, maxima, ld_maxima, workspace,
                                        workspace_bytes, (cudaStream_t)stream);
}

qsa_status qsa_topk_blocks_maxima(const float *scores, int64_t n_q, int64_t ld_scores,
                                  const int32_t *q_pos, int64_t n_full, int64_t k_blk,
                                  const float *maxima, int64_t ld_maxima, int32_t *blocks_out,
                                  int32_t *counts_out, void *workspace, size_t workspace_bytes,
                                  qsa_stream_t stream)
{
    const qsa_status v = check_topk(scores, n_q, ld_scores, n_full, k_blk, blocks_out, counts_out);
    if (v != QSA_OK) return v;
    if (!maxima || !aligned(maxima, 4) || ld_maxima < n_full / 32) return QSA_ERR_INVALID_ARG;
    const size_t need = topk_maxima_workspace_bytes(n_q);
    if (workspace_bytes < need || (need > 0 && (!workspace || !aligned(workspace, 256))))
        return QSA_ERR_INVALID_ARG;
    return from_cuda(launch_topk_maxima(scores, n_q, ld_scores, q_pos, n_full, k_blk, maxima,
                                        ld_maxima, blocks_out, counts_out, workspace,
                                        (cudaStream_t)stream));
}

size_t qsa_topk_blocks_maxima_workspace_size(int64_t n_q) { return topk_maxima_workspace_bytes(n_q); }

qsa_status qsa_expand_block_scores(const float *scores, int64_t n_q, int64_t ld_scores,
                                   int64_t n_full, float *cell_scores, int64_t ld_cells,
                                   qsa_stream_t stream)
{
    if (!scores || !cell_scores) return QSA_ERR_INVALID_ARG;
    if (n_q < 0 || n_full < 0 || ld_scores < n_full || ld_cells < 4 * n_full)
        return QSA_ERR_INVALID_ARG;
    if (!aligned(scores, 4) || !aligned(cell_scores, 4)) return QSA_ERR_INVALID_ARG;
    if (n_q > 65535) return QSA_ERR_UNSUPPORTED;
    return from_cuda(launch_expand_scores(scores, n_q, ld_scores, n_full, cell_scores, ld_cells,
                                          (cudaStream_t)stream));
}

static qsa_status check_gather(const void *K, const void *V, qsa_dtype dtype, int64_t n_kv,
                               int H_kv, int d_k, int d_v, int64_t ld_k, int64_t ld_v,
                               const int32_t *blocks, const int32_t *counts, int64_t n_q,
                               int64_t k_blk, const int32_t *q_pos, int64_t n_ctx, void *K_out,
                               void *V_out, int32_t *pos_out, int32_t *n_cells_out,
                               int64_t max_cells)
{
    if (!blocks || !counts || !pos_out || !n_cells_out) return QSA_ERR_INVALID_ARG;
    if ((K_out && !K) || (V_out && !V)) return QSA_ERR_INVALID_ARG;
    if (!valid_dtype(dtype) || n_kv < 0 || n_q < 0 || k_blk < 1 || max_cells < 4 * k_blk + 3)
        return QSA_ERR_INVALID_ARG;
    if (!q_pos && n_ctx < 0) return QSA_ERR_INVALID_ARG;
    if ((K_out || V_out) && (H_kv < 1 || d_k < 1 || d_v < 1 || ld_k < (int64_t)H_kv * d_k ||
                             ld_v < (int64_t)H_kv * d_v))
        return QSA_ERR_INVALID_ARG;
    if (n_q > 65535 || max_cells > 0x7fffffffLL) return QSA_ERR_UNSUPPORTED;
    return QSA_OK;
}

qsa_status qsa_gather_kv(const void *K, const void *V, qsa_dtype dtype, int64_t n_kv, int H_kv,
                         int d_k, int d_v, int64_t ld_k, int64_t ld_v, const int32_t *blocks,
                         const int32_t *counts, int64_t n_q, int64_t k_blk,
                         const int32_t *q_pos, int64_t n_ctx, void *K_out, void *V_out,
                         int32_t *pos_out, int32_t *n_cells_out, int64_t max_cells,
                         qsa_stream_t stream)
{
    const qsa_status v = check_gather(K, V, dtype, n_kv, H_kv, d_k, d_v, ld_k, ld_v, blocks, counts,
                                      n_q, k_blk, q_pos, n_ctx, K_out, V_out, pos_out, n_cells_out,
                                      max_cells);
    if (v != QSA_OK) return v;
    return from_cuda(launch_gather(K, V, dtype, n_kv, H_kv, d_k, d_v, ld_k, ld_v, blocks, counts,
                                   n_q, k_blk, q_pos, n_ctx, K_out, V_out, pos_out, n_cells_out,
                                   max_cells, (cudaStream_t)stream));
}

size_t qsa_sparse_attn_workspace_size(int64_t n_q, int H_q, int H_kv, int d_v, int64_t max_cells)
{
    if (n_q <= 0 || H_q < 1 || H_kv < 1 || d_v < 1 || max_cells < 0 || H_q % H_kv) return 0;
    return attn_workspace_bytes(n_q, H_q, H_kv, d_v, max_cells);
}

static qsa_status check_attn(const float *q, int64_t n_q, int H_q, int H_kv, int d_k, int d_v,
                             const void *K, const void *V, qsa_dtype dtype, int64_t n_kv,
                             int64_t ld_k, int64_t ld_v, const int32_t *pos,
                             const int32_t *n_cells, int64_t max_cells, float *out,
                             void *workspace, size_t workspace_bytes)
{
    if (!q || !K || !V || !n_cells || !out) return QSA_ERR_INVALID_ARG;
    if (!valid_dtype(dtype) || n_q < 0 || H_q < 1 || H_kv < 1 || H_q % H_kv || d_k < 8 ||
        d_v < 8 || d_k % 8 || d_v % 8 || n_kv < 0 || max_cells < 0 || ld_k % 8 || ld_v % 8)
        return QSA_ERR_INVALID_ARG;
    if (ld_k < (int64_t)H_kv * d_k || ld_v < (int64_t)H_kv * d_v) return QSA_ERR_INVALID_ARG;
    if (!aligned(K, 16) || !aligned(V, 16) || !aligned(q, 4) || !aligned(out, 4))
        return QSA_ERR_INVALID_ARG;
    const int G = H_q / H_kv;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return QSA_ERR_UNSUPPORTED;
    if (attn_smem_bytes_host(G, d_k, d_v, esize_of(dtype)) > kMaxSmem) return QSA_ERR_UNSUPPORTED;
    if (n_q > 65535 || H_kv > 65535) return QSA_ERR_UNSUPPORTED;
    if (n_kv > 0x7fffffffLL || n_q * max_cells > 0x7fffffffLL) return QSA_ERR_UNSUPPORTED;
    // the split-K records the kernel these arguments select really writes (none for the
    // forms that merge in a cluster)
    const size_t need =
        attn_partials_bytes(dtype, n_q, H_q, H_kv, d_k, d_v, K, V, ld_k, ld_v, pos, max_cells);
    if (workspace_bytes < need || (need > 0 && !workspace)) return QSA_ERR_INVALID_ARG;
    if (need > 0 && !aligned(workspace, 16)) return QSA_ERR_INVALID_ARG;
    return QSA_OK;
}

qsa_status qsa_sparse_attn(const float *q, int64_t n_q, int H_q, int H_kv, int d_k, int d_v,
                           float scale, const void *K, const void *V, qsa_dtype dtype,
                           int64_t n_kv, int64_t ld_k, int64_t ld_v, const int32_t *pos,
                           const int32_t *n_cells, int64_t max_cells, float *out,
                           float *lse_out, void *workspace, size_t workspace_bytes,
                           qsa_stream_t stream)
{
    const qsa_status v = check_attn(q, n_q, H_q, H_kv, d_k, d_v, K, V, dtype, n_kv, ld_k, ld_v,
                                    pos, n_cells, max_cells, out, workspace, workspace_bytes);
    if (v != QSA_OK) return v;
    // the latent form reads the query in 8-byte pairs
    if (H_kv == 1 && attn_uses_wide(dtype, d_k, d_v, H_q / H_kv, K, V, ld_k, ld_v) &&
        !aligned(q, 8))
        return QSA_ERR_INVALID_ARG;
    return from_cuda(launch_sparse_attn(q, n_q, H_q, H_kv, d_k, d_v, scale, K, V, dtype, n_kv,
                                        ld_k, ld_v, pos, n_cells, max_cells, out, lse_out,
                                        (float *)workspace, (cudaStream_t)stream));
}

size_t qsa_sparse_attn_union_workspace_size(int64_t n_q, int64_t max_cells)
{
    if (n_q <= 0 || max_cells < 0) return 0;
    return attn_union_workspace_bytes(n_q, max_cells);
}

qsa_status qsa_sparse_attn_union(const float *q, int64_t n_q, int H_q, int H_kv, int d,
                                 float scale, const void *K, const void *V, qsa_dtype dtype,
                                 int64_t n_kv, int64_t ld_k, int64_t ld_v, const int32_t *pos,
                                 const int32_t *n_cells, int64_t max_cells, float *out,
                                 float *lse_out, void *workspace, size_t workspace_bytes,
                                 qsa_stream_t stream)
{
    if (!q || !K || !V || !pos || !n_cells || !out) return QSA_ERR_INVALID_ARG;
    if (n_q < 0 || H_q < 1 || H_kv < 1 || d < 1 || n_kv < 0 || max_cells < 0 || ld_k < 0 ||
        ld_v < 0 || !valid_dtype(dtype))
        return QSA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || (lse_out && !aligned(lse_out, 4)) ||
        !aligned(pos, 4) || !aligned(n_cells, 4))
        return QSA_ERR_INVALID_ARG;
    if (!attn_union_shape_ok(dtype, H_q, H_kv, d, d, K, V, ld_k, ld_v)) return QSA_ERR_UNSUPPORTED;
    if (n_kv < 4 || n_kv > attn_union_max_kv() || max_cells > 2100 || H_kv > 65535 ||
        (n_q + kUnionGroup - 1) / kUnionGroup > 0x7fffffffLL)
        return QSA_ERR_UNSUPPORTED;
    if (n_q == 0) return QSA_OK;
    const size_t need = attn_union_workspace_bytes(n_q, max_cells);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return QSA_ERR_INVALID_ARG;
    return launch_attn_union(q, n_q, H_q, H_kv, scale, K, V, n_kv, ld_k, ld_v, pos, n_cells,
                             max_cells, out, lse_out, workspace, (cudaStream_t)stream);
}

static size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

size_t qsa_decode_step_workspace_size(int64_t n_q, int H_q, int H_kv, int d, int64_t max_cells,
                                      int64_t cap_rows)
{
    if (n_q < 1 || n_q > kMaxStreamQueries || H_q < 1 || H_kv < 1 || d < 1 || max_cells < 0 ||
        H_q % H_kv || cap_rows < 0)
        return 0;
    return align256(attn_workspace_bytes(n_q, H_q, H_kv, d, max_cells)) +
           (size_t)n_q * (kTopkHistBytes + topk_select_workspace_bytes(cap_rows));
}

// A decode step fed from host memory: the new tokens' rows go into the caches and the
// queries into `staging`, and the outputs come back to h_out / h_lse.  A host buffer that
// is mapped into the device's address space is read / written in place by the copy kernel;
// any other goes through a copy-engine transfer (inputs: one copy into `staging`, which the
// copy kernel then scatters).
struct HostFeed {
    const void *h_in;
    size_t in_bytes;
    char *staging;
    int64_t off[5];  // new raw rows, new K rows, new V rows, q_idx, q
    float *h_out;
    float *h_lse;
};

static qsa_status decode_step_impl(const void *raw_k, qsa_dtype raw_dtype, int64_t n_ctx, int H_idx,
                                   int d_idx, const float *norm_w, float eps, double rope_base,
                                   void *pooled, qsa_dtype pooled_dtype, int64_t cap_rows,
                                   int64_t n_valid_full, int64_t n_q, const float *q_idx,
                                   float scale_idx, float *scores, int64_t k_blk, int32_t *blocks,
                                   int32_t *counts, const void *K, const void *V,
                                   qsa_dtype kv_dtype, int64_t n_kv, int H_kv, int d, int64_t ld_kv,
                                   int32_t *pos, int32_t *n_cells, int64_t max_cells,
                                   const float *q, int H_q, float scale, float *out, float *lse_out,
                                   void *workspace, size_t workspace_bytes, qsa_stream_t stream,
                                   const HostFeed *feed)
{
    if (n_q < 1 || n_q > kMaxStreamQueries || n_q > n_ctx) return QSA_ERR_INVALID_ARG;
    const int64_t n_rows = (n_ctx + 3) / 4;
    const int64_t n_full = n_ctx / 4;
    const size_t need = qsa_decode_step_workspace_size(n_q, H_q, H_kv, d, max_cells, cap_rows);
    if (!workspace || need == 0 || workspace_bytes < need || !aligned(workspace, 256))
        return QSA_ERR_INVALID_ARG;
    const size_t attn_bytes = align256(attn_workspace_bytes(n_q, H_q, H_kv, d, max_cells));
    const size_t sel_stride = topk_select_workspace_bytes(cap_rows);
    char *wsb = static_cast<char *>(workspace);
    // workspace: attention partials | n_q histograms | n_q top-k scratch areas (each
    // starting with the query's arrival ticket)
    uint32_t *hist = reinterpret_cast<uint32_t *>(wsb + attn_bytes);
    void *sel = wsb + attn_bytes + (size_t)n_q * kTopkHistBytes;
    qsa_status v = check_pool_update(raw_k, raw_dtype, n_ctx, H_idx, d_idx, norm_w, eps,
                                     rope_base, pooled, pooled_dtype, cap_rows, n_valid_full);
    if (v == QSA_OK)
        v = check_index_score(q_idx, n_q, (int64_t)H_idx * d_idx, pooled, pooled_dtype, n_rows,
                              H_idx, d_idx, scores, n_rows);
    if (v == QSA_OK) v = check_topk(scores, n_q, n_rows, n_full, k_blk, blocks, counts);
    if (v == QSA_OK)
        v = check_gather(K, V, kv_dtype, n_kv, H_kv, d, d, ld_kv, ld_kv, blocks, counts, n_q,
                         k_blk, nullptr, n_ctx, nullptr, nullptr, pos, n_cells, max_cells);
    if (v == QSA_OK)
        v = check_attn(q, n_q, H_q, H_kv, d, d, K, V, kv_dtype, n_kv, ld_kv, ld_kv, pos, n_cells,
                       max_cells, out, workspace, attn_bytes);
    if (v != QSA_OK) return v;
    const cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaSuccess;
    if (feed) {
        // 0. this step's inputs from host memory: the new rows into the caches, the queries
        // into the staging area
        const int64_t re = raw_dtype == QSA_BF16 ? 2 : 4, ke = kv_dtype == QSA_BF16 ? 2 : 4;
        const int64_t hd = (int64_t)H_idx * d_idx, p0 = n_ctx - n_q;
        const char *in = static_cast<const char *>(mapped_host_view(feed->h_in));
        if (!in || !aligned(in, 4)) {
            e = cudaMemcpyAsync(feed->staging, feed->h_in, feed->in_bytes,
                                cudaMemcpyHostToDevice, st);
            if (e != cudaSuccess) return QSA_ERR_CUDA;
            in = feed->staging;
        }
        RowCopy job[4];
        job[0] = {in + feed->off[0], (char *)raw_k + p0 * hd * re, hd * re, hd * re, n_q};
        job[1] = {in + feed->off[1], (char *)K + p0 * ld_kv * ke, (int64_t)H_kv * d * ke,
                  ld_kv * ke, n_q};
        job[2] = {in + feed->off[2], (char *)V + p0 * ld_kv * ke, (int64_t)H_kv * d * ke,
                  ld_kv * ke, n_q};
        const int64_t qb = (int64_t)feed->in_bytes - feed->off[3];
        job[3] = {in + feed->off[3], feed->staging + feed->off[3], qb, qb, 1};
        e = launch_copy_rows(job, in == feed->staging ? 3 : 4, st);
        if (e != cudaSuccess) return QSA_ERR_CUDA;
    }
    // Query i sits at position p_i = n_ctx - n_q + i; its candidates are the blocks complete
    // there.  The score kernel counts each query's candidates into its histogram and resets
    // each query's arrival ticket.
    ScoreSide side;
    side.hist = hist;
    for (int i = 0; i < n_q; ++i) {
        const int64_t p1 = (n_ctx - n_q + i + 1) / 4;
        side.n_hist[i] = p1 < n_full ? p1 : n_full;
    }
    side.ticket = topk_select_ticket(sel);
    side.ticket_stride = (int64_t)(sel_stride / sizeof(uint32_t));
    // 1+2. pooled rows of the new / open blocks, then scores of every row for every query.
    // One kernel when the rows to recompute are few (the decode case), else the
    // pool-update kernel (which also clears the histograms) followed by the score kernel.
    const int64_t row0 = n_valid_full < n_full ? n_valid_full : n_full;
    PoolFuse pf;
    pf.raw = raw_k;
    pf.dt = raw_dtype;
    pf.n_ctx = n_ctx;
    pf.w = norm_w;
    pf.eps = eps;
    pf.row0 = row0;
    pf.row1 = n_rows;
    e = launch_score_pool_fused(q_idx, (int)n_q, pooled, pooled_dtype, n_rows, H_idx, d_idx,
                                scale_idx, scores, n_rows, side, pf, rope_base, st);
    if (e == cudaErrorNotSupported) {
        e = run_pool_update(raw_k, raw_dtype, n_ctx, H_idx, d_idx, norm_w, eps, rope_base, pooled,
                            pooled_dtype, n_valid_full, nullptr, st);
        if (e == cudaSuccess)
            e = launch_index_score(q_idx, n_q, (int64_t)H_idx * d_idx, nullptr, pooled,
                                   pooled_dtype, n_rows, H_idx, d_idx, scale_idx, scores, n_rows,
                                   side, st);
    }
    // 3. top-k from those histograms; the last CTA of each query also writes its cell list
    // (qsa_gather_kv's job).  When a query's blocks are all selected, the one-CTA form does it.
    if (e == cudaSuccess) {
        e = launch_topk_select(scores, n_rows, (int)n_q, n_full, cap_rows, k_blk, n_ctx, hist, sel,
                               blocks, counts, pos, n_cells, max_cells, st);
        if (e == cudaErrorNotSupported)
            e = launch_topk(scores, n_q, n_rows, nullptr, n_full, k_blk, blocks, counts, n_ctx, pos,
                            n_cells, max_cells, hist, st, 1);
    }
    // 4. attention over the listed cells, read in place from the cache.  Fed from host
    // memory, the tensor-core form also writes the outputs straight into mapped page-locked
    // host buffers (no copy kernel after it).
    float *ho_direct = nullptr, *hl_direct = nullptr;
    if (feed && attn_writes_host(kv_dtype, n_q, H_q, H_kv, d, d, K, V, ld_kv, ld_kv, pos,
                                 max_cells)) {
        float *ho = static_cast<float *>(mapped_host_view(feed->h_out));
        float *hl = feed->h_lse ? static_cast<float *>(mapped_host_view(feed->h_lse)) : nullptr;
        if (ho && aligned(ho, 4) && (!feed->h_lse || (hl && aligned(hl, 4)))) {
            ho_direct = ho;
            hl_direct = hl;
        }
    }
    if (e == cudaSuccess)
        e = launch_sparse_attn(q, n_q, H_q, H_kv, d, d, scale, K, V, kv_dtype, n_kv, ld_kv, ld_kv,
                               pos, n_cells, max_cells, out, lse_out, (float *)workspace, st,
                               true, ho_direct, hl_direct);
    // 5. the outputs back to host memory (unless the attention wrote them there)
    if (feed && e == cudaSuccess && !ho_direct) {
        const int64_t ob = (int64_t)sizeof(float) * n_q * H_q * d;
        const int64_t lb = (int64_t)sizeof(float) * n_q * H_q;
        void *ho = mapped_host_view(feed->h_out);
        void *hl = feed->h_lse ? mapped_host_view(feed->h_lse) : nullptr;
        if (ho && aligned(ho, 4) && aligned(out, 4) &&
            (!feed->h_lse || (hl && aligned(hl, 4) && aligned(lse_out, 4)))) {
            RowCopy job[2];
            job[0] = {out, ho, ob, ob, 1};
            job[1] = {lse_out, hl, lb, lb, 1};
            e = launch_copy_rows(job, hl ? 2 : 1, st);
        } else {
            e = cudaMemcpyAsync(feed->h_out, out, (size_t)ob, cudaMemcpyDeviceToHost, st);
            if (e == cudaSuccess && feed->h_lse)
                e = cudaMemcpyAsync(feed->h_lse, lse_out, (size_t)lb, cudaMemcpyDeviceToHost, st);
        }
    }
    return from_cuda(e);
}

qsa_status qsa_decode_step(const void *raw_k, qsa_dtype raw_dtype, int64_t n_ctx, int H_idx,
                           int d_idx, const float *norm_w, float eps, double rope_base,
                           void *pooled, qsa_dtype pooled_dtype, int64_t cap_rows,
                           int64_t n_valid_full, int64_t n_q, const float *q_idx, float scale_idx,
                           float *scores, int64_t k_blk, int32_t *blocks, int32_t *counts,
                           const void *K, const void *V, qsa_dtype kv_dtype, int64_t n_kv,
                           int H_kv, int d, int64_t ld_kv, int32_t *pos, int32_t *n_cells,
                           int64_t max_cells, const float *q, int H_q, float scale, float *out,
                           float *lse_out, void *workspace, size_t workspace_bytes,
                           qsa_stream_t stream)
{
    return decode_step_impl(raw_k, raw_dtype, n_ctx, H_idx, d_idx, norm_w, eps, rope_base, pooled,
                            pooled_dtype, cap_rows, n_valid_full, n_q, q_idx, scale_idx, scores,
                            k_blk, blocks, counts, K, V, kv_dtype, n_kv, H_kv, d, ld_kv, pos,
                            n_cells, max_cells, q, H_q, scale, out, lse_out, workspace,
                            workspace_bytes, stream, nullptr);
}

static int64_t a16(int64_t b) { return (b + 15) & ~(int64_t)15; }

size_t qsa_decode_step_host_layout(int64_t n_q, qsa_dtype raw_dtype, int H_idx, int d_idx,
                                   qsa_dtype kv_dtype, int H_kv, int d, int H_q, int64_t *offsets)
{
    if (n_q < 1 || n_q > kMaxStreamQueries || !valid_dtype(raw_dtype) || !valid_dtype(kv_dtype) ||
        H_idx < 1 || d_idx < 1 || H_kv < 1 || d < 1 || H_q < 1)
        return 0;
    const int64_t re = esize_of(raw_dtype), ke = esize_of(kv_dtype);
    int64_t off[5];
    off[0] = 0;
    off[1] = a16(off[0] + n_q * H_idx * d_idx * re);
    off[2] = a16(off[1] + n_q * H_kv * d * ke);
    off[3] = a16(off[2] + n_q * H_kv * d * ke);
    off[4] = a16(off[3] + n_q * H_idx * d_idx * 4);
    const int64_t total = a16(off[4] + n_q * H_q * d * 4);
    if (offsets)
        for (int i = 0; i < 5; ++i) offsets[i] = off[i];
    return (size_t)total;
}

size_t qsa_decode_step_host_workspace_size(int64_t n_q, int H_q, int H_kv, int d,
                                           int64_t max_cells, int64_t cap_rows,
                                           qsa_dtype raw_dtype, int H_idx, int d_idx,
                                           qsa_dtype kv_dtype)
{
    const size_t ws = qsa_decode_step_workspace_size(n_q, H_q, H_kv, d, max_cells, cap_rows);
    const size_t in = qsa_decode_step_host_layout(n_q, raw_dtype, H_idx, d_idx, kv_dtype, H_kv, d,
                                                  H_q, nullptr);
    if (ws == 0 || in == 0) return 0;
    return align256(ws) + align256(in);
}

qsa_status qsa_decode_step_host(const void *h_in, float *h_out, float *h_lse, void *raw_k,
                                qsa_dtype raw_dtype, int64_t n_ctx, int H_idx, int d_idx,
                                const float *norm_w, float eps, double rope_base, void *pooled,
                                qsa_dtype pooled_dtype, int64_t cap_rows, int64_t n_valid_full,
                                int64_t n_q, float scale_idx, float *scores, int64_t k_blk,
                                int32_t *blocks, int32_t *counts, void *K, void *V,
                                qsa_dtype kv_dtype, int64_t n_kv, int H_kv, int d, int64_t ld_kv,
                                int32_t *pos, int32_t *n_cells, int64_t max_cells, int H_q,
                                float scale, float *out, float *lse_out, void *workspace,
                                size_t workspace_bytes, qsa_stream_t stream)
{
    if (!h_in || !h_out || (h_lse && !lse_out) || !raw_k || !K || !V || !workspace)
        return QSA_ERR_INVALID_ARG;
    HostFeed feed;
    feed.in_bytes = qsa_decode_step_host_layout(n_q, raw_dtype, H_idx, d_idx, kv_dtype, H_kv, d,
                                                H_q, feed.off);
    const size_t ws = qsa_decode_step_workspace_size(n_q, H_q, H_kv, d, max_cells, cap_rows);
    if (feed.in_bytes == 0 || ws == 0) return QSA_ERR_INVALID_ARG;
    if (workspace_bytes < align256(ws) + align256(feed.in_bytes) || !aligned(workspace, 256))
        return QSA_ERR_INVALID_ARG;
    // the new rows land inside the caches (rows n_ctx - n_q .. n_ctx - 1), 4-byte units
    if (n_ctx > n_kv || n_q > n_ctx || ld_kv < (int64_t)H_kv * d) return QSA_ERR_INVALID_ARG;
    const int64_t re = esize_of(raw_dtype), ke = esize_of(kv_dtype);
    if ((H_idx * (int64_t)d_idx * re) % 4 || (H_kv * (int64_t)d * ke) % 4 || (ld_kv * ke) % 4 ||
        !aligned(raw_k, 4) || !aligned(K, 4) || !aligned(V, 4))
        return QSA_ERR_INVALID_ARG;
    feed.h_in = h_in;
    feed.staging = static_cast<char *>(workspace) + align256(ws);
    feed.h_out = h_out;
    feed.h_lse = h_lse;
    const float *q_idx = reinterpret_cast<const float *>(feed.staging + feed.off[3]);
    const float *q = reinterpret_cast<const float *>(feed.staging + feed.off[4]);
    return decode_step_impl(raw_k, raw_dtype, n_ctx, H_idx, d_idx, norm_w, eps, rope_base, pooled,
                            pooled_dtype, cap_rows, n_valid_full, n_q, q_idx, scale_idx, scores,
                            k_blk, blocks, counts, K, V, kv_dtype, n_kv, H_kv, d, ld_kv, pos,
                            n_cells, max_cells, q, H_q, scale, out, lse_out, workspace, ws, stream,
                            &feed);
}

struct qsa_decode_plan {
    void *raw_k;
    qsa_dtype raw_dtype;
    int H_idx, d_idx;
    const float *norm_w;
    float eps;
    double rope_base;
    void *pooled;
    qsa_dtype pooled_dtype;
    int64_t cap_rows, max_queries;
    float scale_idx;
    float *scores;
    int64_t k_blk;
    int32_t *blocks, *counts;
    void *K, *V;
    qsa_dtype kv_dtype;
    int64_t n_kv;
    int H_kv, d;
    int64_t ld_kv;
    int32_t *pos, *n_cells;
    int64_t max_cells;
    int H_q;
    float scale;
    float *out, *lse_out;
    void *workspace;
    size_t workspace_bytes;
    bool host;  // the workspace also holds the host-fed step's staging area
};

qsa_status qsa_decode_plan_create(qsa_decode_plan **plan, void *raw_k, qsa_dtype raw_dtype,
                                  int H_idx, int d_idx, const float *norm_w, float eps,
                                  double rope_base, void *pooled, qsa_dtype pooled_dtype,
                                  int64_t cap_rows, int64_t max_queries, float scale_idx,
                                  float *scores, int64_t k_blk, int32_t *blocks, int32_t *counts,
                                  void *K, void *V, qsa_dtype kv_dtype, int64_t n_kv, int H_kv,
                                  int d, int64_t ld_kv, int32_t *pos, int32_t *n_cells,
                                  int64_t max_cells, int H_q, float scale, float *out,
                                  float *lse_out, void *workspace, size_t workspace_bytes)
{
    if (!plan) return QSA_ERR_INVALID_ARG;
    *plan = nullptr;
    if (!raw_k || !norm_w || !pooled || !scores || !blocks || !counts || !K || !V || !pos ||
        !n_cells || !out || !workspace || !valid_dtype(raw_dtype) ||
        !valid_dtype(pooled_dtype) || !valid_dtype(kv_dtype) || max_queries < 1 ||
        max_queries > kMaxStreamQueries || !aligned(workspace, 256))
        return QSA_ERR_INVALID_ARG;
    const size_t need = qsa_decode_step_workspace_size(max_queries, H_q, H_kv, d, max_cells,
                                                       cap_rows);
    if (need == 0 || workspace_bytes < need) return QSA_ERR_INVALID_ARG;
    const size_t need_host = qsa_decode_step_host_workspace_size(
        max_queries, H_q, H_kv, d, max_cells, cap_rows, raw_dtype, H_idx, d_idx, kv_dtype);
    qsa_decode_plan *p = static_cast<qsa_decode_plan *>(malloc(sizeof(qsa_decode_plan)));
    if (!p) return QSA_ERR_INVALID_ARG;
    *p = qsa_decode_plan{raw_k, raw_dtype, H_idx, d_idx, norm_w, eps, rope_base, pooled,
                         pooled_dtype, cap_rows, max_queries, scale_idx, scores, k_blk, blocks,
                         counts, K, V, kv_dtype, n_kv, H_kv, d, ld_kv, pos, n_cells, max_cells,
                         H_q, scale, out, lse_out, workspace, workspace_bytes,
                         need_host != 0 && workspace_bytes >= need_host};
    *plan = p;
    return QSA_OK;
}

void qsa_decode_plan_destroy(qsa_decode_plan *plan) { free(plan); }

qsa_status qsa_decode_plan_step(const qsa_decode_plan *p, int64_t n_ctx, int64_t n_valid_full,
                                int64_t n_q, const float *q_idx, const float *q,
                                qsa_stream_t stream)
{
    if (!p || n_q > p->max_queries) return QSA_ERR_INVALID_ARG;
    return qsa_decode_step(p->raw_k, p->raw_dtype, n_ctx, p->H_idx, p->d_idx, p->norm_w, p->eps,
                           p->rope_base, p->pooled, p->pooled_dtype, p->cap_rows, n_valid_full,
                           n_q, q_idx, p->scale_idx, p->scores, p->k_blk, p->blocks, p->counts,
                           p->K, p->V, p->kv_dtype, p->n_kv, p->H_kv, p->d, p->ld_kv, p->pos,
                           p->n_cells, p->max_cells, q, p->H_q, p->scale, p->out, p->lse_out,
                           p->workspace, p->workspace_bytes, stream);
}

qsa_status qsa_decode_plan_step_host(const qsa_decode_plan *p, int64_t n_ctx,
                                     int64_t n_valid_full, int64_t n_q, const void *h_in,
                                     float *h_out, float *h_lse, qsa_stream_t stream)
{
    if (!p || !p->host || n_q > p->max_queries) return QSA_ERR_INVALID_ARG;
    return qsa_decode_step_host(h_in, h_out, h_lse, p->raw_k, p->raw_dtype, n_ctx, p->H_idx,
                                p->d_idx, p->norm_w, p->eps, p->rope_base, p->pooled,
                                p->pooled_dtype, p->cap_rows, n_valid_full, n_q, p->scale_idx,
                                p->scores, p->k_blk, p->blocks, p->counts, p->K, p->V,
                                p->kv_dtype, p->n_kv, p->H_kv, p->d, p->ld_kv, p->pos, p->n_cells,
                                p->max_cells, p->H_q, p->scale, p->out, p->lse_out, p->workspace,
                                p->workspace_bytes, stream);
}

qsa_status qsa_mask_to_list(const uint8_t *mask, int64_t n_rows, int64_t n_kv, int64_t ld_mask,
                            int64_t max_list, int32_t *pos_out, int32_t *counts_out,
                            uint64_t *bits_out, qsa_stream_t stream)
{
    if (!mask || !counts_out || (!pos_out && max_list > 0)) return QSA_ERR_INVALID_ARG;
    if (n_rows < 0 || n_kv < 0 || ld_mask < n_kv || max_list < 0) return QSA_ERR_INVALID_ARG;
    if (bits_out && !aligned(bits_out, 8)) return QSA_ERR_INVALID_ARG;
    if (n_kv > 0x7fffffffLL || n_rows > 0x7fffffffLL) return QSA_ERR_UNSUPPORTED;
    return from_cuda(launch_mask_to_list(mask, n_rows, n_kv, ld_mask, max_list, pos_out,
                                         counts_out, bits_out, (cudaStream_t)stream));
}

qsa_status qsa_mask_sparse_attn(const float *q, int64_t n_q, int H_q, int H_kv, int d_k,
                                int d_v, float scale, const void *KV, qsa_dtype dtype,
                                int64_t n_kv, int64_t ld_kv, const uint8_t *mask, int64_t ld_mask,
                                int64_t max_list, int32_t *counts_out, float *out, float *lse_out,
                                qsa_stream_t stream)
{
    if (!q || !KV || !mask || !out) return QSA_ERR_INVALID_ARG;
    if (n_q < 0 || H_q < 1 || H_kv < 1 || H_q % H_kv || n_kv < 0 || ld_kv < (int64_t)H_kv * d_k ||
        ld_mask < n_kv || max_list < 0)
        return QSA_ERR_INVALID_ARG;
    if (!aligned(q, 8) || !aligned(out, 4) || (lse_out && !aligned(lse_out, 4)) ||
        (counts_out && !aligned(counts_out, 4)))
        return QSA_ERR_INVALID_ARG;
    if (dtype != QSA_F32 && dtype != QSA_BF16) return QSA_ERR_INVALID_ARG;
    if (H_kv != 1 || !attn_uses_wide(dtype, d_k, d_v, H_q, KV, KV, ld_kv, ld_kv))
        return QSA_ERR_UNSUPPORTED;  // only the latent shape (bf16, 576 / 512, 16 heads, 1 KV)
    if (n_kv > attn_wide_mask_max_kv() || n_q > 65535 || H_kv > 65535 || max_list > 0x7fffffffLL)
        return QSA_ERR_UNSUPPORTED;
    if (n_q == 0) return QSA_OK;
    return from_cuda(launch_attn_wide_mask(q, n_q, H_q, H_kv, scale, KV, n_kv, ld_kv, mask,
                                           ld_mask, max_list, counts_out, out, lse_out,
                                           (cudaStream_t)stream));
}

qsa_status qsa_mask_sparse_eligible(int has_mask, float max_bias, float softcap, int64_t n_kv,
                                    int64_t max_list)
{
    if (n_kv < 0 || max_list < 0) return QSA_ERR_INVALID_ARG;
    if (!has_mask || max_bias != 0.0f || softcap != 0.0f) return QSA_ERR_UNSUPPORTED;
    if (n_kv < 4096 || n_kv < 2 * max_list) return QSA_ERR_UNSUPPORTED;
    return QSA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------------
// Split-K scratch for callers that cannot allocate: one fixed device array per GPU,
// shared by every call.  Host code must not pass the array's name to a kernel (on the
// host that name is a stand-in, not a device address): every call looks the address up
// with cudaGetSymbolAddress in the caller's current device and context.  The lookup
// allocates nothing, and doing it per call (rather than caching it per device ordinal)
// keeps the address right when the caller switches to another context on the same device
// or after a device reset has reloaded the module.
static __device__ __align__(256) unsigned char g_noalloc_scratch[QSA_NOALLOC_SCRATCH_BYTES];

extern "C" qsa_status qsa_sparse_attn_noalloc(const float *q, int64_t n_q, int H_q, int H_kv,
                                              int d_k, int d_v, float scale, const void *K,
                                              const void *V, qsa_dtype dtype, int64_t n_kv,
                                              int64_t ld_k, int64_t ld_v, const int32_t *pos,
                                              const int32_t *n_cells, int64_t max_cells,
                                              float *out, float *lse_out, qsa_stream_t stream)
{
    // what the path these arguments take really writes (0 for the forms that merge their
    // splits inside a cluster); the argument checks themselves are qsa_sparse_attn's
    if (n_q >= 0 && H_q >= 1 && H_kv >= 1 && d_v >= 1 && max_cells >= 0 && H_q % H_kv == 0 &&
        valid_dtype(dtype) &&
        attn_partials_bytes(dtype, n_q, H_q, H_kv, d_k, d_v, K, V, ld_k, ld_v, pos, max_cells) >
            QSA_NOALLOC_SCRATCH_BYTES)
        return QSA_ERR_UNSUPPORTED;  // this shape needs more scratch than the fixed array
    void *scratch = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
    if (e != cudaSuccess || scratch == nullptr) return QSA_ERR_CUDA;
    return qsa_sparse_attn(q, n_q, H_q, H_kv, d_k, d_v, scale, K, V, dtype, n_kv, ld_k, ld_v, pos,
                           n_cells, max_cells, out, lse_out, scratch, QSA_NOALLOC_SCRATCH_BYTES,
                           stream);
}
