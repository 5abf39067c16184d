// gather.cu -- expand selected blocks to KV cells (plus the open tail) and optionally copy
// the selected K/V rows into compact tensors.
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "selected K/V gather (COMMON-005)" (get_rows of K, V and mask at the selected cells,
// then attention over the compact rows) and section "block-domain top-k (COMMON-006)"
// (expand only the chosen blocks, then append the tail indices).
//
// One warp per output cell: lane 0 writes the cell position, all lanes copy the row with
// 16-byte vectors when the row is 16-byte aligned.  In the fused decode step the
// attention kernel reads rows in place from the position list, so only the index part
// runs (K_out = V_out = NULL).
#include "qsa_internal.cuh"

namespace qsa {
namespace {

__device__ __forceinline__ void copy_row(const char *__restrict__ src, char *__restrict__ dst,
                                         int64_t bytes, int lane)
{
    if ((((uintptr_t)src | (uintptr_t)dst | (uintptr_t)bytes) & 15) == 0) {
        const uint4 *s = reinterpret_cast<const uint4 *>(src);
        uint4 *d = reinterpret_cast<uint4 *>(dst);
        for (int64_t i = lane; i < bytes / 16; i += 32) d[i] = s[i];
    } else if ((((uintptr_t)src | (uintptr_t)dst | (uintptr_t)bytes) & 3) == 0) {
        const uint32_t *s = reinterpret_cast<const uint32_t *>(src);
        uint32_t *d = reinterpret_cast<uint32_t *>(dst);
        for (int64_t i = lane; i < bytes / 4; i += 32) d[i] = s[i];
    } else {
        const uint16_t *s = reinterpret_cast<const uint16_t *>(src);
        uint16_t *d = reinterpret_cast<uint16_t *>(dst);
        for (int64_t i = lane; i < bytes / 2; i += 32) d[i] = s[i];
    }
}

__global__ void __launch_bounds__(256)
gather_kernel(const char *__restrict__ K, const char *__restrict__ V, int esize, int64_t n_kv,
              int64_t row_k_bytes, int64_t row_v_bytes, int64_t ld_k_bytes, int64_t ld_v_bytes,
              const int32_t *__restrict__ blocks, const int32_t *__restrict__ counts,
              int64_t k_blk, const int32_t *__restrict__ q_pos, int64_t n_ctx,
              char *__restrict__ K_out, char *__restrict__ V_out, int32_t *__restrict__ pos_out,
              int32_t *__restrict__ n_cells_out, int64_t max_cells)
{
    pdl_wait();
    QSA_AFTER_WAIT(K);
    QSA_AFTER_WAIT(V);
    QSA_AFTER_WAIT(blocks);
    QSA_AFTER_WAIT(counts);
    QSA_AFTER_WAIT(q_pos);
    pdl_trigger();
    const int64_t qi = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int64_t j = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);

    const int64_t p = q_pos ? (int64_t)q_pos[qi] : n_ctx - 1;
    const int64_t tail0 = 4 * ((p + 1) / 4);
    const int64_t n_tail = p + 1 - tail0;
    int64_t cnt = counts[qi];
    if (cnt < 0) cnt = 0;
    if (cnt > k_blk) cnt = k_blk;
    const int64_t n_cells = 4 * cnt + n_tail;
    if (j == 0 && lane == 0) n_cells_out[qi] = (int32_t)n_cells;
    if (j >= n_cells) return;

    int64_t cell;
    if (j < 4 * cnt) {
        const int64_t b = blocks[qi * k_blk + j / 4];
        cell = (b >= 0 && 4 * b + 3 < n_kv + 3) ? 4 * b + (j & 3) : -1;
    } else {
        cell = tail0 + (j - 4 * cnt);
    }
    if (cell >= n_kv) cell = -1;
    if (lane == 0) pos_out[qi * max_cells + j] = (int32_t)cell;
    if (cell < 0) return;
    const int64_t orow = qi * max_cells + j;
    if (K_out) copy_row(K + cell * ld_k_bytes, K_out + orow * row_k_bytes, row_k_bytes, lane);
    if (V_out) copy_row(V + cell * ld_v_bytes, V_out + orow * row_v_bytes, row_v_bytes, lane);
    (void)esize;
}

// Index-only form (no row copies): thread j writes the four cells of selected block j (one
// 16-byte store when the row allows it); thread cnt writes the open tail.
__global__ void __launch_bounds__(256)
cells_kernel(int64_t n_kv, const int32_t *__restrict__ blocks, const int32_t *__restrict__ counts,
             int64_t k_blk, const int32_t *__restrict__ q_pos, int64_t n_ctx,
             int32_t *__restrict__ pos_out, int32_t *__restrict__ n_cells_out, int64_t max_cells)
{
    pdl_wait();
    QSA_AFTER_WAIT(blocks);
    QSA_AFTER_WAIT(counts);
    QSA_AFTER_WAIT(q_pos);
    pdl_trigger();
    const int64_t qi = blockIdx.y;
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t cnt = counts[qi];
    const int64_t b = j < k_blk ? (int64_t)blocks[qi * k_blk + j] : -1;  // issued with counts
    const int64_t p = q_pos ? (int64_t)q_pos[qi] : n_ctx - 1;
    const int64_t tail0 = 4 * ((p + 1) / 4);
    if (cnt < 0) cnt = 0;
    if (cnt > k_blk) cnt = k_blk;
    const int64_t n_tail = p + 1 - tail0;
    int32_t *row = pos_out + qi * max_cells;
    if (j == 0) n_cells_out[qi] = (int32_t)(4 * cnt + n_tail);
    if (j < cnt) {
        int32_t c[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int64_t cell = b >= 0 ? 4 * b + r : -1;
            c[r] = cell >= n_kv ? -1 : (int32_t)cell;
        }
        int32_t *dst = row + 4 * j;
        if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
            *reinterpret_cast<int4 *>(dst) = make_int4(c[0], c[1], c[2], c[3]);
        } else {
#pragma unroll
            for (int r = 0; r < 4; ++r) dst[r] = c[r];
        }
    } else if (j == cnt) {
        for (int64_t t = 0; t < n_tail; ++t) {
            const int64_t cell = tail0 + t;
            row[4 * cnt + t] = cell >= n_kv ? -1 : (int32_t)cell;
        }
    }
}

}  // namespace

cudaError_t launch_gather(const void *K, const void *V, qsa_dtype dt, int64_t n_kv, int H_kv,
                          int d_k, int d_v, int64_t ld_k, int64_t ld_v, const int32_t *blocks,
                          const int32_t *counts, int64_t n_q, int64_t k_blk,
                          const int32_t *q_pos, int64_t n_ctx, void *K_out, void *V_out,
                          int32_t *pos_out, int32_t *n_cells_out, int64_t max_cells,
                          cudaStream_t st)
{
    if (n_q == 0) return cudaSuccess;
    if (!K_out && !V_out) {
        const dim3 grid((unsigned)((k_blk + 1 + 255) / 256), (unsigned)n_q);  // blocks + tail
        return launch(cells_kernel, grid, dim3(256), 0, st, 1, n_kv, blocks, counts, k_blk, q_pos,
                      n_ctx, pos_out, n_cells_out, max_cells);
    }
    const int esize = dt == QSA_BF16 ? 2 : 4;
    const int warps = 8;
    const dim3 grid((unsigned)((max_cells + warps - 1) / warps), (unsigned)n_q);
    return launch(gather_kernel, grid, dim3(32 * warps), 0, st, 1, (const char *)K,
                  (const char *)V, esize, n_kv, (int64_t)H_kv * d_k * esize,
                  (int64_t)H_kv * d_v * esize, ld_k * esize, ld_v * esize, blocks, counts, k_blk,
                  q_pos, n_ctx, (char *)K_out, (char *)V_out, pos_out, n_cells_out, max_cells);
}

}  // namespace qsa
