// attn_union.cuh -- launcher of the grouped-union sparse attention (attn_union.cu), for the
// C entry points in capi.cu.
#pragma once

#include "qsa_internal.cuh"

namespace qsa {

// Queries per group: 16 queries x 8 query heads of one KV head = the 128 rows of one MMA.
constexpr int kUnionGroup = 16;

// Keys per row of the cache that the union builder's block bitmap covers.
int64_t attn_union_max_kv();

// Workspace bytes: per group, the union's block count, its block list and the per-query
// cell-membership words, for lists of up to max_cells cells.
size_t attn_union_workspace_bytes(int64_t n_q, int64_t max_cells);

// The shape the kernel is built for: bf16 K / V, head dim 128 for keys and values, 8 query
// heads per KV head, row strides that are multiples of 8 elements, 16-byte aligned caches.
bool attn_union_shape_ok(qsa_dtype dt, int H_q, int H_kv, int d_k, int d_v, const void *K,
                         const void *V, int64_t ld_k, int64_t ld_v);

// Both kernels on `st`: the per-group union build, then the attention.  workspace is
// attn_union_workspace_bytes() bytes, 256-byte aligned.
qsa_status launch_attn_union(const float *q, int64_t n_q, int H_q, int H_kv, float scale,
                             const void *K, const void *V, int64_t n_kv, int64_t ld_k,
                             int64_t ld_v, const int32_t *pos, const int32_t *n_cells,
                             int64_t max_cells, float *out, float *lse, void *workspace,
                             cudaStream_t st);

}  // namespace qsa
