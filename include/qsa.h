/*
 * qsa.h -- C ABI of the GB300 (sm_103a) QSA two-stage sparse-attention library.
 *
 * QSA ("Qwen Sparse Attention") first runs a light indexer that picks the important
 * 4-token blocks of a long context, then runs attention over the selected cells only
 * (Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
 * "QSA and the QSA indexer").  One decode step of one QSA layer is the call sequence
 *
 *   qsa_pool_update -> qsa_index_score -> qsa_topk_blocks -> qsa_gather_kv
 *                   -> qsa_sparse_attn
 *
 * and the mask-driven variant is qsa_mask_to_list -> qsa_sparse_attn, or for the latent
 * shape the single call qsa_mask_sparse_attn.
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is device memory owned by the caller (except the host buffers
 *     of qsa_decode_step_host); the library never allocates, frees or keeps a pointer past
 *     the call.  Scratch memory comes from a caller buffer whose size the matching
 *     *_workspace_size() function returns.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and never synchronises with the host.
 *   - The returned status is decided on the host from the arguments before anything is
 *     launched: QSA_ERR_INVALID_ARG / QSA_ERR_UNSUPPORTED mean nothing was enqueued.
 *     QSA_ERR_CUDA means a launch failed (the CUDA error is left for
 *     cudaGetLastError()).  Data-dependent conditions (a list longer than its capacity)
 *     are reported in device outputs, never by a trap.
 *   - Layouts are row-major.  "ld" arguments are element strides between consecutive
 *     rows.  Pointers to fp32 / bf16 data must be aligned to their element size.
 *   - Dtype QSA_BF16 means bfloat16 storage; all arithmetic accumulates in fp32.
 *   - Block b of a context covers tokens 4b .. 4b+3.  With n_ctx tokens there are
 *     n_full = floor(n_ctx/4) complete blocks and n_rows = ceil(n_ctx/4) pooled rows;
 *     the last row is the open (partial) block when n_ctx is not a multiple of 4.
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *qsa_stream_t; /* same type as cudaStream_t */

typedef enum {
    QSA_OK = 0,
    QSA_ERR_INVALID_ARG = 1, /* a pointer, size, stride or alignment is invalid */
    QSA_ERR_UNSUPPORTED = 2, /* valid, but outside what this build implements */
    QSA_ERR_CUDA = 3,        /* a CUDA launch or query failed */
    QSA_ERR_TIMEOUT = 4      /* a bounded device wait gave up (reported in device memory,
                                see qsa_set_wait_options) */
} qsa_status;

typedef enum { QSA_F32 = 0, QSA_BF16 = 1 } qsa_dtype;

typedef enum {
    QSA_PREC_F32 = 0,    /* fp32 operands, fp32 accumulation (CUDA cores) */
    QSA_PREC_BF16_TC = 1 /* operands rounded to bf16 (nearest even), fp32 accumulation
                            on the tcgen05 tensor cores; for multi-query chunks */
} qsa_precision;

/* Human-readable name of a status code (static storage). */
const char *qsa_status_str(qsa_status s);

/* Library ABI version: (major << 16) | minor.  Major 2: pooled-cache dtype arguments,
 * several queries per decode step, the host-fed decode step; minor 1: decode plans;
 * minor 2: qsa_mask_sparse_attn; minor 3: qsa_sparse_attn_union; minor 4:
 * qsa_set_wait_options. */
int qsa_version(void);

/*
 * qsa_set_wait_options -- bounded device waits: how long the kernels launched by later calls
 * from the calling host thread may wait for their own asynchronous work, and where they report
 * giving up.
 *
 * The source pages have no counterpart: it is this library's failure reporting.
 *
 * Kernels that stage data with asynchronous copies or run tcgen05 tensor-core work wait on
 * shared-memory barriers: the attention kernels of qsa_sparse_attn (bf16, 128-dim, 8 query
 * heads per KV head; the many-query form; the latent form), qsa_sparse_attn_union,
 * qsa_mask_sparse_attn and qsa_decode_step / its host-fed and plan forms, and the tensor-core
 * score contraction of qsa_index_score (QSA_PREC_BF16_TC).  No wait is unbounded.  When a
 * wait inside a kernel's pipeline lasts longer than pipeline_limit_ns, the kernel stores
 * QSA_ERR_TIMEOUT into *status_out (when status_out is not NULL), stops issuing work, waits
 * for the copies and MMAs it already issued (bounded by the default limit, which these final
 * waits always use), returns its tensor memory, and writes NaN to the outputs it could not
 * finish (scores: the rows of a tile it never stored stay as they were).  The call itself
 * returned QSA_OK long before: the caller reads the status after synchronising its stream.
 *
 *   status_out         device int32 or NULL; the library only ever stores QSA_ERR_TIMEOUT
 *                      there (clear it before the calls it should cover)
 *   pipeline_limit_ns  QSA_WAIT_DEFAULT_NS (2 s) is the default; 0 makes every pipeline wait
 *                      give up at once, without looking (for testing the failure path: every
 *                      covered kernel then reports QSA_ERR_TIMEOUT and leaves NaN or untouched
 *                      outputs)
 * The settings belong to the calling host thread and apply to every later launch from it
 * (a CUDA graph captured meanwhile keeps the values of its capture) until changed.
 */
#define QSA_WAIT_DEFAULT_NS 2000000000ull
void qsa_set_wait_options(int32_t *status_out, uint64_t pipeline_limit_ns);

/*
 * qsa_pool_update -- incremental pooled-key cache update.
 *
 * Source: same page, sections "QSA and the QSA indexer" (4-token average pooling ->
 * RMS norm -> RoPE of the pooled summary) and "incremental pooled-key cache
 * (COMMON-004)" (a persistent cache of completed-block rows; only newly completed or
 * invalidated blocks, and the open block, are recomputed).
 *
 * For every block b in [n_valid_full, n_rows):
 *   p   = mean of the raw indexer keys of the tokens of block b present in n_ctx
 *   y_h = p_h / sqrt(mean_j p_h[j]^2 + eps) * norm_w        (each indexer head h)
 *   z_h = RoPE(y_h, position 4b): dims i and i + d/2 rotate by 4b * base^(-2i/d)
 *   pooled[b][h*d .. h*d+d) = z_h  (the angle is formed in fp64; computed in fp32 and
 *                                   stored as fp32, or as bf16 rounded to nearest even)
 * Rows below n_valid_full are not touched.  Invalidation after a state load, a
 * sequence edit or a rolled-back speculative write is done by passing a smaller
 * n_valid_full (e.g. floor(first_changed_position / 4)).
 *
 *   raw_k      [n_ctx][H][d] raw indexer keys, dtype raw_dtype (row stride H*d)
 *   norm_w     [d] fp32 RMS-norm weight shared by all indexer heads
 *   pooled     [cap_rows][H*d] cache of type pooled_dtype (QSA_F32, or QSA_BF16: half
 *              the bytes for the score scan to read), updated in place
 *   n_valid_full  rows [0, n_valid_full) are known to be valid; 0 <= n_valid_full
 *              (values above n_full are clamped to n_full)
 * Errors: INVALID_ARG for null pointers, n_ctx < 0, H < 1, d < 2 or odd d,
 * n_valid_full < 0, an unknown dtype, a misaligned pooled pointer, or
 * n_rows > cap_rows.
 */
qsa_status qsa_pool_update(const void *raw_k, qsa_dtype raw_dtype, int64_t n_ctx, int H, int d,
                           const float *norm_w, float eps, double rope_base, void *pooled,
                           qsa_dtype pooled_dtype, int64_t cap_rows, int64_t n_valid_full,
                           qsa_stream_t stream);

/*
 * qsa_index_score -- indexer score of every pooled row against each query.
 *
 * Source: same page, section "QSA and the QSA indexer" (the query is scored against
 * every pooled block summary; the top blocks are then selected).
 *
 *   scores[i][b] = scale * sum_{h,j} q[i][h*d+j] * pooled[b][h*d+j],  b < n_rows
 * When q_pos is not NULL (prefill chunk), row b is visible to query i only if the
 * block is complete at the query's position (4b + 3 <= q_pos[i]); other rows get
 * -inf.  When q_pos is NULL (decode), every row including the open one is scored.
 * Up to four queries share one pass over the cache (each row is read once for all).
 *
 *   q          [n_q][ld_q] fp32 indexer queries (already position-encoded by the caller)
 *   q_pos      [n_q] int32 device positions, or NULL
 *   pooled     [n_rows][H*d] of type pooled_dtype (fp32 or bf16; the products and sums
 *              are fp32 either way)
 *   scores     [n_q][ld_scores] fp32 output, ld_scores >= n_rows
 *   precision  QSA_PREC_F32 or QSA_PREC_BF16_TC (q and an fp32 cache rounded to bf16
 *              for the tensor cores; needs the workspace)
 *   workspace  caller scratch of qsa_index_score_workspace_size() bytes (may be NULL
 *              when that size is 0)
 * Errors: INVALID_ARG for null pointers, sizes < 0, ld_q < H*d, ld_scores < n_rows, an
 * unknown dtype, a misaligned pointer, or a workspace smaller than required.
 */
qsa_status qsa_index_score(const float *q, int64_t n_q, int64_t ld_q, const int32_t *q_pos,
                           const void *pooled, qsa_dtype pooled_dtype, int64_t n_rows, int H,
                           int d, float scale, float *scores, int64_t ld_scores,
                           qsa_precision precision, void *workspace, size_t workspace_bytes,
                           qsa_stream_t stream);

/* Workspace bytes of qsa_index_score (0 for QSA_PREC_F32; a bf16 cache needs no copy). */
size_t qsa_index_score_workspace_size(int64_t n_q, int64_t n_rows, int H, int d,
                                      qsa_dtype pooled_dtype, qsa_precision precision);

/*
 * qsa_topk_blocks -- block-domain top-k.
 *
 * Source: same page, section "block-domain top-k (COMMON-006)" (top-k is taken over
 * the block scores and only the chosen blocks are expanded to cells) and section
 * "QSA and the QSA indexer" (indexer_top_k = 2048 tokens = 512 blocks).
 *
 * For each query i, the candidates are the complete blocks b < n_full_i, where
 * n_full_i = n_full when q_pos is NULL, else min(n_full, floor((q_pos[i]+1)/4)).
 * The open block never competes (it is appended as the tail by qsa_gather_kv).
 * Output: the min(k_blk, n_full_i) best candidates by score, ties to the lower block
 * index, NaN ranked as -inf, written in ascending block order to
 * blocks_out[i][0 .. count), count to counts_out[i].  Entries past the count are not
 * written.
 *
 *   scores     [n_q][ld_scores] fp32 (as written by qsa_index_score)
 *   blocks_out [n_q][k_blk] int32;  counts_out [n_q] int32
 * Errors: INVALID_ARG for null pointers, n_q < 0, k_blk < 1, n_full < 0,
 * ld_scores < n_full; UNSUPPORTED when n_full exceeds qsa_topk_max_candidates().
 */
qsa_status qsa_topk_blocks(const float *scores, int64_t n_q, int64_t ld_scores,
                           const int32_t *q_pos, int64_t n_full, int64_t k_blk,
                           int32_t *blocks_out, int32_t *counts_out, qsa_stream_t stream);

int64_t qsa_topk_max_candidates(void);

/*
 * qsa_index_score_maxima / qsa_topk_blocks_maxima -- the prefill selection with a per-row
 * summary written by the score contraction and read by the top-k.
 *
 * Source: same page, section "block-domain top-k (COMMON-006)" (the top-k over block
 * scores) with section "QSA and the QSA indexer" (every query of a prefill chunk scored
 * against every pooled block).  The pages do not describe how a chunk's top-k is fed; this
 * library's reading: the score kernel's epilogue, which holds each query's scores of 32
 * consecutive rows at once, also stores their maximum, and the top-k takes its threshold
 * from those maxima instead of sampling or scanning the whole row.
 *
 * qsa_index_score_maxima is qsa_index_score with precision QSA_PREC_BF16_TC (same
 * arguments, scores and workspace, same errors) that also writes
 *   maxima[i][g] = max { scores[i][b] : 32g <= b < min(32g + 32, n_rows) }
 * for g < ceil(n_rows / 32): -inf when every score of the group is -inf (rows the query
 * cannot see), NaN scores left out.  maxima: [n_q][ld_maxima] fp32, ld_maxima >=
 * ceil(n_rows / 32), 4-byte aligned; INVALID_ARG otherwise.
 *
 * qsa_topk_blocks_maxima returns exactly what qsa_topk_blocks returns for the same
 * arguments (same candidates, order, ties and errors), given maxima as written above for
 * these scores (ld_maxima >= n_full / 32, rounded down; INVALID_ARG otherwise).  For a query
 * with at least 32 * k_blk candidates (and n_full <= 131,072), the k_blk-th largest maximum
 * of the groups that hold only candidates bounds its threshold from below, only the groups
 * whose maximum reaches that bound are read, and four queries share an SM; a query whose
 * bound leaves more than 2,048 candidates, and every other query, takes the general form.
 * Maxima that are not those of the scores give an unspecified (but in-bounds) selection.
 *   workspace  device scratch of qsa_topk_blocks_maxima_workspace_size(n_q) bytes, 256-byte
 *              aligned (INVALID_ARG when smaller or misaligned)
 */
qsa_status qsa_index_score_maxima(const float *q, int64_t n_q, int64_t ld_q,
                                  const int32_t *q_pos, const void *pooled,
                                  qsa_dtype pooled_dtype, int64_t n_rows, int H, int d,
                                  float scale, float *scores, int64_t ld_scores, float *maxima,
                                  int64_t ld_maxima, void *workspace, size_t workspace_bytes,
                                  qsa_stream_t stream);

qsa_status qsa_topk_blocks_maxima(const float *scores, int64_t n_q, int64_t ld_scores,
                                  const int32_t *q_pos, int64_t n_full, int64_t k_blk,
                                  const float *maxima, int64_t ld_maxima, int32_t *blocks_out,
                                  int32_t *counts_out, void *workspace, size_t workspace_bytes,
                                  qsa_stream_t stream);

size_t qsa_topk_blocks_maxima_workspace_size(int64_t n_q);

/*
 * qsa_expand_block_scores -- the selection input of the pages' earlier path, kept for A/B
 * measurement: each full block's score copied to its four cells.
 *
 * Source: same page, section "block-domain top-k (COMMON-006)" (before it, block scores were
 * expanded to every cell through a cell -> block map and the top-k ran over cells; that
 * expansion cost 0.45 / 0.91 ms per layer at 128k / 256k on the pages' GPU).
 *
 *   cell_scores[i][c] = scores[i][floor(c / 4)]   for c < 4 * n_full
 * qsa_topk_blocks over cell_scores with 4 * n_full candidates and k = 4 * k_blk then
 * selects cells; since a block's four cells tie and ties go to the lower index, whole
 * blocks are selected, the same ones as the block-domain top-k unless a tie straddles its
 * boundary.  The decode path does not use this call.
 *
 *   scores       [n_q][ld_scores] fp32, ld_scores >= n_full
 *   cell_scores  [n_q][ld_cells] fp32 output, ld_cells >= 4 * n_full; entries from 4*n_full
 *                on are not written
 * Errors: INVALID_ARG for null or misaligned pointers, negative sizes or short strides;
 * UNSUPPORTED for n_q > 65535.
 */
qsa_status qsa_expand_block_scores(const float *scores, int64_t n_q, int64_t ld_scores,
                                   int64_t n_full, float *cell_scores, int64_t ld_cells,
                                   qsa_stream_t stream);

/*
 * qsa_gather_kv -- expand selected blocks to KV cells and (optionally) copy the rows.
 *
 * Source: same page, section "selected K/V gather (COMMON-005)" (get_rows of K, V and
 * mask at the ~2051 selected cells into compact tensors) and section "block-domain
 * top-k (COMMON-006)" (expand only the selected blocks to cell indices, then append
 * the tail indices); section "why Flash Attention scaled" gives 2048 + 4 - 1 = 2051.
 *
 * For query i at position p_i (q_pos[i], or n_ctx - 1 when q_pos is NULL):
 *   cells = 4b, 4b+1, 4b+2, 4b+3 for each b in blocks[i][0 .. counts[i]) in order,
 *           then the tail 4*floor((p_i+1)/4) .. p_i
 *   pos_out[i][j] = cells[j];  n_cells_out[i] = 4*counts[i] + tail length
 * If K_out / V_out are not NULL, row j of query i is copied:
 *   K_out[(i*max_cells + j)][0 .. H_kv*d_k) = K[cells[j]*ld_k + 0 .. H_kv*d_k)
 *   V_out likewise with d_v and ld_v (K_out / V_out are packed: row stride H_kv*d_k,
 *   H_kv*d_v).  Entries past n_cells_out[i] are not written.
 *
 *   K, V       [n_kv][ld] caches, dtype `dtype` (may be NULL when K_out/V_out are NULL)
 *   blocks     [n_q][k_blk] int32; counts [n_q] int32 (from qsa_topk_blocks)
 *   max_cells  capacity per query; must be >= 4*k_blk + 3
 * Errors: INVALID_ARG for null required pointers, bad sizes or max_cells too small.
 * Block indices outside [0, n_kv/4) produce position -1 rows that are not copied.
 */
qsa_status qsa_gather_kv(const void *K, const void *V, qsa_dtype dtype, int64_t n_kv, int H_kv,
                         int d_k, int d_v, int64_t ld_k, int64_t ld_v, const int32_t *blocks,
                         const int32_t *counts, int64_t n_q, int64_t k_blk,
                         const int32_t *q_pos, int64_t n_ctx, void *K_out, void *V_out,
                         int32_t *pos_out, int32_t *n_cells_out, int64_t max_cells,
                         qsa_stream_t stream);

/*
 * qsa_sparse_attn -- attention of each query token over its listed cells only.
 *
 * Source: same page, section "selected K/V gather (COMMON-005)" (attention over the
 * compact ~2051 rows; the Flash Attention kernel then no longer scales with context)
 * and devotd.net, "llama.cpp CDNA sparse attention", sections 2-3 (attention over the
 * listed key positions only; DKQ 576 with 16 query columns per KV head).
 *
 * For query i and head h (KV head g = floor(h*H_kv/H_q)), over j < n_cells[i]:
 *   c_j    = pos[i*max_cells + j]  (pos != NULL: rows of the full cache K, V)
 *          = i*max_cells + j       (pos == NULL: K, V are already compact)
 *   logit_j = scale * sum_t q[i][h][t] * K[c_j*ld_k + g*d_k + t]
 *   out[i][h][:] = sum_j softmax(logit)_j * V[c_j*ld_v + g*d_v + :]
 *   lse_out[i][h] = log(sum_j exp(logit_j))   (natural log; optional)
 * Computed as split-K flash decoding (online softmax per split, then a log-sum-exp
 * combine).  Cells whose position is outside [0, n_kv) are skipped.  An empty list
 * gives out = 0 and lse = -inf.  n_cells[i] > max_cells (a truncated list, e.g. a
 * mask with more set positions than the list holds) gives out = NaN and lse = NaN for
 * that query: the result must not be used.
 *
 *   q        [n_q][H_q][d_k] fp32;  out [n_q][H_q][d_v] fp32;  lse_out [n_q][H_q] or NULL
 *   K, V     dtype `dtype`, row strides ld_k, ld_v (V may alias K, e.g. V = K[:, :d_v])
 *   n_cells  [n_q] int32 device counts
 *   workspace  caller scratch for the split-K partial records, 16-byte aligned: at least
 *            the bytes the kernel these arguments select writes (0 for the forms that merge
 *            their splits inside a thread-block cluster); qsa_sparse_attn_workspace_size()
 *            is always enough.  INVALID_ARG when smaller than the kernel needs.
 * Requirements: H_q % H_kv == 0, d_k and d_v multiples of 8, ld_k and ld_v multiples
 * of 8, K and V 16-byte aligned; for the latent shape (bf16, d_k 576, d_v 512, 16 query
 * heads on one KV head, V = K with the same stride) q 8-byte aligned (checked:
 * INVALID_ARG otherwise).
 */
qsa_status qsa_sparse_attn(const float *q, int64_t n_q, int H_q, int H_kv, int d_k, int d_v,
                           float scale, const void *K, const void *V, qsa_dtype dtype,
                           int64_t n_kv, int64_t ld_k, int64_t ld_v, const int32_t *pos,
                           const int32_t *n_cells, int64_t max_cells, float *out,
                           float *lse_out, void *workspace, size_t workspace_bytes,
                           qsa_stream_t stream);

/* Workspace bytes of qsa_sparse_attn: the split-K partial records of the general kernels.
 * It depends on the shape only, so it is an upper bound: the forms that merge their splits
 * inside a cluster (see qsa_sparse_attn_noalloc) leave the workspace untouched. */
size_t qsa_sparse_attn_workspace_size(int64_t n_q, int H_q, int H_kv, int d_v,
                                      int64_t max_cells);

/*
 * qsa_sparse_attn_union -- qsa_sparse_attn for many consecutive queries (a prefill chunk),
 * computed group by group over the union of each group's lists.
 *
 * Source: same page as qsa_pool_update, section on profiling the Vulkan build (its table of
 * r2 with "QSA union" off / on: 221.44 -> 263.28 tok/s of prompt processing, token
 * generation unchanged) and the COMMON-004 results section (r2's grouped-union keeps long
 * prompt processing ahead).  The pages do not describe the mechanism; here queries of a
 * chunk that selected the same blocks read each such block once.
 *
 * Queries are taken in groups of 16 consecutive ones (the last group may be short).  For a
 * group, the union of the 4-cell blocks its listed cells fall in is staged once, as dense
 * tiles, and every query attends over the whole tile sequence with its own cells only (the
 * others masked).  Result: out[i][h][:] and lse_out[i][h] as qsa_sparse_attn over the same
 * lists (up to rounding; a cell listed twice in one list counts once here), including the
 * conventions for empty lists (out 0, lse -inf), truncated lists (n_cells[i] > max_cells:
 * NaN) and cells outside [0, n_kv) (skipped).  The union wins over qsa_sparse_attn when the
 * queries of a group share much of their selection; with independent selections it moves
 * the same bytes and does about 16 times the arithmetic.
 *
 *   q, out   [n_q][H_q][128] fp32, 16-byte aligned;  lse_out [n_q][H_q] or NULL
 *   K, V     bf16 caches, row strides ld_k, ld_v (multiples of 8 elements), 16-byte aligned;
 *            KV head g of row c at K[c*ld_k + g*128]
 *   pos      [n_q][max_cells] int32 cell lists;  n_cells [n_q] int32 device counts
 *   workspace  qsa_sparse_attn_union_workspace_size(n_q, max_cells) bytes, 256-byte aligned
 * Only this shape runs: bf16, d_k = d_v = 128, H_q = 8 * H_kv (QSA_ERR_UNSUPPORTED
 * otherwise), 4 <= n_kv <= 2^20 (UNSUPPORTED), max_cells <= 2100 (UNSUPPORTED).  The union of
 * one group may hold at most 16 * (ceil(max_cells/4) + 1) blocks -- always the case for
 * lists of whole blocks plus one open block, as qsa_gather_kv writes; a group beyond it gets
 * NaN outputs.  Errors: INVALID_ARG for null pointers, negative sizes, misaligned pointers or
 * a short workspace.
 */
qsa_status qsa_sparse_attn_union(const float *q, int64_t n_q, int H_q, int H_kv, int d,
                                 float scale, const void *K, const void *V, qsa_dtype dtype,
                                 int64_t n_kv, int64_t ld_k, int64_t ld_v, const int32_t *pos,
                                 const int32_t *n_cells, int64_t max_cells, float *out,
                                 float *lse_out, void *workspace, size_t workspace_bytes,
                                 qsa_stream_t stream);

size_t qsa_sparse_attn_union_workspace_size(int64_t n_q, int64_t max_cells);

/*
 * qsa_decode_step -- one decode step of one QSA layer: the five calls above in order,
 * validated together before anything is enqueued, issued from one host call.
 *
 * Source: same page as qsa_pool_update, sections "incremental pooled-key cache
 * (COMMON-004)", "selected K/V gather (COMMON-005)" and "block-domain top-k
 * (COMMON-006)" (the decode path: cached pooled keys -> scores -> block top-k -> selected
 * cells -> attention over them).  Several query tokens per step (n_q > 1) serve
 * speculative decoding, where a token and the draft tokens that follow it are verified
 * in one pass (the pages' runs use multi-token prediction with two drafts): the queries
 * are the last n_q tokens of the context and share one scan of the pooled cache.
 *
 * Query i (0 <= i < n_q) sits at position p_i = n_ctx - n_q + i.  Equivalent to, on
 * `stream`, with q_pos[i] = p_i:
 *   qsa_pool_update(raw_k, raw_dtype, n_ctx, H_idx, d_idx, norm_w, eps, rope_base, pooled,
 *                   pooled_dtype, cap_rows, n_valid_full)
 *   qsa_index_score(q_idx, n_q, H_idx*d_idx, NULL, pooled, pooled_dtype, n_rows, H_idx,
 *                   d_idx, scale_idx, scores, n_rows, QSA_PREC_F32)
 *   qsa_topk_blocks(scores, n_q, n_rows, q_pos, n_full, k_blk, blocks, counts)
 *   qsa_gather_kv(K, V, kv_dtype, n_kv, H_kv, d, d, ld_kv, ld_kv, blocks, counts, n_q,
 *                 k_blk, q_pos, n_ctx, NULL, NULL, pos, n_cells, max_cells)  (cell lists)
 *   qsa_sparse_attn(q, n_q, H_q, H_kv, d, d, scale, K, V, kv_dtype, n_kv, ld_kv, ld_kv, pos,
 *                   n_cells, max_cells, out, lse_out, workspace, workspace_bytes)
 * with n_rows = ceil(n_ctx/4), n_full = floor(n_ctx/4).  So every query scores every row,
 * but query i selects only among the blocks complete at p_i, and its tail ends at p_i.
 * With n_q = 1, q_pos = {n_ctx - 1} is the same as q_pos = NULL.
 *   q_idx [n_q][H_idx*d_idx], scores [n_q][n_rows], blocks [n_q][k_blk], counts [n_q],
 *   pos [n_q][max_cells], n_cells [n_q], q [n_q][H_q][d], out [n_q][H_q][d],
 *   lse_out [n_q][H_q] (nullable); all packed.  1 <= n_q <= 4 and n_q <= n_ctx.
 * Results are identical to those calls; the work is fused differently: when at most 4
 * pooled rows need recomputing (every decode step), the score kernel recomputes them
 * itself; it also counts the top 12 bits of the score key of each query's candidate
 * blocks into a histogram per query kept in the workspace, which the top-k kernel starts
 * from (and clears for the next step); the top-k is one kernel whose CTAs each classify
 * 1024 blocks of one query against its histogram and whose last CTA to finish for a
 * query settles its threshold bucket, orders its output and writes its cell list; the
 * attention kernel reads the listed K/V rows in place.  Three launches in all.
 * workspace: qsa_decode_step_workspace_size() bytes, 256-byte aligned.  Its contents need
 * no initialisation: a histogram whose total disagrees with the block count (a workspace
 * never cleared) is rebuilt from the scores, which only makes that call slower; filling
 * it with zeros once avoids that.  Steps that share a workspace must not overlap in time.
 * Returns the first failing validation status without enqueuing anything (INVALID_ARG
 * for n_q outside [1, 4] or above n_ctx, and for a workspace sized for fewer queries or
 * rows).
 */
qsa_status qsa_decode_step(const void *raw_k, qsa_dtype raw_dtype, int64_t n_ctx, int H_idx,
                           int d_idx, const float *norm_w, float eps, double rope_base,
                           void *pooled, qsa_dtype pooled_dtype, int64_t cap_rows,
                           int64_t n_valid_full, int64_t n_q, const float *q_idx, float scale_idx,
                           float *scores, int64_t k_blk, int32_t *blocks, int32_t *counts,
                           const void *K, const void *V, qsa_dtype kv_dtype, int64_t n_kv,
                           int H_kv, int d, int64_t ld_kv, int32_t *pos, int32_t *n_cells,
                           int64_t max_cells, const float *q, int H_q, float scale, float *out,
                           float *lse_out, void *workspace, size_t workspace_bytes,
                           qsa_stream_t stream);

/* Workspace bytes of qsa_decode_step for n_q queries and a cache of up to cap_rows pooled
 * rows (0 for an invalid shape). */
size_t qsa_decode_step_workspace_size(int64_t n_q, int H_q, int H_kv, int d, int64_t max_cells,
                                      int64_t cap_rows);

/*
 * qsa_decode_step_host -- qsa_decode_step fed from host memory: the step's new cache rows
 * and queries come from one packed host buffer, and its output goes back to host memory.
 *
 * Source: same passages as qsa_decode_step (the decode step appends the new tokens, then
 * scores, selects and attends); the host transfer is this library's service.
 *
 * On `stream`, in order: a copy kernel writing the new tokens' rows into the caches --
 * raw indexer keys to raw_k rows n_ctx - n_q .. n_ctx - 1 (row stride H_idx*d_idx), K and
 * V rows to the same rows of K and V (row stride ld_kv) -- and the queries into a staging
 * area at the end of the workspace; then exactly qsa_decode_step with q_idx and q read from
 * the staging area; then out (n_q*H_q*d floats) into h_out and, if h_lse is not NULL,
 * lse_out (n_q*H_q floats) into h_lse.  When h_in is page-locked memory mapped into the
 * current device's address space (cudaHostAlloc'd or registered memory on a unified-address
 * system; torch's pin_memory() buffers are), the copy kernel reads it in place over the
 * host link; otherwise one host-to-device copy of h_in (qsa_decode_step_host_layout()
 * bytes) into the staging area comes first.  Likewise mapped h_out / h_lse are written in
 * place: by the attention kernel itself (bf16 K/V, d 128, 8 query heads per KV head, where
 * it also writes out / lse_out), else by a copy kernel after it; other host buffers by
 * device-to-host copies.  The call returns without waiting: synchronise the stream before
 * reading h_out or reusing h_in.
 *
 *   h_in    packed inputs, sections at the byte offsets qsa_decode_step_host_layout()
 *           reports: [n_q][H_idx*d_idx] raw-key rows (raw_dtype), [n_q][H_kv*d] K rows and
 *           [n_q][H_kv*d] V rows (kv_dtype), [n_q][H_idx*d_idx] fp32 q_idx, [n_q][H_q][d]
 *           fp32 q
 *   raw_k, K, V   the caches, written at the new tokens' rows (n_ctx <= n_kv)
 *   workspace     qsa_decode_step_host_workspace_size() bytes, 256-byte aligned
 * Other arguments, results and errors as qsa_decode_step, plus INVALID_ARG for null host
 * pointers, h_lse without lse_out, rows that are not whole 4-byte units, n_ctx > n_kv, or a
 * workspace without room for the staging area.
 */
qsa_status qsa_decode_step_host(const void *h_in, float *h_out, float *h_lse, void *raw_k,
                                qsa_dtype raw_dtype, int64_t n_ctx, int H_idx, int d_idx,
                                const float *norm_w, float eps, double rope_base, void *pooled,
                                qsa_dtype pooled_dtype, int64_t cap_rows, int64_t n_valid_full,
                                int64_t n_q, float scale_idx, float *scores, int64_t k_blk,
                                int32_t *blocks, int32_t *counts, void *K, void *V,
                                qsa_dtype kv_dtype, int64_t n_kv, int H_kv, int d, int64_t ld_kv,
                                int32_t *pos, int32_t *n_cells, int64_t max_cells, int H_q,
                                float scale, float *out, float *lse_out, void *workspace,
                                size_t workspace_bytes, qsa_stream_t stream);

/*
 * qsa_decode_plan -- a sequence's decode steps with the arguments that stay the same from
 * step to step bound once.
 *
 * Source: same passages as qsa_decode_step; the plan is this library's service (it only
 * saves the caller from passing some thirty unchanged arguments per step).
 *
 * qsa_decode_plan_create checks and copies the fixed arguments -- those of qsa_decode_step
 * other than n_ctx, n_valid_full, n_q, q_idx and q -- into a host object (allocated with
 * malloc; nothing on the device), for steps of up to max_queries query tokens (1..4).
 * The buffers stay the caller's and must outlive the plan; the plan keeps no state between
 * steps (the caller passes n_valid_full each step, as to qsa_decode_step).
 *   workspace  at least qsa_decode_step_workspace_size(max_queries, ...) bytes, 256-byte
 *              aligned; qsa_decode_plan_step_host also needs the staging area, i.e.
 *              qsa_decode_step_host_workspace_size(max_queries, ...) bytes.
 *   scores     room for [max_queries][cap_rows] floats.
 * qsa_decode_plan_step(plan, n_ctx, n_valid_full, n_q, q_idx, q, stream) is
 * qsa_decode_step with the plan's fixed arguments; qsa_decode_plan_step_host(plan, n_ctx,
 * n_valid_full, n_q, h_in, h_out, h_lse, stream) is qsa_decode_step_host likewise (raw_k, K
 * and V are the caches the new rows go into).  Results, validation and errors are those of
 * the two calls, plus INVALID_ARG for a null plan, n_q above max_queries, and a host step
 * on a plan whose workspace has no staging area.  qsa_decode_plan_create returns
 * INVALID_ARG (and sets *plan to NULL) for a null plan pointer, null required buffers,
 * unknown dtypes, max_queries outside [1, 4], or a workspace too small or misaligned; it
 * launches nothing.  qsa_decode_plan_destroy(NULL) does nothing.
 */
typedef struct qsa_decode_plan qsa_decode_plan;

qsa_status qsa_decode_plan_create(qsa_decode_plan **plan, void *raw_k, qsa_dtype raw_dtype,
                                  int H_idx, int d_idx, const float *norm_w, float eps,
                                  double rope_base, void *pooled, qsa_dtype pooled_dtype,
                                  int64_t cap_rows, int64_t max_queries, float scale_idx,
                                  float *scores, int64_t k_blk, int32_t *blocks, int32_t *counts,
                                  void *K, void *V, qsa_dtype kv_dtype, int64_t n_kv, int H_kv,
                                  int d, int64_t ld_kv, int32_t *pos, int32_t *n_cells,
                                  int64_t max_cells, int H_q, float scale, float *out,
                                  float *lse_out, void *workspace, size_t workspace_bytes);

void qsa_decode_plan_destroy(qsa_decode_plan *plan);

qsa_status qsa_decode_plan_step(const qsa_decode_plan *plan, int64_t n_ctx, int64_t n_valid_full,
                                int64_t n_q, const float *q_idx, const float *q,
                                qsa_stream_t stream);

qsa_status qsa_decode_plan_step_host(const qsa_decode_plan *plan, int64_t n_ctx,
                                     int64_t n_valid_full, int64_t n_q, const void *h_in,
                                     float *h_out, float *h_lse, qsa_stream_t stream);

/* Total bytes of qsa_decode_step_host's packed input (0 for an invalid shape); offsets
 * (nullable, [5]) receives the byte offsets of its sections: raw-key rows, K rows, V rows,
 * q_idx, q (each 16-byte aligned). */
size_t qsa_decode_step_host_layout(int64_t n_q, qsa_dtype raw_dtype, int H_idx, int d_idx,
                                   qsa_dtype kv_dtype, int H_kv, int d, int H_q, int64_t *offsets);

/* Workspace bytes of qsa_decode_step_host: the decode step's, then the staging area. */
size_t qsa_decode_step_host_workspace_size(int64_t n_q, int H_q, int H_kv, int d,
                                           int64_t max_cells, int64_t cap_rows,
                                           qsa_dtype raw_dtype, int H_idx, int d_idx,
                                           qsa_dtype kv_dtype);

/*
 * qsa_sparse_attn_noalloc -- qsa_sparse_attn for callers that cannot allocate device
 * memory.
 *
 * The source pages have no counterpart of this call: it is a service of this library.
 *
 * qsa_sparse_attn needs a caller-provided workspace for its split-K partial results.
 * Some callers cannot obtain one: a plugin running inside a host framework that owns
 * every device allocation and hands its plugins no allocator, or a real-time loop that
 * must not risk the latency or the failure of a cudaMalloc.  This entry point takes no
 * workspace.  Its scratch is a fixed array of QSA_NOALLOC_SCRATCH_BYTES bytes that the
 * library defines in device memory; every GPU that loads the library keeps that array
 * until the process exits.
 *
 * Arguments, layouts and results are those of qsa_sparse_attn without workspace and
 * workspace_bytes.  The call allocates nothing and calls no allocating routine.  Every
 * call looks the array's device address up (cudaGetSymbolAddress, in the caller's current
 * device and context; the lookup allocates nothing), so calls may come from any context
 * and survive a device reset; the first lookup in a context loads the library's device
 * code there if that has not happened yet, so make a first call before any stream
 * capture.  All calls share the one array, which keeps whatever the previous call wrote
 * there; nothing in it has to start at zero, because every call writes each partial
 * record before reading it.  Calls that run at the same time on the GPU (on different
 * streams, or in parallel branches of a graph) race on the array: the caller must order
 * them.
 *
 * Errors: those of qsa_sparse_attn, plus QSA_ERR_UNSUPPORTED when the split-K scratch the
 * shape's kernel really uses is larger than QSA_NOALLOC_SCRATCH_BYTES, and QSA_ERR_CUDA
 * when the address lookup fails.  The forms that merge their splits inside a thread-block
 * cluster use none (bf16 with 8 query heads per KV head and d 128, e.g. the decode shape
 * 32 / 4 heads; the latent shape; many-query bf16 4 x 8 heads); the others use about
 * qsa_sparse_attn_workspace_size() bytes (e.g. fp32 K/V, 32 / 4 heads, d 128, 2051 cells:
 * 0.6 MB), which is an upper bound for every form.
 */
#define QSA_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)
qsa_status qsa_sparse_attn_noalloc(const float *q, int64_t n_q, int H_q, int H_kv, int d_k,
                                   int d_v, float scale, const void *K, const void *V,
                                   qsa_dtype dtype, int64_t n_kv, int64_t ld_k, int64_t ld_v,
                                   const int32_t *pos, const int32_t *n_cells, int64_t max_cells,
                                   float *out, float *lse_out, qsa_stream_t stream);

/*
 * qsa_mask_to_list -- build each mask row's list of attendable key positions.
 *
 * Source: devotd.net, "llama.cpp CDNA sparse attention", section 2 (attendable key
 * positions are gathered from the mask into a list before the sparse kernel runs; the
 * per-lane selection is kept as a 64-bit mask and the count uses the same words).
 *
 * For row r: bit t of word w is (mask[r*ld_mask + 64w + t] != 0), least significant
 * bit first (each 64-bit word is built from two 32-lane warp ballots); the set
 * positions are written in ascending order to pos_out[r][0 .. min(count, max_list));
 * counts_out[r] = the true number of set positions, even when it exceeds max_list.
 *
 *   mask      [n_rows][ld_mask] uint8, nonzero = attend
 *   pos_out   [n_rows][max_list] int32;  counts_out [n_rows] int32
 *   bits_out  [n_rows][ceil(n_kv/64)] uint64, or NULL
 * Errors: INVALID_ARG for null required pointers, n_kv < 0, ld_mask < n_kv,
 * max_list < 0; UNSUPPORTED for n_kv > 2^31 - 1.
 */
qsa_status qsa_mask_to_list(const uint8_t *mask, int64_t n_rows, int64_t n_kv, int64_t ld_mask,
                            int64_t max_list, int32_t *pos_out, int32_t *counts_out,
                            uint64_t *bits_out, qsa_stream_t stream);

/*
 * qsa_mask_sparse_attn -- the mask-driven sparse attention in one call: each query's key
 * list is taken from its mask row inside the attention kernel instead of a separate
 * qsa_mask_to_list launch.
 *
 * Source: devotd.net, "llama.cpp CDNA sparse attention", section 2 (the attendable
 * positions are listed from the mask before the sparse kernel runs) and section 3 (the
 * sparse matrix-op kernel over the listed keys, for DKQ 576 with 16 query columns per KV
 * group; here d_v 512 on one latent KV head).
 *
 * For query i the list is the ascending set positions of mask row i (nonzero bytes of
 * mask[i*ld_mask + 0 .. n_kv)), exactly the list qsa_mask_to_list writes, and the result
 * equals qsa_sparse_attn over that list (same cells per split, same order: bit for bit).
 * counts_out[i] (nullable) = the true count; a count above max_list gives out = NaN and
 * lse = NaN for that query (the caller must not use it), as in the two-call path.
 *
 *   q       [n_q][H_q][576] fp32, 8-byte aligned;  out [n_q][H_q][512] fp32
 *   KV      [n_kv] rows of ld_kv bf16 elements (16-byte aligned, ld_kv*2 a multiple of 16):
 *           the key is a row's first 576 columns, the value its first 512
 *   mask    [n_q][ld_mask] uint8, nonzero = attend;  lse_out [n_q][H_q] or NULL
 * Only the latent shape runs here: bf16, d_k 576, d_v 512, H_q = 16 on H_kv = 1
 * (QSA_ERR_UNSUPPORTED otherwise), n_kv <= 65536 (QSA_ERR_UNSUPPORTED above).
 * Errors: INVALID_ARG for null q / KV / mask / out, a misaligned q, out, lse_out or
 * counts_out, n_q < 0, H_q not a multiple of H_kv, ld_kv < H_kv * d_k, ld_mask < n_kv,
 * max_list < 0, a dtype other than QSA_F32 / QSA_BF16.  No workspace: the splits of a query combine inside a thread-block cluster.
 * Eligibility (qsa_mask_sparse_eligible) stays the caller's decision.
 */
qsa_status qsa_mask_sparse_attn(const float *q, int64_t n_q, int H_q, int H_kv, int d_k,
                                int d_v, float scale, const void *KV, qsa_dtype dtype,
                                int64_t n_kv, int64_t ld_kv, const uint8_t *mask, int64_t ld_mask,
                                int64_t max_list, int32_t *counts_out, float *out, float *lse_out,
                                qsa_stream_t stream);

/*
 * qsa_mask_sparse_eligible -- host-side check of when the mask-driven sparse path
 * applies.
 *
 * Source: devotd.net, "llama.cpp CDNA sparse attention", section 3 (the sparse path is
 * a candidate when a mask is present and bias and softcap are 0; on CDNA the key length
 * must be at least 4096 and at least twice the maximum list length).
 *
 * Returns QSA_OK when has_mask != 0, max_bias == 0, softcap == 0, n_kv >= 4096 and
 * n_kv >= 2*max_list; QSA_ERR_UNSUPPORTED otherwise (this library has no dense
 * fallback: the caller runs its own dense attention).  Launches nothing.
 */
qsa_status qsa_mask_sparse_eligible(int has_mask, float max_bias, float softcap, int64_t n_kv,
                                    int64_t max_list);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H */
