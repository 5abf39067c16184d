// topk.cu -- block-domain top-k: one CTA per query, radix select over score keys.
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "block-domain top-k (COMMON-006)": select over the block scores instead of expanding
// every block score to its cells first (the expansion cost grew with context:
// 0.45 -> 0.91 ms per layer from 128k to 256k on the pages' GPU), then expand only the
// selected blocks to cell indices and append the tail.
//
// Scores become order-preserving 32-bit keys.  The k-th largest key T is found by radix
// select in three digits (12 + 10 + 10 bits):
//   1. a 4096-bin histogram of the top 12 bits -- either accumulated by the score kernel
//      as it writes the scores (decode step, no extra pass; this kernel clears it again)
//      or built here from one read;
//   2. one read of the scores classifies every candidate: above the threshold bucket
//      (selected: a bit in a shared-memory bitmap), inside it (appended to a candidate
//      list in shared memory), or below (dropped);
//   3. the remaining digits are resolved on the candidate list alone (a few hundred to a
//      few thousand keys), stopping early once a bucket holds exactly the keys still
//      needed;
//   4. the candidates above T join the bitmap, the ones equal to T go to a tie bitmap;
//   5. a block-wide scan over the bitmap words writes the selected blocks in ascending
//      order -- ties taken lowest index first -- and, when asked, their cells and the
//      open tail.
// If the candidate list would overflow shared memory (pathological score
// distributions), steps 3-4 re-read the scores instead.  No inter-CTA communication,
// no global scratch beyond the optional histogram, no spin-waits.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int NT = kTopkThreads;
constexpr int kBins1 = 1 << kTopkHistBits;  // 4096
constexpr int kMaxSmemBytes = 220 * 1024;
constexpr int kFixedWords = kBins1 + 2 * (NT / 32) + 32;
constexpr int64_t kMaxN = 640 * 1024;           // candidates per query
constexpr int kCandCapMax = 16384;

__device__ __forceinline__ void put_cells(int32_t *dst, int32_t b, bool vec)
{
    if (vec) {
        *reinterpret_cast<int4 *>(dst) = make_int4(4 * b, 4 * b + 1, 4 * b + 2, 4 * b + 3);
    } else {
        dst[0] = 4 * b;
        dst[1] = 4 * b + 1;
        dst[2] = 4 * b + 2;
        dst[3] = 4 * b + 3;
    }
}

// Exclusive prefix sum over the block (NT threads); *total gets the block total.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *warp_s, uint32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_s[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < NT / 32 ? warp_s[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < NT / 32) warp_s[lane] = w;
    }
    __syncthreads();
    const uint32_t r = (warp == 0 ? 0u : warp_s[warp - 1]) + x - v;
    *total = warp_s[NT / 32 - 1];
    __syncthreads();
    return r;
}

// Bucket holding the k_rem-th largest of the histogram h[0..nb) (bins scanned from the
// top).  Returns via misc: [0] bin, [1] keys in higher bins, [2] keys in the bin.
__device__ __forceinline__ void find_bucket(const uint32_t *h, int nb, uint32_t k_rem,
                                            uint32_t *warp_s, uint32_t *misc)
{
    const int per = nb / NT;  // 4 or 1
    uint32_t cnt[4];
    uint32_t mine = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        cnt[j] = j < per ? h[nb - 1 - threadIdx.x * per - j] : 0u;
        mine += cnt[j];
    }
    uint32_t tot;
    uint32_t above = block_excl_scan(mine, warp_s, &tot);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (j < per) {
            if (above < k_rem && above + cnt[j] >= k_rem) {
                misc[0] = (uint32_t)(nb - 1 - threadIdx.x * per - j);
                misc[1] = above;
                misc[2] = cnt[j];
            }
            above += cnt[j];
        }
    }
    __syncthreads();
}

// Apply f(key, index) to every score of the row.  Each thread first loads 8 16-byte
// vectors (all in flight at once), then applies f to their 32 keys.
template <typename F>
__device__ __forceinline__ void for_each_key(const float *__restrict__ row, int64_t n, F f)
{
    constexpr int U = 8;
    if ((reinterpret_cast<uintptr_t>(row) & 15) == 0) {
        const int64_t n4 = n / 4;
        const float4 *r4 = reinterpret_cast<const float4 *>(row);
        for (int64_t base = threadIdx.x; base < n4; base += (int64_t)NT * U) {
            float4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = base + (int64_t)u * NT;
                v[u] = i < n4 ? r4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = base + (int64_t)u * NT;
                if (i < n4) {
                    f(score_key(v[u].x), 4 * i);
                    f(score_key(v[u].y), 4 * i + 1);
                    f(score_key(v[u].z), 4 * i + 2);
                    f(score_key(v[u].w), 4 * i + 3);
                }
            }
        }
        for (int64_t i = 4 * n4 + threadIdx.x; i < n; i += NT) f(score_key(row[i]), i);
    } else {
        for (int64_t base = threadIdx.x; base < n; base += (int64_t)NT * U) {
            float v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = base + (int64_t)u * NT;
                v[u] = i < n ? row[i] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = base + (int64_t)u * NT;
                if (i < n) f(score_key(v[u]), i);
            }
        }
    }
}

__global__ void __launch_bounds__(NT)
topk_kernel(const float *__restrict__ scores, int64_t ld, const int32_t *__restrict__ q_pos,
            int64_t n_full_cap, int k_blk, int32_t *__restrict__ blocks_out,
            int32_t *__restrict__ counts_out, int64_t n_ctx, int32_t *__restrict__ pos_out,
            int32_t *__restrict__ n_cells_out, int64_t max_cells, uint32_t *__restrict__ ext_hist,
            int cand_cap, const TopkPre pre)
{
    extern __shared__ __align__(16) uint32_t smem[];
    uint32_t *hist = smem;                      // [4096]
    uint32_t *warp_s = hist + kBins1;           // [2][NT/32]
    uint32_t *misc = warp_s + 2 * (NT / 32);    // [32]
    uint32_t *selw = misc + 32;                 // [nw] selected blocks bitmap
    const int64_t qi = blockIdx.x;
    const uint32_t *pre_meta = pre.meta, *pre_bitmap = pre.bitmap;
    const uint2 *pre_cand = pre.cand;
    const int32_t *pre_cnt = pre.cand_cnt;

    pdl_wait();
    QSA_AFTER_WAIT(scores);
    QSA_AFTER_WAIT(q_pos);
    QSA_AFTER_WAIT(ext_hist);
    QSA_AFTER_WAIT(pre_meta);
    QSA_AFTER_WAIT(pre_bitmap);
    QSA_AFTER_WAIT(pre_cand);
    QSA_AFTER_WAIT(pre_cnt);
    pdl_trigger();

    const int64_t p = q_pos ? (int64_t)q_pos[qi] : n_ctx - 1;  // the query's position
    int64_t n = n_full_cap;
    if (q_pos) {
        const int64_t p1 = (p + 1) / 4;
        n = p1 < n ? p1 : n;
    }
    if (n < 0) n = 0;
    const int64_t k = (int64_t)k_blk < n ? (int64_t)k_blk : n;
    int32_t *out = blocks_out + qi * (int64_t)k_blk;
    int32_t *pout = pos_out ? pos_out + qi * max_cells : nullptr;
    const bool pvec = (reinterpret_cast<uintptr_t>(pout) & 15) == 0;
    uint32_t *ehist = ext_hist ? ext_hist + qi * (int64_t)kBins1 : nullptr;
    if (threadIdx.x < 4) {
        const int64_t tail0 = 4 * ((p + 1) / 4);
        const int64_t n_tail = p + 1 - tail0;
        if (threadIdx.x == 0) counts_out[qi] = (int32_t)k;
        if (pout) {
            if (threadIdx.x == 0) n_cells_out[qi] = (int32_t)(4 * k + n_tail);
            if (threadIdx.x < n_tail) pout[4 * k + threadIdx.x] = (int32_t)(tail0 + threadIdx.x);
        }
    }
    if (n <= k_blk) {  // every candidate is selected
        for (int64_t i = threadIdx.x; i < n; i += NT) {
            out[i] = (int32_t)i;
            if (pout) put_cells(pout + 4 * i, (int32_t)i, pvec);
        }
        if (ehist)  // leave the histogram cleared for the next step
            for (int i = threadIdx.x; i < kBins1; i += NT) ehist[i] = 0u;
        return;
    }
    const int64_t nw = (n + 31) / 32;
    uint32_t *eqw = selw + nw;                               // [nw] tie bitmap
    uint32_t *cand_key = eqw + nw;                           // [cand_cap]
    int32_t *cand_idx = reinterpret_cast<int32_t *>(cand_key + cand_cap);
    const float *srow = scores + qi * ld;

    uint32_t prefix = 0, k_rem = 0;
    int fixed = kTopkHistBits;
    bool whole = false;
    bool pre_ok = false;
    if (pre_meta) {
        // ---- 1-2 done by the classify pass: take its decision, bitmap and candidates
        const int c = threadIdx.x;
        uint32_t my = 0;
        bool over = false;
        if (c < pre.n_cta) {
            my = (uint32_t)pre_cnt[c];
            over = my > (uint32_t)pre.cap;
        }
        const bool any_over = __syncthreads_or(over);
        uint32_t n_cand;
        const uint32_t cbase = block_excl_scan(my, warp_s, &n_cand);
        pre_ok = pre_meta[3] != 0 && !any_over && n_cand <= (uint32_t)cand_cap;
        if (pre_ok) {
            prefix = pre_meta[0];
            k_rem = (uint32_t)k - pre_meta[1];
            whole = pre_meta[2] != 0;
            for (int64_t w = threadIdx.x; w < nw; w += NT) {
                selw[w] = pre_bitmap[w];
                eqw[w] = 0u;
            }
            for (uint32_t j = 0; j < my; ++j) {
                const uint2 e = pre_cand[(int64_t)c * pre.cap + j];
                cand_key[cbase + j] = e.x;
                cand_idx[cbase + j] = (int32_t)e.y;
            }
            if (threadIdx.x == 0) misc[8] = n_cand;
        }
        if (ehist)  // leave the histogram cleared for the next step
            for (int i = threadIdx.x; i < kBins1; i += NT) ehist[i] = 0u;
        __syncthreads();
    }
    if (!pre_ok) {
        // ---- 1. histogram of the top 12 bits: take the one the score kernel accumulated
        // (and clear it for the next step) unless its total disagrees with the candidate
        // count -- a workspace that was never cleared -- in which case build it here
        bool have = false;
        if (ehist && !pre_meta) {
            uint32_t part = 0;
            for (int i = threadIdx.x; i < kBins1; i += NT) {
                const uint32_t v = ehist[i];
                hist[i] = v;
                ehist[i] = 0u;
                part += v;
            }
            uint32_t tot;
            block_excl_scan(part, warp_s, &tot);
            have = tot == (uint32_t)n;
        }
        if (!have) {
            for (int i = threadIdx.x; i < kBins1; i += NT) hist[i] = 0u;
            __syncthreads();
            for_each_key(srow, n, [&](uint32_t key, int64_t) {
                atomicAdd(&hist[key >> (32 - kTopkHistBits)], 1u);
            });
        }
        for (int64_t i = threadIdx.x; i < 2 * nw; i += NT) selw[i] = 0u;
        if (threadIdx.x == 0) misc[8] = 0u;  // candidate count
        __syncthreads();
        find_bucket(hist, kBins1, (uint32_t)k, warp_s, misc);
        prefix = misc[0];
        k_rem = (uint32_t)k - misc[1];
        whole = misc[2] == k_rem;
        __syncthreads();

        // ---- 2. classify every candidate (one read)
        const uint32_t B1c = prefix;
        const uint32_t lo_key = B1c << (32 - kTopkHistBits);  // smallest key with digit B1
        for_each_key(srow, n, [&](uint32_t key, int64_t i) {
            if (key < lo_key) return;  // below the threshold bucket: the common case
            const uint32_t d = key >> (32 - kTopkHistBits);
            if (d > B1c || whole) {
                atomicOr(&selw[i >> 5], 1u << (i & 31));
            } else {
                const uint32_t slot = atomicAdd(&misc[8], 1u);
                if (slot < (uint32_t)cand_cap) {
                    cand_key[slot] = key;
                    cand_idx[slot] = (int32_t)i;
                }
            }
        });
        __syncthreads();
    }
    const uint32_t B1 = prefix;

    if (!whole) {
        const uint32_t n_cand = misc[8];
        const bool in_smem = n_cand <= (uint32_t)cand_cap;
        // ---- 3. remaining digits on the candidates
        bool exact = false;
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            const int bits = 10;
            const int shift = 32 - fixed - bits;
            const int nb = 1 << bits;
            for (int i = threadIdx.x; i < nb; i += NT) hist[i] = 0u;
            __syncthreads();
            const uint32_t pf = prefix;
            const int fx = fixed;
            auto add = [&](uint32_t key, int64_t) {
                if ((key >> (32 - fx)) == pf) atomicAdd(&hist[(key >> shift) & (uint32_t)(nb - 1)], 1u);
            };
            if (in_smem) {
                for (uint32_t c = threadIdx.x; c < n_cand; c += NT) add(cand_key[c], 0);
            } else {
                for_each_key(srow, n, add);
            }
            __syncthreads();
            find_bucket(hist, nb, k_rem, warp_s, misc);
            k_rem -= misc[1];
            prefix = (prefix << bits) | misc[0];
            fixed += bits;
            exact = misc[2] == k_rem;
            __syncthreads();
            if (exact) break;
        }
        // ---- 4. mark the candidates above the threshold and the ties
        const int drop = 32 - fixed;
        const uint32_t T = prefix;
        auto mark = [&](uint32_t key, int64_t i) {
            if ((key >> (32 - kTopkHistBits)) != B1) return;
            const uint32_t kp = key >> drop;
            if (kp > T || (exact && kp == T)) atomicOr(&selw[i >> 5], 1u << (i & 31));
            else if (kp == T) atomicOr(&eqw[i >> 5], 1u << (i & 31));
        };
        if (in_smem) {
            for (uint32_t c = threadIdx.x; c < n_cand; c += NT) mark(cand_key[c], cand_idx[c]);
        } else {
            for_each_key(srow, n, mark);
        }
        if (exact) k_rem = 0;
        __syncthreads();
    } else {
        k_rem = 0;
    }

    // ---- 5. ordered output: ties lowest index first, then a scan over bitmap words
    const int64_t wpt = (nw + NT - 1) / NT;
    const int64_t w0 = (int64_t)threadIdx.x * wpt;
    const int64_t w1 = w0 + wpt < nw ? w0 + wpt : nw;
    uint32_t n_eq = 0;
    for (int64_t w = w0; w < w1; ++w) n_eq += __popc(eqw[w]);
    uint32_t tot;
    uint32_t eq_before = block_excl_scan(n_eq, warp_s, &tot);
    uint32_t n_sel = 0;
    for (int64_t w = w0; w < w1; ++w) {
        uint32_t e = eqw[w];
        uint32_t keep = 0;
        while (e && eq_before < k_rem) {
            const uint32_t bit = e & (0u - e);
            keep |= bit;
            e ^= bit;
            ++eq_before;
        }
        const uint32_t f = selw[w] | keep;
        selw[w] = f;
        n_sel += __popc(f);
    }
    uint32_t o = block_excl_scan(n_sel, warp_s + NT / 32, &tot);
    for (int64_t w = w0; w < w1; ++w) {
        uint32_t f = selw[w];
        while (f) {
            const int b = __ffs(f) - 1;
            f &= f - 1;
            const int32_t blk = (int32_t)(32 * w + b);
            if (o < (uint32_t)k) {
                out[o] = blk;
                if (pout) put_cells(pout + 4 * o, blk, pvec);
            }
            ++o;
        }
    }
}

// Classify pass (decode, one query): every CTA derives the threshold digit from the score
// kernel's histogram, then one warp per bitmap word classifies 32 consecutive blocks with
// two ballots -- the word of blocks above the threshold bucket is written as is, blocks
// inside it are appended to this CTA's candidate list.  CTA 0 publishes the decision.
__global__ void __launch_bounds__(NT)
topk_classify_kernel(const float *__restrict__ scores, int64_t n, int64_t k,
                     const uint32_t *__restrict__ hist, uint32_t *__restrict__ meta,
                     uint32_t *__restrict__ bitmap, uint2 *__restrict__ cand,
                     int32_t *__restrict__ cand_cnt, int cap)
{
    __shared__ uint32_t h[kBins1];
    __shared__ uint32_t warp_s[2 * (NT / 32)];
    __shared__ uint32_t misc[32];
    pdl_wait();
    QSA_AFTER_WAIT(scores);
    QSA_AFTER_WAIT(hist);
    pdl_trigger();
    uint32_t part = 0;
    for (int i = threadIdx.x; i < kBins1; i += NT) {
        const uint32_t v = hist[i];
        h[i] = v;
        part += v;
    }
    uint32_t tot;
    block_excl_scan(part, warp_s, &tot);
    if (threadIdx.x == 0) misc[8] = 0u;
    if (tot != (uint32_t)n) {  // not this step's histogram: the resolve pass does it all
        if (blockIdx.x == 0 && threadIdx.x == 0) meta[3] = 0u;
        return;
    }
    find_bucket(h, kBins1, (uint32_t)k, warp_s, misc);
    const uint32_t B1 = misc[0];
    const uint32_t above_n = misc[1];
    const bool whole = misc[2] == (uint32_t)k - above_n;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        meta[0] = B1;
        meta[1] = above_n;
        meta[2] = whole ? 1u : 0u;
        meta[3] = 1u;
    }
    const int lane = threadIdx.x & 31;
    const int64_t nw = (n + 31) / 32;
    const int64_t wi = (int64_t)blockIdx.x * kClsWordsPerCta + (threadIdx.x >> 5);
    if (wi < nw) {
        const int64_t i = wi * 32 + lane;
        const bool valid = i < n;
        const uint32_t key = valid ? score_key(scores[i]) : 0u;
        const uint32_t d = key >> (32 - kTopkHistBits);
        const bool above = valid && (d > B1 || (whole && d == B1));
        const bool is_cand = valid && !whole && d == B1;
        const uint32_t word = __ballot_sync(0xffffffffu, above);
        if (lane == 0) bitmap[wi] = word;
        const uint32_t cm = __ballot_sync(0xffffffffu, is_cand);
        uint32_t base = 0;
        if (lane == 0 && cm) base = atomicAdd(&misc[8], (uint32_t)__popc(cm));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (is_cand) {
            const uint32_t slot = base + __popc(cm & ((1u << lane) - 1u));
            if (slot < (uint32_t)cap) cand[(int64_t)blockIdx.x * cap + slot] = make_uint2(key, (uint32_t)i);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) cand_cnt[blockIdx.x] = (int32_t)misc[8];
}

size_t topk_smem_bytes(int64_t n, int *cand_cap)
{
    const int64_t nw = (n + 31) / 32;
    int64_t words = kFixedWords + 2 * nw;
    int64_t cap = (kMaxSmemBytes / 4 - words) / 2;
    if (cap > kCandCapMax) cap = kCandCapMax;
    if (cap < 0) cap = 0;
    *cand_cap = (int)cap;
    return sizeof(uint32_t) * (size_t)(words + 2 * cap);
}

}  // namespace

int64_t topk_max_candidates() { return kMaxN; }

size_t topk_pre_workspace_bytes(int64_t n_full_cap)
{
    const int64_t nw = (n_full_cap + 31) / 32;
    const int64_t g = (nw + kClsWordsPerCta - 1) / kClsWordsPerCta;
    // meta (256 B) | counts | candidates | bitmap, each 256-byte aligned
    auto al = [](int64_t b) { return (b + 255) & ~(int64_t)255; };
    return (size_t)(256 + al(4 * g) + al(8 * g * kClsCap) + al(4 * nw));
}

cudaError_t launch_topk_classify(const float *scores, int64_t n_full, int64_t k_blk,
                                 const uint32_t *hist, uint32_t *meta, uint32_t *bitmap,
                                 uint2 *cand, int32_t *cand_cnt, TopkPre *pre, cudaStream_t st)
{
    const int64_t nw = (n_full + 31) / 32;
    const int64_t g = (nw + kClsWordsPerCta - 1) / kClsWordsPerCta;
    if (n_full <= k_blk || g < 1 || g > NT) return cudaErrorNotSupported;
    cudaError_t e = launch(topk_classify_kernel, dim3((unsigned)g), dim3(NT), 0, st, 1, scores,
                           n_full, k_blk, hist, meta, bitmap, cand, cand_cnt, kClsCap);
    if (e != cudaSuccess) return e;
    pre->meta = meta;
    pre->bitmap = bitmap;
    pre->cand = cand;
    pre->cand_cnt = cand_cnt;
    pre->n_cta = (int)g;
    pre->cap = kClsCap;
    return cudaSuccess;
}

cudaError_t launch_topk(const float *scores, int64_t n_q, int64_t ld, const int32_t *q_pos,
                        int64_t n_full, int64_t k_blk, int32_t *blocks_out, int32_t *counts_out,
                        int64_t n_ctx, int32_t *pos_out, int32_t *n_cells_out,
                        int64_t max_cells, uint32_t *ext_hist, cudaStream_t st,
                        const TopkPre &pre)
{
    if (n_q == 0) return cudaSuccess;
    int cand_cap = 0;
    const size_t smem = topk_smem_bytes(n_full, &cand_cap);
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kMaxSmemBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    return launch(topk_kernel, dim3((unsigned)n_q), dim3(NT), smem, st, 1, scores, ld, q_pos,
                  n_full, (int)k_blk, blocks_out, counts_out, n_ctx, pos_out, n_cells_out,
                  max_cells, ext_hist, cand_cap, pre);
}

}  // namespace qsa
