// topk.cu -- block-domain top-k: radix select over order-preserving score keys.
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "block-domain top-k (COMMON-006)": select over the block scores instead of expanding
// every block score to its cells first (the expansion cost grew with context:
// 0.45 -> 0.91 ms per layer from 128k to 256k on the pages' GPU), then expand only the
// selected blocks to cell indices and append the tail.
//
// Scores become order-preserving 32-bit keys.  The k-th largest key T is found by radix
// select, first digit 12 bits (a 4096-bin histogram), then digits of 10 bits.
//
// General form (qsa_topk_blocks, prefill): one 1024-thread CTA per query.
//   1. the 4096-bin histogram -- built here from one read of the scores, or taken from
//      the score kernel when it accumulated one (and cleared again for the next step);
//   2. one read of the scores classifies every block: above the threshold bucket
//      (selected: a bit in a shared-memory bitmap), inside it (a candidate list in
//      shared memory), or below (dropped);
//   3. the remaining digits are resolved on the candidate list alone, stopping early
//      once a bucket holds exactly the keys still needed;
//   4. the candidates above T join the bitmap, the ones equal to T go to a tie bitmap;
//   5. a block-wide scan over the bitmap words writes the selected blocks in ascending
//      order -- ties taken lowest index first -- and, when asked, their cells and the
//      open tail.
// If the candidate list would overflow shared memory (pathological score
// distributions), steps 3-4 re-read the scores instead.
//
// Decode form (inside qsa_decode_step, 1-4 queries): one kernel of ceil(n/1024) CTAs per
// query.  Every CTA finds the threshold bucket in its query's histogram (built by the
// score kernel) with a two-level warp search, classifies its 1024 blocks with ballots
// (bitmap words for the blocks above the bucket, a per-CTA list for the blocks inside it),
// then takes its query's ticket; the last CTA to arrive settles the bucket with a second
// 8-bit digit and ranks the few candidates left against each other (key descending, index
// ascending), writes the selection, the cells and the tail, and clears the histogram.  No CTA waits for another: the ticket decides which CTA
// finishes the work, so there is no spin-wait.  A histogram whose total disagrees with
// the block count (a workspace never cleared), or a bucket holding more than 1024
// candidates, sends the last CTA through the general form instead.
#include "qsa_internal.cuh"
#include "prefill_select.cuh"

namespace qsa {
namespace {

constexpr int NT = kTopkThreads;
constexpr int kBins1 = 1 << kTopkHistBits;  // 4096
constexpr int kMaxSmemBytes = 220 * 1024;
constexpr int kFixedWords = kBins1 + 2 * (NT / 32) + 32;
constexpr int64_t kMaxN = 640 * 1024;           // candidates per query
constexpr int kCandCapMax = 16384;
constexpr int64_t kSampledMinN = 16384;  // below this the sampled form saves nothing

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

// The float whose key is T, for a T above the key of -inf (score_key is monotone and maps
// NaN to -inf and -0 to +0): for such T, score_key(x) >= T exactly when x >= key_float(T)
// as floats (a NaN x compares false, and its key, that of -inf, is below T).  A T in the
// NaN range above +inf gives a NaN, which no x reaches, as no key reaches T.
__device__ __forceinline__ float key_float(uint32_t T)
{
    return __uint_as_float((T & 0x80000000u) ? (T & 0x7fffffffu) : ~T);
}
constexpr uint32_t kKeyNegInf = 0x007fffffu;  // score_key(-inf), also that of NaN

// Apply f(key, index) to the scores of the row with key >= T, T > kKeyNegInf: one float
// compare per score (four per vector on the common path) instead of a key per score.
template <typename F>
__device__ __forceinline__ void for_each_key_at_least(const float *__restrict__ row, int64_t n,
                                                      uint32_t T, F f)
{
    constexpr int U = 8;
    const float lo = key_float(T);
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
                const float4 x = v[u];
                // fmaxf drops NaN operands, so the maximum reaches lo iff some lane does
                if (i < n4 && fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)) >= lo) {
                    if (x.x >= lo) f(score_key(x.x), 4 * i);
                    if (x.y >= lo) f(score_key(x.y), 4 * i + 1);
                    if (x.z >= lo) f(score_key(x.z), 4 * i + 2);
                    if (x.w >= lo) f(score_key(x.w), 4 * i + 3);
                }
            }
        }
        for (int64_t i = 4 * n4 + threadIdx.x; i < n; i += NT)
            if (row[i] >= lo) f(score_key(row[i]), i);
    } else {
        for (int64_t i = threadIdx.x; i < n; i += NT)
            if (row[i] >= lo) f(score_key(row[i]), i);
    }
}

// The sampled form's candidate pass over a 16-byte aligned row (T > kKeyNegInf): every
// score >= key_float(T) goes to the candidate list (key, block), slots past cap counted
// but not stored, and into hist, the candidates' histogram of the first 12-bit digit.  Each round a thread loads U vectors, folds them into a 4U-bit hit mask
// and lets them die; a warp scan and one shared atomic per warp reserve the round's slots;
// the hits are then read again (lines just fetched) and stored.  Keeping the vectors live
// across the stores (a lambda per hit) measured 9.8 us per 64k-block row against 5.6 us
// this way.  All threads of the CTA call it; the round loop is uniform (full-warp shuffles).
__device__ __forceinline__ void collect_at_least(const float *__restrict__ row, int64_t n,
                                                 uint32_t T, uint32_t *counter,
                                                 uint32_t *cand_key, int32_t *cand_idx,
                                                 uint32_t cap, uint32_t *hist)
{
    constexpr int U = 8;
    const float lo = key_float(T);
    const int lane = threadIdx.x & 31;
    const int n4 = (int)(n / 4);  // n <= kMaxN: int indices
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
    const float4 pad = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);  // < lo
    for (int b0 = 0; b0 < n4; b0 += NT * U) {
        float4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = b0 + (int)threadIdx.x + u * NT;
            v[u] = i < n4 ? r4[i] : pad;
        }
        uint32_t hit = 0;
#pragma unroll
        for (int u = 0; u < U; ++u)
            hit |= ((uint32_t)(v[u].x >= lo) | ((uint32_t)(v[u].y >= lo) << 1) |
                    ((uint32_t)(v[u].z >= lo) << 2) | ((uint32_t)(v[u].w >= lo) << 3)) << (4 * u);
        const uint32_t c = __popc(hit);
        uint32_t inc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        const uint32_t tot = __shfl_sync(0xffffffffu, inc, 31);
        uint32_t s = 0;
        if (lane == 31 && tot) s = atomicAdd(counter, tot);
        s = __shfl_sync(0xffffffffu, s, 31) + inc - c;
        while (hit) {
            const int bit = __ffs(hit) - 1;
            hit &= hit - 1;
            const int b = 4 * (b0 + (int)threadIdx.x + (bit >> 2) * NT) + (bit & 3);
            const uint32_t key = score_key(row[b]);
            atomicAdd(&hist[key >> (32 - kTopkHistBits)], 1u);
            if (s < cap) {
                cand_key[s] = key;
                cand_idx[s] = b;
            }
            ++s;
        }
    }
    for (int64_t i = 4 * (int64_t)n4 + threadIdx.x; i < n; i += NT)
        if (row[i] >= lo) {
            const uint32_t key = score_key(row[i]);
            atomicAdd(&hist[key >> (32 - kTopkHistBits)], 1u);
            const uint32_t slot = atomicAdd(counter, 1u);
            if (slot < cap) {
                cand_key[slot] = key;
                cand_idx[slot] = (int32_t)i;
            }
        }
}

// Step 5 of the general form: fold the ties (lowest index first, k_rem of them) into the
// selected bitmap, then write the selected blocks in ascending order.
__device__ void write_selection(uint32_t *selw, const uint32_t *eqw, int64_t nw, uint32_t k_rem,
                                int64_t k, int32_t *out, int32_t *pout, bool pvec,
                                uint32_t *warp_s)
{
    const int64_t wpt = (nw + NT - 1) / NT;
    const int64_t w0 = (int64_t)threadIdx.x * wpt;
    const int64_t w1 = w0 + wpt < nw ? w0 + wpt : nw;
    uint32_t tot;
    uint32_t n_sel = 0;
    if (eqw) {
        uint32_t n_eq = 0;
        for (int64_t w = w0; w < w1; ++w) n_eq += __popc(eqw[w]);
        uint32_t eq_before = block_excl_scan(n_eq, warp_s, &tot);
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
    } else {
        for (int64_t w = w0; w < w1; ++w) n_sel += __popc(selw[w]);
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

// Counts and the open tail of one query (threads 0-3 of the CTA).
__device__ __forceinline__ void write_count_tail(int64_t k, int64_t p, int32_t *count_out,
                                                 int32_t *pout, int32_t *n_cells_out)
{
    if (threadIdx.x < 4) {
        const int64_t tail0 = 4 * ((p + 1) / 4);
        const int64_t n_tail = p + 1 - tail0;
        if (threadIdx.x == 0) *count_out = (int32_t)k;
        if (pout) {
            if (threadIdx.x == 0) *n_cells_out = (int32_t)(4 * k + n_tail);
            if (threadIdx.x < n_tail) pout[4 * k + threadIdx.x] = (int32_t)(tail0 + threadIdx.x);
        }
    }
}

// The general form for one query whose n candidates outnumber k (steps 1-5).  smem:
// hist [4096] | warp_s [2][32] | misc [32] | selw [nw] | eqw [nw] | keys [cap] | idx [cap].
// ehist (nullable): the score kernel's histogram of this query, cleared here.
__device__ void topk_query(const float *srow, int64_t n, int64_t k, int32_t *out, int32_t *pout,
                           bool pvec, uint32_t *ehist, int cand_cap, uint32_t *smem)
{
    uint32_t *hist = smem;
    uint32_t *warp_s = hist + kBins1;
    uint32_t *misc = warp_s + 2 * (NT / 32);
    uint32_t *selw = misc + 32;
    const int64_t nw = (n + 31) / 32;
    uint32_t *eqw = selw + nw;
    uint32_t *cand_key = eqw + nw;
    int32_t *cand_idx = reinterpret_cast<int32_t *>(cand_key + cand_cap);

    // ---- 1. histogram of the top 12 bits: take the one the score kernel accumulated
    // (and clear it for the next step) unless its total disagrees with the candidate
    // count -- a workspace that was never cleared -- in which case build it here
    bool have = false;
    if (ehist) {
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
    uint32_t prefix = misc[0];
    uint32_t k_rem = (uint32_t)k - misc[1];
    const bool whole = misc[2] == k_rem;
    int fixed = kTopkHistBits;
    __syncthreads();

    // ---- 2. classify every candidate (one read)
    const uint32_t B1 = prefix;
    const uint32_t lo_key = B1 << (32 - kTopkHistBits);  // smallest key with digit B1
    auto classify = [&](uint32_t key, int64_t i) {
        if (key < lo_key) return;  // below the threshold bucket: the common case
        const uint32_t d = key >> (32 - kTopkHistBits);
        if (d > B1 || whole) {
            atomicOr(&selw[i >> 5], 1u << (i & 31));
        } else {
            const uint32_t slot = atomicAdd(&misc[8], 1u);
            if (slot < (uint32_t)cand_cap) {
                cand_key[slot] = key;
                cand_idx[slot] = (int32_t)i;
            }
        }
    };
    if (lo_key > kKeyNegInf) for_each_key_at_least(srow, n, lo_key, classify);
    else for_each_key(srow, n, classify);
    __syncthreads();

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

    // ---- 5. ordered output
    write_selection(selw, eqw, nw, k_rem, k, out, pout, pvec, warp_s);
}

// Steps 3-6 of the candidate forms: the exact top k of the m candidates (cand_key / cand_idx;
// hist holds their first-digit histogram): first 12-bit digit, second 8-bit digit, a (key,
// index) rank inside the last bin, then the ordered output.  Returns false (nothing written)
// when the last bin holds more than kBins1 candidates.  All threads of the CTA call it.
__device__ bool select_candidates(int64_t k, uint32_t m, uint32_t *hist, uint32_t *warp_s,
                                  uint32_t *misc, uint32_t *selw, int64_t nw,
                                  const uint32_t *cand_key, const int32_t *cand_idx,
                                  int32_t *out, int32_t *pout, bool pvec)
{
    const int tid = threadIdx.x;
    // ---- 3. first digit over the candidates (their histogram came with the pass)
    find_bucket(hist, kBins1, (uint32_t)k, warp_s, misc);
    const uint32_t B1 = misc[0];
    const uint32_t k_rem = (uint32_t)k - misc[1];
    const bool whole1 = misc[2] == k_rem;
    __syncthreads();
    // ---- 4. above the bucket: selected; inside it: the second digit
    if (tid < 256) hist[tid] = 0u;
    __syncthreads();
    for (uint32_t c = tid; c < m; c += NT) {
        const uint32_t key = cand_key[c];
        const uint32_t d1 = key >> (32 - kTopkHistBits);
        if (d1 > B1 || (whole1 && d1 == B1)) {
            const int32_t i = cand_idx[c];
            atomicOr(&selw[i >> 5], 1u << (i & 31));
        } else if (d1 == B1) {
            atomicAdd(&hist[(key >> 12) & 255u], 1u);
        }
    }
    __syncthreads();
    if (!whole1) {
        {
            const uint32_t c2 = tid < 256 ? hist[255 - tid] : 0u;  // top bin first
            uint32_t tot;
            const uint32_t above2 = block_excl_scan(c2, warp_s, &tot);
            if (tid < 256 && above2 < k_rem && above2 + c2 >= k_rem) {
                misc[3] = 255u - (uint32_t)tid;
                misc[4] = above2;
                misc[5] = c2;
            }
        }
        __syncthreads();
        const uint32_t F = misc[3], k_rem2 = k_rem - misc[4], n_last = misc[5];
        const bool whole2 = n_last == k_rem2;
        if (n_last > (uint32_t)kBins1) return false;  // uniform: the general form takes it
        // ---- 5. above the last bin: selected; its members (the histogram area holds their
        // candidate slots) are ranked by (key descending, index ascending) among themselves
        uint32_t *last = hist;
        if (tid == 0) misc[9] = 0u;
        __syncthreads();
        for (uint32_t c = tid; c < m; c += NT) {
            const uint32_t key = cand_key[c];
            if ((key >> (32 - kTopkHistBits)) != B1) continue;
            const uint32_t d2 = (key >> 12) & 255u;
            if (d2 > F || (whole2 && d2 == F)) {
                const int32_t i = cand_idx[c];
                atomicOr(&selw[i >> 5], 1u << (i & 31));
            } else if (d2 == F) {
                const uint32_t slot = atomicAdd(&misc[9], 1u);
                if (slot < (uint32_t)kBins1) last[slot] = c;
            }
        }
        __syncthreads();
        if (!whole2) {
            for (uint32_t t = tid; t < n_last; t += NT) {
                const uint32_t c = last[t];
                const uint32_t key = cand_key[c];
                const int32_t i = cand_idx[c];
                uint32_t rank = 0;
                for (uint32_t u = 0; u < n_last; ++u) {
                    const uint32_t c2 = last[u];
                    const uint32_t k2 = cand_key[c2];
                    rank += (k2 > key || (k2 == key && cand_idx[c2] < i)) ? 1u : 0u;
                }
                if (rank < k_rem2) atomicOr(&selw[i >> 5], 1u << (i & 31));
            }
            __syncthreads();
        }
    }
    // ---- 6. ordered output
    write_selection(selw, nullptr, nw, 0u, k, out, pout, pvec, warp_s);
    return true;
}

// The general form for one query when n is large and no histogram comes with the scores:
// a strided sample (1024 positions over the row's capacity n_cap, the ones below n kept)
// sets a threshold T at the 12-bit digit that holds the sample's r-th largest key (r a
// margin above the k/n share); one pass keeps every key >= T
// as a candidate (the top k are among them whenever at least k are); the candidates are
// then selected exactly: first 12-bit digit, second 8-bit digit, and a (key, index) rank
// inside the last bin.  Returns false (nothing written) when the sample missed -- fewer
// than k or more than cand_cap candidates -- and the caller runs topk_query instead.
// smem: the layout of topk_query.
__device__ bool topk_query_sampled(const float *srow, int64_t n, int64_t k, int32_t *out,
                                   int32_t *pout, bool pvec, int cand_cap, uint32_t *smem,
                                   float sample, int64_t n_cap)
{
    uint32_t *hist = smem;
    uint32_t *warp_s = hist + kBins1;
    uint32_t *misc = warp_s + 2 * (NT / 32);
    uint32_t *selw = misc + 32;
    const int64_t nw = (n + 31) / 32;
    uint32_t *cand_key = selw + 2 * nw;
    int32_t *cand_idx = reinterpret_cast<int32_t *>(cand_key + cand_cap);
    const int tid = threadIdx.x;

    // ---- 1. the sample's histogram and the threshold digit.  sample: this thread's score at
    // (tid * n_cap) >> 10, loaded by the caller before the query's block count n was known;
    // the ns samples below n stand for the row (ns >= 1: thread 0 samples block 0).
    for (int i = tid; i < kBins1; i += NT) hist[i] = 0u;
    for (int64_t w = tid; w < nw; w += NT) selw[w] = 0u;
    if (tid == 0) misc[8] = 0u;
    __syncthreads();
    const bool in_row = (((int64_t)tid * n_cap) >> 10) < n;
    if (in_row) atomicAdd(&hist[score_key(sample) >> (32 - kTopkHistBits)], 1u);
    const int64_t ns = __syncthreads_count(in_row);
    int64_t r = (k * ns + n - 1) / n + 8;
    if (r > ns) r = ns;
    find_bucket(hist, kBins1, (uint32_t)r, warp_s, misc);
    const uint32_t T = misc[0] << (32 - kTopkHistBits);
    for (int i = tid; i < kBins1; i += NT) hist[i] = 0u;  // find_bucket has read it
    __syncthreads();

    // ---- 2. one pass: every key >= T is a candidate, and the candidates' first-digit
    // histogram
    auto keep = [&](uint32_t key, int64_t i) {
        if (key >= T) {
            atomicAdd(&hist[key >> (32 - kTopkHistBits)], 1u);
            const uint32_t slot = atomicAdd(&misc[8], 1u);
            if (slot < (uint32_t)cand_cap) {
                cand_key[slot] = key;
                cand_idx[slot] = (int32_t)i;
            }
        }
    };
    if (T > kKeyNegInf && (reinterpret_cast<uintptr_t>(srow) & 15) == 0)
        collect_at_least(srow, n, T, &misc[8], cand_key, cand_idx, (uint32_t)cand_cap, hist);
    else if (T > kKeyNegInf)
        for_each_key_at_least(srow, n, T, keep);
    else
        for_each_key(srow, n, keep);
    __syncthreads();
    const uint32_t m = misc[8];
    if (m < (uint32_t)k || m > (uint32_t)cand_cap) return false;  // uniform

    return select_candidates(k, m, hist, warp_s, misc, selw, nw, cand_key, cand_idx, out, pout,
                             pvec);
}

// One query of the general kernel (all threads of a 1024-thread CTA): query qi of n_q.
__device__ void topk_one(int64_t qi, int64_t n_q, const float *__restrict__ scores, int64_t ld,
                         const int32_t *__restrict__ q_pos, int64_t n_full_cap, int k_blk,
                         int32_t *__restrict__ blocks_out, int32_t *__restrict__ counts_out,
                         int64_t n_ctx, int32_t *__restrict__ pos_out,
                         int32_t *__restrict__ n_cells_out, int64_t max_cells,
                         uint32_t *__restrict__ ext_hist, int cand_cap, int64_t p_step,
                         uint32_t *smem)
{
    // the sampled form's strided sample over the row's capacity, in flight while the query's
    // position is read (samples past its own block count are dropped there)
    const float sample = (!ext_hist && n_full_cap >= kSampledMinN)
                             ? scores[qi * ld + (((int64_t)threadIdx.x * n_full_cap) >> 10)]
                             : 0.0f;

    // the query's position: q_pos[qi], else n_ctx - 1 - p_step * (n_q - 1 - qi) (the last
    // n_q tokens of the context when p_step = 1; every query at n_ctx - 1 when it is 0)
    const int64_t p = q_pos ? (int64_t)q_pos[qi] : n_ctx - 1 - p_step * (n_q - 1 - qi);
    int64_t n = n_full_cap;
    if (q_pos || p_step) {
        const int64_t p1 = (p + 1) / 4;
        n = p1 < n ? p1 : n;
    }
    if (n < 0) n = 0;
    const int64_t k = (int64_t)k_blk < n ? (int64_t)k_blk : n;
    int32_t *out = blocks_out + qi * (int64_t)k_blk;
    int32_t *pout = pos_out ? pos_out + qi * max_cells : nullptr;
    const bool pvec = (reinterpret_cast<uintptr_t>(pout) & 15) == 0;
    uint32_t *ehist = ext_hist ? ext_hist + qi * (int64_t)kBins1 : nullptr;
    write_count_tail(k, p, counts_out + qi, pout, n_cells_out ? n_cells_out + qi : nullptr);
    if (n <= k_blk) {  // every candidate is selected
        for (int64_t i = threadIdx.x; i < n; i += NT) {
            out[i] = (int32_t)i;
            if (pout) put_cells(pout + 4 * i, (int32_t)i, pvec);
        }
        if (ehist)  // leave the histogram cleared for the next step
            for (int i = threadIdx.x; i < kBins1; i += NT) ehist[i] = 0u;
        return;
    }
    if (!ehist && n >= kSampledMinN &&
        topk_query_sampled(scores + qi * ld, n, k, out, pout, pvec, cand_cap, smem, sample,
                           n_full_cap))
        return;
    topk_query(scores + qi * ld, n, k, out, pout, pvec, ehist, cand_cap, smem);
}

__global__ void __launch_bounds__(NT)
topk_kernel(const float *__restrict__ scores, int64_t ld, const int32_t *__restrict__ q_pos,
            int64_t n_full_cap, int k_blk, int32_t *__restrict__ blocks_out,
            int32_t *__restrict__ counts_out, int64_t n_ctx, int32_t *__restrict__ pos_out,
            int32_t *__restrict__ n_cells_out, int64_t max_cells, uint32_t *__restrict__ ext_hist,
            int cand_cap, int64_t p_step)
{
    extern __shared__ __align__(16) uint32_t smem[];
    pdl_wait();
    QSA_AFTER_WAIT(scores);
    QSA_AFTER_WAIT(q_pos);
    QSA_AFTER_WAIT(ext_hist);
    pdl_trigger();
    topk_one(blockIdx.x, gridDim.x, scores, ld, q_pos, n_full_cap, k_blk, blocks_out, counts_out,
             n_ctx, pos_out, n_cells_out, max_cells, ext_hist, cand_cap, p_step, smem);
}

// The queries listed in list[0 .. *count) (queries the maxima form handed back), each by the
// general kernel's logic; a persistent grid takes them in turn.
__global__ void __launch_bounds__(NT)
topk_listed_kernel(const float *__restrict__ scores, int64_t ld, const int32_t *__restrict__ q_pos,
                   int64_t n_q, int64_t n_full_cap, int k_blk, int32_t *__restrict__ blocks_out,
                   int32_t *__restrict__ counts_out, const uint32_t *__restrict__ count,
                   const int32_t *__restrict__ list, int cand_cap)
{
    extern __shared__ __align__(16) uint32_t smem[];
    pdl_wait();
    QSA_AFTER_WAIT(scores);
    QSA_AFTER_WAIT(count);
    QSA_AFTER_WAIT(list);
    pdl_trigger();
    const uint32_t cnt = *count;
    for (uint32_t j = blockIdx.x; j < cnt; j += gridDim.x) {
        topk_one(list[j], n_q, scores, ld, q_pos, n_full_cap, k_blk, blocks_out, counts_out, 0,
                 nullptr, nullptr, 0, nullptr, cand_cap, 0, smem);
        __syncthreads();  // the next query reuses the shared memory
    }
}

// Byte offset of a pointer (the per-query copies of the decode top-k's scratch).
template <typename P>
__device__ __forceinline__ P *byte_shift(P *p, int64_t bytes)
{
    return reinterpret_cast<P *>(reinterpret_cast<char *>(p) + bytes);
}

// The decode form (n > k for every query): see the file comment.  Grid ceil(n_full / 1024)
// x n_q CTAs of 1024 threads; CTA (c, i) classifies blocks [1024c, 1024c + 1024) of query
// i, the query at position p_i = n_ctx - n_q + i, whose candidates are the blocks
// b < n_i = min(n_full, floor((p_i+1)/4)).  hist: the score kernel's histograms of those
// blocks (2^kTopkHistBits words per query); ticket: set to 0 by the score kernel of this
// step.  Scratch per query (query i's at byte offset i * q_stride): bitmap [ceil(n/32)]
// words, cand [grid.x][1024] (key, block), cand_cnt [grid.x].
// BPT blocks per thread: CTA c classifies blocks [c * 1024 * BPT, (c + 1) * 1024 * BPT).
template <int BPT>
__global__ void __launch_bounds__(NT)
topk_select_kernel(const float *__restrict__ scores, int64_t ld_scores, int n_q, int64_t n_full,
                   int k_blk, int64_t n_ctx, uint32_t *__restrict__ hist,
                   uint32_t *__restrict__ ticket, uint32_t *__restrict__ bitmap,
                   uint2 *__restrict__ cand, int32_t *__restrict__ cand_cnt, int64_t q_stride,
                   int32_t *__restrict__ blocks_out, int32_t *__restrict__ counts_out,
                   int32_t *__restrict__ pos_out, int32_t *__restrict__ n_cells_out,
                   int64_t max_cells, int cand_cap)
{
    extern __shared__ __align__(16) uint32_t smem[];
    __shared__ uint32_t wtot[NT / 32];
    __shared__ uint32_t sh[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) sh[6] = 0u;  // this CTA's candidate count
    pdl_wait();
    QSA_AFTER_WAIT(scores);
    QSA_AFTER_WAIT(hist);
    QSA_AFTER_WAIT(ticket);
    QSA_AFTER_WAIT(bitmap);
    QSA_AFTER_WAIT(cand);
    QSA_AFTER_WAIT(cand_cnt);
    pdl_trigger();

    // this CTA's query
    const int qi = (int)blockIdx.y;
    const int64_t p_q = n_ctx - n_q + qi;
    const int64_t n = (p_q + 1) / 4 < n_full ? (p_q + 1) / 4 : n_full;
    scores += qi * ld_scores;
    hist += (int64_t)qi << kTopkHistBits;
    ticket = byte_shift(ticket, qi * q_stride);
    bitmap = byte_shift(bitmap, qi * q_stride);
    cand = byte_shift(cand, qi * q_stride);
    cand_cnt = byte_shift(cand_cnt, qi * q_stride);
    blocks_out += (int64_t)qi * k_blk;
    counts_out += qi;
    if (pos_out) pos_out += qi * max_cells;
    if (n_cells_out) n_cells_out += qi;

    const int64_t k = k_blk;
    const int64_t nw = (n + 31) / 32;
    constexpr int kSpan = NT * BPT;  // blocks of one CTA
    const int64_t i0 = (int64_t)blockIdx.x * kSpan + tid;  // this thread's blocks: i0 + j*NT
    float sv[BPT];
#pragma unroll
    for (int j = 0; j < BPT; ++j) sv[j] = i0 + j * NT < n ? scores[i0 + j * NT] : 0.0f;
    // ---- threshold bucket, two-level: thread t holds bins 4095-4t .. 4092-4t (top first)
    uint32_t c[4], mine = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        c[j] = hist[kBins1 - 1 - 4 * tid - j];
        mine += c[j];
    }
    uint32_t inc = mine;  // inclusive scan within the warp, top bins first
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) wtot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const uint32_t w = wtot[lane];
        uint32_t winc = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, winc, o);
            if (lane >= o) winc += y;
        }
        const uint32_t ball = __ballot_sync(0xffffffffu, winc >= (uint32_t)k);
        const int wl = ball ? __ffs(ball) - 1 : 0;
        const uint32_t before = __shfl_sync(0xffffffffu, winc - w, wl);
        const uint32_t total = __shfl_sync(0xffffffffu, winc, 31);
        if (lane == 0) {
            sh[0] = (total == (uint32_t)n && ball != 0u) ? 1u : 0u;  // the histogram is usable
            sh[1] = (uint32_t)wl;
            sh[2] = before;
        }
    }
    __syncthreads();
    const bool valid = sh[0] != 0u;
    if (valid && warp == (int)sh[1]) {
        uint32_t above = sh[2] + inc - mine;  // keys in the bins above this thread's
        if (above < (uint32_t)k && above + mine >= (uint32_t)k) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (above + c[j] >= (uint32_t)k) {
                    sh[3] = (uint32_t)(kBins1 - 1 - 4 * tid - j);
                    sh[4] = above;
                    sh[5] = c[j];
                    break;
                }
                above += c[j];
            }
        }
    }
    __syncthreads();
    const uint32_t B1 = sh[3], above_n = sh[4];
    const uint32_t k_rem = (uint32_t)k - above_n;
    const bool whole = valid && sh[5] == k_rem;

    // ---- classify this CTA's blocks
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
        const int64_t i = i0 + j * NT;
        const uint32_t key = score_key(sv[j]);
        const uint32_t dg = key >> (32 - kTopkHistBits);
        const bool in = valid && i < n;
        const bool above = in && (dg > B1 || (whole && dg == B1));
        const bool is_cand = in && !whole && dg == B1;
        const uint32_t word = __ballot_sync(0xffffffffu, above);
        const int64_t wi = (int64_t)blockIdx.x * (kSpan / 32) + j * (NT / 32) + warp;
        if (lane == 0 && wi < nw) bitmap[wi] = word;
        const uint32_t cm = __ballot_sync(0xffffffffu, is_cand);
        uint32_t base = 0;
        if (lane == 0 && cm) base = atomicAdd(&sh[6], (uint32_t)__popc(cm));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (is_cand)
            cand[(int64_t)blockIdx.x * kSpan + base + __popc(cm & ((1u << lane) - 1u))] =
                make_uint2(key, (uint32_t)i);
    }
    // Arrival: the barrier orders this CTA's writes before thread 0's ticket, an
    // acquire-release atomic at device scope: it publishes them, and the last arrival
    // acquires everything the others published (the grid-barrier pattern, without the wait).
    __syncthreads();
    if (tid == 0) {
        cand_cnt[blockIdx.x] = (int32_t)sh[6];
        uint32_t old;
        asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                     : "=r"(old)
                     : "l"(ticket)
                     : "memory");
        sh[7] = old == gridDim.x - 1 ? 1u : 0u;
    }
    __syncthreads();
    if (!sh[7]) return;

    // ---- the last CTA: every other CTA's bitmap words and candidates are visible
    int32_t *pout = pos_out;
    const bool pvec = (reinterpret_cast<uintptr_t>(pout) & 15) == 0;
    write_count_tail(k, p_q, counts_out, pout, n_cells_out);
    // the general form's layout, its histogram area holding the candidates and the lists
    // cp [1024]: candidates packed as key << 32 | ~block, so that one unsigned comparison
    // orders them by key descending, then block ascending
    unsigned long long *cp = reinterpret_cast<unsigned long long *>(smem);
    uint32_t *lo = smem + 2 * NT;                               // [grid] list offsets
    uint32_t *lc = smem + 3 * NT;                               // [grid] list lengths
    uint32_t *warp_s = smem + kBins1;
    uint32_t *selw = warp_s + 2 * (NT / 32) + 32;
    uint32_t n_cand = 0;
    if (valid) {
        const int G = (int)gridDim.x;
        const uint32_t my = tid < G ? (uint32_t)__ldcg(cand_cnt + tid) : 0u;
        // Lists warp and warp + 32 (all of them when the grid has at most 64 CTAs): their
        // first 32 entries are read together with the counts, before the offsets exist.
        constexpr int kSpec = 2;
        uint2 spec[kSpec];
#pragma unroll
        for (int r = 0; r < kSpec; ++r) {
            const int cta = warp + 32 * r;
            spec[r] = cta < G ? __ldcg(cand + (int64_t)cta * kSpan + lane) : make_uint2(0u, 0u);
        }
        for (int64_t w = tid; w < nw; w += NT) selw[w] = __ldcg(bitmap + w);
        const uint32_t off = block_excl_scan(my, warp_s, &n_cand);
        if (tid < G) {
            lo[tid] = off;
            lc[tid] = my;
        }
        __syncthreads();
        if (n_cand <= (uint32_t)NT) {
#pragma unroll
            for (int r = 0; r < kSpec; ++r) {
                const int cta = warp + 32 * r;
                if (cta < G && (uint32_t)lane < lc[cta])
                    cp[lo[cta] + lane] = ((unsigned long long)spec[r].x << 32) | (uint32_t)~spec[r].y;
            }
            for (int cta = warp; cta < G; cta += NT / 32) {
                const uint32_t j0 = cta < 32 * kSpec ? 32u : 0u;  // entries already placed
                for (uint32_t j = j0 + lane; j < lc[cta]; j += 32) {
                    const uint2 e = __ldcg(cand + (int64_t)cta * kSpan + j);
                    cp[lo[cta] + j] = ((unsigned long long)e.x << 32) | (uint32_t)~e.y;
                }
            }
            __syncthreads();
            // Second digit (key bits 12-19) over the candidates: a 256-bin histogram, then
            // the bin holding the k_rem-th; candidates above it are in, the ones inside it
            // (few) are ranked against each other by (key, index).
            uint32_t *h2 = lo;                                     // [256]
            uint32_t *sub = lc;                                    // [n_cand] indices into cp
            if (tid < 256) h2[tid] = 0u;
            if (tid == 0) sh[5] = 0u;
            __syncthreads();
            if ((uint32_t)tid < n_cand) atomicAdd(&h2[(uint32_t)(cp[tid] >> 44) & 255u], 1u);
            __syncthreads();
            {
                const uint32_t c2n = tid < 256 ? h2[255 - tid] : 0u;  // top bin first
                uint32_t tot;
                const uint32_t above2 = block_excl_scan(c2n, warp_s, &tot);
                if (tid < 256 && above2 < k_rem && above2 + c2n >= k_rem) {
                    sh[0] = 255u - (uint32_t)tid;
                    sh[1] = above2;
                    sh[2] = c2n;
                }
            }
            __syncthreads();
            const uint32_t F = sh[0], k_rem2 = k_rem - sh[1];
            const bool whole2 = sh[2] == k_rem2;
            if ((uint32_t)tid < n_cand) {
                const unsigned long long v = cp[tid];
                const uint32_t d2 = (uint32_t)(v >> 44) & 255u, it = ~(uint32_t)v;
                if (d2 > F || (whole2 && d2 == F)) atomicOr(&selw[it >> 5], 1u << (it & 31));
                else if (d2 == F) sub[atomicAdd(&sh[5], 1u)] = (uint32_t)tid;
            }
            __syncthreads();
            if (!whole2) {
                const uint32_t m = sh[5];
                if ((uint32_t)tid < m) {
                    const unsigned long long v = cp[sub[tid]];
                    uint32_t r = 0;
                    for (uint32_t j = 0; j < m; ++j) r += cp[sub[j]] > v ? 1u : 0u;
                    if (r < k_rem2) {
                        const uint32_t it = ~(uint32_t)v;
                        atomicOr(&selw[it >> 5], 1u << (it & 31));
                    }
                }
                __syncthreads();
            }
            write_selection(selw, nullptr, nw, 0u, k, blocks_out, pout, pvec, warp_s);
            for (int j = tid; j < kBins1; j += NT) hist[j] = 0u;  // cleared for the next step
            return;
        }
        __syncthreads();
    }
    // unusable histogram or an oversized bucket: the general form (clears the histogram)
    topk_query(scores, n, k, blocks_out, pout, pvec, hist, cand_cap, smem);
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

cudaError_t set_max_smem()
{
    cudaError_t e = ensure_kernel_attrs<topk_kernel>(kMaxSmemBytes);
    if (e == cudaSuccess) e = ensure_kernel_attrs<topk_select_kernel<1>>(kMaxSmemBytes);
    if (e == cudaSuccess) e = ensure_kernel_attrs<topk_select_kernel<2>>(kMaxSmemBytes);
    return e;
}

}  // namespace

int64_t topk_max_candidates() { return kMaxN; }

// CTA slots of the decode top-k's scratch: enough for one or two blocks per thread.
static int64_t select_slots(int64_t n) { return 2 * ((n + 2 * NT - 1) / (2 * NT)); }

size_t topk_select_workspace_bytes(int64_t n_full_cap)
{
    const int64_t nw = (n_full_cap + 31) / 32;
    const int64_t g = select_slots(n_full_cap);
    // ticket (256 B) | counts | candidates | bitmap, each 256-byte aligned
    auto al = [](int64_t b) { return (b + 255) & ~(int64_t)255; };
    return (size_t)(256 + al(4 * g) + al(8 * g * NT) + al(4 * nw));
}

cudaError_t launch_topk_select(const float *scores, int64_t ld_scores, int n_q, int64_t n_full,
                               int64_t n_full_cap, int64_t k_blk, int64_t n_ctx, uint32_t *hist,
                               void *scratch, int32_t *blocks_out, int32_t *counts_out,
                               int32_t *pos_out, int32_t *n_cells_out, int64_t max_cells,
                               cudaStream_t st)
{
    // the first query has the fewest candidates
    const int64_t p0 = n_ctx - n_q;
    const int64_t n_min = (p0 + 1) / 4 < n_full ? (p0 + 1) / 4 : n_full;
    if (n_q < 1 || n_q > 65535 || n_min <= k_blk || n_full > kMaxN || n_full > n_full_cap)
        return cudaErrorNotSupported;
    const int64_t nw = (n_full + 31) / 32;
    const int64_t g = select_slots(n_full);
    auto al = [](int64_t b) { return (b + 255) & ~(int64_t)255; };
    char *b = static_cast<char *>(scratch);
    uint32_t *ticket = reinterpret_cast<uint32_t *>(b);
    int32_t *cand_cnt = reinterpret_cast<int32_t *>(b + 256);
    uint2 *cand = reinterpret_cast<uint2 *>(b + 256 + al(4 * g));
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(b + 256 + al(4 * g) + al(8 * g * NT));
    // Shared memory for the fast path and the general form without a candidate list (it
    // re-reads the scores instead): every CTA of the grid carries this allocation, and a
    // large one would shrink the L1 of SMs still running the score kernel.
    const int cand_cap = 0;
    const size_t smem = sizeof(uint32_t) * (size_t)(kFixedWords + 2 * nw);
    cudaError_t e = set_max_smem();
    if (e != cudaSuccess) return e;
    const int64_t q_stride = (int64_t)topk_select_workspace_bytes(n_full_cap);
    // One CTA per SM (registers): when the queries' CTAs would need a second wave, each
    // CTA takes two blocks per thread.
    const int64_t g1 = (n_full + NT - 1) / NT;
    if (n_q * g1 > device_sm_count()) {
        const int64_t g2 = (n_full + 2 * NT - 1) / (2 * NT);
        return launch(topk_select_kernel<2>, dim3((unsigned)g2, (unsigned)n_q), dim3(NT), smem,
                      st, 1, scores, ld_scores, n_q, n_full, (int)k_blk, n_ctx, hist, ticket,
                      bitmap, cand, cand_cnt, q_stride, blocks_out, counts_out, pos_out,
                      n_cells_out, max_cells, cand_cap);
    }
    return launch(topk_select_kernel<1>, dim3((unsigned)g1, (unsigned)n_q), dim3(NT), smem, st, 1,
                  scores, ld_scores, n_q, n_full, (int)k_blk, n_ctx, hist, ticket, bitmap, cand,
                  cand_cnt, q_stride, blocks_out, counts_out, pos_out, n_cells_out, max_cells,
                  cand_cap);
}

uint32_t *topk_select_ticket(void *scratch) { return static_cast<uint32_t *>(scratch); }

cudaError_t launch_topk(const float *scores, int64_t n_q, int64_t ld, const int32_t *q_pos,
                        int64_t n_full, int64_t k_blk, int32_t *blocks_out, int32_t *counts_out,
                        int64_t n_ctx, int32_t *pos_out, int32_t *n_cells_out,
                        int64_t max_cells, uint32_t *ext_hist, cudaStream_t st, int64_t p_step)
{
    if (n_q == 0) return cudaSuccess;
    int cand_cap = 0;
    const size_t smem = topk_smem_bytes(n_full, &cand_cap);
    cudaError_t e = set_max_smem();
    if (e != cudaSuccess) return e;
    return launch(topk_kernel, dim3((unsigned)n_q), dim3(NT), smem, st, 1, scores, ld, q_pos,
                  n_full, (int)k_blk, blocks_out, counts_out, n_ctx, pos_out, n_cells_out,
                  max_cells, ext_hist, cand_cap, p_step);
}

cudaError_t launch_topk_listed(const float *scores, int64_t n_q, int64_t ld, const int32_t *q_pos,
                               int64_t n_full, int64_t k_blk, int32_t *blocks_out,
                               int32_t *counts_out, const uint32_t *count, const int32_t *list,
                               cudaStream_t st)
{
    if (n_q == 0) return cudaSuccess;
    int cand_cap = 0;
    const size_t smem = topk_smem_bytes(n_full, &cand_cap);
    cudaError_t e = set_max_smem();
    if (e == cudaSuccess) e = ensure_kernel_attrs<topk_listed_kernel>(kMaxSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t grid = n_q < device_sm_count() ? n_q : device_sm_count();
    return launch(topk_listed_kernel, dim3((unsigned)grid), dim3(NT), smem, st, 1, scores, ld,
                  q_pos, n_q, n_full, (int)k_blk, blocks_out, counts_out, count, list, cand_cap);
}

}  // namespace qsa
