// topk_maxima.cu -- block-domain top-k of a prefill chunk fed by the score kernel's group
// maxima: maxima[i][g] is the largest score of blocks 32g .. 32g + 31 of query i (written by
// the tensor-core score kernel's epilogue).
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "block-domain top-k (COMMON-006)" (the top-k runs over block scores; ties to the lower
// block index as in qsa_topk_blocks) and section "QSA and the QSA indexer" (indexer_top_k =
// 2048 tokens = 512 blocks).  The pages do not say how a chunk's top-k is fed; here the
// contraction's epilogue summarises each 32-block group by its maximum, and the top-k takes
// its threshold from those maxima.
//
// Why a second kernel: the general top-k keeps one 1024-thread CTA (and up to 220 KB of
// candidate lists) per query, so each SM works one query at a time through a chain of
// dependent phases.  With the maxima the threshold is tight (a few hundred candidates beyond
// k), so a query needs 256 threads and ~40 KB, and four queries share an SM.
//
// Per query (one 256-thread CTA), with the n candidates b < n and G = n / 32 groups that
// hold only candidates:
//   1. the groups' keys (score_key of their maxima, at most 16 per thread): the k-th largest
//      lies in a 12-bit first-digit bin, then an 8-bit second-digit bin; T = that 20-bit
//      prefix.  At least k groups have key >= T, each at a candidate, so at least k
//      candidates have key >= T;
//   2. one pass reads only the groups whose maximum reaches T (32 groups per round per warp,
//      eight 16-byte loads in flight per lane) and the partial last group, keeping every
//      candidate with key >= T and their first-digit histogram;
//   3. the exact top k of those: first 12-bit digit, second 8-bit digit, (key, index) rank
//      inside the last bin, ordered output from a bitmap.
// A query it cannot settle -- fewer than k groups, T at -inf, more candidates than its
// lists hold, maxima that do not match the scores -- is appended to a list that the general
// kernel (topk.cu) then takes, so every query gets the same selection as qsa_topk_blocks.
#include "prefill_select.cuh"

namespace qsa {
namespace {

constexpr int MT = 256;                          // threads per query
constexpr int kMWarps = MT / 32;
constexpr int kMPer = 16;                        // group keys per thread
constexpr int64_t kMMaxN = (int64_t)MT * kMPer * 32;  // 131,072 candidate blocks
constexpr int kMCap = 2048;                      // candidates kept
constexpr int kMBins = 1 << kTopkHistBits;       // 4096
constexpr uint32_t kNegInfKey = 0x007fffffu;     // score_key(-inf), also that of NaN

// The float whose key is T (T above the key of -inf): score_key(x) >= T exactly when
// x >= key_float(T) as floats; a NaN x compares false.
__device__ __forceinline__ float key_float_m(uint32_t T)
{
    return __uint_as_float((T & 0x80000000u) ? (T & 0x7fffffffu) : ~T);
}

// Exclusive prefix sum over the CTA; *total gets the CTA's total.
__device__ __forceinline__ uint32_t scan_m(uint32_t v, uint32_t *warp_s, uint32_t *total)
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
        uint32_t w = lane < kMWarps ? warp_s[lane] : 0u;
#pragma unroll
        for (int o = 1; o < kMWarps; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kMWarps) warp_s[lane] = w;
    }
    __syncthreads();
    const uint32_t r = (warp == 0 ? 0u : warp_s[warp - 1]) + x - v;
    *total = warp_s[kMWarps - 1];
    __syncthreads();
    return r;
}

// Bin of h[0 .. nb) (nb = 4096 or 256, scanned from the top) holding the k_rem-th largest;
// misc[0] bin, misc[1] entries in higher bins, misc[2] entries in the bin.
template <int NB>
__device__ __forceinline__ void bucket_m(const uint32_t *h, uint32_t k_rem, uint32_t *warp_s,
                                         uint32_t *misc)
{
    constexpr int per = NB / MT;  // 16 or 1
    uint32_t cnt[per];
    uint32_t mine = 0;
#pragma unroll
    for (int j = 0; j < per; ++j) {
        cnt[j] = h[NB - 1 - threadIdx.x * per - j];
        mine += cnt[j];
    }
    uint32_t tot;
    uint32_t above = scan_m(mine, warp_s, &tot);
#pragma unroll
    for (int j = 0; j < per; ++j) {
        if (above < k_rem && above + cnt[j] >= k_rem) {
            misc[0] = (uint32_t)(NB - 1 - threadIdx.x * per - j);
            misc[1] = above;
            misc[2] = cnt[j];
        }
        above += cnt[j];
    }
    __syncthreads();
}

__global__ void __launch_bounds__(MT, 4)
topk_maxima_kernel(const float *__restrict__ scores, int64_t ld, const int32_t *__restrict__ q_pos,
                   int64_t n_full, int k_blk, const float *__restrict__ maxima, int64_t ld_max,
                   int32_t *__restrict__ blocks_out, int32_t *__restrict__ counts_out,
                   uint32_t *__restrict__ fb_count, int32_t *__restrict__ fb_list)
{
    extern __shared__ __align__(16) uint32_t sm[];
    pdl_wait();
    QSA_AFTER_WAIT(scores);
    QSA_AFTER_WAIT(q_pos);
    QSA_AFTER_WAIT(maxima);
    QSA_AFTER_WAIT(fb_count);
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t qi = blockIdx.x;
    int64_t n = n_full;
    if (q_pos) {
        const int64_t p1 = ((int64_t)q_pos[qi] + 1) / 4;
        n = p1 < n ? p1 : n;
    }
    if (n < 0) n = 0;
    const int64_t k = (int64_t)k_blk < n ? (int64_t)k_blk : n;
    int32_t *out = blocks_out + qi * (int64_t)k_blk;
    if (tid == 0) counts_out[qi] = (int32_t)k;
    if (n <= k_blk) {  // every candidate is selected
        for (int64_t i = tid; i < n; i += MT) out[i] = (int32_t)i;
        return;
    }
    auto hand_back = [&]() {  // the general kernel takes this query
        if (tid == 0) fb_list[atomicAdd(fb_count, 1u)] = (int32_t)qi;
    };
    const int64_t G = n / 32;
    if (G < k || n > kMMaxN) {  // uniform
        hand_back();
        return;
    }
    const int ng = (int)G;
    const int nw = (int)((n + 31) / 32);
    uint32_t *hist = sm;                          // [4096]
    uint32_t *warp_s = hist + kMBins;             // [2 * warps]
    uint32_t *misc = warp_s + 2 * kMWarps;        // [32]
    uint32_t *selw = misc + 32;                   // [nw] the pass's group list, then the
                                                  // selected-block bitmap
    uint32_t *cand_key = selw + nw;               // [kMCap]
    int32_t *cand_idx = reinterpret_cast<int32_t *>(cand_key + kMCap);
    const float *srow = scores + qi * ld;
    const float *gm = maxima + qi * ld_max;

    // ---- 1. the groups' keys: thread t holds groups t + u * MT (warp w: the 32 groups
    // u * MT + 32w .. of each round u)
    const int n_u = (ng + MT - 1) / MT;  // <= kMPer
    uint32_t gk[kMPer];
#pragma unroll
    for (int u = 0; u < kMPer; ++u) {
        const int g = tid + u * MT;
        gk[u] = (u < n_u && g < ng) ? score_key(gm[g]) : 0u;  // 0: below every key
    }
    for (int i = tid; i < kMBins; i += MT) hist[i] = 0u;
    if (tid < 32) misc[tid] = 0u;
    __syncthreads();
    // one shared atomic per distinct bin of a warp (the maxima crowd a few bins)
    auto add_bin = [&](bool take, uint32_t bin) {
        const uint32_t same = __match_any_sync(0xffffffffu, take ? bin : 0xffffffffu);
        if (take && (same & ((1u << lane) - 1u)) == 0)
            atomicAdd(&hist[bin], (uint32_t)__popc(same));
    };
#pragma unroll
    for (int u = 0; u < kMPer; ++u)
        if (u < n_u) add_bin(gk[u] != 0u, gk[u] >> (32 - kTopkHistBits));
    __syncthreads();
    bucket_m<kMBins>(hist, (uint32_t)k, warp_s, misc);
    const uint32_t B1 = misc[0];
    const uint32_t k2 = (uint32_t)k - misc[1];
    if (tid < 256) hist[tid] = 0u;
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kMPer; ++u)
        if (u < n_u)
            add_bin(gk[u] != 0u && (gk[u] >> (32 - kTopkHistBits)) == B1, (gk[u] >> 12) & 255u);
    __syncthreads();
    bucket_m<256>(hist, k2, warp_s, misc);
    const uint32_t T = (B1 << (32 - kTopkHistBits)) | (misc[0] << 12);
    if (T <= kNegInfKey) {  // uniform: the k-th largest maximum is -inf or NaN
        hand_back();
        return;
    }
    for (int i = tid; i < kMBins; i += MT) hist[i] = 0u;
    __syncthreads();

    // ---- 2. the pass: every candidate with key >= T, and their first-digit histogram.
    // The groups whose maximum reaches T are listed first (at most G <= nw entries, in the
    // bitmap's area), then each warp reads 32 listed groups a round: lane / 8 picks one of
    // four groups per 16-byte load, lane % 8 its 16 bytes, eight loads in flight per lane.
    const float lo = key_float_m(T);
    uint32_t *glist = selw;
#pragma unroll
    for (int u = 0; u < kMPer; ++u) {
        if (u >= n_u) break;  // uniform
        const bool take = gk[u] >= T;  // 0 keys fail
        const uint32_t b = __ballot_sync(0xffffffffu, take);
        uint32_t base = 0;
        if (lane == 0 && b) base = atomicAdd(&misc[10], (uint32_t)__popc(b));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (take) glist[base + __popc(b & ((1u << lane) - 1u))] = (uint32_t)(tid + u * MT);
    }
    __syncthreads();
    const uint32_t n_list = misc[10];
    const bool vec = ((reinterpret_cast<uintptr_t>(srow)) & 15) == 0;
    for (uint32_t r0 = 32 * (uint32_t)warp; r0 < n_list; r0 += 32 * kMWarps) {  // warp-uniform
        float4 v[8];
        int g_of[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t idx = r0 + 4 * j + (lane >> 3);
            const int g = idx < n_list ? (int)glist[idx] : -1;
            g_of[j] = g;
            const float *src = srow + 32 * (int64_t)(g < 0 ? 0 : g) + 4 * (lane & 7);
            if (g < 0)
                v[j] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            else if (vec)
                v[j] = *reinterpret_cast<const float4 *>(src);
            else
                v[j] = make_float4(src[0], src[1], src[2], src[3]);
        }
        uint32_t hit = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            hit |= ((uint32_t)(v[j].x >= lo) | ((uint32_t)(v[j].y >= lo) << 1) |
                    ((uint32_t)(v[j].z >= lo) << 2) | ((uint32_t)(v[j].w >= lo) << 3)) << (4 * j);
        const uint32_t c = __popc(hit);
        uint32_t inc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        const uint32_t tot = __shfl_sync(0xffffffffu, inc, 31);
        uint32_t s = 0;
        if (lane == 31 && tot) s = atomicAdd(&misc[8], tot);
        s = __shfl_sync(0xffffffffu, s, 31) + inc - c;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t h4 = (hit >> (4 * j)) & 15u;
            if (!h4) continue;
            const float e4[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (!((h4 >> e) & 1u)) continue;
                const uint32_t key = score_key(e4[e]);
                atomicAdd(&hist[key >> (32 - kTopkHistBits)], 1u);
                if (s < (uint32_t)kMCap) {
                    cand_key[s] = key;
                    cand_idx[s] = 32 * g_of[j] + 4 * (lane & 7) + e;
                }
                ++s;
            }
        }
    }
    if (warp == kMWarps - 1 && 32 * G < n) {  // the partial group: blocks 32G .. n - 1
        const int64_t b = 32 * G + lane;
        const float x = b < n ? srow[b] : -INFINITY;
        const bool take = x >= lo;
        const uint32_t bl = __ballot_sync(0xffffffffu, take);
        uint32_t base = 0;
        if (lane == 0 && bl) base = atomicAdd(&misc[8], (uint32_t)__popc(bl));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (take) {
            const uint32_t key = score_key(x);
            atomicAdd(&hist[key >> (32 - kTopkHistBits)], 1u);
            const uint32_t slot = base + __popc(bl & ((1u << lane) - 1u));
            if (slot < (uint32_t)kMCap) {
                cand_key[slot] = key;
                cand_idx[slot] = (int32_t)b;
            }
        }
    }
    __syncthreads();
    const uint32_t m = misc[8];
    if (m < (uint32_t)k || m > (uint32_t)kMCap) {  // uniform
        hand_back();
        return;
    }
    for (int w = tid; w < nw; w += MT) selw[w] = 0u;  // the list's area becomes the bitmap
    __syncthreads();

    // ---- 3. the exact top k of the m candidates: first digit (histogram from the pass)
    bucket_m<kMBins>(hist, (uint32_t)k, warp_s, misc);
    const uint32_t C1 = misc[0];
    const uint32_t k_rem = (uint32_t)k - misc[1];
    const bool whole1 = misc[2] == k_rem;
    if (tid < 256) hist[tid] = 0u;
    __syncthreads();
    for (uint32_t c = tid; c < m; c += MT) {
        const uint32_t key = cand_key[c];
        const uint32_t d1 = key >> (32 - kTopkHistBits);
        if (d1 > C1 || (whole1 && d1 == C1)) {
            const int32_t i = cand_idx[c];
            atomicOr(&selw[i >> 5], 1u << (i & 31));
        } else if (d1 == C1) {
            atomicAdd(&hist[(key >> 12) & 255u], 1u);
        }
    }
    __syncthreads();
    if (!whole1) {
        bucket_m<256>(hist, k_rem, warp_s, misc);
        const uint32_t F = misc[0], k_rem2 = k_rem - misc[1], n_last = misc[2];
        const bool whole2 = n_last == k_rem2;
        // above the last bin: selected; its members (slots in the histogram area, n_last <=
        // m <= kMCap < 4096) ranked by (key descending, index ascending) among themselves
        uint32_t *last = hist;
        if (tid == 0) misc[9] = 0u;
        __syncthreads();
        for (uint32_t c = tid; c < m; c += MT) {
            const uint32_t key = cand_key[c];
            if ((key >> (32 - kTopkHistBits)) != C1) continue;
            const uint32_t d2 = (key >> 12) & 255u;
            if (d2 > F || (whole2 && d2 == F)) {
                const int32_t i = cand_idx[c];
                atomicOr(&selw[i >> 5], 1u << (i & 31));
            } else if (d2 == F) {
                last[atomicAdd(&misc[9], 1u)] = c;
            }
        }
        __syncthreads();
        if (!whole2) {
            for (uint32_t t = tid; t < n_last; t += MT) {
                const uint32_t c = last[t];
                const uint32_t key = cand_key[c];
                const int32_t i = cand_idx[c];
                uint32_t rank = 0;
                for (uint32_t u = 0; u < n_last; ++u) {
                    const uint32_t c2 = last[u];
                    const uint32_t k2b = cand_key[c2];
                    rank += (k2b > key || (k2b == key && cand_idx[c2] < i)) ? 1u : 0u;
                }
                if (rank < k_rem2) atomicOr(&selw[i >> 5], 1u << (i & 31));
            }
            __syncthreads();
        }
    }
    // ---- ordered output: each thread a run of bitmap words
    const int wpt = (nw + MT - 1) / MT;
    const int w0 = tid * wpt, w1 = w0 + wpt < nw ? w0 + wpt : nw;
    uint32_t n_sel = 0;
    for (int w = w0; w < w1; ++w) n_sel += __popc(selw[w]);
    uint32_t tot;
    uint32_t o = scan_m(n_sel, warp_s, &tot);
    for (int w = w0; w < w1; ++w) {
        uint32_t f = selw[w];
        while (f) {
            const int b = __ffs(f) - 1;
            f &= f - 1;
            if (o < (uint32_t)k) out[o] = 32 * w + b;
            ++o;
        }
    }
}

}  // namespace

size_t topk_maxima_workspace_bytes(int64_t n_q)
{
    return n_q <= 0 ? 0 : 256 + (((size_t)n_q * 4 + 255) & ~(size_t)255);
}

cudaError_t launch_topk_maxima(const float *scores, int64_t n_q, int64_t ld, const int32_t *q_pos,
                               int64_t n_full, int64_t k_blk, const float *maxima,
                               int64_t ld_maxima, int32_t *blocks_out, int32_t *counts_out,
                               void *workspace, cudaStream_t st)
{
    if (n_q == 0) return cudaSuccess;
    if (n_full > kMMaxN || n_q > 0x7fffffffLL)  // the general kernel for every query
        return launch_topk(scores, n_q, ld, q_pos, n_full, k_blk, blocks_out, counts_out, 0,
                           nullptr, nullptr, 0, nullptr, st, 0);
    uint32_t *count = static_cast<uint32_t *>(workspace);
    int32_t *list = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + 256);
    cudaError_t e = cudaMemsetAsync(count, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    const int64_t nw = (n_full + 31) / 32;
    const size_t smem = sizeof(uint32_t) * (size_t)(kMBins + 2 * kMWarps + 32 + nw + 2 * kMCap);
    e = ensure_kernel_attrs<topk_maxima_kernel>(smem);
    if (e != cudaSuccess) return e;
    e = launch(topk_maxima_kernel, dim3((unsigned)n_q), dim3(MT), smem, st, 1, scores, ld, q_pos,
               n_full, (int)k_blk, maxima, ld_maxima, blocks_out, counts_out, count, list);
    if (e != cudaSuccess) return e;
    return launch_topk_listed(scores, n_q, ld, q_pos, n_full, k_blk, blocks_out, counts_out,
                              count, list, st);
}

}  // namespace qsa
