// topk.cu -- block-domain top-k by cluster-wide radix select.
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "block-domain top-k (COMMON-006)": select over the block scores instead of expanding
// every block score to its cells first (the expansion cost grew with context:
// 0.45 -> 0.91 ms per layer from 128k to 256k on the pages' GPU).
//
// One thread-block cluster of 8 CTAs per query.  Each CTA keeps 1/8 of the candidates
// (contiguous block indices) as order-preserving 32-bit keys in shared memory.  Three
// radix passes (11 + 11 + 10 bits) find the k-th largest key T: every CTA histograms its
// slice, the histograms are summed across the cluster through distributed shared memory,
// and every CTA picks the same bucket.  The final pass keeps keys > T and the first
// (lowest-index) keys == T until k are taken, writing them in ascending block order from
// a cluster-wide exclusive scan of per-thread counts.  No grid-wide synchronisation and no
// global scratch: cluster barriers are hardware barriers.
#include <cooperative_groups.h>

#include "qsa_internal.cuh"

namespace cg = cooperative_groups;

namespace qsa {
namespace {

constexpr int CL = kTopkCluster;
constexpr int NT = kTopkThreads;
constexpr int kBins = 2048;
constexpr int kSmemFixedWords = 2 * kBins + 64 + 2 * NT;
constexpr int kMaxSmemBytes = 220 * 1024;
constexpr int64_t kMaxSlice = (kMaxSmemBytes / 4) - kSmemFixedWords;

// Higher score <=> larger key.  NaN ranks as -inf; -0 and +0 are the same score.
__device__ __forceinline__ uint32_t score_key(float s)
{
    uint32_t u = __float_as_uint(s);
    if ((u & 0x7fffffffu) > 0x7f800000u) u = 0xff800000u;  // NaN -> -inf
    if (u == 0x80000000u) u = 0u;                           // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the block (NT threads); returns the total in *total.
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
        if (lane < NT / 32) warp_s[lane] = w;  // inclusive per-warp totals
    }
    __syncthreads();
    const uint32_t warp_before = warp == 0 ? 0u : warp_s[warp - 1];
    *total = warp_s[NT / 32 - 1];
    const uint32_t r = warp_before + x - v;
    __syncthreads();  // warp_s is reused by the caller's next scan
    return r;
}

__global__ void __launch_bounds__(NT)
topk_cluster_kernel(const float *__restrict__ scores, int64_t ld, const int32_t *__restrict__ q_pos,
                    int64_t n_full_cap, int k_blk, int32_t *__restrict__ blocks_out,
                    int32_t *__restrict__ counts_out)
{
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int64_t qi = blockIdx.x / CL;

    extern __shared__ uint32_t smem[];
    uint32_t *hist = smem;              // [kBins] this CTA's histogram
    uint32_t *ghist = hist + kBins;     // [kBins] cluster-summed histogram
    uint32_t *misc = ghist + kBins;     // [64] bucket choice, CTA totals
    uint32_t *warp_s = misc + 64;       // [NT/32] scan scratch (x2)
    uint32_t *keys = warp_s + 2 * NT;   // [slice]

    pdl_wait();
    pdl_trigger();

    int64_t n = n_full_cap;
    if (q_pos) {
        const int64_t p1 = ((int64_t)q_pos[qi] + 1) / 4;
        n = p1 < n ? p1 : n;
    }
    if (n < 0) n = 0;
    const int64_t k = (int64_t)k_blk < n ? (int64_t)k_blk : n;
    int32_t *out = blocks_out + qi * (int64_t)k_blk;
    if (rank == 0 && threadIdx.x == 0) counts_out[qi] = (int32_t)k;

    const int64_t slice = (n + CL - 1) / CL;
    const int64_t lo = (int64_t)rank * slice;
    const int64_t hi = lo + slice < n ? lo + slice : n;
    const int64_t len = hi > lo ? hi - lo : 0;

    if (n <= k_blk) {  // every candidate is selected (uniform across the cluster)
        for (int64_t i = threadIdx.x; i < len; i += NT) out[lo + i] = (int32_t)(lo + i);
        return;
    }

    const float *srow = scores + qi * ld;
    for (int64_t i = threadIdx.x; i < len; i += NT) keys[i] = score_key(srow[lo + i]);

    uint32_t prefix = 0;     // bits of T fixed so far
    int fixed = 0;           // number of fixed high bits
    uint32_t k_rem = (uint32_t)k;
#pragma unroll
    for (int pass = 0; pass < 3; ++pass) {
        const int bits = pass == 2 ? 10 : 11;
        const int shift = 32 - fixed - bits;
        const int nb = 1 << bits;
        for (int i = threadIdx.x; i < nb; i += NT) hist[i] = 0u;
        __syncthreads();
        for (int64_t i = threadIdx.x; i < len; i += NT) {
            const uint32_t key = keys[i];
            const bool match = fixed == 0 || (key >> (32 - fixed)) == prefix;
            if (match) atomicAdd(&hist[(key >> shift) & (uint32_t)(nb - 1)], 1u);
        }
        cluster.sync();  // every CTA's histogram is complete
        for (int i = threadIdx.x; i < nb; i += NT) {
            uint32_t s = 0;
#pragma unroll
            for (int r = 0; r < CL; ++r) s += cluster.map_shared_rank(hist, r)[i];
            ghist[i] = s;
        }
        cluster.sync();  // remote reads of hist are done before it is cleared again
        // Bucket of the k_rem-th largest key: scan bins from the top.  Thread t owns
        // bins nb-1-t*per .. nb-per-t*per (per = nb/NT, descending).
        const int per = nb / NT;
        uint32_t mine = 0;
        for (int j = 0; j < per; ++j) mine += ghist[nb - 1 - threadIdx.x * per - j];
        uint32_t tot;
        uint32_t above = block_excl_scan(mine, warp_s, &tot);
        for (int j = 0; j < per; ++j) {
            const int bin = nb - 1 - threadIdx.x * per - j;
            const uint32_t c = ghist[bin];
            if (above < k_rem && above + c >= k_rem) {
                misc[0] = (uint32_t)bin;
                misc[1] = above;
            }
            above += c;
        }
        __syncthreads();
        const uint32_t bucket = misc[0];
        k_rem -= misc[1];
        prefix = (prefix << bits) | bucket;
        fixed += bits;
        __syncthreads();
    }
    const uint32_t T = prefix;   // the k-th largest key
    const uint32_t k_eq = k_rem; // keys == T to take, lowest block index first

    // Contiguous chunk per thread so that the output comes out in index order.
    const int64_t chunk = (len + NT - 1) / NT;
    const int64_t c0 = (int64_t)threadIdx.x * chunk;
    const int64_t c1 = c0 + chunk < len ? c0 + chunk : len;
    uint32_t n_gt = 0, n_eq = 0;
    for (int64_t i = c0; i < c1; ++i) {
        const uint32_t key = keys[i];
        n_gt += key > T;
        n_eq += key == T;
    }
    uint32_t tot_gt, tot_eq;
    uint32_t gt_before = block_excl_scan(n_gt, warp_s, &tot_gt);
    uint32_t eq_before = block_excl_scan(n_eq, warp_s + NT, &tot_eq);
    if (threadIdx.x == 0) {
        misc[2] = tot_gt;
        misc[3] = tot_eq;
    }
    cluster.sync();
    for (int r = 0; r < rank; ++r) {
        const uint32_t *rm = cluster.map_shared_rank(misc, r);
        gt_before += rm[2];
        eq_before += rm[3];
    }
    for (int64_t i = c0; i < c1; ++i) {
        const uint32_t key = keys[i];
        if (key > T) {
            out[gt_before + (eq_before < k_eq ? eq_before : k_eq)] = (int32_t)(lo + i);
            ++gt_before;
        } else if (key == T) {
            if (eq_before < k_eq) out[gt_before + eq_before] = (int32_t)(lo + i);
            ++eq_before;
        }
    }
    cluster.sync();  // keep this CTA's shared memory alive until every remote read is done
}

}  // namespace

int64_t topk_max_candidates() { return kMaxSlice * CL; }

cudaError_t launch_topk(const float *scores, int64_t n_q, int64_t ld, const int32_t *q_pos,
                        int64_t n_full, int64_t k_blk, int32_t *blocks_out, int32_t *counts_out,
                        cudaStream_t st)
{
    if (n_q == 0) return cudaSuccess;
    const int64_t slice = (n_full + CL - 1) / CL;
    const size_t smem = sizeof(uint32_t) * ((size_t)kSmemFixedWords + (size_t)slice);
    static size_t attr_bytes = 0;
    if (smem > 48 * 1024 && attr_bytes < smem) {
        cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kMaxSmemBytes);
        if (e != cudaSuccess) return e;
        attr_bytes = kMaxSmemBytes;
    }
    return launch(topk_cluster_kernel, dim3((unsigned)(n_q * CL)), dim3(NT), smem, st, CL,
                  scores, ld, q_pos, n_full, (int)k_blk, blocks_out, counts_out);
}

}  // namespace qsa
