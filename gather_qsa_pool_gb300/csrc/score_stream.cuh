// score_stream.cuh -- the streaming scan of the pooled-key cache shared by the decode score
// kernels (index_score.cu, score_pool.cu).  Only those two files include it.
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "QSA and the QSA indexer" (each query is scored against every pooled block summary) and
// section "incremental pooled-key cache (COMMON-004)" (after the cache fix this scan is
// the one step left whose cost grows with context).
//
// A pooled row is H*d values of type TP (fp32, or bf16 storage: half the bytes).  Each
// lane of a warp owns 16-byte chunks lane, lane+32, ... of a row (CH of them), issues the
// loads of R rows before reducing any, and scores NQ queries from every row it reads
// (several query tokens of one decode step share the pass).  Per lane the products go
// into four fp32 running sums with fmaf in chunk order; the sums are added pairwise and
// then across the warp.  A row held in shared memory is scored with exactly that order
// (score_row_smem), so a recomputed row scores the same bits as the streamed one.
#pragma once

#include "qsa_internal.cuh"

namespace qsa {

template <typename TP>
struct RowChunk;
template <>
struct RowChunk<float> {
    using V = float4;  // 4 values
};
template <>
struct RowChunk<__nv_bfloat16> {
    using V = uint4;   // 8 values: value 2m in the low half of word m, 2m+1 in the high half
};

// Streaming loads as volatile asms: they stay in program order with the other volatile
// asms, so a row's loads are all issued before the code that follows them.
__device__ __forceinline__ float4 ld_row_chunk_ordered(const float4 *p)
{
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_row_chunk_ordered(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Shared-memory image of one query, hd/4 float4 words.  fp32 rows: word c holds query
// values 4c..4c+3 (chunk c of a row).  bf16 rows: word c holds values 8c..8c+3 and word
// hd/8 + c values 8c+4..8c+7, so that lanes reading consecutive chunks read consecutive
// words of each plane.  Called by the whole CTA (no barrier inside).
template <typename TP>
__device__ __forceinline__ void stage_query(const float *__restrict__ q, int hd, float4 *q_s)
{
    const float4 *q4 = reinterpret_cast<const float4 *>(q);
    if constexpr (sizeof(TP) == 4) {
        for (int c = threadIdx.x; c < hd / 4; c += blockDim.x) q_s[c] = q4[c];
    } else {
        const int h8 = hd / 8;
        for (int c = threadIdx.x; c < h8; c += blockDim.x) {
            q_s[c] = q4[2 * c];
            q_s[h8 + c] = q4[2 * c + 1];
        }
    }
}

__device__ __forceinline__ void dot_acc(float4 &a, const float4 v, const float4 qa)
{
    a.x = fmaf(v.x, qa.x, a.x);
    a.y = fmaf(v.y, qa.y, a.y);
    a.z = fmaf(v.z, qa.z, a.z);
    a.w = fmaf(v.w, qa.w, a.w);
}

// Eight values lo (values 0..3) and hi (values 4..7) of a chunk against its two query words.
__device__ __forceinline__ void dot_acc8(float4 &a, const float4 lo, const float4 hi,
                                         const float4 qa, const float4 qb)
{
    dot_acc(a, lo, qa);
    dot_acc(a, hi, qb);
}

__device__ __forceinline__ void dot_acc(float4 &a, const uint4 v, const float4 qa, const float4 qb)
{
    dot_acc8(a, make_float4(bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y)),
             make_float4(bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w)), qa, qb);
}

__device__ __forceinline__ float finish_dot(const float4 a) { return warp_sum((a.x + a.y) + (a.z + a.w)); }

// Score sc of row `row` for query qi: store it, and count it in the query's histogram.
__device__ __forceinline__ void put_score(float sc, int qi, int64_t row, float *__restrict__ scores,
                                          int64_t ld_s, const ScoreSide &side)
{
    scores[qi * ld_s + row] = sc;
    if (side.hist && row < side.n_hist[qi])
        atomicAdd(&side.hist[((int64_t)qi << kTopkHistBits) + (score_key(sc) >> (32 - kTopkHistBits))],
                  1u);
}

// Rows in flight per warp for the 2048-wide rows (16 indexer heads x 128), as measured
// fastest for each row type and query count on GB300.
template <typename TP, int NQ>
constexpr int stream_rows()
{
    return sizeof(TP) == 4 ? (NQ == 2 ? 2 : 1) : (NQ == 4 ? 4 : 2);
}

// Rows [0, n_rows) walked by warps gw, gw + nw, ... of the grid, R rows per warp in
// flight.  q_s: NQ query images of hd/4 words each (hd = CH * 32 * 16 / sizeof(TP)).
// lim[qi]: rows b < lim[qi] are visible to query qi, the others score -inf.
template <typename TP, int CH, int NQ, int R>
__device__ __forceinline__ void score_stream(const float4 *q_s, const TP *__restrict__ pooled,
                                             int64_t n_rows, int64_t gw, int64_t nw, float scale,
                                             float *__restrict__ scores, int64_t ld_s,
                                             const int64_t *lim, const ScoreSide &side)
{
    using V = typename RowChunk<TP>::V;
    constexpr int kHd = CH * 32 * (16 / (int)sizeof(TP));
    constexpr int kQ4 = kHd / 4;     // query words per query
    constexpr int kPlane = CH * 32;  // bf16: offset of the high plane
    // The row loads are issued first, unconditionally and in program order (volatile), and
    // each chunk's query words are read only after the previous chunk's products (an empty
    // asm with a memory clobber between chunks).  Left to itself the compiler either
    // interleaves loads with the arithmetic (fewer bytes in flight) or loads every query
    // word of the row up front (64 registers per query) and spills; paced, the scan runs
    // at the copy bandwidth of the part.  A row past the end loads the last row instead
    // (its results are dropped), which keeps the loads free of branches.
    const int lane = threadIdx.x & 31;
    for (int64_t r0 = gw; r0 < n_rows; r0 += nw * R) {
        V v[R][CH];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            int64_t row = r0 + (int64_t)r * nw;
            row = row < n_rows ? row : n_rows - 1;
            const V *rp = reinterpret_cast<const V *>(pooled + row * kHd) + lane;
#pragma unroll
            for (int j = 0; j < CH; ++j) v[r][j] = ld_row_chunk_ordered(rp + 32 * j);
        }
        float4 acc[R][NQ];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) acc[r][qi] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < CH; ++j) {
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                const float4 *qw = q_s + qi * kQ4 + lane + 32 * j;
                const float4 qa = qw[0];
                if constexpr (sizeof(TP) == 4) {
#pragma unroll
                    for (int r = 0; r < R; ++r) dot_acc(acc[r][qi], v[r][j], qa);
                } else {
                    const float4 qb = qw[kPlane];
#pragma unroll
                    for (int r = 0; r < R; ++r) dot_acc(acc[r][qi], v[r][j], qa, qb);
                }
            }
            asm volatile("" ::: "memory");
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = r0 + (int64_t)r * nw;
            if (row >= n_rows) continue;  // the same for the whole warp
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                const float tot = finish_dot(acc[r][qi]);
                if (lane == qi) put_score(row < lim[qi] ? tot * scale : -INFINITY, qi, row, scores,
                                          ld_s, side);
            }
        }
    }
}

// The NQ scores (before the scale) of one row held in shared memory as fp32 values
// ([hd], 16-byte aligned), with score_stream's order.  Called by one whole warp; every lane
// gets every result.
template <typename TP, int CH, int NQ>
__device__ __forceinline__ void score_row_smem(const float4 *q_s, const float *row_s, float *out)
{
    constexpr int kHd = CH * 32 * (16 / (int)sizeof(TP));
    constexpr int kQ4 = kHd / 4;
    constexpr int kPlane = CH * 32;
    const int lane = threadIdx.x & 31;
    const float4 *r4 = reinterpret_cast<const float4 *>(row_s);
    float4 acc[NQ];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) acc[qi] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < CH; ++j) {
        const int c = lane + 32 * j;
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
            const float4 *qw = q_s + qi * kQ4 + c;
            if constexpr (sizeof(TP) == 4) {
                dot_acc(acc[qi], r4[c], qw[0]);
            } else {
                dot_acc8(acc[qi], r4[2 * c], r4[2 * c + 1], qw[0], qw[kPlane]);
            }
        }
    }
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) out[qi] = finish_dot(acc[qi]);
}

}  // namespace qsa
