// index_score_tc.cu -- index scores of a prefill chunk (many queries) on the tcgen05 tensor
// cores: scores[i][b] = scale * sum_e bf16(q[i][e]) * bf16(z[b][e]), fp32 accumulation in
// tensor memory, with the causal block visibility rule (4b + 3 <= q_pos[i]) applied in the
// epilogue.
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "QSA and the QSA indexer" (each query is scored against every pooled block); the pages
// leave prefill on the old full path ("selected K/V gather (COMMON-005)": decode only),
// so the chunk form -- every query of a 1024-token ubatch against 64k pooled rows, a
// [1024 x 2048] x [2048 x 64052] contraction -- is this library's.
//
// Design:
//   - prologue kernels round the queries and (for an fp32 cache) the pooled rows to bf16
//     (nearest even) into the workspace, so that both operands can be staged by TMA; a
//     bf16 cache is already the operand and is read in place;
//   - the score kernel is persistent and runs as CTA pairs (clusters of two, one CTA per
//     SM) sharing each tcgen05.mma of M 256 (128 queries in each CTA), N 256, K 16: per
//     stage each CTA stages by TMA its 128 x 64 query tile and half (128 x 64) of the pooled
//     tile (128-byte swizzle, six stages in flight), both completing on the leader CTA's
//     barrier; the leader's warp 1 issues the MMAs (four per stage) into one of two
//     256-column accumulators held in both CTAs' tensor memory and frees each stage in both
//     CTAs with a multicast commit; warps 2-5 of each CTA drain the other accumulator
//     (tcgen05.ld, scale, causal mask, store: each warp turns its 32 x 32 chunks through
//     shared memory so that every store writes whole 128-byte lines) while the next tile
//     computes.  Against one CTA per M 128 tile this halves the pooled bytes each SM stages
//     per MMA (32 KB a stage instead of 48 KB), so the same shared memory keeps 1.5 times
//     the MMA time in flight;
//   - when the query blocks of 256 pair up, clusters of four CTAs run two pairs on adjacent
//     query blocks against the same pooled tile: each CTA stages a quarter (64 rows) of the
//     half its pair position needs and multicasts it into the CTA of the same position in
//     both pairs, so a pooled tile leaves L2 once per two query blocks (the stage is freed
//     by both pairs' commits); this cuts the operands each SM pulls from L2 by a quarter,
//     which is what bounds the contraction once the scores are stored as well;
//   - tiles are ordered query-block-fastest, so the clusters working at the same time share
//     a pooled tile and all but the first read it from L2;
//   - every mbarrier wait is bounded (the pipeline's by the caller's limit, the final ones by
//     2 s): on a timeout the kernel reports it (qsa_set_wait_options), stops issuing, waits
//     for what every CTA of the cluster already issued, and always returns its tensor
//     memory.
#include <cuda.h>

#include "prefill_select.cuh"

namespace qsa {
namespace {

constexpr int kTcWarps = 6;
constexpr int kTcThreads = 32 * kTcWarps;
constexpr int kBM = 128;     // queries per CTA; the CTA pair's MMA covers 256
constexpr int kBN = 256;     // pooled rows per tile (MMA N); each CTA stages half of them
constexpr int kBK = 64;      // k per stage: one 128-byte swizzle row of bf16
constexpr int kStages = 6;
constexpr int kTileA = kBM * kBK * 2;        // 16 KB: this CTA's 128 queries
constexpr int kTileB = (kBN / 2) * kBK * 2;  // 16 KB: this CTA's 128 pooled rows
constexpr uint32_t kTmemCols = 512;          // two accumulators of 256 columns
constexpr int kEpiWarps = 4;                 // warps 2-5

// Each epilogue warp's staging buffer: its 32 rows x 32 columns of a chunk, rows padded to
// 36 floats (16-byte aligned, banks spread), through which the chunk is turned so that every
// store instruction writes whole 128-byte lines of four rows.
constexpr int kEpRow = 36;
constexpr size_t kEpBytes = (size_t)kEpiWarps * 32 * kEpRow * sizeof(float);

__host__ __device__ constexpr size_t tc_smem_bytes()
{
    return 1024 /* alignment slack */ + (size_t)kStages * (kTileA + kTileB) + 256 /* barriers */ +
           kEpBytes;
}

// 64-bit shared-memory matrix descriptor of a K-major tile in the 128-byte swizzle:
// start address, leading byte offset (unused for this layout: 16), stride byte offset
// 1024 (one 8-row swizzle atom), descriptor version 1, layout type 2 (128-byte swizzle).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(16u >> 4) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor: fp32 accumulator, bf16 A and B, both K-major, N = 256, M = 256
// (the CTA pair: 128 rows in each CTA's tensor memory).
__host__ __device__ constexpr uint32_t idesc_bf16_m256_n256()
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
           ((uint32_t)((2 * kBM) >> 4) << 24);
}

// One M256 x N256 x K16 MMA of the CTA pair: A and B are read from the same shared-memory
// offsets in both CTAs, D is written to the same tensor-memory columns of both.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the barrier at this shared-memory offset in every CTA of `mask` once the pair
// MMAs issued so far by this thread have completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar, uint16_t mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(mask)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(const void *p, uint32_t rank)
{
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    return a;
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// 2-D tiled TMA load of the box at (x, y) into this CTA's shared memory, completing its bytes
// on the barrier at cluster address bar (the leader CTA's, for either CTA of the pair).
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map, int x, int y,
                                                 uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
        "bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// The same load multicast into every CTA of `mask` (the same shared-memory offset in each),
// each destination's bytes completing on the barrier at bar's offset in the leader of that
// destination's pair (bar: the issuing CTA's pair leader's barrier, even rank).
__device__ __forceinline__ void tma_load_2d_pair_mc(void *dst, const CUtensorMap *map, int x,
                                                    int y, uint32_t bar, uint16_t mask)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
        "bytes.multicast::cluster [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "h"(mask)
        : "memory");
}

// Remote (or local) arrival on a barrier given by its cluster address.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
                 : "memory");
}

// Complete `bytes` transaction bytes of the barrier's current phase without a copy.
__device__ __forceinline__ void mbar_complete_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Store a word into the shared memory of another CTA of the cluster (cluster address).
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Prologue: q (fp32, row stride ld_q) -> bf16 rows of K elements, nearest even.  One CTA
// per row at a time; four elements per thread and step when every row starts on a 16-byte
// boundary (vec), else one.
__global__ void __launch_bounds__(256)
q_to_bf16_kernel(const float *__restrict__ q, int64_t n_q, int64_t ld_q, int K,
                 __nv_bfloat16 *__restrict__ qb, int vec)
{
    pdl_wait();
    QSA_AFTER_WAIT(q);
    pdl_trigger();
    for (int64_t i = blockIdx.x; i < n_q; i += gridDim.x) {
        const float *src = q + i * ld_q;
        __nv_bfloat16 *dst = qb + i * (int64_t)K;
        if (vec) {
            for (int k4 = threadIdx.x; k4 < K / 4; k4 += blockDim.x) {
                const float4 v = reinterpret_cast<const float4 *>(src)[k4];
                reinterpret_cast<uint2 *>(dst)[k4] =
                    make_uint2(bf16x2(v.x, v.y), bf16x2(v.z, v.w));
            }
        } else {
            for (int k = threadIdx.x; k < K; k += blockDim.x) dst[k] = __float2bfloat16_rn(src[k]);
        }
    }
}

// Prologue: the pooled rows (fp32, contiguous, n4 float4) -> bf16, nearest even.
__global__ void __launch_bounds__(256)
rows_to_bf16_kernel(const float4 *__restrict__ src, int64_t n4, uint2 *__restrict__ dst)
{
    pdl_wait();
    QSA_AFTER_WAIT(src);
    pdl_trigger();
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n4;
         e += (int64_t)gridDim.x * blockDim.x) {
        const float4 v = ld_stream_f4(src + e);
        dst[e] = make_uint2(bf16x2(v.x, v.y), bf16x2(v.z, v.w));
    }
}

// CL: CTAs per cluster.  2: one CTA pair.  4: two pairs working on adjacent query blocks
// against the same pooled tile, each CTA staging a 1/(CL/2) share (64 rows) of the tile's
// half its pair position needs and multicasting it into every pair.
template <int CL>
__global__ void __launch_bounds__(kTcThreads, 1)
score_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                int64_t n_q, const int32_t *__restrict__ q_pos, int64_t n_rows, int K,
                float scale, float *__restrict__ scores, int64_t ld_scores,
                float *__restrict__ gmax, int64_t ld_gmax, const WaitCtl wc)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    // 1024-byte aligned operand area (the swizzle is a function of address bits 4-9); the
    // same offsets in both CTAs of the pair, as the pair MMA requires
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *sA = base;                              // [kStages][128 queries][128 B]
    unsigned char *sB = base + kStages * kTileA;           // [kStages][128 rows][128 B]
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + kStages * kTileB);  // [kStages] leader
    uint64_t *empty = full + kStages;                      // [kStages] both CTAs
    uint64_t *accf = empty + kStages;                      // [2] accumulator ready, both CTAs
    uint64_t *acce = accf + 2;                             // [2] accumulator drained, leader
    uint64_t *drain = acce + 2;                            // every MMA issued has finished
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    uint32_t *issued_all = tmem_slot + 1;                  // leader: k-steps each CTA issued
    float *ep_buf = reinterpret_cast<float *>(sB + kStages * kTileB + 256);  // [warp][32][36]

    static_assert(CL == 2 || CL == 4, "one pair or two");
    constexpr int kPairs = CL / 2;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_rank();
    const uint32_t lrank = rank & ~1u;  // the pair's leader (even rank), which issues its MMAs
    const bool leader = rank == lrank;
    const uint32_t half = rank & 1u;    // which 128 queries (and pooled rows) of the pair
    const uint32_t pq = rank >> 1;      // the pair's place in the cluster

    pdl_wait();
    QSA_AFTER_WAIT(q_pos);
    pdl_trigger();

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kPairs);  // a commit from each pair's MMAs
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&accf[j], 1);
            mbar_init(&acce[j], 2 * kEpiWarps);
        }
        mbar_init(drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        // both CTAs of the pair allocate together: the same columns in each
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncwarp();
    cluster_sync_all();  // barriers initialised and tensor memory allocated in both CTAs
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    // unit u: pooled tile u / n_mg against query blocks (u % n_mg) * kPairs + (0 .. kPairs-1),
    // one per pair (a block past the queries reads zeros and stores nothing)
    const int64_t n_mb = (n_q + 2 * kBM - 1) / (2 * kBM);
    const int64_t n_mg = (n_mb + kPairs - 1) / kPairs;
    const int64_t n_nb = (n_rows + kBN - 1) / kBN;
    const int64_t n_units = n_mg * n_nb;
    const int64_t grp = blockIdx.x / CL, n_grp = gridDim.x / CL;
    const int n_k = K / kBK;
    bool ok = true;
    uint32_t issued = 0;  // producer: k-steps whose copies this CTA issued

    if (warp == 0) {
        // ---- producer, in each CTA: its 128 queries and its share of the pooled rows of
        // every stage (with one pair its 128 rows; with two, a quarter of them, multicast
        // into the CTA of the same half in both pairs), all completing on the barriers of the
        // pair leaders
        if (lane == 0) {
            // k-step `it` of this CTA's sequence uses stage it % kStages for the
            // (it / kStages)-th time; every CTA of the cluster runs the same sequence
            uint32_t it = 0;
            for (int64_t u = grp; u < n_units && ok; u += n_grp) {
                const int m0 = (int)(((u % n_mg) * kPairs + pq) * (2 * kBM) + half * kBM);
                const int n0 = (int)((u / n_mg) * kBN + half * (kBN / 2) + pq * (kBN / CL));
                for (int kb = 0; kb < n_k; ++kb, ++it) {
                    const uint32_t stage = it % kStages, use = it / kStages;
                    if (use > 0 && !mbar_wait(&empty[stage], (use - 1) & 1u, wc.limit_ns)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(&full[stage], 2 * (kTileA + kTileB));
                    const uint32_t fb = map_to_rank(&full[stage], lrank);
                    tma_load_2d_pair(sA + stage * kTileA, &tmA, kb * kBK, m0, fb);
                    if constexpr (CL > 2)
                        tma_load_2d_pair_mc(sB + stage * kTileB + pq * (kTileB / kPairs), &tmB,
                                            kb * kBK, n0, fb,
                                            (uint16_t)((0x5555u & ((1u << CL) - 1u)) << half));
                    else
                        tma_load_2d_pair(sB + stage * kTileB, &tmB, kb * kBK, n0, fb);
                }
            }
            issued = it;
            // this CTA's count goes to every pair leader (read there after the cluster
            // barrier below)
#pragma unroll
            for (int l = 0; l < CL; l += 2) st_cluster_u32(map_to_rank(issued_all + rank, l), it);
        }
    } else if (warp == 1) {
        // ---- MMA issuer: one thread of the leader; accumulators alternate between the two
        // tensor-memory halves
        if (leader && lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_m256_n256();
            uint32_t it = 0;
            int64_t t = 0;
            for (int64_t u = grp; u < n_units && ok; u += n_grp, ++t) {
                const int j = (int)(t & 1);
                if (t >= 2 && !mbar_wait(&acce[j], (uint32_t)((t >> 1) - 1) & 1u, wc.limit_ns)) {
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                for (int kb = 0; kb < n_k; ++kb, ++it) {
                    const uint32_t stage = it % kStages;
                    if (!mbar_wait(&full[stage], (it / kStages) & 1u, wc.limit_ns)) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t a0 = smem_u32(sA + stage * kTileA);
                    const uint32_t b0 = smem_u32(sB + stage * kTileB);
#pragma unroll
                    for (int k16 = 0; k16 < kBK / 16; ++k16)
                        umma_bf16_pair(tmem + (uint32_t)(j * kBN), sw128_desc(a0 + k16 * 32),
                                       sw128_desc(b0 + k16 * 32), idesc, (kb | k16) ? 1u : 0u);
                    // the stage is free (as far as this pair is concerned) in every CTA
                    umma_commit_pair(&empty[stage], (uint16_t)((1u << CL) - 1u));
                }
                if (!ok) break;
                umma_commit_pair(&accf[j], (uint16_t)(3u << lrank));
            }
            umma_commit_pair(drain, (uint16_t)(1u << lrank));
            if (!mbar_wait(drain, 0)) ok = false;
        }
    } else {
        // ---- epilogue, in each CTA: warp w reads tensor-memory lanes 32*(w%4) .. +31 (its
        // queries), then reports the accumulator half drained to the leader
        const int quarter = warp & 3;
        const uint32_t acce_leader[2] = {map_to_rank(&acce[0], lrank),
                                         map_to_rank(&acce[1], lrank)};
        int64_t t = 0;
        for (int64_t u = grp; u < n_units && ok; u += n_grp, ++t) {
            const int j = (int)(t & 1);
            if (!mbar_wait(&accf[j], (uint32_t)(t >> 1) & 1u, wc.limit_ns)) {
                ok = false;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int64_t m0 = ((u % n_mg) * kPairs + pq) * (2 * kBM) + half * kBM;
            const int64_t n0 = (u / n_mg) * kBN;
            const int64_t qi = m0 + quarter * 32 + lane;
            const int64_t p = (qi < n_q && q_pos) ? (int64_t)q_pos[qi] : INT64_MAX;
            // blocks complete at position p: b with 4b + 3 <= p
            const int64_t vis_rows = p >= 3 ? (p - 3) / 4 + 1 : 0;
            // every row of the scores starts on a 16-byte boundary (the transposed stores)
            const bool rows_vec =
                ld_scores % 4 == 0 && (reinterpret_cast<uintptr_t>(scores) & 15) == 0;
            // the tile's eight group maxima of this query, shifted in one per chunk (index cc
            // ends in m8[cc]), stored together after the chunks: two 16-byte stores a tile
            float m8[kBN / 32];
#pragma unroll
            for (int e = 0; e < kBN / 32; ++e) m8[e] = -INFINITY;
#pragma unroll 1
            for (int cc = 0; cc < kBN / 32; ++cc) {
                uint32_t v[32];
                const uint32_t taddr =
                    tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(j * kBN + cc * 32);
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                    "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                    "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                    : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                      "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
                      "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
                      "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
                      "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]),
                      "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                    : "r"(taddr));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                const int64_t b0 = n0 + cc * 32;
                // rows b0 + e, e < lim, exist and are visible (4b + 3 <= p); the others are
                // -inf (those past n_rows are not stored)
                const int64_t lim64 = (vis_rows < n_rows ? vis_rows : n_rows) - b0;
                const int lim = lim64 < 0 ? 0 : (lim64 > 32 ? 32 : (int)lim64);
                float o[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    o[e] = e < lim ? __uint_as_float(v[e]) * scale : -INFINITY;
                if (gmax) {  // the group's largest visible score
                    float m16[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) m16[e] = fmaxf(o[e], o[e + 16]);
#pragma unroll
                    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                        for (int e = 0; e < w; ++e) m16[e] = fmaxf(m16[e], m16[e + w]);
#pragma unroll
                    for (int e = 0; e + 1 < kBN / 32; ++e) m8[e] = m8[e + 1];
                    m8[kBN / 32 - 1] = m16[0];
                }
                if (b0 + 32 <= n_rows && rows_vec) {
                    // a whole chunk (warp-uniform): each lane's row into the warp's buffer,
                    // then four rows of 32 scores per store instruction (eight lanes a row)
                    float *buf = ep_buf + (warp - 2) * 32 * kEpRow;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(buf + lane * kEpRow + e) =
                            make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
                    __syncwarp();
                    const int c4 = (lane & 7) * 4;
#pragma unroll
                    for (int pass = 0; pass < 8; ++pass) {
                        const int rr = pass * 4 + (lane >> 3);
                        const int64_t qr = m0 + quarter * 32 + rr;
                        const float4 val = *reinterpret_cast<const float4 *>(buf + rr * kEpRow + c4);
                        if (qr < n_q)
                            *reinterpret_cast<float4 *>(scores + qr * ld_scores + b0 + c4) = val;
                    }
                    __syncwarp();  // the buffer is rewritten by the next chunk
                } else if (qi < n_q) {
                    float *dst = scores + qi * ld_scores + b0;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (b0 + e < n_rows) dst[e] = o[e];
                }
            }
            if (gmax && qi < n_q) {  // groups n0 / 32 .. + 7 of this query (those that exist)
                float *gd = gmax + qi * ld_gmax + (n0 >> 5);
                const int64_t n_g = (n_rows + 31) / 32 - (n0 >> 5);
                if (n_g >= kBN / 32 && (reinterpret_cast<uintptr_t>(gd) & 15) == 0) {
                    *reinterpret_cast<float4 *>(gd) = make_float4(m8[0], m8[1], m8[2], m8[3]);
                    *reinterpret_cast<float4 *>(gd + 4) = make_float4(m8[4], m8[5], m8[6], m8[7]);
                } else {
#pragma unroll
                    for (int e = 0; e < kBN / 32; ++e)
                        if (e < n_g) gd[e] = m8[e];
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acce_leader[j]);  // this half may be overwritten
        }
    }

    if (!ok) report_timeout(wc);
    // Every copy lands on the barrier of the leader of the pair it lands in, so each leader
    // sees all of its pair's bytes land before any CTA of the cluster may leave.  After a wait
    // gave up, the producers may have stopped at different k-steps: a phase the leader armed
    // (for the whole stage) gets the bytes of the copies never issued completed by the
    // leader; a phase copied into but never armed is armed for the bytes that did land.  The
    // producers run at most kStages k-steps apart (each waits for every pair's MMAs to free
    // a stage), so each stage has at most one such phase, and the phase before it completed.
    cluster_sync_all();  // every CTA's count is in each leader's shared memory
    if (warp == 0 && lane == 0 && leader) {
        uint32_t lo = issued, hi = issued;
        for (int c = 0; c < CL; ++c) {
            const uint32_t n = issued_all[c];
            lo = n < lo ? n : lo;
            hi = n > hi ? n : hi;
        }
        for (uint32_t x = lo; x < hi; ++x) {
            const uint32_t stage = x % kStages, use = x / kStages;
            if (use > 0) (void)mbar_wait(&full[stage], (use - 1) & 1u);
            // bytes of k-step x that landed in this pair: each CTA's query tile lands in its
            // own CTA, its pooled rows in the CTA(s) of its half
            uint32_t landed = 0;
            for (int c = 0; c < CL; ++c)
                if (x < issued_all[c])
                    landed += ((uint32_t)c >> 1 == pq ? (uint32_t)kTileA : 0u) +
                              (uint32_t)(kTileB / kPairs);
            if (x < issued) {
                if (landed < 2u * (kTileA + kTileB))
                    mbar_complete_tx(&full[stage], 2u * (kTileA + kTileB) - landed);
            } else {
                mbar_arrive_expect_tx(&full[stage], landed);
            }
        }
        for (uint32_t s = 0; s < kStages; ++s) {
            const uint32_t uses = hi / kStages + (s < hi % kStages ? 1u : 0u);
            if (uses > 0 && !mbar_wait(&full[s], (uses - 1) & 1u)) report_timeout(wc);
        }
    }
    // neither CTA leaves (or frees its tensor memory) while the pair's MMAs, copies or
    // remote arrivals may still touch it
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncwarp();
    cluster_sync_all();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Tensor map of a row-major bf16 matrix [rows][K]: boxes of 64 x box_rows, 128-byte
// swizzle, zero fill outside the matrix.
bool make_map(CUtensorMap *m, const void *base, int64_t rows, int K, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t al256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace

size_t index_score_tc_workspace(int64_t n_q, int64_t n_rows, int H, int d, qsa_dtype pdt)
{
    // bf16 copies of the queries and (for an fp32 cache) of the pooled rows; a bf16 cache is
    // read in place
    const size_t K = (size_t)H * (size_t)d;
    const size_t rows = pdt == QSA_BF16 ? 0 : al256((size_t)n_rows * K * 2);
    return al256((size_t)n_q * K * 2) + rows;
}

// Persistent launch of the score kernel in clusters of CL CTAs: as many clusters as fit on
// the GPU at once (one CTA per SM), at most one per unit of work.
template <int CL>
static cudaError_t launch_score_tc(const CUtensorMap &tmA, const CUtensorMap &tmB, int64_t n_q,
                                  const int32_t *q_pos, int64_t n_rows, int K, float scale,
                                  float *scores, int64_t ld_scores, float *gmax, int64_t ld_gmax,
                                  cudaStream_t st)
{
    cudaError_t e = ensure_kernel_attrs<score_tc_kernel<CL>>(tc_smem_bytes());
    if (e != cudaSuccess) return e;
    const int64_t n_mb = (n_q + 2 * kBM - 1) / (2 * kBM);
    const int64_t n_units = ((n_mb + CL / 2 - 1) / (CL / 2)) * ((n_rows + kBN - 1) / kBN);
    int64_t groups = device_sm_count() / CL;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(CL * groups));
        cfg.blockDim = dim3(kTcThreads);
        cfg.dynamicSmemBytes = tc_smem_bytes();
        cudaLaunchAttribute a;
        a.id = cudaLaunchAttributeClusterDimension;
        a.val.clusterDim.x = CL;
        a.val.clusterDim.y = 1;
        a.val.clusterDim.z = 1;
        cfg.attrs = &a;
        cfg.numAttrs = 1;
        int resident = 0;
        if (cudaOccupancyMaxActiveClusters(&resident, score_tc_kernel<CL>, &cfg) != cudaSuccess)
            (void)cudaGetLastError();
        else if (resident > 0 && resident < groups)
            groups = resident;
    }
    if (groups > n_units) groups = n_units;
    if (groups < 1) groups = 1;
    return launch(score_tc_kernel<CL>, dim3((unsigned)(CL * groups)), dim3(kTcThreads),
                  tc_smem_bytes(), st, CL, tmA, tmB, n_q, q_pos, n_rows, K, scale, scores,
                  ld_scores, gmax, ld_gmax, current_wait_ctl());
}

static qsa_status score_tc(const float *q, int64_t n_q, int64_t ld_q, const int32_t *q_pos,
                           const void *pooled, qsa_dtype pdt, int64_t n_rows, int H, int d,
                           float scale, float *scores, int64_t ld_scores, float *gmax,
                           int64_t ld_gmax, void *workspace, size_t ws_bytes, cudaStream_t st)
{
    const int K = H * d;
    if (K % kBK != 0) return QSA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(pooled) & 15) || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return QSA_ERR_INVALID_ARG;
    if (n_q == 0 || n_rows == 0) return QSA_OK;
    if (n_q > 0x7fffffffLL || n_rows > 0x7fffffffLL) return QSA_ERR_UNSUPPORTED;
    const size_t need = index_score_tc_workspace(n_q, n_rows, H, d, pdt);
    if (ws_bytes < need) return QSA_ERR_INVALID_ARG;
    char *ws = static_cast<char *>(workspace);
    __nv_bfloat16 *qb = reinterpret_cast<__nv_bfloat16 *>(ws);
    const bool convert_rows = pdt != QSA_BF16;
    const __nv_bfloat16 *pb =
        convert_rows ? reinterpret_cast<__nv_bfloat16 *>(ws + al256((size_t)n_q * K * 2))
                     : static_cast<const __nv_bfloat16 *>(pooled);
    // two CTA pairs share each pooled tile when the query blocks of 256 pair up exactly
    const int64_t n_mb = (n_q + 2 * kBM - 1) / (2 * kBM);
    const int cl = n_mb % 2 == 0 ? 4 : 2;
    CUtensorMap tmA, tmB;
    if (!make_map(&tmA, qb, n_q, K, kBM) || !make_map(&tmB, pb, n_rows, K, (uint32_t)(kBN / cl)))
        return QSA_ERR_CUDA;
    const int qvec = ld_q % 4 == 0 && (reinterpret_cast<uintptr_t>(q) & 15) == 0;
    const int64_t qgrid = n_q < (int64_t)device_sm_count() * 8 ? n_q : (int64_t)device_sm_count() * 8;
    cudaError_t e = launch(q_to_bf16_kernel, dim3((unsigned)qgrid), dim3(256), 0, st, 1, q, n_q,
                           ld_q, K, qb, qvec);
    if (e == cudaSuccess && convert_rows) {
        const int64_t n4 = n_rows * (int64_t)K / 4;
        e = launch(rows_to_bf16_kernel, dim3((unsigned)(device_sm_count() * 8)), dim3(256), 0, st,
                   1, reinterpret_cast<const float4 *>(pooled), n4,
                   reinterpret_cast<uint2 *>(const_cast<__nv_bfloat16 *>(pb)));
    }
    if (e != cudaSuccess) return QSA_ERR_CUDA;
    e = cl == 4 ? launch_score_tc<4>(tmA, tmB, n_q, q_pos, n_rows, K, scale, scores, ld_scores,
                                     gmax, ld_gmax, st)
                : launch_score_tc<2>(tmA, tmB, n_q, q_pos, n_rows, K, scale, scores, ld_scores,
                                     gmax, ld_gmax, st);
    return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}

qsa_status launch_index_score_tc(const float *q, int64_t n_q, int64_t ld_q,
                                 const int32_t *q_pos, const void *pooled, qsa_dtype pdt,
                                 int64_t n_rows, int H, int d, float scale, float *scores,
                                 int64_t ld_scores, void *workspace, size_t ws_bytes,
                                 cudaStream_t st)
{
    return score_tc(q, n_q, ld_q, q_pos, pooled, pdt, n_rows, H, d, scale, scores, ld_scores,
                    nullptr, 0, workspace, ws_bytes, st);
}

qsa_status launch_index_score_tc_maxima(const float *q, int64_t n_q, int64_t ld_q,
                                        const int32_t *q_pos, const void *pooled,
                                        qsa_dtype pdt, int64_t n_rows, int H, int d, float scale,
                                        float *scores, int64_t ld_scores, float *maxima,
                                        int64_t ld_maxima, void *workspace, size_t ws_bytes,
                                        cudaStream_t st)
{
    return score_tc(q, n_q, ld_q, q_pos, pooled, pdt, n_rows, H, d, scale, scores, ld_scores,
                    maxima, ld_maxima, workspace, ws_bytes, st);
}

}  // namespace qsa
