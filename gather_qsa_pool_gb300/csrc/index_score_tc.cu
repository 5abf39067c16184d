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
// Design (one CTA per SM, persistent over work items):
//   - a work item is 512 queries x 128 pooled rows; its four 128 x 128 fp32 accumulators
//     fill the SM's 512 tensor-memory columns;
//   - the K = H*d reduction runs in stages of 64: the query tile (bf16, converted once by a
//     prologue kernel) arrives by cp.async, the pooled tile (fp32 in HBM) is loaded into
//     registers one stage ahead, rounded to bf16 (nearest even) and stored; both tiles use
//     the 128-byte-swizzled K-major layout the MMA descriptors describe;
//   - one thread issues 16 tcgen05.mma (4 accumulators x 4 k-steps of 16) per stage and
//     commits them to the stage's mbarrier, which releases the buffer two stages later;
//   - after the last stage a commit to a second mbarrier hands the accumulators to the
//     epilogue: every warp reads its 32 tensor-memory lanes (tcgen05.ld), scales, masks and
//     writes the scores.
// Work items alternate the two query halves on the same pooled tile so that the second
// read of each pooled tile is an L2 hit.  Every mbarrier wait is bounded: on a timeout the
// kernel records an error word and stops issuing work (no hang), and it always returns its
// tensor memory.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kTcThreads = 128;
constexpr int kBM = 128;          // rows per MMA (queries)
constexpr int kMT = 4;            // accumulators per work item (512 queries)
constexpr int kBN = 128;          // pooled rows per work item
constexpr int kBK = 64;           // k per stage (one 128-byte swizzle row of bf16)
constexpr int kStages = 2;
constexpr int kTileA = kMT * kBM * kBK * 2;  // 64 KB per stage
constexpr int kTileB = kBN * kBK * 2;        // 16 KB per stage
constexpr uint32_t kTmemCols = 512;

__host__ __device__ constexpr size_t tc_smem_bytes()
{
    return 1024 /* alignment slack */ + (size_t)kStages * (kTileA + kTileB) + 64;
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

// Instruction descriptor: fp32 accumulator, bf16 A and B, both K-major, N = 128, M = 128.
__host__ __device__ constexpr uint32_t idesc_bf16_m128_n128()
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
           ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid)
{
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
                 : "memory");
}

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Prologue: q (fp32, row stride ld_q) -> bf16 rows of K elements, nearest even.
__global__ void __launch_bounds__(256)
q_to_bf16_kernel(const float *__restrict__ q, int64_t n_q, int64_t ld_q, int K,
                 __nv_bfloat16 *__restrict__ qb)
{
    pdl_wait();
    QSA_AFTER_WAIT(q);
    pdl_trigger();
    const int64_t total = n_q * (int64_t)K;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = e / K, k = e - i * K;
        qb[e] = __float2bfloat16_rn(q[i * ld_q + k]);
    }
}

__global__ void __launch_bounds__(kTcThreads, 1)
score_tc_kernel(const __nv_bfloat16 *__restrict__ qb, int64_t n_q,
                const int32_t *__restrict__ q_pos, const float *__restrict__ pooled,
                int64_t n_rows, int K, float scale, float *__restrict__ scores, int64_t ld_scores,
                int *__restrict__ err)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    // 1024-byte aligned operand area (the swizzle is a function of address bits 4-9)
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *sA = base;                             // [kStages][kMT*kBM rows][128 B]
    unsigned char *sB = base + kStages * kTileA;          // [kStages][kBN rows][128 B]
    uint64_t *bar = reinterpret_cast<uint64_t *>(sB + kStages * kTileB);  // [kStages] + acc
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + kStages + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    pdl_wait();
    QSA_AFTER_WAIT(qb);
    QSA_AFTER_WAIT(q_pos);
    QSA_AFTER_WAIT(pooled);
    pdl_trigger();

    if (tid == 0) {
        for (int s = 0; s <= kStages; ++s) mbar_init(&bar[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    const int64_t n_mb = (n_q + kMT * kBM - 1) / (kMT * kBM);
    const int64_t n_nt = (n_rows + kBN - 1) / kBN;
    const int64_t n_items = n_mb * n_nt;
    const int n_k = K / kBK;
    constexpr uint32_t idesc = idesc_bf16_m128_n128();

    uint32_t use_count[kStages] = {0, 0};  // commits issued to each stage barrier
    uint32_t acc_count = 0;
    bool ok = true;

    // The pooled tile of a stage is 128 rows x 16 float4; thread tid loads float4
    // f = j*128 + tid (row f/16, column group f%16): coalesced, one stage ahead.
    float4 breg[kBK / 4];
    auto load_b = [&](int64_t it, int ks) {
        const int64_t n0b = (it / n_mb) * kBN;
#pragma unroll
        for (int j = 0; j < kBK / 4; ++j) {
            const int f = j * kTcThreads + tid;
            const int64_t row = n0b + (f >> 4);
            breg[j] = row < n_rows
                          ? ld_stream_f4(reinterpret_cast<const float4 *>(
                                pooled + row * (int64_t)K + (int64_t)ks * kBK) + (f & 15))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    // Fill buffer sb with stage (it, ks): query tile by cp.async, pooled tile from the
    // registers (fp32 -> bf16, nearest even), both in the 128-byte swizzle; then load the
    // pooled registers of the following stage.
    auto fill = [&](int sb, int64_t it, int ks) {
        unsigned char *a_s = sA + sb * kTileA;
        unsigned char *b_s = sB + sb * kTileB;
        const int64_t m0 = (it % n_mb) * (kMT * kBM);
        for (int e = tid; e < kMT * kBM * 8; e += kTcThreads) {
            const int r = e >> 3, c = e & 7;
            const int64_t qi = m0 + r;
            const bool valid = qi < n_q;
            const __nv_bfloat16 *src = qb + (valid ? qi : 0) * (int64_t)K + (int64_t)ks * kBK + c * 8;
            cp_async16(smem_u32(a_s + r * 128 + ((c ^ (r & 7)) << 4)), src, valid);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
#pragma unroll
        for (int j = 0; j < kBK / 4; ++j) {
            const int f = j * kTcThreads + tid;
            const int r = f >> 4, c4 = f & 15;
            const uint2 v = make_uint2(bf16x2(breg[j].x, breg[j].y), bf16x2(breg[j].z, breg[j].w));
            *reinterpret_cast<uint2 *>(b_s + r * 128 + (((c4 >> 1) ^ (r & 7)) << 4) + (c4 & 1) * 8) = v;
        }
        int64_t nit = it;
        int nks = ks + 1;
        if (nks == n_k) {
            nit = it + gridDim.x;
            nks = 0;
        }
        if (nit < n_items) load_b(nit, nks);
    };

    // Pipeline over the flattened (work item, k stage) sequence of this CTA: the copies of
    // stage g+1 are in flight while the tensor cores run stage g.
    int64_t item = blockIdx.x;
    const int64_t my_items = item < n_items ? (n_items - 1 - item) / gridDim.x + 1 : 0;
    const int64_t n_stages = my_items * n_k;
    if (n_stages > 0) {
        load_b(item, 0);
        fill(0, item, 0);
    }
    for (int64_t gs = 0; gs < n_stages && ok; ++gs) {
        const int sb = (int)(gs % kStages);
        const int ks = (int)(gs % n_k);
        const int64_t it = blockIdx.x + (gs / n_k) * gridDim.x;
        asm volatile("cp.async.wait_group 0;" ::: "memory");  // this stage's query tile
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t a0 = smem_u32(sA + sb * kTileA), b0 = smem_u32(sB + sb * kTileB);
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt) {
#pragma unroll
                for (int k16 = 0; k16 < kBK / 16; ++k16) {
                    const uint64_t ad = sw128_desc(a0 + mt * (kBM * 128) + k16 * 32);
                    const uint64_t bd = sw128_desc(b0 + k16 * 32);
                    umma_bf16(tmem + mt * kBN, ad, bd, idesc, (ks > 0 || k16 > 0) ? 1u : 0u);
                }
            }
            umma_commit(&bar[sb]);
            if (ks == n_k - 1) umma_commit(&bar[kStages]);
        }
        ++use_count[sb];
        // refill the other buffer with stage gs+1 once the MMAs that last read it are done
        if (gs + 1 < n_stages) {
            const int nb = (int)((gs + 1) % kStages);
            if (use_count[nb] > 0 && !mbar_wait(&bar[nb], (use_count[nb] - 1) & 1)) ok = false;
            if (__syncthreads_or(!ok)) {
                ok = false;
                break;
            }
            if (ks + 1 < n_k) fill(nb, it, ks + 1);
            else fill(nb, it + gridDim.x, 0);
        }
        if (ks == n_k - 1) {
            // epilogue of work item `it`: wait for its accumulators, read this warp's lanes
            const int64_t m0 = (it % n_mb) * (kMT * kBM), n0 = (it / n_mb) * kBN;
            if (!mbar_wait(&bar[kStages], acc_count & 1)) ok = false;
            ++acc_count;
            if (__syncthreads_or(!ok)) {
                ok = false;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll 1
            for (int mt = 0; mt < kMT; ++mt) {
                const int64_t qi = m0 + mt * kBM + warp * 32 + lane;
                const int64_t p = (qi < n_q && q_pos) ? (int64_t)q_pos[qi] : INT64_MAX;
#pragma unroll 1
                for (int cc = 0; cc < kBN / 32; ++cc) {
                    uint32_t v[32];
                    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(mt * kBN + cc * 32);
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
                    if (qi < n_q) {
                        float *dst = scores + qi * ld_scores + n0 + cc * 32;
                        const int64_t b0 = n0 + cc * 32;
                        float o[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            o[j] = 4 * (b0 + j) + 3 <= p ? __uint_as_float(v[j]) * scale : -INFINITY;
                        if (b0 + 32 <= n_rows && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
                            for (int j = 0; j < 32; j += 4)
                                *reinterpret_cast<float4 *>(dst + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (b0 + j < n_rows) dst[j] = o[j];
                        }
                    }
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncthreads();  // accumulators read: the next item's MMAs may overwrite them
        }
    }
    if (!ok && tid == 0) atomicExch(err, 1);
    // drain: the last commits must have landed before tensor memory is returned
    __syncthreads();
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s)
            if (use_count[s] > 0) mbar_wait(&bar[s], (use_count[s] - 1) & 1);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

}  // namespace

size_t index_score_tc_workspace(int64_t n_q, int64_t n_rows, int H, int d)
{
    (void)n_rows;
    // bf16 copy of the queries, then one error word (256-byte aligned)
    const size_t qb = ((size_t)n_q * (size_t)H * (size_t)d * 2 + 255) & ~(size_t)255;
    return qb + 256;
}

qsa_status launch_index_score_tc(const float *q, int64_t n_q, int64_t ld_q,
                                 const int32_t *q_pos, const float *pooled, int64_t n_rows,
                                 int H, int d, float scale, float *scores, int64_t ld_scores,
                                 void *workspace, size_t ws_bytes, cudaStream_t st)
{
    const int K = H * d;
    if (K % kBK != 0) return QSA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(pooled) & 15) || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return QSA_ERR_INVALID_ARG;
    if (n_q == 0 || n_rows == 0) return QSA_OK;
    const size_t need = index_score_tc_workspace(n_q, n_rows, H, d);
    if (ws_bytes < need) return QSA_ERR_INVALID_ARG;
    __nv_bfloat16 *qb = static_cast<__nv_bfloat16 *>(workspace);
    int *err = reinterpret_cast<int *>(static_cast<char *>(workspace) + need - 256);
    cudaError_t e = launch(q_to_bf16_kernel, dim3(1024), dim3(256), 0, st, 1, q, n_q, ld_q, K, qb);
    if (e != cudaSuccess) return QSA_ERR_CUDA;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(score_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)tc_smem_bytes()) != cudaSuccess)
            return QSA_ERR_CUDA;
        attr = true;
    }
    const int64_t n_items = ((n_q + kMT * kBM - 1) / (kMT * kBM)) * ((n_rows + kBN - 1) / kBN);
    int64_t grid = device_sm_count();
    if (grid > n_items) grid = n_items;
    e = launch(score_tc_kernel, dim3((unsigned)grid), dim3(kTcThreads), tc_smem_bytes(), st, 1,
               (const __nv_bfloat16 *)qb, n_q, q_pos, pooled, n_rows, K, scale, scores, ld_scores,
               err);
    return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}

}  // namespace qsa
