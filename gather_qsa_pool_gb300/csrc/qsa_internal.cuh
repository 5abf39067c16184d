// qsa_internal.cuh -- shared device helpers and launcher declarations of the sm_103a
// QSA library.  Only the library's own .cu files include this header.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "../../include/qsa.h"

namespace qsa {

// GB300: 152 SMs.  Split counts that must be known without a device (workspace sizes)
// are derived from this constant; launch grids query the device.
constexpr int kTargetSMs = 152;

// ------------------------------------------------------------------ element loads

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// 16-byte streaming load: read once, do not keep in L1, ask L2 for 256-byte sectors.
__device__ __forceinline__ float4 ld_stream_f4(const float4 *p)
{
    float4 v;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.f32 {%0,%1,%2,%3}, [%4];"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ------------------------------------------------------------------ programmatic launch
// Every kernel waits for the preceding grid in the stream before touching memory that grid
// may write (a no-op when it was launched without the programmatic-serialisation
// attribute), then lets its successor launch: the successor's CTAs become resident as this
// grid's CTAs retire and block in their own wait until this grid has completed and
// flushed, which hides the launch gap between the small kernels of a decode step.  Every
// kernel triggers right after its own wait, so a running kernel knows that all grids
// before its immediate predecessor have completed: inputs written before that
// predecessor may be read before the wait.

// Bit i (i < 4) set when byte i of x is nonzero: the bytes' nonzero flags (0 or 1 each), times
// a constant that moves byte i's flag to bit 28 + i with no carry into those bits.
__device__ __forceinline__ uint32_t nonzero_byte_bits(uint32_t x)
{
    const uint32_t m = __vcmpne4(x, 0u) & 0x01010101u;
    return (m * 0x10204080u) >> 28;
}

// Index (0-31) of the j-th lowest set bit of x, j < popc(x): five halving steps.
__device__ __forceinline__ int select_set_bit(uint32_t x, int j)
{
    int b = 0;
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const int c = __popc((x >> b) & ((1u << w) - 1u));
        if (j >= c) {
            j -= c;
            b += w;
        }
    }
    return b;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// A load through a const __restrict__ pointer may be compiled as an invariant load, which
// the compiler is free to issue before griddepcontrol.wait (an asm with a memory clobber
// does not order it).  QSA_AFTER_WAIT(p), placed after the wait, passes p through an
// empty volatile asm: every later load through p then depends on a value produced after
// the wait.  Each kernel applies it to every pointer it reads after its wait.
#define QSA_AFTER_WAIT(p) asm volatile("" : "+l"(p))

// ------------------------------------------------------------------ mbarrier / bulk copy
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // a wait that lasts 2 s is declared lost

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait until the barrier's phase with the given parity has completed; false once the wait
// has lasted limit_ns (the caller then records an error and winds down).  limit_ns == 0:
// false at once, without looking (a way to drive the failure path on purpose).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    if (limit_ns == 0) return false;
    const uint32_t a = smem_u32(bar);
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
        if ((i & 1023) == 0) {
            const uint64_t t = global_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > limit_ns) return false;
        }
    }
}

// The same with the library's default limit (the drains that let every copy or MMA a kernel
// issued complete before it exits always use it).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    return mbar_wait(bar, parity, kWaitLimitNs);
}

// Bounded waits of one launch: where a kernel reports that a wait gave up (nullable) and the
// limit of the waits inside its pipeline, as qsa_set_wait_options() set them on the launching
// host thread.
struct WaitCtl {
    int32_t *status;
    uint64_t limit_ns;
};
WaitCtl current_wait_ctl();

__device__ __forceinline__ void report_timeout(const WaitCtl &w)
{
    if (w.status) atomicExch(reinterpret_cast<int *>(w.status), (int)QSA_ERR_TIMEOUT);
}

// One plain arrival on the barrier.
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One arrival on the barrier that also expects `bytes` more transaction bytes this phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Bulk copy global -> this CTA's shared memory, completing `bytes` transaction bytes on bar.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   cudaStream_t stream, int cluster_x, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (unsigned)n;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e == cudaErrorNotSupported || e == cudaErrorInvalidValue) {
        // a stream that does not take programmatic serialisation: launch plainly
        (void)cudaGetLastError();
        cfg.attrs = attr + 1;
        cfg.numAttrs = (unsigned)(n - 1);
        e = cudaLaunchKernelEx(&cfg, kernel, args...);
    }
    return e;
}

int device_sm_count();

// Kernel attributes are per device: raise the kernel's dynamic shared-memory limit to at
// least `smem` bytes (and, when asked, allow non-portable cluster sizes) on the current
// device, once per (kernel, device) and size.
template <auto Kernel>
cudaError_t ensure_kernel_attrs(size_t smem, bool nonportable_cluster = false)
{
    constexpr int kMaxDevices = 64;
    static std::atomic<size_t> smem_set[kMaxDevices];  // zero before first use (static)
    static std::atomic<bool> cluster_set[kMaxDevices];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = -1;
    if (dev >= 0 && smem_set[dev].load() >= smem && (!nonportable_cluster || cluster_set[dev].load()))
        return cudaSuccess;
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024)
        e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && nonportable_cluster)
        e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess && dev >= 0) {
        size_t cur = smem_set[dev].load();
        while (cur < smem && !smem_set[dev].compare_exchange_weak(cur, smem)) {
        }
        if (nonportable_cluster) cluster_set[dev].store(true);
    }
    return e;
}

// Resident CTAs of Kernel per SM for `threads` threads and `smem` dynamic bytes, on the
// current device (asked once per device; at least 1).
template <auto Kernel>
int occupancy_blocks(int threads, size_t smem)
{
    constexpr int kMaxDevices = 64;
    static std::atomic<int> blocks_of[kMaxDevices];  // 0: not yet asked
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = -1;
    int b = dev >= 0 ? blocks_of[dev].load() : 0;
    if (b > 0) return b;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, Kernel, threads, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        b = 1;
    }
    if (b < 1) b = 1;
    if (dev >= 0) blocks_of[dev].store(b);
    return b;
}

// ------------------------------------------------------------------ RoPE frequencies
// Inverse frequencies theta_i = base^(-2i/d), i < d/2, computed on the host in fp64 and
// passed by value as a kernel parameter.
constexpr int kRopeMaxHalf = 256;  // d <= 512
struct RopeTable {
    double theta[kRopeMaxHalf];
};
constexpr double kTwoPi = 6.283185307179586;
constexpr double kInvTwoPi = 0.15915494309189535;
void make_rope_table(RopeTable *tab, int d, double base);

// Storage of one pooled-cache value: fp32 as is, bf16 rounded to nearest even.
__device__ __forceinline__ float stored_value(float v, const float *) { return v; }
__device__ __forceinline__ float stored_value(float v, const __nv_bfloat16 *)
{
    return __bfloat162float(__float2bfloat16_rn(v));
}
__device__ __forceinline__ void store_pooled(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_pooled(__nv_bfloat16 *p, float v)
{
    *p = __float2bfloat16_rn(v);
}

// One pooled-key row b, computed by the whole CTA: mean of the block's present raw keys
// -> per-head RMS norm -> rotation at position 4b.  The row is stored to out_row (global,
// element type TP: fp32, or bf16 rounded to nearest even) and p_s (shared, [H*d] fp32)
// ends up holding exactly the stored values.  cs / sn: shared [d/2] scratch.  Every
// element's arithmetic is independent of the CTA size, so every kernel that calls this
// produces the same bits.  Contains __syncthreads().
template <typename T, typename TP>
__device__ __forceinline__ void pool_row(const T *__restrict__ raw, int64_t n_ctx, int H, int d,
                                         const float *__restrict__ w, float eps,
                                         const RopeTable &tab, int64_t b, float *p_s, float *cs,
                                         float *sn, TP *__restrict__ out_row)
{
    const int hd = H * d;
    const int half = d / 2;
    const int64_t t0 = 4 * b;
    const int c = (int)min((int64_t)4, n_ctx - t0);  // tokens present in this block (1..4)
    const float inv_c = 1.0f / (float)c;
    const T *rb = raw + t0 * hd;
#pragma unroll 4
    for (int e = threadIdx.x; e < hd; e += blockDim.x) {
        float v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) v[t] = t < c ? to_f32(rb[(int64_t)t * hd + e]) : 0.0f;
        p_s[e] = ((v[0] + v[1]) + (v[2] + v[3])) * inv_c;
    }
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        // the angle 4b * theta_i, formed and reduced modulo 2 pi in fp64; fp32 sincos of
        // the reduced angle (|r| <= pi)
        const double phi = (4.0 * (double)b) * tab.theta[i];
        const double k = rint(phi * kInvTwoPi);
        const float r = (float)fma(-k, kTwoPi, phi);
        float sv, cv;
        sincosf(r, &sv, &cv);
        cs[i] = cv;
        sn[i] = sv;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    for (int h = threadIdx.x >> 5; h < H; h += nwarps) {
        float *ph = p_s + h * d;
        float ss = 0.0f;
        for (int j = lane; j < d; j += 32) ss = fmaf(ph[j], ph[j], ss);
        ss = warp_sum(ss);
        const float inv = 1.0f / sqrtf(ss / (float)d + eps);
        TP *o = out_row + (int64_t)h * d;
        for (int i = lane; i < half; i += 32) {
            const float ya = ph[i] * inv * w[i];
            const float yb = ph[i + half] * inv * w[i + half];
            const float za = ya * cs[i] - yb * sn[i];
            const float zb = ya * sn[i] + yb * cs[i];
            ph[i] = stored_value(za, o);
            ph[i + half] = stored_value(zb, o);
            store_pooled(o + i, za);
            store_pooled(o + i + half, zb);
        }
    }
    __syncthreads();
}

// ------------------------------------------------------------------ launchers
// Host-side launchers, one per kernel family; arguments are already validated.

// zero_hist (nullable): a top-k histogram that the kernel clears (the launch then has at
// least one CTA even when no row needs recomputing).
// pooled: [rows][H*d] of type pdt (QSA_F32 or QSA_BF16).
cudaError_t launch_pool_update(const void *raw_k, qsa_dtype dt, int64_t n_ctx, int H, int d,
                               const float *norm_w, float eps, double rope_base,
                               void *pooled, qsa_dtype pdt, int64_t row0, int64_t row1,
                               uint32_t *zero_hist, cudaStream_t st);

// Up to this many queries share one streaming pass over the pooled cache.
constexpr int kMaxStreamQueries = 4;

// Where the decode score kernels send their results besides scores[i][b]:
// hist (nullable): per query i, rows b < n_hist[i] also enter a histogram of the top
// kTopkHistBits bits of their score key (hist + i * 2^kTopkHistBits), for the top-k's
// first radix digit.  ticket (nullable): the word ticket + i * ticket_stride (uint32
// units) is set to 0 once the kernel runs, for each query i (the decode top-k's arrival
// counters).
struct ScoreSide {
    uint32_t *hist = nullptr;
    int64_t n_hist[kMaxStreamQueries] = {0, 0, 0, 0};
    uint32_t *ticket = nullptr;
    int64_t ticket_stride = 0;
};

// Pooled-row recomputation fused into the decode score kernel (rows [row0, row1)).
struct PoolFuse {
    const void *raw;
    qsa_dtype dt;
    int64_t n_ctx;
    const float *w;
    float eps;
    int64_t row0, row1;
};
constexpr int kMaxFusedPoolRows = 4;
// Decode score kernel for n_q <= kMaxStreamQueries queries ([n_q][H*d], packed) with the
// pool update of rows [pf.row0, pf.row1) folded in, when the shape allows it (returns
// cudaErrorNotSupported otherwise, without launching).  scores [n_q][ld_scores].
cudaError_t launch_score_pool_fused(const float *q, int n_q, void *pooled, qsa_dtype pdt,
                                    int64_t n_rows, int H, int d, float scale, float *scores,
                                    int64_t ld_scores, const ScoreSide &side, const PoolFuse &pf,
                                    double rope_base, cudaStream_t st);

// pooled of type pdt.  side: see ScoreSide (hist and tickets for the decode top-k; only
// used with q_pos == NULL and n_q <= kMaxStreamQueries).
cudaError_t launch_index_score(const float *q, int64_t n_q, int64_t ld_q, const int32_t *q_pos,
                               const void *pooled, qsa_dtype pdt, int64_t n_rows, int H, int d,
                               float scale, float *scores, int64_t ld_scores,
                               const ScoreSide &side, cudaStream_t st);

qsa_status launch_index_score_tc(const float *q, int64_t n_q, int64_t ld_q,
                                 const int32_t *q_pos, const void *pooled, qsa_dtype pdt,
                                 int64_t n_rows, int H, int d, float scale, float *scores,
                                 int64_t ld_scores, void *workspace, size_t ws_bytes,
                                 cudaStream_t st);
size_t index_score_tc_workspace(int64_t n_q, int64_t n_rows, int H, int d, qsa_dtype pdt);

// Order-preserving key of a score: higher score <=> larger key.  NaN ranks as -inf;
// -0 and +0 are the same score.
__device__ __forceinline__ uint32_t score_key(float s)
{
    uint32_t u = __float_as_uint(s);
    if ((u & 0x7fffffffu) > 0x7f800000u) u = 0xff800000u;  // NaN -> -inf
    if (u == 0x80000000u) u = 0u;                           // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kTopkThreads = 1024;
constexpr int kTopkHistBits = 12;  // first radix digit: histogram of key >> 20
constexpr size_t kTopkHistBytes = sizeof(uint32_t) << kTopkHistBits;
int64_t topk_max_candidates();

// pos_out / n_cells_out (nullable): also write each query's cell list -- the selected
// blocks' 4 cells in order, then the open tail of the query.
// The position of query i: q_pos[i]; without q_pos, n_ctx - 1 - p_step * (n_q - 1 - i):
// with p_step = 1 the queries are the last n_q tokens (their candidates are then limited
// to the blocks complete at their position, as with q_pos), with p_step = 0 every query
// sits at n_ctx - 1 and every one of the n_full blocks competes.
// ext_hist (nullable): per-query histograms accumulated by the score kernel, cleared here.
cudaError_t launch_topk(const float *scores, int64_t n_q, int64_t ld, const int32_t *q_pos,
                        int64_t n_full, int64_t k_blk, int32_t *blocks_out, int32_t *counts_out,
                        int64_t n_ctx, int32_t *pos_out, int32_t *n_cells_out,
                        int64_t max_cells, uint32_t *ext_hist, cudaStream_t st,
                        int64_t p_step = 0);
// The decode form of the top-k (one query whose n_full blocks outnumber k_blk): many CTAs
// classify against the score kernel's histogram, the last to finish resolves and writes
// blocks, count, cells and tail.  scratch: topk_select_workspace_bytes(n_full) bytes,
// 256-byte aligned, whose first word (the ticket) the step's score kernel sets to 0.
// Returns cudaErrorNotSupported, without launching, when n_full <= k_blk or n_full is
// above topk_max_candidates().
// Several queries (n_q <= kMaxStreamQueries, the last n_q tokens of the context: query i
// at position n_ctx - n_q + i, candidates b < min(n_full, floor((p_i+1)/4))) run as
// grid.y = n_q: query i reads scores + i*ld_scores and hist + i*2^kTopkHistBits, uses
// the scratch at scratch + i*topk_select_workspace_bytes(n_full_cap) and writes
// blocks_out + i*k_blk, counts_out + i, pos_out + i*max_cells, n_cells_out + i.
// Returns cudaErrorNotSupported when some query has no more candidates than k_blk.
cudaError_t launch_topk_select(const float *scores, int64_t ld_scores, int n_q, int64_t n_full,
                               int64_t n_full_cap, int64_t k_blk, int64_t n_ctx, uint32_t *hist,
                               void *scratch, int32_t *blocks_out, int32_t *counts_out,
                               int32_t *pos_out, int32_t *n_cells_out, int64_t max_cells,
                               cudaStream_t st);
size_t topk_select_workspace_bytes(int64_t n_full_cap);
uint32_t *topk_select_ticket(void *scratch);

// Row blocks copied from contiguous sources to strided destinations, one per grid row (the
// host transfers of a host-fed decode step).  Every address, row size and stride must be a
// multiple of 4 bytes; src / dst may be device views of mapped host memory.
constexpr int kMaxCopyJobs = 4;
struct RowCopy {
    const void *src;
    void *dst;
    int64_t row_bytes;  // bytes per row, rows contiguous in the source
    int64_t dst_ld;     // bytes between rows in the destination
    int64_t rows;
};
cudaError_t launch_copy_rows(const RowCopy *jobs, int n_jobs, cudaStream_t st);

// The address through which kernels on the current device reach host buffer h, or NULL
// when h is not page-locked memory mapped for it (pageable memory, another device's).
void *mapped_host_view(const void *h);

// cells[i][c] = scores[i][c / 4] for c < 4 * n_full (the pre-block-domain selection input).
cudaError_t launch_expand_scores(const float *scores, int64_t n_q, int64_t ld_s, int64_t n_full,
                                 float *cells, int64_t ld_c, cudaStream_t st);

cudaError_t launch_gather(const void *K, const void *V, qsa_dtype dt, int64_t n_kv, int H_kv,
                          int d_k, int d_v, int64_t ld_k, int64_t ld_v, const int32_t *blocks,
                          const int32_t *counts, int64_t n_q, int64_t k_blk,
                          const int32_t *q_pos, int64_t n_ctx, void *K_out, void *V_out,
                          int32_t *pos_out, int32_t *n_cells_out, int64_t max_cells,
                          cudaStream_t st);

// Many queries (a prefill chunk) of the bf16 128-dim form with 4 KV heads x 8 query heads
// and a position list: one CTA per query stages whole cell rows (all four heads).
bool attn_uses_rows4(qsa_dtype dt, int64_t n_q, int H_q, int H_kv, int d_k, int d_v,
                     const void *K, const void *V, int64_t ld_k, int64_t ld_v,
                     const int32_t *pos, int64_t max_cells);
cudaError_t launch_attn_rows4(const float *q, int64_t n_q, int H_q, float scale, const void *K,
                              const void *V, int64_t n_kv, int64_t ld_k, int64_t ld_v,
                              const int32_t *pos, const int32_t *n_cells, int64_t max_cells,
                              float *out, float *lse, cudaStream_t st);
// The latent-KV form (bf16, DKQ 576, d_v 512, 16 query heads per KV head, V the first
// 512 columns of each K row: K == V, same stride) has its own tensor-core kernel.
bool attn_uses_wide(qsa_dtype dt, int d_k, int d_v, int G, const void *K, const void *V,
                    int64_t ld_k, int64_t ld_v);
cudaError_t launch_attn_wide(const float *q, int64_t n_q, int H_q, int H_kv, float scale,
                             const void *KV, int64_t n_kv, int64_t ld, const int32_t *pos,
                             const int32_t *n_cells, int64_t max_cells, float *out, float *lse,
                             cudaStream_t st);
// The same kernel listing each query's cells from its mask row itself (rows of at most
// attn_wide_mask_max_kv() positions); counts_out (nullable) gets each row's true count.
int64_t attn_wide_mask_max_kv();
cudaError_t launch_attn_wide_mask(const float *q, int64_t n_q, int H_q, int H_kv, float scale,
                                  const void *KV, int64_t n_kv, int64_t ld, const uint8_t *mask,
                                  int64_t ld_mask, int64_t max_list, int32_t *counts_out,
                                  float *out, float *lse, cudaStream_t st);
int attn_num_splits(int64_t n_q, int H_kv, int64_t max_cells);
size_t attn_smem_bytes_host(int G, int d_k, int d_v, int esize);
size_t attn_workspace_bytes(int64_t n_q, int H_q, int H_kv, int d_v, int64_t max_cells);
// Split-K scratch the path launch_sparse_attn takes for these arguments really uses: 0 for
// the forms that merge their splits inside a cluster (rows4, latent, bf16 8-head mma),
// attn_workspace_bytes() otherwise.
size_t attn_partials_bytes(qsa_dtype dt, int64_t n_q, int H_q, int H_kv, int d_k, int d_v,
                           const void *K, const void *V, int64_t ld_k, int64_t ld_v,
                           const int32_t *pos, int64_t max_cells);
cudaError_t launch_sparse_attn(const float *q, int64_t n_q, int H_q, int H_kv, int d_k, int d_v,
                               float scale, const void *K, const void *V, qsa_dtype dt,
                               int64_t n_kv, int64_t ld_k, int64_t ld_v, const int32_t *pos,
                               const int32_t *n_cells, int64_t max_cells, float *out,
                               float *lse, float *partials, cudaStream_t st,
                               bool early_q = false,  // q written before the predecessor
                               float *out_host = nullptr, float *lse_host = nullptr);
// (out_host / lse_host: device views of page-locked host buffers that also receive out /
// lse; only the bf16 8-head tensor-core form writes them, attn_writes_host() says when.)
bool attn_writes_host(qsa_dtype dt, int64_t n_q, int H_q, int H_kv, int d_k, int d_v,
                      const void *K, const void *V, int64_t ld_k, int64_t ld_v,
                      const int32_t *pos, int64_t max_cells);

cudaError_t launch_mask_to_list(const uint8_t *mask, int64_t n_rows, int64_t n_kv,
                                int64_t ld_mask, int64_t max_list, int32_t *pos_out,
                                int32_t *counts_out, uint64_t *bits_out, cudaStream_t st);

}  // namespace qsa
