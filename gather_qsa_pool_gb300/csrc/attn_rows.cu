// attn_rows.cu -- sparse attention of one query over its listed cells for all four KV heads
// at once (bf16, head dim 128, 8 query heads per KV head), one CTA per query: the form the
// prefill chunk takes, where 1024 queries each attend over their own ~2051 cells.
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "selected K/V gather (COMMON-005)" (attention over the gathered rows of the selected
// cells) applied per query of a chunk; the pages leave prefill on the dense path.
//
// A listed cell's K row holds the four KV heads contiguously (1 KB in bf16), and so does its
// V row: one bulk copy per row and tensor stages all four heads, four times fewer requests
// than one copy per KV head.  The query's whole position list is read into shared memory
// first, so no stage waits on a position load.  Cells go in
// stages of 32, three stages in flight; warp w works on KV head w/2 and on cells
// 16*(w%2) .. +15 of each stage, with the same tensor-core arithmetic as the per-head
// kernel (mma.m16n8k16 over the two bf16 halves of the query and of P).  The two warps of
// a head merge their online-softmax states at the end.  Rows are padded to 1040 bytes so
// that the eight rows of every ldmatrix fall in distinct banks.
#include "mma_frag.cuh"

namespace qsa {
namespace {

constexpr int kRHkv = 4;               // KV heads
constexpr int kRG = 8;                 // query heads per KV head
constexpr int kRD = 128;               // head dim
constexpr int kRWarps = 8;             // two per KV head
constexpr int kRNT = 32 * kRWarps;
constexpr int kRTC = 32;               // cells per stage
constexpr int kRStages = 3;
constexpr int kRRow = kRHkv * kRD;     // bf16 elements of one cell row (all heads)
constexpr int kRLD = kRRow + 8;        // padded row: 1040 bytes
constexpr size_t kRStageBytes = (size_t)kRTC * kRLD * 2;
constexpr int kRMaxList = 4096;        // the query's whole position list stays in shared memory
constexpr size_t kRSmem = 2 * kRStages * kRStageBytes + (size_t)kRMaxList * 4;
static_assert((size_t)kRWarps * kRG * (kRD + 2) * 4 <= kRSmem, "merge area fits the stages");
static_assert(2 * kRTC <= kRNT, "one thread per row and tensor of a stage");

__global__ void __launch_bounds__(kRNT, 1)
attn_rows4_kernel(const float *__restrict__ q, int H_q, float scale_log2,
                  const __nv_bfloat16 *__restrict__ K, const __nv_bfloat16 *__restrict__ V,
                  int64_t n_kv, int64_t ld_k, int64_t ld_v, const int32_t *__restrict__ pos,
                  const int32_t *__restrict__ n_cells, int64_t max_cells,
                  float *__restrict__ out, float *__restrict__ lse)
{
    constexpr int G = kRG, D = kRD, TC = kRTC, LD = kRLD, NS = kRStages, NT = kRNT;
    extern __shared__ __align__(16) char smem_raw[];
    __nv_bfloat16 *Ks = reinterpret_cast<__nv_bfloat16 *>(smem_raw);       // [NS][TC][LD]
    __nv_bfloat16 *Vs = Ks + (size_t)NS * TC * LD;                          // [NS][TC][LD]
    float *mrg = reinterpret_cast<float *>(smem_raw);  // [warps][G][D + 2], after the loop
    int32_t *plist_s = reinterpret_cast<int32_t *>(smem_raw + 2 * NS * kRStageBytes);  // [n]
    __shared__ int32_t rows[NS * TC];
    __shared__ __align__(8) uint64_t sbar[NS];

    const int64_t qi = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = warp >> 1, half = warp & 1;  // KV head, cell half of each stage
    const int hr = lane >> 2, qc = (lane & 3) * 2;
    const int mi = lane >> 3, mj = lane & 7;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&sbar[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_wait();
    QSA_AFTER_WAIT(q);
    QSA_AFTER_WAIT(K);
    QSA_AFTER_WAIT(V);
    QSA_AFTER_WAIT(pos);
    QSA_AFTER_WAIT(n_cells);
    pdl_trigger();

    // A fragments of this warp's KV head's 8 query heads: rows 0-7 hi, rows 8-15 lo
    uint32_t qa[8][4];
    {
        const float *qh = q + (qi * H_q + (int64_t)g * G + hr) * D;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const float2 x0 = *reinterpret_cast<const float2 *>(qh + ks * 16 + qc);
            const float2 x1 = *reinterpret_cast<const float2 *>(qh + ks * 16 + 8 + qc);
            float h0, l0, h1, l1, h2, l2, h3, l3;
            split_bf16(x0.x * scale_log2, h0, l0);
            split_bf16(x0.y * scale_log2, h1, l1);
            split_bf16(x1.x * scale_log2, h2, l2);
            split_bf16(x1.y * scale_log2, h3, l3);
            qa[ks][0] = pack_bf16(h0, h1);
            qa[ks][1] = pack_bf16(l0, l1);
            qa[ks][2] = pack_bf16(h2, h3);
            qa[ks][3] = pack_bf16(l2, l3);
        }
    }
    float o[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;
    float m = -INFINITY, lsum = 0.0f;

    // the list length and the whole position list (up to kRMaxList entries, checked by the
    // launcher) in one round trip; entries past the length are dropped once it arrives
    int64_t n = n_cells[qi];
    const int32_t *plist = pos + qi * max_cells;
    int32_t pre[kRMaxList / kRNT];
#pragma unroll
    for (int j = 0; j < kRMaxList / kRNT; ++j) {
        const int e = j * NT + tid;
        pre[j] = e < max_cells ? plist[e] : -1;
    }
    const bool overflow = n > max_cells;  // truncated list: the result must not be used
    if (overflow || n < 0) n = 0;
    const int ntiles = (int)((n + TC - 1) / TC);
#pragma unroll
    for (int j = 0; j < kRMaxList / kRNT; ++j) {
        const int e = j * NT + tid;
        int64_t row = e < n ? pre[j] : -1;
        if (row < 0 || row >= n_kv) row = -1;
        plist_s[e] = (int32_t)row;
    }
    __syncthreads();
    if (tid < NS * TC) rows[tid] = plist_s[tid];
    __syncthreads();

    uint32_t sphase = 0;
    bool lost = false;
    uint32_t lost_at = 0;
    auto load_rows = [&](int it, int buf) {
        if (tid < TC) rows[buf * TC + tid] = plist_s[it * TC + tid];
        __syncthreads();
    };
    // one bulk copy per listed row and tensor (all four heads, 1 KB); the V rows of skipped
    // slots are zero-filled (P = 0 multiplies them; stale data could hold a NaN pattern)
    auto copy_rows = [&](int buf) {
        const int32_t *rb = rows + buf * TC;
        __nv_bfloat16 *ks = Ks + (size_t)buf * TC * LD;
        __nv_bfloat16 *vs = Vs + (size_t)buf * TC * LD;
        for (int e = tid; e < TC * (kRRow / 8); e += NT) {
            const int slot = e / (kRRow / 8), c = e - slot * (kRRow / 8);
            if (rb[slot] < 0) *reinterpret_cast<uint4 *>(vs + slot * LD + c * 8) = make_uint4(0u, 0u, 0u, 0u);
        }
        const int nv = __syncthreads_count(tid < TC && rb[tid] >= 0);
        if (tid == 0) mbar_arrive_expect_tx(&sbar[buf], (uint32_t)nv * 2u * kRRow * 2u);
        if (tid < 2 * TC) {
            const int slot = tid >> 1;
            const int64_t row = rb[slot];
            if (row >= 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                if (tid & 1) bulk_g2s(vs + slot * LD, V + row * ld_v, kRRow * 2, &sbar[buf]);
                else bulk_g2s(ks + slot * LD, K + row * ld_k, kRRow * 2, &sbar[buf]);
            }
        }
    };
    auto wait_rows = [&](int buf) {
        if (!lost && !mbar_wait(&sbar[buf], (sphase >> buf) & 1u)) {
            lost = true;
            lost_at = (uint32_t)buf | (((sphase >> buf) & 1u) << 2);
        }
        sphase ^= 1u << buf;
        __syncthreads();
    };

    for (int s = 0; s < NS && s < ntiles; ++s) copy_rows(s);
    for (int it = 0; it < ntiles; ++it) {
        const int buf = it % NS;
        if (it >= 1 && it + NS - 1 < ntiles) {
            const int nb = (it + NS - 1) % NS;  // consumed at iteration it - 1
            load_rows(it + NS - 1, nb);
            copy_rows(nb);
        }
        wait_rows(buf);
        const int tc = (int)min((int64_t)TC, n - (int64_t)it * TC);
        const __nv_bfloat16 *ks = Ks + (size_t)buf * TC * LD + g * D;
        const __nv_bfloat16 *vs = Vs + (size_t)buf * TC * LD + g * D;
        const int32_t *rw = rows + buf * TC;
        const int s0 = half * 16;
        if (s0 < tc) {
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t b[4];
                const int cell = s0 + (mi >> 1) * 8 + mj;
                ldsm_x4(b, ks + cell * LD + kk * 16 + (mi & 1) * 8);
                mma_16816(sc[0], qa[kk], b[0], b[1]);
                mma_16816(sc[1], qa[kk], b[2], b[3]);
            }
            float x[4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int slot = s0 + nt * 8 + qc + u;
                    const bool ok = slot < tc && rw[slot] >= 0;
                    x[nt * 2 + u] = ok ? sc[nt][u] + sc[nt][u + 2] : -INFINITY;
                }
            }
            float cmax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
            cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 1));
            cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 2));
            const float m_new = fmaxf(m, cmax);
            const bool live = m_new != -INFINITY;
            if (__any_sync(0xffffffffu, live)) {
                const float alpha = live ? exp2f(m - m_new) : 1.0f;
                float p[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) p[u] = live ? exp2f(x[u] - m_new) : 0.0f;
                if (live) {
                    lsum = lsum * alpha + ((p[0] + p[1]) + (p[2] + p[3]));
                    m = m_new;
                }
                if (alpha != 1.0f) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        o[j][0] *= alpha;
                        o[j][1] *= alpha;
                        o[j][2] *= alpha;
                        o[j][3] *= alpha;
                    }
                }
                float ph[4], pl[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) split_bf16(p[u], ph[u], pl[u]);
                uint32_t pa[4];
                pa[0] = pack_bf16(ph[0], ph[1]);
                pa[1] = pack_bf16(pl[0], pl[1]);
                pa[2] = pack_bf16(ph[2], ph[3]);
                pa[3] = pack_bf16(pl[2], pl[3]);
#pragma unroll
                for (int dp = 0; dp < 8; ++dp) {
                    uint32_t b[4];
                    const int cell = s0 + (mi & 1) * 8 + mj;
                    ldsm_x4_t(b, vs + cell * LD + dp * 16 + (mi >> 1) * 8);
                    mma_16816(o[2 * dp], pa, b[0], b[1]);
                    mma_16816(o[2 * dp + 1], pa, b[2], b[3]);
                }
            }
        }
        __syncthreads();  // this stage is refilled by a later copy
    }
    lost = __syncthreads_or(lost);

    // per-warp states -> shared memory (the stage area is free now), then the two warps of
    // each KV head merge into the output
    {
        float l4 = lsum;
        l4 += __shfl_xor_sync(0xffffffffu, l4, 1);
        l4 += __shfl_xor_sync(0xffffffffu, l4, 2);
        float *mw = mrg + ((size_t)warp * G + hr) * (D + 2);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            mw[8 * j + qc] = o[j][0] + o[j][2];
            mw[8 * j + qc + 1] = o[j][1] + o[j][3];
        }
        if ((lane & 3) == 0) {
            mw[D] = m;
            mw[D + 1] = l4;
        }
    }
    __syncthreads();
    for (int e = tid; e < kRHkv * G * D; e += NT) {
        const int hq = e / D, c = e - hq * D;  // query head of this query, dim
        const int gg = hq / G, h = hq - gg * G;
        const float *r0 = mrg + ((size_t)(2 * gg) * G + h) * (D + 2);
        const float *r1 = mrg + ((size_t)(2 * gg + 1) * G + h) * (D + 2);
        const float M = fmaxf(r0[D], r1[D]);
        float acc = 0.0f, L = 0.0f;
        if (M != -INFINITY) {
            const float f0 = exp2f(r0[D] - M), f1 = exp2f(r1[D] - M);
            acc = fmaf(f0, r0[c], f1 * r1[c]);
            L = fmaf(f0, r0[D + 1], f1 * r1[D + 1]);
        }
        float v = L > 0.0f ? acc / L : 0.0f;
        if (overflow || lost) v = __int_as_float(0x7fc00000);
        out[(qi * H_q + hq) * (int64_t)D + c] = v;
        if (lse && c == 0)
            lse[qi * H_q + hq] = (overflow || lost) ? __int_as_float(0x7fc00000)
                                 : (L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY);
    }
    if (lost) (void)mbar_wait(&sbar[lost_at & 3u], lost_at >> 2);
}

}  // namespace

bool attn_uses_rows4(qsa_dtype dt, int64_t n_q, int H_q, int H_kv, int d_k, int d_v,
                     const void *K, const void *V, int64_t ld_k, int64_t ld_v,
                     const int32_t *pos, int64_t max_cells)
{
    return dt == QSA_BF16 && H_kv == kRHkv && H_q == kRHkv * kRG && d_k == kRD && d_v == kRD &&
           pos != nullptr && n_q * H_kv >= kTargetSMs && ld_k >= kRRow && ld_v >= kRRow &&
           max_cells <= kRMaxList &&
           (ld_k * 2) % 16 == 0 && (ld_v * 2) % 16 == 0 &&
           ((reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V)) & 15) == 0;
}

cudaError_t launch_attn_rows4(const float *q, int64_t n_q, int H_q, float scale, const void *K,
                              const void *V, int64_t n_kv, int64_t ld_k, int64_t ld_v,
                              const int32_t *pos, const int32_t *n_cells, int64_t max_cells,
                              float *out, float *lse, cudaStream_t st)
{
    const cudaError_t e = ensure_kernel_attrs<attn_rows4_kernel>(kRSmem);
    if (e != cudaSuccess) return e;
    return launch(attn_rows4_kernel, dim3((unsigned)n_q), dim3(kRNT), kRSmem, st, 1, q, H_q,
                  scale * kLog2e, (const __nv_bfloat16 *)K, (const __nv_bfloat16 *)V, n_kv, ld_k,
                  ld_v, pos, n_cells, max_cells, out, lse);
}

}  // namespace qsa
