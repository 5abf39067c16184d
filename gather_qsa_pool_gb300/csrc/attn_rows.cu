// attn_rows.cu -- sparse attention of one query over its listed cells for all four KV heads
// at once (bf16, head dim 128, 8 query heads per KV head), one CTA per query: the form the
// prefill chunk takes, where 1024 queries each attend over their own ~2051 cells.
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "selected K/V gather (COMMON-005)" (attention over the gathered rows of the selected
// cells) applied per query of a chunk; the pages leave prefill on the dense path.
//
// Warp-specialised: a producer warp streams the listed K and V rows into a ring of three
// 32-cell stages while eight consumer warps compute, the two sides handing stages over
// through per-stage full / empty barriers (no block-wide barrier in the loop).  A listed
// cell's K row holds the four KV heads contiguously (1 KB in bf16), and so does its V row.
// The selection lists whole 4-token blocks, so a stage is eight groups of four cells, and a
// group whose four cells are consecutive rows of a contiguous cache is one 4 KB bulk copy
// (four times fewer copies than one per row; the copy engine, not the memory, limits how
// fast rows arrive); other groups take one copy per row.  Groups sit 4 KB + 16 bytes apart in
// shared memory, so the eight cells an ldmatrix reads -- the same row of eight groups -- fall
// in distinct banks.  The query's whole position list is read into shared memory first.
// Consumer warp w works on KV head w/2 and on rows 2*(w%2), 2*(w%2)+1 of every group of a
// stage (16 cells), with mma.m16n8k16 over the two bf16 halves of the query and of P; the two
// warps of a head merge their online-softmax states at the end.
#include "mma_frag.cuh"

namespace qsa {
namespace {

constexpr int kRHkv = 4;               // KV heads
constexpr int kRG = 8;                 // query heads per KV head
constexpr int kRD = 128;               // head dim
constexpr int kRWarps = 8;             // consumer warps, two per KV head
constexpr int kRNT = 32 * kRWarps;     // consumer threads
constexpr int kRThreads = kRNT + 32;   // plus the producer warp
constexpr int kRTC = 32;               // cells per stage: eight groups of four
constexpr int kRGroups = kRTC / 4;
constexpr int kRStages = 3;
constexpr int kRRow = kRHkv * kRD;     // bf16 elements of one cell row (all heads)
constexpr int kRGroupElems = 4 * kRRow + 8;               // 4 KB + 16 bytes
constexpr int kRStageElems = kRGroups * kRGroupElems;     // one tensor's stage
constexpr size_t kRStageBytes = (size_t)kRStageElems * 2;
constexpr int kRMaxList = 4096;        // the query's whole position list stays in shared memory
constexpr size_t kRSmem = 2 * kRStages * kRStageBytes + (size_t)kRMaxList * 4;
static_assert((size_t)kRHkv * kRG * (kRD + 2) * 4 <= 2 * kRStages * kRStageBytes,
              "merge area fits the stages");
static_assert(kRMaxList % kRNT == 0, "the list is read in whole rounds");

__global__ void __launch_bounds__(kRThreads, 1)
attn_rows4_kernel(const float *__restrict__ q, int H_q, float scale_log2,
                  const __nv_bfloat16 *__restrict__ K, const __nv_bfloat16 *__restrict__ V,
                  int64_t n_kv, int64_t ld_k, int64_t ld_v, const int32_t *__restrict__ pos,
                  const int32_t *__restrict__ n_cells, int64_t max_cells,
                  float *__restrict__ out, float *__restrict__ lse, const WaitCtl wc)
{
    constexpr int G = kRG, D = kRD, TC = kRTC, NS = kRStages, NT = kRNT;
    constexpr int GE = kRGroupElems, SE = kRStageElems;
    extern __shared__ __align__(16) char smem_raw[];
    __nv_bfloat16 *Ks = reinterpret_cast<__nv_bfloat16 *>(smem_raw);       // [NS][8][GE]
    __nv_bfloat16 *Vs = Ks + (size_t)NS * SE;                               // [NS][8][GE]
    float *mrg = reinterpret_cast<float *>(smem_raw);  // [KV heads][G][D + 2], after the loop
    int32_t *plist_s = reinterpret_cast<int32_t *>(smem_raw + 2 * NS * kRStageBytes);  // [4096]
    __shared__ __align__(8) uint64_t full[NS];
    __shared__ __align__(8) uint64_t empty[NS];

    const int64_t qi = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);          // the producer's arrival (+ the copies' bytes)
            mbar_init(&empty[s], kRWarps);   // one arrival per consumer warp
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_wait();
    QSA_AFTER_WAIT(q);
    QSA_AFTER_WAIT(K);
    QSA_AFTER_WAIT(V);
    QSA_AFTER_WAIT(pos);
    QSA_AFTER_WAIT(n_cells);
    pdl_trigger();

    // the list length and the whole position list (up to kRMaxList entries, checked by the
    // launcher) in one round trip; entries past the length, or outside the cache, become -1
    int64_t n = n_cells[qi];
    int32_t pre[kRMaxList / kRNT];
    if (tid < NT) {
        const int32_t *plist = pos + qi * max_cells;
#pragma unroll
        for (int j = 0; j < kRMaxList / kRNT; ++j) {
            const int e = j * NT + tid;
            pre[j] = e < max_cells ? plist[e] : -1;
        }
    }
    const bool overflow = n > max_cells;  // truncated list: the result must not be used
    if (overflow || n < 0) n = 0;
    const int ntiles = (int)((n + TC - 1) / TC);
    if (tid < NT) {
#pragma unroll
        for (int j = 0; j < kRMaxList / kRNT; ++j) {
            const int e = j * NT + tid;
            const int64_t row = e < n ? pre[j] : -1;
            plist_s[e] = (row < 0 || row >= n_kv) ? -1 : (int32_t)row;
        }
    }
    __syncthreads();

    bool lost = false;
    if (warp == kRWarps) {
        // ---- producer: lanes 0-7 copy the K rows of group `lane` of each stage, lanes 8-15
        // the V rows; V rows of empty slots are zeroed (P = 0 multiplies them, and stale data
        // could hold a NaN pattern)
        const int j = lane & 7;
        const bool act = lane < 16, isv = lane >= 8;
        const __nv_bfloat16 *src = isv ? V : K;
        const int64_t ldt = isv ? ld_v : ld_k;
        const bool runs = ldt == kRRow;  // consecutive rows are one contiguous run
        int armed = 0;
        for (int it = 0; it < ntiles; ++it, ++armed) {
            const int s = it % NS;
            const uint32_t use = (uint32_t)(it / NS);
            bool ok = use == 0 || mbar_wait(&empty[s], (use - 1) & 1u, wc.limit_ns);
            if (!__all_sync(0xffffffffu, ok)) {
                lost = true;
                break;
            }
            __nv_bfloat16 *dst = (isv ? Vs : Ks) + (size_t)s * SE + j * GE;
            int32_t p[4];
            int nv = 0;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                p[r] = plist_s[it * TC + j * 4 + r];
                nv += p[r] >= 0;
            }
            const bool whole = runs && nv == 4 && p[1] == p[0] + 1 && p[2] == p[0] + 2 &&
                               p[3] == p[0] + 3;
            if (act && isv)
#pragma unroll 1
                for (int r = 0; r < 4; ++r)
                    if (p[r] < 0)
                        for (int c = 0; c < kRRow / 8; ++c)
                            *reinterpret_cast<uint4 *>(dst + r * kRRow + c * 8) =
                                make_uint4(0u, 0u, 0u, 0u);
            const uint32_t bytes =
                __reduce_add_sync(0xffffffffu, act ? (uint32_t)nv * kRRow * 2u : 0u);
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&full[s], bytes);
            __syncwarp();
            if (act) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                if (whole) {
                    bulk_g2s(dst, src + (int64_t)p[0] * ldt, 4 * kRRow * 2, &full[s]);
                } else {
#pragma unroll 1
                    for (int r = 0; r < 4; ++r)
                        if (p[r] >= 0)
                            bulk_g2s(dst + r * kRRow, src + (int64_t)p[r] * ldt, kRRow * 2,
                                     &full[s]);
                }
            }
        }
        // every copy issued lands before the CTA leaves: the last phase armed on each stage
        // (a stage is re-armed only after every consumer saw its previous phase complete, so
        // no earlier phase can be outstanding)
        if (lane == 0)
            for (int s = 0; s < NS && s < armed; ++s) {
                const int uses = armed / NS + (s < armed % NS ? 1 : 0);
                (void)mbar_wait(&full[s], (uint32_t)(uses - 1) & 1u);
            }
    } else {
        // ---- consumers
        const int g = warp >> 1, half = warp & 1;  // KV head; rows 2*half, 2*half+1 of groups
        const int hr = lane >> 2, qc = (lane & 3) * 2;
        const int mi = lane >> 3, mj = lane & 7;
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
        for (int jj = 0; jj < 16; ++jj) o[jj][0] = o[jj][1] = o[jj][2] = o[jj][3] = 0.0f;
        float m = -INFINITY, lsum = 0.0f;
        // n-tile t of this warp = row 2*half + t of the stage's eight groups; column c of a
        // tile = group c.  ldmatrix lane addresses: group mj, tile / k-half from mi.
        const int krow = (2 * half + (mi >> 1)) * kRRow + g * D + (mi & 1) * 8;
        const int vrow = (2 * half + (mi & 1)) * kRRow + g * D + (mi >> 1) * 8;

        for (int it = 0; it < ntiles; ++it) {
            const int s = it % NS;
            const bool ok = !lost && mbar_wait(&full[s], (uint32_t)(it / NS) & 1u, wc.limit_ns);
            if (!__all_sync(0xffffffffu, ok)) lost = true;
            // a warp that gave up neither reads the stage (copies may still be landing) nor
            // releases it, so the producer stops too
            if (lost) continue;
            const __nv_bfloat16 *kst = Ks + (size_t)s * SE + mj * GE + krow;
            const __nv_bfloat16 *vst = Vs + (size_t)s * SE + mj * GE + vrow;
            // two accumulator chains per tile (even / odd k steps) halve the MMA dependency
            float sc[2][2][4] = {};
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t b[4];
                ldsm_x4(b, kst + kk * 16);
                mma_16816(sc[0][kk & 1], qa[kk], b[0], b[1]);
                mma_16816(sc[1][kk & 1], qa[kk], b[2], b[3]);
            }
            float x[4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int li = it * TC + (qc + u) * 4 + 2 * half + nt;  // list index
                    const bool valid = li < n && plist_s[li] >= 0;
                    const float hi = sc[nt][0][u] + sc[nt][1][u];
                    const float lo = sc[nt][0][u + 2] + sc[nt][1][u + 2];
                    x[nt * 2 + u] = valid ? hi + lo : -INFINITY;
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
                    for (int jj = 0; jj < 16; ++jj) {
                        o[jj][0] *= alpha;
                        o[jj][1] *= alpha;
                        o[jj][2] *= alpha;
                        o[jj][3] *= alpha;
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
                    ldsm_x4_t(b, vst + dp * 16);
                    mma_16816(o[2 * dp], pa, b[0], b[1]);
                    mma_16816(o[2 * dp + 1], pa, b[2], b[3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage
        }
        // per-warp state, kept in registers until every warp has left the ring; the second
        // warp of each KV head leaves its state in shared memory, the first merges it with
        // its own in registers and writes the head group's outputs
        __syncthreads();
        float l4 = lsum;
        l4 += __shfl_xor_sync(0xffffffffu, l4, 1);
        l4 += __shfl_xor_sync(0xffffffffu, l4, 2);
        float *mw = mrg + ((size_t)g * G + hr) * (D + 2);
        if (half == 1) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                mw[8 * jj + qc] = o[jj][0] + o[jj][2];
                mw[8 * jj + qc + 1] = o[jj][1] + o[jj][3];
            }
            if ((lane & 3) == 0) {
                mw[D] = m;
                mw[D + 1] = l4;
            }
        }
        lost = __syncthreads_or(lost);  // also orders those writes before the reads below
        if (half == 0) {
            const float m1 = mw[D], l1 = mw[D + 1];
            const float M = fmaxf(m, m1);
            float f0 = 0.0f, f1 = 0.0f, L = 0.0f;
            if (M != -INFINITY) {
                f0 = exp2f(m - M);
                f1 = exp2f(m1 - M);
                L = fmaf(f0, l4, f1 * l1);
            }
            const int64_t hq = qi * H_q + (int64_t)g * G + hr;
            float *orow = out + hq * D;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const float r0 = o[jj][u] + o[jj][u + 2];
                    const float acc =
                        M != -INFINITY ? fmaf(f0, r0, f1 * mw[8 * jj + qc + u]) : 0.0f;
                    float v = L > 0.0f ? acc / L : 0.0f;
                    if (overflow || lost) v = __int_as_float(0x7fc00000);
                    orow[8 * jj + qc + u] = v;
                }
            }
            if (lse && (lane & 3) == 0)
                lse[hq] = (overflow || lost) ? __int_as_float(0x7fc00000)
                          : (L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY);
        }
    }
    if (warp == kRWarps) {
        __syncthreads();                // pairs with the consumers' two barriers above
        lost = __syncthreads_or(lost);
        if (lost && lane == 0) report_timeout(wc);
    }
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
    return launch(attn_rows4_kernel, dim3((unsigned)n_q), dim3(kRThreads), kRSmem, st, 1, q, H_q,
                  scale * kLog2e, (const __nv_bfloat16 *)K, (const __nv_bfloat16 *)V, n_kv, ld_k,
                  ld_v, pos, n_cells, max_cells, out, lse, current_wait_ctl());
}

}  // namespace qsa
