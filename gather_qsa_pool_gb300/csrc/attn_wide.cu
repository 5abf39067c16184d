// attn_wide.cu -- sparse attention of 16 query heads on one latent KV head: DKQ 576,
// d_v 512, V the first 512 columns of each K row (one row read serves both), bf16.
//
// Source: devotd.net, "llama.cpp CDNA sparse attention", sections 2-3: the sparse
// matrix-op kernel attends the 16 query columns of one KV group only over the key positions
// listed from the mask (DKQ 576 / ncols2 16 on the pages' model).
//
// Grid (S, H_kv, n_q): the S CTAs of one (query, KV head) split the list and, for S > 1,
// form a thread-block cluster that merges their (o, m, l) states in distributed shared
// memory.  A CTA walks its cells in stages of 64: one bulk copy per cell brings the
// 1152-byte row into shared memory (rows padded to 1168 bytes so that ldmatrix rows fall
// in distinct banks), counted on the stage's mbarrier.  Per stage:
//   S = Q K^T  -- warp w takes cells 8w..8w+7: 36 k-steps of mma.m16n8k16 over the two
//                 halves of the query (bf16 rounding of the pre-scaled query in one
//                 16-row tile, the bf16 rounding of the remainder in the other);
//   softmax    -- per-head maxima and sums meet in shared memory; P is written there as
//                 bf16 hi / lo halves;
//   O += P V   -- warp w owns output dims 64w..64w+63 for all 16 heads: 4 k-steps over
//                 the 64 cells x 8 n-tiles, hi and lo halves of P into one accumulator.
// K and V are exact bf16, so only the query and P are rounded (to ~2^-17 relative).
#include "mma_frag.cuh"

#include <cooperative_groups.h>

namespace cg = cooperative_groups;

namespace qsa {
namespace {

constexpr int kWG = 16;           // query heads per KV head
constexpr int kWDK = 576;         // key / query head dim
constexpr int kWDV = 512;         // value head dim (the first columns of the key row)
constexpr int kWWarps = 8;
constexpr int kWNT = 32 * kWWarps;
constexpr int kWTC = 64;          // cells per stage (8 per warp for Q K^T)
constexpr int kWLD = kWDK + 8;    // padded row, bf16 elements (1168 bytes)
constexpr int kWPLD = kWTC + 8;   // padded P row, bf16 elements
constexpr int kWOLD = kWDV + 4;   // padded output-state row, floats
constexpr int kWMaxCluster = 16;

// shared memory: Q hi/lo [32][kWLD] | rows [2][kWTC] stages [2][kWTC][kWLD] | P [32][kWPLD]
constexpr size_t kWQBytes = 32 * (size_t)kWLD * 2;
constexpr size_t kWStageBytes = (size_t)kWTC * kWLD * 2;
constexpr size_t kWPBytes = 32 * (size_t)kWPLD * 2;
constexpr size_t kWSmem = kWQBytes + 2 * kWStageBytes + kWPBytes;
static_assert((size_t)kWG * kWOLD * 4 <= 2 * kWStageBytes, "output state fits the stages");
static_assert(kWQBytes % 16 == 0 && kWStageBytes % 16 == 0, "16-byte aligned regions");

// Mask mode: the mask row's 64-bit ballot words (bit t of word w: position 64w + t is set)
// and their exclusive prefix counts, built by every CTA of the query in shared memory; the
// list index L is the L-th set position in ascending order, the list the separate
// mask-to-list call writes.  Rows of up to kWMaskWords * 64 positions.
constexpr int kWMaskWords = 1024;
constexpr int kWWordsPerThread = kWMaskWords / kWNT;  // 4

// Builds words[0, nw) and pre[0, nw) of one mask row (all threads call it); returns the
// row's set-position count.  Thread t owns words [t * wpt, (t + 1) * wpt).
__device__ int64_t build_mask_words(const uint8_t *__restrict__ row, int64_t n_kv,
                                    unsigned long long *words, uint32_t *pre, uint32_t *wsum)
{
    constexpr int NT = kWNT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nw = (int)((n_kv + 63) / 64);
    const int wpt = (nw + NT - 1) / NT;  // <= kWWordsPerThread
    const int w0 = tid * wpt;
    unsigned long long wv[kWWordsPerThread];
    const bool vec = n_kv % 64 == 0 && (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    if (vec) {
        // whole words: four 16-byte loads per word, all of the thread's loads in flight
        uint4 u[kWWordsPerThread][4];
#pragma unroll
        for (int i = 0; i < kWWordsPerThread; ++i)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                u[i][k] = (i < wpt && w0 + i < nw)
                              ? reinterpret_cast<const uint4 *>(row + 64 * (int64_t)(w0 + i))[k]
                              : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int i = 0; i < kWWordsPerThread; ++i) {
            unsigned long long w = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                w |= (unsigned long long)nonzero_byte_bits(u[i][k].x) << (16 * k);
                w |= (unsigned long long)nonzero_byte_bits(u[i][k].y) << (16 * k + 4);
                w |= (unsigned long long)nonzero_byte_bits(u[i][k].z) << (16 * k + 8);
                w |= (unsigned long long)nonzero_byte_bits(u[i][k].w) << (16 * k + 12);
            }
            wv[i] = w;
        }
    } else {
        // a ragged or unaligned row: byte loads, positions past n_kv read as zero
#pragma unroll
        for (int i = 0; i < kWWordsPerThread; ++i) {
            unsigned long long w = 0;
            if (i < wpt && w0 + i < nw) {
                const int64_t p0 = 64 * (int64_t)(w0 + i);
                uint8_t b[64];
#pragma unroll
                for (int t = 0; t < 64; ++t) b[t] = p0 + t < n_kv ? row[p0 + t] : (uint8_t)0;
#pragma unroll
                for (int t = 0; t < 64; ++t) w |= (unsigned long long)(b[t] != 0) << t;
            }
            wv[i] = w;
        }
    }
    // exclusive scan of the per-thread counts (threads own consecutive words)
    uint32_t c = 0;
#pragma unroll
    for (int i = 0; i < kWWordsPerThread; ++i) c += __popcll(wv[i]);
    uint32_t x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    uint32_t before = 0, total = 0;
#pragma unroll
    for (int k = 0; k < NT / 32; ++k) {
        before += k < warp ? wsum[k] : 0u;
        total += wsum[k];
    }
    uint32_t run = before + x - c;
#pragma unroll
    for (int i = 0; i < kWWordsPerThread; ++i)
        if (i < wpt && w0 + i < nw) {
            words[w0 + i] = wv[i];
            pre[w0 + i] = run;
            run += __popcll(wv[i]);
        }
    __syncthreads();
    return total;
}

// The L-th set position (L < the row's count): the last word whose prefix is <= L holds it.
__device__ __forceinline__ int64_t mask_position(const unsigned long long *words,
                                                 const uint32_t *pre, int nw, uint32_t L)
{
    int lo = 0, hi = nw - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= L) lo = mid;
        else hi = mid - 1;
    }
    const unsigned long long w = words[lo];
    int j = (int)(L - pre[lo]);
    const uint32_t w_lo = (uint32_t)w;
    const int c_lo = __popc(w_lo);
    const int bit = j < c_lo ? select_set_bit(w_lo, j) : 32 + select_set_bit((uint32_t)(w >> 32), j - c_lo);
    return 64 * (int64_t)lo + bit;
}

template <bool kMask>
__global__ void __launch_bounds__(kWNT, 1)
attn_wide_kernel(const float *__restrict__ q, int H_q, int H_kv, float scale_log2,
                 const __nv_bfloat16 *__restrict__ KV, int64_t n_kv, int64_t ld,
                 const int32_t *__restrict__ pos, const int32_t *__restrict__ n_cells,
                 int64_t max_cells, float *__restrict__ out, float *__restrict__ lse,
                 const uint8_t *__restrict__ mask, int64_t ld_mask,
                 int32_t *__restrict__ counts_out, const WaitCtl wc)
{
    constexpr int G = kWG, DK = kWDK, DV = kWDV, TC = kWTC, LD = kWLD, NT = kWNT;
    extern __shared__ __align__(16) char smem_raw[];
    __nv_bfloat16 *Qs = reinterpret_cast<__nv_bfloat16 *>(smem_raw);
    __nv_bfloat16 *St = reinterpret_cast<__nv_bfloat16 *>(smem_raw + kWQBytes);
    __nv_bfloat16 *Ps = reinterpret_cast<__nv_bfloat16 *>(smem_raw + kWQBytes + 2 * kWStageBytes);
    float *ost = reinterpret_cast<float *>(St);  // [G][kWOLD] after the last stage
    __shared__ int32_t rows[2 * TC];
    __shared__ __align__(8) uint64_t sbar[2];
    __shared__ float red[kWWarps][G];
    __shared__ float run_m[G], run_l[G], new_m[G], alpha[G];

    const int S = gridDim.x, s_idx = blockIdx.x, g = blockIdx.y;
    const int64_t qi = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hr = lane >> 2;       // fragment rows hr and hr + 8 = heads
    const int qc = (lane & 3) * 2;  // fragment columns qc, qc + 1
    const int mi = lane >> 3, mj = lane & 7;

    if (tid == 0) {
        mbar_init(&sbar[0], 1);
        mbar_init(&sbar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < G) {
        run_m[tid] = -INFINITY;
        run_l[tid] = 0.0f;
    }
    pdl_wait();
    QSA_AFTER_WAIT(q);
    QSA_AFTER_WAIT(KV);
    QSA_AFTER_WAIT(pos);
    QSA_AFTER_WAIT(n_cells);
    QSA_AFTER_WAIT(mask);
    pdl_trigger();

    // this split's cells; positions of its first two stages load with the list length
    const int64_t chunk = (max_cells + S - 1) / S;
    const int64_t c0 = (int64_t)s_idx * chunk;
    const int64_t c1max = c0 + chunk < max_cells ? c0 + chunk : max_cells;
    __shared__ unsigned long long mwords[kMask ? kWMaskWords : 1];
    __shared__ uint32_t mpre[kMask ? kWMaskWords : 1];
    __shared__ uint32_t mwsum[kWWarps];
    const int mnw = (int)((n_kv + 63) / 64);
    int64_t n;
    int64_t first_row = -1;
    if constexpr (kMask) {
        n = build_mask_words(mask + qi * ld_mask, n_kv, mwords, mpre, mwsum);
        if (counts_out && s_idx == 0 && g == 0 && tid == 0) counts_out[qi] = (int32_t)n;
        if (tid < 2 * TC && c0 + tid < c1max && c0 + tid < n)
            first_row = mask_position(mwords, mpre, mnw, (uint32_t)(c0 + tid));
    } else {
        n = n_cells[qi];
        if (tid < 2 * TC && c0 + tid < c1max)
            first_row = pos ? (int64_t)pos[qi * max_cells + c0 + tid] : qi * max_cells + c0 + tid;
    }
    const bool overflow = n > max_cells;  // truncated list: the result must not be used
    if (overflow || n < 0) n = 0;
    const int64_t c1 = c1max < n ? c1max : n;
    const int ntiles = c1 > c0 ? (int)((c1 - c0 + TC - 1) / TC) : 0;
    if (tid < 2 * TC) {
        int64_t row = c0 + tid < c1 ? first_row : -1;
        if (row < 0 || row >= n_kv) row = -1;
        rows[tid] = (int32_t)row;
    }
    __syncthreads();

    // phases armed on / seen complete by each stage buffer's barrier (the same in every
    // thread); a wait that gave up stops the stage loop (the outputs become NaN)
    int armed0 = 0, armed1 = 0, done0 = 0, done1 = 0;
    bool lost = false;
    auto load_rows = [&](int it, int buf) {
        const int64_t base = c0 + (int64_t)it * TC;
        const int tc = (int)min((int64_t)TC, c1 - base);
        if (tid < TC) {
            int64_t row = -1;
            if (tid < tc) {
                const int64_t cell = base + tid;
                if constexpr (kMask) row = mask_position(mwords, mpre, mnw, (uint32_t)cell);
                else row = pos ? (int64_t)pos[qi * max_cells + cell] : qi * max_cells + cell;
                if (row < 0 || row >= n_kv) row = -1;
            }
            rows[buf * TC + tid] = (int32_t)row;
        }
        __syncthreads();
    };
    // one bulk copy per listed row; the value columns of skipped rows are zero-filled
    // (P = 0 multiplies them, and stale shared memory could hold a NaN pattern)
    auto copy_rows = [&](int buf) {
        const int32_t *rb = rows + buf * TC;
        __nv_bfloat16 *st = St + (size_t)buf * TC * LD;
        for (int e = tid; e < TC * (DV / 8); e += NT) {
            const int slot = e / (DV / 8), c = e - slot * (DV / 8);
            if (rb[slot] < 0) *reinterpret_cast<uint4 *>(st + slot * LD + c * 8) = make_uint4(0u, 0u, 0u, 0u);
        }
        const int nv = __syncthreads_count(tid < TC && rb[tid] >= 0);
        if (tid == 0) mbar_arrive_expect_tx(&sbar[buf], (uint32_t)nv * DK * 2u);
        if (buf) ++armed1;
        else ++armed0;
        if (tid < TC && rb[tid] >= 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            bulk_g2s(st + tid * LD, KV + (int64_t)rb[tid] * ld, DK * 2, &sbar[buf]);
        }
    };
    auto wait_rows = [&](int buf) {
        const uint32_t par = (uint32_t)((buf ? done1 : done0) & 1);
        const bool ok_w = !lost && mbar_wait(&sbar[buf], par, wc.limit_ns);
        lost = __syncthreads_or(lost || !ok_w) != 0;
        if (!lost) {
            if (buf) ++done1;
            else ++done0;
        }
    };

    float o[8][4];  // heads hr / hr + 8, dims 64 * warp + 8j + qc + {0, 1}
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;

    if (ntiles > 0) copy_rows(0);
    if (ntiles > 1) copy_rows(1);
    // the query, while the first rows are in flight: rows 0-15 = bf16(q * scale), rows 16-31
    // = bf16 of the remainder
    {
        const float *qh = q + (qi * H_q + (int64_t)g * G) * DK;
        constexpr int kPer = G * DK / 2 / NT;  // float pairs per thread, all loaded at once
        static_assert(kPer * NT * 2 == G * DK, "the query splits evenly over the threads");
        float2 x[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k)
            x[k] = *reinterpret_cast<const float2 *>(qh + 2 * (int64_t)(tid + k * NT));
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int e = tid + k * NT;
            const int h = (2 * e) / DK, c = 2 * e - h * DK;
            float h0, l0, h1, l1;
            split_bf16(x[k].x * scale_log2, h0, l0);
            split_bf16(x[k].y * scale_log2, h1, l1);
            *reinterpret_cast<uint32_t *>(Qs + h * LD + c) = pack_bf16(h0, h1);
            *reinterpret_cast<uint32_t *>(Qs + (G + h) * LD + c) = pack_bf16(l0, l1);
        }
    }
    __syncthreads();  // the query images are complete
    for (int it = 0; it < ntiles; ++it) {
        const int buf = it & 1;
        if (it >= 1 && it + 1 < ntiles) {
            load_rows(it + 1, buf ^ 1);
            copy_rows(buf ^ 1);
        }
        wait_rows(buf);
        if (lost) break;  // issue nothing more; what was issued is drained below
        const int tc = (int)min((int64_t)TC, c1 - (c0 + (int64_t)it * TC));
        const __nv_bfloat16 *st = St + (size_t)buf * TC * LD;
        const int32_t *rw = rows + buf * TC;

        // ---- S = Q K^T for this warp's 8 cells
        float shi[4] = {0.f, 0.f, 0.f, 0.f}, slo[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const __nv_bfloat16 *kb = st + (warp * 8 + (lane & 7)) * LD + ((lane >> 3) & 1) * 8;
            const __nv_bfloat16 *qa = Qs + (lane & 15) * LD + (lane >> 4) * 8;
#pragma unroll 4
            for (int kk = 0; kk < DK / 16; ++kk) {
                uint32_t a_hi[4], a_lo[4], b[2];
                ldsm_x4(a_hi, qa + kk * 16);
                ldsm_x4(a_lo, qa + G * LD + kk * 16);
                ldsm_x2(b, kb + kk * 16);
                mma_16816(shi, a_hi, b[0], b[1]);
                mma_16816(slo, a_lo, b[0], b[1]);
            }
        }
        // logits of heads hr (x[0..1]) and hr + 8 (x[2..3]) for cells warp*8 + qc + {0,1}
        float x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int slot = warp * 8 + qc + (u & 1);
            const bool ok = slot < tc && rw[slot] >= 0;
            x[u] = ok ? shi[u] + slo[u] : -INFINITY;
        }
        float m0 = fmaxf(x[0], x[1]), m1 = fmaxf(x[2], x[3]);
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
        if ((lane & 3) == 0) {
            red[warp][hr] = m0;
            red[warp][hr + 8] = m1;
        }
        __syncthreads();
        if (tid < G) {
            float M = run_m[tid];
#pragma unroll
            for (int w = 0; w < kWWarps; ++w) M = fmaxf(M, red[w][tid]);
            new_m[tid] = M;
            alpha[tid] = M == -INFINITY ? 1.0f : exp2f(run_m[tid] - M);
        }
        __syncthreads();
        // ---- P = 2^(S - M), its hi / lo bf16 halves into shared memory, partial row sums
        {
            const float M0 = new_m[hr], M1 = new_m[hr + 8];
            float p[4];
            p[0] = M0 == -INFINITY ? 0.0f : exp2f(x[0] - M0);
            p[1] = M0 == -INFINITY ? 0.0f : exp2f(x[1] - M0);
            p[2] = M1 == -INFINITY ? 0.0f : exp2f(x[2] - M1);
            p[3] = M1 == -INFINITY ? 0.0f : exp2f(x[3] - M1);
            float ph[4], pl[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) split_bf16(p[u], ph[u], pl[u]);
            const int cell = warp * 8 + qc;
            *reinterpret_cast<uint32_t *>(Ps + hr * kWPLD + cell) = pack_bf16(ph[0], ph[1]);
            *reinterpret_cast<uint32_t *>(Ps + (hr + 8) * kWPLD + cell) = pack_bf16(ph[2], ph[3]);
            *reinterpret_cast<uint32_t *>(Ps + (G + hr) * kWPLD + cell) = pack_bf16(pl[0], pl[1]);
            *reinterpret_cast<uint32_t *>(Ps + (G + hr + 8) * kWPLD + cell) = pack_bf16(pl[2], pl[3]);
            float s0 = p[0] + p[1], s1 = p[2] + p[3];
            s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
            s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
            s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
            s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
            __syncwarp();
            if ((lane & 3) == 0) {
                red[warp][hr] = s0;
                red[warp][hr + 8] = s1;
            }
        }
        __syncthreads();
        if (tid < G) {
            float L = run_l[tid] * alpha[tid];
#pragma unroll
            for (int w = 0; w < kWWarps; ++w) L += red[w][tid];
            run_l[tid] = L;
            run_m[tid] = new_m[tid];
        }
        // ---- O = alpha O + P V over this warp's 64 output dims
        {
            const float a0 = alpha[hr], a1 = alpha[hr + 8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                o[j][0] *= a0;
                o[j][1] *= a0;
                o[j][2] *= a1;
                o[j][3] *= a1;
            }
#pragma unroll
            for (int ks = 0; ks < TC / 16; ++ks) {
                uint32_t p_hi[4], p_lo[4];
                ldsm_x4(p_hi, Ps + (lane & 15) * kWPLD + ks * 16 + (lane >> 4) * 8);
                ldsm_x4(p_lo, Ps + (G + (lane & 15)) * kWPLD + ks * 16 + (lane >> 4) * 8);
#pragma unroll
                for (int dp = 0; dp < 4; ++dp) {
                    uint32_t b[4];
                    const int cell = ks * 16 + (mi & 1) * 8 + mj;
                    ldsm_x4_t(b, st + cell * LD + warp * 64 + dp * 16 + (mi >> 1) * 8);
                    mma_16816(o[2 * dp], p_hi, b[0], b[1]);
                    mma_16816(o[2 * dp], p_lo, b[0], b[1]);
                    mma_16816(o[2 * dp + 1], p_hi, b[2], b[3]);
                    mma_16816(o[2 * dp + 1], p_lo, b[2], b[3]);
                }
            }
        }
        __syncthreads();  // this stage and P are refilled next
    }
    // every copy issued lands before the stage area is reused or the CTA leaves (a buffer is
    // re-armed only after its previous phase was seen complete: at most one outstanding)
    if (armed0 > done0) (void)mbar_wait(&sbar[0], (uint32_t)(done0 & 1));
    if (armed1 > done1) (void)mbar_wait(&sbar[1], (uint32_t)(done1 & 1));
    lost = __syncthreads_or(lost);
    if (lost && tid == 0) report_timeout(wc);

    // the CTA's state: unnormalised o (stage area, now free), m and l per head
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int c = warp * 64 + 8 * j + qc;
        ost[hr * kWOLD + c] = o[j][0];
        ost[hr * kWOLD + c + 1] = o[j][1];
        ost[(hr + 8) * kWOLD + c] = o[j][2];
        ost[(hr + 8) * kWOLD + c + 1] = o[j][3];
    }
    if (tid < G && lost) run_l[tid] = -1.0f;  // a negative weight sum marks a lost stage
    __syncthreads();
    if (S == 1) {
        for (int e = tid; e < G * DV; e += NT) {
            const int h = e / DV, c = e - h * DV;
            const float L = run_l[h];
            float v = L > 0.0f ? ost[h * kWOLD + c] / L : 0.0f;
            if (overflow || lost) v = __int_as_float(0x7fc00000);
            out[(qi * H_q + (int64_t)g * G + h) * DV + c] = v;
            if (lse && c == 0)
                lse[qi * H_q + g * G + h] = (overflow || lost) ? __int_as_float(0x7fc00000)
                                           : (L > 0.0f ? (run_m[h] + log2f(L)) * kLn2 : -INFINITY);
        }
        return;
    }

    // cluster combine: CTA s owns outputs [s*per, (s+1)*per) of G*DV.  First the weights of
    // the heads in that slice (one round of remote loads of every split's maximum and sum),
    // then every output sums its S partials, all S remote loads in flight at once.
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int per = (G * DV + S - 1) / S;
    const int e_begin = s_idx * per, e_end = min((s_idx + 1) * per, G * DV);
    const int h_first = e_begin / DV;
    const int nh = e_end > e_begin ? (e_end - 1) / DV - h_first + 1 : 0;
    // the query images are no longer read: their space holds the weights
    float *wf = reinterpret_cast<float *>(Qs);   // [nh][kWMaxCluster] split weights
    float *wm = wf + G * kWMaxCluster;           // [nh][kWMaxCluster] split maxima, then [nh] M
    float *hM = wm + G * kWMaxCluster;           // [nh] head maximum
    float *hL = hM + G;                          // [nh] head weight sum (< 0: a lost stage)
    for (int x = tid; x < nh * S; x += NT) {
        const int hh = x / S, r = x - hh * S;
        const int h = h_first + hh;
        wm[hh * kWMaxCluster + r] = cluster.map_shared_rank(run_m, r)[h];
        wf[hh * kWMaxCluster + r] = cluster.map_shared_rank(run_l, r)[h];
    }
    __syncthreads();
    if (tid < nh) {
        float M = -INFINITY;
        bool bad = false;
        for (int r = 0; r < S; ++r) {
            M = fmaxf(M, wm[tid * kWMaxCluster + r]);
            bad = bad || wf[tid * kWMaxCluster + r] < 0.0f;
        }
        float L = 0.0f;
        for (int r = 0; r < S; ++r) {
            const float f = M != -INFINITY ? exp2f(wm[tid * kWMaxCluster + r] - M) : 0.0f;
            L = fmaf(f, wf[tid * kWMaxCluster + r], L);
            wf[tid * kWMaxCluster + r] = f;
        }
        hM[tid] = M;
        hL[tid] = bad ? -1.0f : L;
    }
    __syncthreads();
    for (int e = e_begin + tid; e < e_end; e += NT) {
        const int h = e / DV, c = e - h * DV, hh = h - h_first;
        const float *f = wf + hh * kWMaxCluster;
        float ov[kWMaxCluster];
#pragma unroll
        for (int r = 0; r < kWMaxCluster; ++r)
            ov[r] = r < S ? cluster.map_shared_rank(ost, r)[h * kWOLD + c] : 0.0f;
        float acc = 0.0f;
#pragma unroll
        for (int r = 0; r < kWMaxCluster; ++r)
            if (r < S) acc = fmaf(f[r], ov[r], acc);
        const float L = hL[hh];
        const bool bad = L < 0.0f || overflow;
        float v = L > 0.0f ? acc / L : 0.0f;
        if (bad) v = __int_as_float(0x7fc00000);
        out[(qi * H_q + (int64_t)g * G + h) * DV + c] = v;
        if (lse && c == 0)
            lse[qi * H_q + g * G + h] = bad ? __int_as_float(0x7fc00000)
                                       : (L > 0.0f ? (hM[hh] + log2f(L)) * kLn2 : -INFINITY);
    }
    cluster.sync();  // keep this CTA's state alive until every remote read is done
}

}  // namespace

bool attn_uses_wide(qsa_dtype dt, int d_k, int d_v, int G, const void *K, const void *V,
                    int64_t ld_k, int64_t ld_v)
{
    return dt == QSA_BF16 && d_k == kWDK && d_v == kWDV && G == kWG && K == V && ld_k == ld_v &&
           (ld_k * 2) % 16 == 0 && reinterpret_cast<uintptr_t>(K) % 16 == 0;
}

int attn_wide_splits(int64_t n_q, int H_kv, int64_t max_cells)
{
    const int64_t groups = n_q * (int64_t)H_kv;
    if (groups >= kTargetSMs) return 1;
    int64_t S = (max_cells + 2 * kWTC - 1) / (2 * kWTC);  // about two stages per CTA
    const int64_t fill = (kTargetSMs + groups - 1) / groups;
    if (S > fill) S = fill;
    if (S > kWMaxCluster) S = kWMaxCluster;
    if (S < 1) S = 1;
    return (int)S;
}

cudaError_t launch_attn_wide(const float *q, int64_t n_q, int H_q, int H_kv, float scale,
                             const void *KV, int64_t n_kv, int64_t ld, const int32_t *pos,
                             const int32_t *n_cells, int64_t max_cells, float *out, float *lse,
                             cudaStream_t st)
{
    const cudaError_t ea = ensure_kernel_attrs<attn_wide_kernel<false>>(kWSmem, true);
    if (ea != cudaSuccess) return ea;
    const int S = attn_wide_splits(n_q, H_kv, max_cells);
    const dim3 grid((unsigned)S, (unsigned)H_kv, (unsigned)n_q);
    return launch(attn_wide_kernel<false>, grid, dim3(kWNT), kWSmem, st, S > 1 ? S : 1, q, H_q,
                  H_kv, scale * kLog2e, (const __nv_bfloat16 *)KV, n_kv, ld, pos, n_cells,
                  max_cells, out, lse, (const uint8_t *)nullptr, (int64_t)0, (int32_t *)nullptr,
                  current_wait_ctl());
}

int64_t attn_wide_mask_max_kv() { return (int64_t)kWMaskWords * 64; }

cudaError_t launch_attn_wide_mask(const float *q, int64_t n_q, int H_q, int H_kv, float scale,
                                  const void *KV, int64_t n_kv, int64_t ld, const uint8_t *mask,
                                  int64_t ld_mask, int64_t max_list, int32_t *counts_out,
                                  float *out, float *lse, cudaStream_t st)
{
    const cudaError_t ea = ensure_kernel_attrs<attn_wide_kernel<true>>(kWSmem, true);
    if (ea != cudaSuccess) return ea;
    const int S = attn_wide_splits(n_q, H_kv, max_list);
    const dim3 grid((unsigned)S, (unsigned)H_kv, (unsigned)n_q);
    return launch(attn_wide_kernel<true>, grid, dim3(kWNT), kWSmem, st, S > 1 ? S : 1, q, H_q,
                  H_kv, scale * kLog2e, (const __nv_bfloat16 *)KV, n_kv, ld,
                  (const int32_t *)nullptr, (const int32_t *)nullptr, max_list, out, lse, mask,
                  ld_mask, counts_out, current_wait_ctl());
}

}  // namespace qsa
