// attn.cu -- attention of each query token over its listed KV cells only (split-K flash
// decoding with an online softmax per split and a log-sum-exp combine).
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "selected K/V gather (COMMON-005)" (attention over the ~2051 selected rows instead of
// the full KV: 2.939 ms -> 42 us per layer at 256k on the pages' GPU) and devotd.net,
// "llama.cpp CDNA sparse attention", sections 2-3 (attention over the listed key
// positions; DKQ 576 with 16 query heads per KV head).
//
// Every kernel here reads the listed rows straight from the full cache into shared memory
// (the gather happens on the way in: no compact copy round-trips through HBM).
//   - attn_mma_kernel: the decode form (bf16, head dim 128, 8 query heads per KV head):
//     tensor-core mma.sync, bulk-copy staging, the splits of one (query, KV head) combined
//     inside a thread-block cluster.  See the comment above it.
//   - attn128_kernel: head dim 128 for other dtypes and group sizes.
//   - sparse_attn_kernel: any shape.  Grid (split, kv head, query); each CTA stages 32
//     listed rows of K and V at a time with 16-byte cp.async, double-buffered so the next
//     tile's loads overlap this tile's math.  Logits: one warp per cell, lanes split the
//     head dim, one warp reduction per query head of the group.  Softmax: one warp per
//     head, one lane per cell.  P.V: each thread owns G*d_v/128 output entries.  fp32.
//   - attn_combine_kernel: the log-sum-exp merge of the splits of the last two.
#include <cooperative_groups.h>

#include "mma_frag.cuh"

namespace cg = cooperative_groups;

namespace qsa {
namespace {

constexpr int kAttnThreads = 128;
constexpr int kTile = 32;

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc, bool valid)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem_dst);
    const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zeroed
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gsrc), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Four consecutive elements as fp32.
__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16 *p)
{
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

struct AttnSmem {
    float *q;      // [G][d_k]   query rows, pre-scaled by scale*log2(e)
    float *o;      // [G][d_v]   unnormalised output accumulators
    float *p;      // [G][kTile] logits, then probabilities
    float *m;      // [G]        running max (log2 domain)
    float *l;      // [G]        running sum
    float *a;      // [G]        rescale factor of the current tile
    int32_t *row;  // [2][kTile] cache row of each staged cell (-1 = skipped)
    char *k;       // [2][kTile][d_k]
    char *v;       // [2][kTile][d_v]
};

__host__ __device__ inline size_t attn_smem_bytes(int G, int d_k, int d_v, int esize)
{
    size_t f = (size_t)G * d_k + (size_t)G * d_v + (size_t)G * kTile + 3 * (size_t)G;
    size_t bytes = f * 4 + 2 * kTile * 4;
    bytes = (bytes + 15) & ~(size_t)15;
    bytes += 2 * (size_t)kTile * ((size_t)d_k + d_v) * esize;
    return bytes;
}

__device__ inline AttnSmem carve(char *base, int G, int d_k, int d_v, int esize)
{
    AttnSmem s;
    float *f = reinterpret_cast<float *>(base);
    s.q = f;
    f += (size_t)G * d_k;
    s.o = f;
    f += (size_t)G * d_v;
    s.p = f;
    f += (size_t)G * kTile;
    s.m = f;
    s.l = f + G;
    s.a = f + 2 * G;
    f += 3 * G;
    s.row = reinterpret_cast<int32_t *>(f);
    size_t off = (size_t)((char *)(s.row + 2 * kTile) - base);
    off = (off + 15) & ~(size_t)15;
    s.k = base + off;
    s.v = s.k + 2 * (size_t)kTile * d_k * esize;
    (void)esize;
    return s;
}

template <typename T, int G>
__global__ void __launch_bounds__(kAttnThreads)
sparse_attn_kernel(const float *__restrict__ q, int H_q, int H_kv, int d_k, int d_v,
                   float scale_log2, const T *__restrict__ K, const T *__restrict__ V,
                   int64_t n_kv, int64_t ld_k, int64_t ld_v, const int32_t *__restrict__ pos,
                   const int32_t *__restrict__ n_cells, int64_t max_cells,
                   float *__restrict__ out, float *__restrict__ lse, float *__restrict__ part)
{
    extern __shared__ __align__(16) char smem_raw[];
    const int S = gridDim.x;
    const int s_idx = blockIdx.x;
    const int g = blockIdx.y;
    const int64_t qi = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NW = kAttnThreads / 32;
    AttnSmem sm = carve(smem_raw, G, d_k, d_v, (int)sizeof(T));

    pdl_wait();
    QSA_AFTER_WAIT(q);
    QSA_AFTER_WAIT(K);
    QSA_AFTER_WAIT(V);
    QSA_AFTER_WAIT(pos);
    QSA_AFTER_WAIT(n_cells);
    pdl_trigger();

    int64_t n = n_cells[qi];
    if (n > max_cells) {  // truncated list: the result must not be used
        if (S == 1) {
            for (int e = tid; e < G * d_v; e += kAttnThreads)
                out[(qi * H_q + (int64_t)g * G) * d_v + e] = __int_as_float(0x7fc00000);
            if (lse && tid < G) lse[qi * H_q + g * G + tid] = __int_as_float(0x7fc00000);
        }
        return;  // with S > 1 the combine kernel writes the NaN result
    }
    if (n < 0) n = 0;
    const int64_t chunk = (n + S - 1) / S;
    const int64_t c0 = (int64_t)s_idx * chunk;
    const int64_t c1 = c0 + chunk < n ? c0 + chunk : n;
    const int64_t n_my = c1 > c0 ? c1 - c0 : 0;
    const int ntiles = (int)((n_my + kTile - 1) / kTile);

    const float *qg = q + (qi * H_q + (int64_t)g * G) * d_k;
    for (int e = tid; e < G * d_k; e += kAttnThreads) sm.q[e] = qg[e] * scale_log2;
    for (int e = tid; e < G * d_v; e += kAttnThreads) sm.o[e] = 0.0f;
    if (tid < G) {
        sm.m[tid] = -INFINITY;
        sm.l[tid] = 0.0f;
    }

    const int kchunks = d_k * (int)sizeof(T) / 16;  // 16-byte pieces per K row
    const int vchunks = d_v * (int)sizeof(T) / 16;
    auto issue_tile = [&](int it, int buf) {
        const int64_t base_cell = c0 + (int64_t)it * kTile;
        const int tc = (int)min((int64_t)kTile, c1 - base_cell);
        T *ks = reinterpret_cast<T *>(sm.k) + (size_t)buf * kTile * d_k;
        T *vs = reinterpret_cast<T *>(sm.v) + (size_t)buf * kTile * d_v;
        const int per_row = kchunks + vchunks;
        // cache rows of the tile first (one load each), so the copies below do not wait on
        // a position load apiece
        int32_t *rb = sm.row + buf * kTile;
        for (int slot = tid; slot < kTile; slot += kAttnThreads) {
            int64_t row = -1;
            if (slot < tc) {
                const int64_t cell = base_cell + slot;
                row = pos ? (int64_t)pos[qi * max_cells + cell] : qi * max_cells + cell;
                if (row < 0 || row >= n_kv) row = -1;
            }
            rb[slot] = (int32_t)row;
        }
        __syncthreads();
        for (int e = tid; e < kTile * per_row; e += kAttnThreads) {
            const int slot = e / per_row;
            const int c = e - slot * per_row;
            const int64_t row = rb[slot];
            const bool ok = row >= 0;
            if (c < kchunks) {
                const T *src = K + (ok ? row : 0) * ld_k + (int64_t)g * d_k + c * (16 / sizeof(T));
                cp_async16(ks + (size_t)slot * d_k + c * (16 / sizeof(T)), src, ok);
            } else {
                const int cv = c - kchunks;
                const T *src = V + (ok ? row : 0) * ld_v + (int64_t)g * d_v + cv * (16 / sizeof(T));
                cp_async16(vs + (size_t)slot * d_v + cv * (16 / sizeof(T)), src, ok);
            }
        }
        cp_async_commit();
    };

    if (ntiles > 0) issue_tile(0, 0);
    __syncthreads();  // q, o, m, l initialised

    for (int it = 0; it < ntiles; ++it) {
        const int buf = it & 1;
        if (it + 1 < ntiles) {
            issue_tile(it + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int tc = (int)min((int64_t)kTile, c1 - (c0 + (int64_t)it * kTile));
        const T *ks = reinterpret_cast<const T *>(sm.k) + (size_t)buf * kTile * d_k;
        const T *vs = reinterpret_cast<const T *>(sm.v) + (size_t)buf * kTile * d_v;
        const int32_t *rows = sm.row + buf * kTile;

        // logits (log2 domain)
        for (int slot = warp; slot < tc; slot += NW) {
            float acc[G];
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h] = 0.0f;
            const T *kr = ks + (size_t)slot * d_k;
            for (int t = lane * 4; t < d_k; t += 128) {
                const float4 kv = ld4(kr + t);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float4 qq = *reinterpret_cast<const float4 *>(sm.q + h * d_k + t);
                    acc[h] = fmaf(kv.x, qq.x, fmaf(kv.y, qq.y, fmaf(kv.z, qq.z, fmaf(kv.w, qq.w, acc[h]))));
                }
            }
            const bool ok = rows[slot] >= 0;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float v = warp_sum(acc[h]);
                if (lane == 0) sm.p[h * kTile + slot] = ok ? v : -INFINITY;
            }
        }
        __syncthreads();

        // online softmax: one warp per head, one lane per cell
        for (int h = warp; h < G; h += NW) {
            const float x = lane < tc ? sm.p[h * kTile + lane] : -INFINITY;
            const float m_old = sm.m[h];
            const float m_new = fmaxf(m_old, warp_max(x));
            float p = 0.0f, alpha = 1.0f;
            if (m_new != -INFINITY) {
                p = x == -INFINITY ? 0.0f : exp2f(x - m_new);
                alpha = m_old == -INFINITY ? 0.0f : exp2f(m_old - m_new);
            }
            const float psum = warp_sum(p);
            if (lane < kTile) sm.p[h * kTile + lane] = p;
            if (lane == 0) {
                sm.m[h] = m_new;
                sm.l[h] = sm.l[h] * alpha + psum;
                sm.a[h] = alpha;
            }
        }
        __syncthreads();

        // o = o * alpha + P . V
        for (int e = tid; e < G * d_v; e += kAttnThreads) {
            const int h = e / d_v;
            const int c = e - h * d_v;
            const float *ph = sm.p + h * kTile;
            float acc = 0.0f;
            for (int slot = 0; slot < tc; ++slot) acc = fmaf(ph[slot], to_f32(vs[(size_t)slot * d_v + c]), acc);
            sm.o[e] = sm.o[e] * sm.a[h] + acc;
        }
        __syncthreads();
    }

    if (S == 1) {
        for (int e = tid; e < G * d_v; e += kAttnThreads) {
            const int h = e / d_v;
            const float l = sm.l[h];
            out[(qi * H_q + (int64_t)g * G) * d_v + e] = l > 0.0f ? sm.o[e] / l : 0.0f;
        }
        if (lse && tid < G) {
            const float l = sm.l[tid];
            lse[qi * H_q + g * G + tid] = l > 0.0f ? (sm.m[tid] + log2f(l)) * kLn2 : -INFINITY;
        }
    } else {
        const int rec = d_v + 4;
        float *pr = part + (((qi * H_kv + g) * (int64_t)S + s_idx) * G) * rec;
        for (int e = tid; e < G * d_v; e += kAttnThreads) {
            const int h = e / d_v;
            pr[(int64_t)h * rec + 4 + (e - h * d_v)] = sm.o[e];
        }
        if (tid < G) {
            pr[(int64_t)tid * rec + 0] = sm.m[tid];
            pr[(int64_t)tid * rec + 1] = sm.l[tid];
        }
    }
}

// ---------------------------------------------------------------------------------
// Head dim 128, up to 8 query heads per KV head (the decode and prefill shapes).
// CTA = (split, kv head g, query); 4 warps share the CTA's cells (warp w takes every 4th
// staged cell).  A warp covers all G heads of the group: lane = (head hl = lane / LPH,
// slice sl = lane % LPH) with LPH = 32 / G lanes per head, each holding DPL = 128 / LPH
// consecutive dims of its head's query and output in registers.  Per cell: DPL fused
// multiply-adds, log2(LPH) shuffles for the logit, DPL more for P.V; cells go in chunks
// of 4 with one online-softmax rescale per chunk.  The 4 warps' (m, l, o) are merged in
// shared memory at the end.
template <typename T>
struct Tile128 {
    static constexpr int kCells = sizeof(T) == 2 ? 64 : 32;  // cells per stage
};

template <typename T, int G>
__global__ void __launch_bounds__(128)
attn128_kernel(const float *__restrict__ q, int H_q, int H_kv, float scale_log2,
               const T *__restrict__ K, const T *__restrict__ V, int64_t n_kv, int64_t ld_k,
               int64_t ld_v, const int32_t *__restrict__ pos, const int32_t *__restrict__ n_cells,
               int64_t max_cells, float *__restrict__ out, float *__restrict__ lse,
               float *__restrict__ part)
{
    constexpr int D = 128;
    constexpr int LPH = 32 / G;
    constexpr int DPL = D / LPH;
    constexpr int TC = Tile128<T>::kCells;
    constexpr int EPC = 16 / sizeof(T);  // elements per 16-byte chunk
    constexpr int CPR = D / EPC;         // chunks per row
    constexpr int NW = 4;
    constexpr int CH = 4;                // cells per softmax chunk
    extern __shared__ __align__(16) char smem_raw[];
    T *Ks = reinterpret_cast<T *>(smem_raw);                  // [2][TC][D]
    T *Vs = Ks + 2 * TC * D;                                  // [2][TC][D]
    int32_t *rows = reinterpret_cast<int32_t *>(Vs + 2 * TC * D);  // [2][TC]
    float *mrg = reinterpret_cast<float *>(rows + 2 * TC);    // [NW][G][D + 2]

    const int S = gridDim.x, s_idx = blockIdx.x, g = blockIdx.y;
    const int64_t qi = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hl = lane / LPH, sl = lane % LPH;

    pdl_wait();
    QSA_AFTER_WAIT(q);
    QSA_AFTER_WAIT(K);
    QSA_AFTER_WAIT(V);
    QSA_AFTER_WAIT(pos);
    QSA_AFTER_WAIT(n_cells);
    pdl_trigger();

    int64_t n = n_cells[qi];
    if (n > max_cells) {
        if (S == 1) {
            for (int e = tid; e < G * D; e += 128)
                out[(qi * H_q + (int64_t)g * G) * D + e] = __int_as_float(0x7fc00000);
            if (lse && tid < G) lse[qi * H_q + g * G + tid] = __int_as_float(0x7fc00000);
        }
        return;
    }
    if (n < 0) n = 0;
    const int64_t chunk = (n + S - 1) / S;
    const int64_t c0 = (int64_t)s_idx * chunk;
    const int64_t c1 = c0 + chunk < n ? c0 + chunk : n;
    const int ntiles = c1 > c0 ? (int)((c1 - c0 + TC - 1) / TC) : 0;

    float qr[DPL], o[DPL];
    {
        const float *qh = q + ((qi * H_q + (int64_t)g * G + hl) * D) + sl * DPL;
#pragma unroll
        for (int j = 0; j < DPL; j += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(qh + j);
            qr[j] = v.x * scale_log2;
            qr[j + 1] = v.y * scale_log2;
            qr[j + 2] = v.z * scale_log2;
            qr[j + 3] = v.w * scale_log2;
        }
    }
#pragma unroll
    for (int j = 0; j < DPL; ++j) o[j] = 0.0f;
    float m = -INFINITY, l = 0.0f;

    auto issue = [&](int it, int buf) {
        const int64_t base = c0 + (int64_t)it * TC;
        const int tc = (int)min((int64_t)TC, c1 - base);
        T *ks = Ks + buf * TC * D;
        T *vs = Vs + buf * TC * D;
        // cache rows of the tile first (one load each), then the copies
        int32_t *rb = rows + buf * TC;
        for (int slot = tid; slot < TC; slot += 128) {
            int64_t row = -1;
            if (slot < tc) {
                const int64_t cell = base + slot;
                row = pos ? (int64_t)pos[qi * max_cells + cell] : qi * max_cells + cell;
                if (row < 0 || row >= n_kv) row = -1;
            }
            rb[slot] = (int32_t)row;
        }
        __syncthreads();
        for (int e = tid; e < TC * 2 * CPR; e += 128) {
            const int slot = e / (2 * CPR);
            const int c = e - slot * 2 * CPR;
            const int64_t row = rb[slot];
            const bool ok = row >= 0;
            if (c < CPR) {
                cp_async16(ks + slot * D + c * EPC, K + (ok ? row : 0) * ld_k + (int64_t)g * D + c * EPC, ok);
            } else {
                const int cv = c - CPR;
                cp_async16(vs + slot * D + cv * EPC, V + (ok ? row : 0) * ld_v + (int64_t)g * D + cv * EPC, ok);
            }
        }
        cp_async_commit();
    };

    if (ntiles > 0) issue(0, 0);
    for (int it = 0; it < ntiles; ++it) {
        const int buf = it & 1;
        if (it + 1 < ntiles) {
            issue(it + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int tc = (int)min((int64_t)TC, c1 - (c0 + (int64_t)it * TC));
        const T *ks = Ks + buf * TC * D;
        const T *vs = Vs + buf * TC * D;
        const int32_t *rw = rows + buf * TC;
        for (int s0 = warp * CH; s0 < tc; s0 += NW * CH) {
            float sc[CH];
#pragma unroll
            for (int u = 0; u < CH; ++u) {
                const int slot = s0 + u;
                float a = 0.0f;
                if (slot < tc) {
                    const T *kr = ks + slot * D + sl * DPL;
#pragma unroll
                    for (int j = 0; j < DPL; j += 4) {
                        const float4 kv = ld4(kr + j);
                        a = fmaf(kv.x, qr[j], fmaf(kv.y, qr[j + 1], fmaf(kv.z, qr[j + 2], fmaf(kv.w, qr[j + 3], a))));
                    }
                }
#pragma unroll
                for (int off = LPH / 2; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
                sc[u] = (slot < tc && rw[slot] >= 0) ? a : -INFINITY;
            }
            float cmax = sc[0];
#pragma unroll
            for (int u = 1; u < CH; ++u) cmax = fmaxf(cmax, sc[u]);
            const float m_new = fmaxf(m, cmax);
            if (m_new == -INFINITY) continue;  // nothing valid yet
            const float alpha = exp2f(m - m_new);  // m = -inf -> 0
            float p[CH];
            float psum = 0.0f;
#pragma unroll
            for (int u = 0; u < CH; ++u) {
                p[u] = exp2f(sc[u] - m_new);
                psum += p[u];
            }
            l = l * alpha + psum;
            m = m_new;
#pragma unroll
            for (int j = 0; j < DPL; ++j) o[j] *= alpha;
#pragma unroll
            for (int u = 0; u < CH; ++u) {
                const int slot = s0 + u;
                if (p[u] != 0.0f) {
                    const T *vr = vs + slot * D + sl * DPL;
#pragma unroll
                    for (int j = 0; j < DPL; j += 4) {
                        const float4 vv = ld4(vr + j);
                        o[j] = fmaf(p[u], vv.x, o[j]);
                        o[j + 1] = fmaf(p[u], vv.y, o[j + 1]);
                        o[j + 2] = fmaf(p[u], vv.z, o[j + 2]);
                        o[j + 3] = fmaf(p[u], vv.w, o[j + 3]);
                    }
                }
            }
        }
        __syncthreads();  // this stage is refilled by the next issue()
    }

    // merge the 4 warps' states
    float *mw = mrg + (size_t)warp * G * (D + 2);
    if (sl == 0) {
        mw[hl * (D + 2) + D] = m;
        mw[hl * (D + 2) + D + 1] = l;
    }
#pragma unroll
    for (int j = 0; j < DPL; ++j) mw[hl * (D + 2) + sl * DPL + j] = o[j];
    __syncthreads();
    for (int e = tid; e < G * D; e += 128) {
        const int h = e / D, c = e - h * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, mrg[(w * G + h) * (D + 2) + D]);
        float acc = 0.0f, L = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float *r = mrg + (w * G + h) * (D + 2);
                const float f = exp2f(r[D] - M);
                acc = fmaf(f, r[c], acc);
                L = fmaf(f, r[D + 1], L);
            }
        }
        if (S == 1) {
            out[(qi * H_q + (int64_t)g * G + h) * D + c] = L > 0.0f ? acc / L : 0.0f;
            if (lse && c == 0)
                lse[qi * H_q + g * G + h] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
        } else {
            constexpr int rec = D + 4;
            float *pr = part + ((((qi * H_kv + g) * (int64_t)S + s_idx) * G) + h) * rec;
            pr[4 + c] = acc;
            if (c == 0) {
                pr[0] = M;
                pr[1] = L;
            }
        }
    }
}

template <typename T, int G>
size_t attn128_smem()
{
    constexpr int TC = Tile128<T>::kCells;
    return 2 * 2 * (size_t)TC * 128 * sizeof(T) + 2 * TC * sizeof(int32_t) +
           4 * (size_t)G * (128 + 2) * sizeof(float);
}

// ---------------------------------------------------------------------------------
// bf16 K/V, head dim 128, 8 query heads per KV head: QK^T and P.V on the tensor cores
// with warp-level mma.m16n8k16 (bf16 operands, fp32 accumulation).  The 16 rows of the A
// operand are the 8 heads twice: rows 0-7 hold the bf16 rounding of the (pre-scaled)
// query, rows 8-15 the bf16 rounding of what that left over, so row h + row h+8 carries
// the fp32 query to ~2^-17 relative; K and V are exact bf16.  The probabilities are split
// the same way for P.V.  Per 16 cells a warp issues 16 + 16 MMAs and 8 + 8 ldmatrix loads
// (vs. ~2700 CUDA-core instructions).  K and V tiles live in shared memory with rows
// padded to 272 bytes so that the 8 rows of every ldmatrix fall in distinct banks.
constexpr int kMmaWarps = 8;
constexpr int kMmaTC = 16 * kMmaWarps;  // cells per stage: 16 per warp
constexpr int kMmaLd = 136;             // padded smem row in bf16 elements = 272 bytes
constexpr int kMmaMaxCluster = 16;      // splits of one (query, KV head) merged in-cluster

// Shared memory of the tensor-core kernel with NW warps (16 cells each per stage) and NB
// stage buffers: K and V stages, cell rows, per-warp states, the CTA's merged state.  With
// one stage buffer the per-warp states reuse the stage area once the cells are done.
// Rows of a stage buffer: 16 per warp, and with one buffer 16 more, so that a split a few
// cells longer than a stage (the last of 2,051 cells over 16 splits holds 131) is still
// one stage (its last warp takes the extra cells).
template <int NW, int NB>
__host__ __device__ constexpr int attn_mma_stage_rows()
{
    return 16 * NW + (NB == 1 ? 16 : 0);
}
template <int NW, int NB>
__host__ __device__ constexpr size_t attn_mma_stage_bytes()
{
    return 2 * (size_t)NB * attn_mma_stage_rows<NW, NB>() * kMmaLd * 2;
}
template <int NW>
__host__ __device__ constexpr size_t attn_mma_merge_bytes()
{
    return (size_t)NW * 8 * (128 + 2) * 4;
}
template <int NW, int NB>
__host__ __device__ constexpr size_t attn_mma_smem()
{
    return (NB == 1 ? (attn_mma_stage_bytes<NW, NB>() > attn_mma_merge_bytes<NW>()
                           ? attn_mma_stage_bytes<NW, NB>()
                           : attn_mma_merge_bytes<NW>())
                    : attn_mma_stage_bytes<NW, NB>() + attn_mma_merge_bytes<NW>()) +
           2 * (size_t)(16 * NW) * 4 + (size_t)8 * (128 + 2) * 4;
}

// Grid (S, H_kv, n_q).  With S > 1 the S CTAs of one (query, KV head) form a thread-block
// cluster: each merges its warps into one (m, l, o) per head in shared memory, then every
// CTA combines a slice of the 8 x 128 outputs from all S states through distributed shared
// memory -- no partials in global memory and no second kernel.
// NW warps per CTA (stages of 16 * NW cells), NB stage buffers (2: the next stage's rows
// load while this one computes; 1: every split is one stage, and two CTAs fit an SM).
template <int NW, int NB>
__global__ void __launch_bounds__(32 * NW, (NB == 1 ? 2 : 0))
attn_mma_kernel(const float *__restrict__ q, int H_q, int H_kv, float scale_log2,
                const __nv_bfloat16 *__restrict__ K, const __nv_bfloat16 *__restrict__ V,
                int64_t n_kv, int64_t ld_k, int64_t ld_v, const int32_t *__restrict__ pos,
                const int32_t *__restrict__ n_cells, int64_t max_cells, float *__restrict__ out,
                float *__restrict__ lse, int early_q, const WaitCtl wc,
                float *__restrict__ out_host, float *__restrict__ lse_host)
{
    // out_host / lse_host (nullable): a second copy of out / lse, written in place into the
    // caller's page-locked host memory (the host-fed decode step), so that no copy kernel
    // follows this one.
    constexpr int G = 8, D = 128, TC = 16 * NW, LD = kMmaLd, NT = 32 * NW;
    constexpr int TX = attn_mma_stage_rows<NW, NB>();  // rows of a stage buffer
    static_assert(NT == 2 * TC, "one thread per cell of the first two stages");
    static_assert(TX <= 2 * TC, "the preloaded rows cover a whole stage buffer");
    static_assert(NB == 1 || NB == 2, "one or two stage buffers");
    constexpr size_t kStage = attn_mma_stage_bytes<NW, NB>();
    constexpr size_t kMerge = attn_mma_merge_bytes<NW>();
    extern __shared__ __align__(16) char smem_raw[];
    __nv_bfloat16 *Ks = reinterpret_cast<__nv_bfloat16 *>(smem_raw);  // [NB][TX][LD]
    __nv_bfloat16 *Vs = Ks + NB * TX * LD;                               // [NB][TX][LD]
    char *tail = smem_raw + (NB == 1 ? (kStage > kMerge ? kStage : kMerge) : kStage + kMerge);
    int32_t *rows = reinterpret_cast<int32_t *>(tail);                   // [2][TC]
    // [NW][G][D+2] per-warp states: after the stages (two buffers) or over them (one)
    float *mrg = reinterpret_cast<float *>(NB == 1 ? smem_raw : smem_raw + kStage);
    float *cta = reinterpret_cast<float *>(rows + 2 * TC);               // [G][D+2]: o, m, l

    const int S = gridDim.x, s_idx = blockIdx.x, g = blockIdx.y;
    const int64_t qi = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hr = lane >> 2;       // head of this lane's fragment rows
    const int qc = (lane & 3) * 2;  // first column of this lane's fragment pairs
    const int mi = lane >> 3, mj = lane & 7;  // ldmatrix: matrix and row this lane addresses

    // Inside a decode step the preceding kernel only produces the cell list, so the query
    // fragments are built before waiting on it (early_q); a standalone call waits first.
    if (!early_q) {
        pdl_wait();
        QSA_AFTER_WAIT(q);
    }
    // A fragments of the query: rows 0-7 = hi, rows 8-15 = lo, for 8 k-steps of 16 dims
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

    if (early_q) pdl_wait();  // the cell list is complete from here on
    QSA_AFTER_WAIT(pos);
    QSA_AFTER_WAIT(n_cells);
    QSA_AFTER_WAIT(K);
    QSA_AFTER_WAIT(V);
    pdl_trigger();
    // One barrier per stage buffer: a phase completes when every K and V row of the stage
    // has landed (bulk copies count their bytes on it).
    __shared__ __align__(8) uint64_t sbar[2];
    if (tid == 0) {
        mbar_init(&sbar[0], 1);
        mbar_init(&sbar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // phases armed on / seen complete by each stage buffer's barrier (the same in every
    // thread); a wait that gave up stops the CTA's stage loop (its outputs become NaN)
    int armed0 = 0, armed1 = 0, done0 = 0, done1 = 0;
    bool lost = false;
    // A split's cell range is fixed by max_cells, so the positions of its first two stages
    // are loaded together with the list length; entries past the length are dropped once
    // it arrives.  A range a few cells longer than a stage (2,051 cells over 16 splits:
    // 129) would cost every split a second stage: then every split but the last takes
    // whole stages and the last the few cells left.
    int64_t chunk = (max_cells + S - 1) / S;
    if (chunk > TC && chunk % TC != 0 && chunk % TC <= 8) chunk -= chunk % TC;
    const int64_t c0 = (int64_t)s_idx * chunk;
    const int64_t c1max =
        (s_idx == S - 1 || c0 + chunk >= max_cells) ? max_cells : c0 + chunk;
    int64_t n = n_cells[qi];
    int64_t first_row = -1;  // cell c0 + tid: stage tid / TC, slot tid % TC
    if (c0 + tid < c1max)
        first_row = pos ? (int64_t)pos[qi * max_cells + c0 + tid] : qi * max_cells + c0 + tid;
    const bool overflow = n > max_cells;  // truncated list: the result must not be used
    if (overflow || n < 0) n = 0;
    const int64_t c1 = c1max < n ? c1max : n;
    // cells per stage: a split that fits the one-buffer form's wider buffer is one stage
    const int SC = (NB == 1 && c1max - c0 <= TX) ? TX : TC;
    const int ntiles = c1 > c0 ? (int)((c1 - c0 + SC - 1) / SC) : 0;
    {
        int64_t row = c0 + tid < c1 ? first_row : -1;
        if (row < 0 || row >= n_kv) row = -1;
        rows[tid] = (int32_t)row;
    }
    __syncthreads();

    // rows of stage `it` into row buffer `buf` (stages from the third on)
    auto load_rows = [&](int it, int buf) {
        const int64_t base = c0 + (int64_t)it * SC;
        const int tc = (int)min((int64_t)SC, c1 - base);
        int32_t *rb = rows + buf * TC;
        for (int slot = tid; slot < TC; slot += NT) {
            int64_t row = -1;
            if (slot < tc) {
                const int64_t cell = base + slot;
                row = pos ? (int64_t)pos[qi * max_cells + cell] : qi * max_cells + cell;
                if (row < 0 || row >= n_kv) row = -1;
            }
            rb[slot] = (int32_t)row;
        }
        __syncthreads();
    };
    // K and V rows of buffer `buf` into shared memory: one bulk copy of this KV head's 256
    // bytes per row and tensor, all counted on the buffer's barrier.  A skipped row's K is
    // never used (its logit is masked by a select), but its V row is multiplied by p = 0
    // inside the MMA, so it is zero-filled: stale shared memory could hold a NaN pattern.
    auto copy_rows = [&](int buf) {
        const int32_t *rb = rows + buf * TC;
        __nv_bfloat16 *ks = Ks + buf * TX * LD;
        __nv_bfloat16 *vs = Vs + buf * TX * LD;
        for (int e = tid; e < SC * (D / 8); e += NT) {
            const int slot = e / (D / 8), c = e - slot * (D / 8);
            if (rb[slot] < 0) *reinterpret_cast<uint4 *>(vs + slot * LD + c * 8) = make_uint4(0u, 0u, 0u, 0u);
        }
        const int nv = __syncthreads_count(tid < SC && rb[tid] >= 0);
        if (tid == 0) mbar_arrive_expect_tx(&sbar[buf], (uint32_t)nv * 2u * D * 2u);
        if (buf) ++armed1;
        else ++armed0;
        // one thread per row and tensor (NT = 2 * TC); the rows past TC of a wider stage
        // go to the first threads once more
        for (int t = tid; t < 2 * SC; t += NT) {
            const int slot = t >> 1;
            const int64_t row = rb[slot];
            if (row >= 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                if (t & 1)
                    bulk_g2s(vs + slot * LD, V + row * ld_v + (int64_t)g * D, D * 2, &sbar[buf]);
                else
                    bulk_g2s(ks + slot * LD, K + row * ld_k + (int64_t)g * D, D * 2, &sbar[buf]);
            }
        }
    };
    // Wait for buffer `buf`'s stage (bounded), then make its zero-filled rows visible; the
    // CTA agrees on whether any thread's wait gave up.
    auto wait_rows = [&](int buf) {
        const uint32_t par = (uint32_t)((buf ? done1 : done0) & 1);
        const bool ok_w = !lost && mbar_wait(&sbar[buf], par, wc.limit_ns);
        lost = __syncthreads_or(lost || !ok_w) != 0;
        if (!lost) {
            if (buf) ++done1;
            else ++done0;
        }
    };

    if (ntiles > 0) copy_rows(0);
    if (NB == 2 && ntiles > 1) copy_rows(1);
    for (int it = 0; it < ntiles; ++it) {
        const int buf = NB == 2 ? (it & 1) : 0;
        if (NB == 2) {
            if (it >= 1 && it + 1 < ntiles) {
                load_rows(it + 1, buf ^ 1);
                copy_rows(buf ^ 1);
            }
        } else if (it >= 1) {  // one buffer: the previous stage is done (barrier below)
            load_rows(it, 0);
            copy_rows(0);
        }
        wait_rows(buf);
        if (lost) break;  // issue nothing more; what was issued is drained below
        const int tc = (int)min((int64_t)SC, c1 - (c0 + (int64_t)it * SC));
        const __nv_bfloat16 *ks = Ks + buf * TX * LD;
        const __nv_bfloat16 *vs = Vs + buf * TX * LD;
        const int32_t *rw = rows + buf * TC;
        // cells s0 .. s0+15 of the stage into this warp's online-softmax state
        auto group = [&](const int s0) {
        if (s0 < tc) {
            // S = Q K^T for cells s0..s0+15 as two n-tiles of 8 cells
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t b[4];
                const int cell = s0 + (mi >> 1) * 8 + mj;
                ldsm_x4(b, ks + cell * LD + kk * 16 + (mi & 1) * 8);
                mma_16816(sc[0], qa[kk], b[0], b[1]);
                mma_16816(sc[1], qa[kk], b[2], b[3]);
            }
            // logits of head hr for cells s0 + nt*8 + qc + {0,1}: hi row + lo row
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
            // warp-uniform branch: every lane takes part in the MMAs below
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
                // A fragment of P (rows 0-7 hi, 8-15 lo); the K dim is the 16 cells
                float ph[4], pl[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) split_bf16(p[u], ph[u], pl[u]);
                uint32_t pa[4];
                pa[0] = pack_bf16(ph[0], ph[1]);
                pa[1] = pack_bf16(pl[0], pl[1]);
                pa[2] = pack_bf16(ph[2], ph[3]);
                pa[3] = pack_bf16(pl[2], pl[3]);
                // O += P V over 16 dim tiles of 8; ldmatrix.trans gives V^T fragments
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
        };
        group(warp * 16);
        if (NB == 1 && warp == NW - 1) group(TC);  // the extra rows of a wider stage
        __syncthreads();  // this stage is refilled by the next issue()
    }
    // every copy issued lands before the stage area is reused or the CTA leaves (a buffer is
    // re-armed only after its previous phase was seen complete: at most one outstanding)
    if (armed0 > done0) (void)mbar_wait(&sbar[0], (uint32_t)(done0 & 1));
    if (armed1 > done1) (void)mbar_wait(&sbar[1], (uint32_t)(done1 & 1));
    lost = __syncthreads_or(lost);
    if (lost && tid == 0) report_timeout(wc);
    // per-warp state -> shared memory: head hr, dims 8j + qc + {0,1}
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
    __syncthreads();
    // merge the warps: per head the maximum M over the warps and each warp's weight
    // 2^(m_w - M) once, then every output is one weighted sum over the warps
    __shared__ float wf[NW * G];  // warp weights
    __shared__ float hm[G], hl[G];  // per head: M and the weighted l
    if (tid < G) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, mrg[(w * G + tid) * (D + 2) + D]);
        float L = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float *r = mrg + (w * G + tid) * (D + 2);
            const float f = M != -INFINITY ? exp2f(r[D] - M) : 0.0f;
            wf[w * G + tid] = f;
            L = fmaf(f, r[D + 1], L);
        }
        hm[tid] = M;
        hl[tid] = L;
    }
    __syncthreads();
    for (int e = tid; e < G * D; e += NT) {
        const int h = e / D, c = e - h * D;
        float acc = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w) acc = fmaf(wf[w * G + h], mrg[(w * G + h) * (D + 2) + c], acc);
        const float M = hm[h], L = hl[h];
        if (S == 1) {
            float v = L > 0.0f ? acc / L : 0.0f;
            if (overflow || lost) v = __int_as_float(0x7fc00000);
            const int64_t oi = (qi * H_q + (int64_t)g * G + h) * D + c;
            out[oi] = v;
            if (out_host) out_host[oi] = v;
            if (lse && c == 0) {
                const float lv_ = (overflow || lost) ? __int_as_float(0x7fc00000)
                                  : (L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY);
                lse[qi * H_q + g * G + h] = lv_;
                if (lse_host) lse_host[qi * H_q + g * G + h] = lv_;
            }
        } else {
            float *r = cta + h * (D + 2);
            r[c] = acc;
            if (c == 0) {
                r[D] = M;
                r[D + 1] = lost ? -1.0f : L;  // a negative weight sum marks a lost stage
            }
        }
    }
    if (S == 1) return;

    // combine the S CTAs of the cluster: CTA s owns outputs [s*per, (s+1)*per) of G*D.
    // Four threads per output, each reading (m, l, o) of a quarter of the remote states in
    // one round of distributed shared-memory loads; the maximum and the sums meet through
    // two shuffles.
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();  // every CTA's merged state is in its shared memory
    const int per = (G * D + S - 1) / S;
    const int part = tid & 3;
    for (int base = s_idx * per; base < (s_idx + 1) * per; base += NT / 4) {
        const int e0 = base + (tid >> 2);
        const bool live = e0 < (s_idx + 1) * per && e0 < G * D;
        const int e = live ? e0 : 0;
        const int h = e / D, c = e - h * D;
        constexpr int RQ = kMmaMaxCluster / 4;
        float mv[RQ], lv[RQ], ov[RQ];
        float M = -INFINITY;
#pragma unroll
        for (int j = 0; j < RQ; ++j) {
            const int r = part + 4 * j;
            mv[j] = -INFINITY;
            lv[j] = ov[j] = 0.0f;
            if (r < S) {
                const float *rc = cluster.map_shared_rank(cta, r) + h * (D + 2);
                mv[j] = rc[D];
                lv[j] = rc[D + 1];
                ov[j] = rc[c];
            }
            M = fmaxf(M, mv[j]);
        }
        bool bad = false;
#pragma unroll
        for (int j = 0; j < RQ; ++j) bad = bad || lv[j] < 0.0f;
        bad = __any_sync(0xffffffffu, bad && live) || overflow;  // any lost stage of the group
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 1));
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 2));
        float acc = 0.0f, L = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int j = 0; j < RQ; ++j) {
                const float f = exp2f(mv[j] - M);
                acc = fmaf(f, ov[j], acc);
                L = fmaf(f, lv[j], L);
            }
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        L += __shfl_xor_sync(0xffffffffu, L, 1);
        L += __shfl_xor_sync(0xffffffffu, L, 2);
        if (part == 0 && live) {
            float v = L > 0.0f ? acc / L : 0.0f;
            if (bad) v = __int_as_float(0x7fc00000);
            const int64_t oi = (qi * H_q + (int64_t)g * G + h) * D + c;
            out[oi] = v;
            if (out_host) out_host[oi] = v;
            if (lse && c == 0) {
                const float lv_ = bad ? __int_as_float(0x7fc00000)
                                  : (L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY);
                lse[qi * H_q + g * G + h] = lv_;
                if (lse_host) lse_host[qi * H_q + g * G + h] = lv_;
            }
        }
    }
    cluster.sync();  // keep this CTA's state alive until every remote read is done
}

// Combine the S split partials of one (query, head): log-sum-exp weighting.  The split
// maxima and weights go through shared memory once; every output dim then sums its S
// partials with eight independent loads in flight.
__global__ void __launch_bounds__(128)
attn_combine_kernel(const float *__restrict__ part, int S, int H_q, int H_kv, int d_v,
                    const int32_t *__restrict__ n_cells, int64_t max_cells,
                    float *__restrict__ out, float *__restrict__ lse)
{
    extern __shared__ float wsm[];  // [S] weights, [S] sums, [8] reduction scratch
    const int h = blockIdx.x;
    const int64_t qi = blockIdx.y;
    const int G = H_q / H_kv;
    const int g = h / G, hh = h - g * G;
    const int rec = d_v + 4;
    const int64_t stride = (int64_t)G * rec;
    pdl_wait();
    QSA_AFTER_WAIT(part);
    QSA_AFTER_WAIT(n_cells);
    pdl_trigger();
    float *o = out + (qi * H_q + h) * (int64_t)d_v;
    if ((int64_t)n_cells[qi] > max_cells) {
        for (int c = threadIdx.x; c < d_v; c += blockDim.x) o[c] = __int_as_float(0x7fc00000);
        if (lse && threadIdx.x == 0) lse[qi * H_q + h] = __int_as_float(0x7fc00000);
        return;
    }
    const float *pr = part + ((qi * H_kv + g) * (int64_t)S * G + hh) * rec;  // split s: + s*stride
    float *ls = wsm + S;
    float *red = wsm + 2 * S;
    float mx = -INFINITY;
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
        const float mv = pr[s * stride];
        wsm[s] = mv;
        ls[s] = pr[s * stride + 1];
        mx = fmaxf(mx, mv);
    }
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
        const float mv = wsm[s];
        wsm[s] = mv == -INFINITY ? 0.0f : exp2f(mv - mx);
    }
    __syncthreads();
    float L = 0.0f;
    for (int s = 0; s < S; ++s) L = fmaf(wsm[s], ls[s], L);
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    for (int c = threadIdx.x; c < d_v; c += blockDim.x) {
        const float *pc = pr + 4 + c;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        int s = 0;
        for (; s + 8 <= S; s += 8) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = pc[(s + u) * stride];
#pragma unroll
            for (int u = 0; u < 8; ++u) acc[u] = fmaf(wsm[s + u], v[u], acc[u]);
        }
        for (; s < S; ++s) acc[0] = fmaf(wsm[s], pc[s * stride], acc[0]);
        o[c] = (((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]))) * inv;
    }
    if (lse && threadIdx.x == 0) lse[qi * H_q + h] = L > 0.0f ? (mx + log2f(L)) * kLn2 : -INFINITY;
}

// Splits for the tensor-core kernel: about one 128-cell stage per CTA, at most one
// cluster (16 CTAs) per (query, KV head); one split per group when there are many groups.
int attn_mma_splits(int64_t n_q, int H_kv, int64_t max_cells)
{
    const int64_t groups = n_q * (int64_t)H_kv;
    if (groups >= kTargetSMs) return 1;
    int64_t S = (max_cells + kMmaTC - 1) / kMmaTC;
    if (S > kMmaMaxCluster) S = kMmaMaxCluster;
    if (S < 1) S = 1;
    return (int)S;
}

template <int NW, int NB>
cudaError_t launch_attn_mma_t(int S, const float *q, int64_t n_q, int H_q, int H_kv, float scale,
                              const void *K, const void *V, int64_t n_kv, int64_t ld_k,
                              int64_t ld_v, const int32_t *pos, const int32_t *n_cells,
                              int64_t max_cells, float *out, float *lse, cudaStream_t st,
                              bool early_q, float *out_host, float *lse_host)
{
    auto k = attn_mma_kernel<NW, NB>;
    const size_t smem = attn_mma_smem<NW, NB>();
    cudaError_t ea = ensure_kernel_attrs<attn_mma_kernel<NW, NB>>(smem, true);
    if (ea != cudaSuccess) return ea;
    const dim3 grid((unsigned)S, (unsigned)H_kv, (unsigned)n_q);
    return launch(k, grid, dim3(32 * NW), smem, st, S > 1 ? S : 1, q, H_q, H_kv,
                  scale * kLog2e, (const __nv_bfloat16 *)K, (const __nv_bfloat16 *)V, n_kv, ld_k,
                  ld_v, pos, n_cells, max_cells, out, lse, early_q ? 1 : 0, current_wait_ctl(),
                  out_host, lse_host);
}

cudaError_t launch_attn_mma(const float *q, int64_t n_q, int H_q, int H_kv, float scale,
                            const void *K, const void *V, int64_t n_kv, int64_t ld_k, int64_t ld_v,
                            const int32_t *pos, const int32_t *n_cells, int64_t max_cells,
                            float *out, float *lse, cudaStream_t st, bool early_q,
                            float *out_host, float *lse_host)
{
    const int S = attn_mma_splits(n_q, H_kv, max_cells);
    // Several queries per step: n_q * H_kv clusters of S CTAs at one CTA per SM would need a
    // second wave.  With one stage buffer two CTAs share an SM and the step fits one wave.
    // (With one wave either way the two-buffer form is kept: the one-buffer form measured
    // 0.2-0.4 us faster with an fp32 pooled cache but ~3 us slower with a bf16 one.)
    const int64_t ctas = n_q * (int64_t)H_kv * S;
    if (S > 1 && ctas > device_sm_count() && ctas <= 2 * (int64_t)device_sm_count())
        return launch_attn_mma_t<kMmaWarps, 1>(S, q, n_q, H_q, H_kv, scale, K, V, n_kv, ld_k, ld_v,
                                               pos, n_cells, max_cells, out, lse, st, early_q,
                                               out_host, lse_host);
    return launch_attn_mma_t<kMmaWarps, 2>(S, q, n_q, H_q, H_kv, scale, K, V, n_kv, ld_k, ld_v, pos,
                                           n_cells, max_cells, out, lse, st, early_q, out_host,
                                           lse_host);
}

template <typename T, int G>
cudaError_t launch_attn128_t(const float *q, int64_t n_q, int H_q, int H_kv, float scale,
                             const void *K, const void *V, int64_t n_kv, int64_t ld_k, int64_t ld_v,
                             const int32_t *pos, const int32_t *n_cells, int64_t max_cells,
                             float *out, float *lse, float *part, int S, cudaStream_t st)
{
    auto k = attn128_kernel<T, G>;
    const size_t smem = attn128_smem<T, G>();
    cudaError_t ea = ensure_kernel_attrs<attn128_kernel<T, G>>(smem);
    if (ea != cudaSuccess) return ea;
    const dim3 grid((unsigned)S, (unsigned)H_kv, (unsigned)n_q);
    cudaError_t e = launch(k, grid, dim3(128), smem, st, 1, q, H_q, H_kv, scale * kLog2e,
                           (const T *)K, (const T *)V, n_kv, ld_k, ld_v, pos, n_cells, max_cells,
                           out, lse, part);
    if (e != cudaSuccess || S == 1) return e;
    const size_t csmem = sizeof(float) * (2 * (size_t)S + 8);
    return launch(attn_combine_kernel, dim3((unsigned)H_q, (unsigned)n_q), dim3(128), csmem, st,
                  1, (const float *)part, S, H_q, H_kv, 128, n_cells, max_cells, out, lse);
}

template <typename T, int G>
cudaError_t launch_attn_t(const float *q, int64_t n_q, int H_q, int H_kv, int d_k, int d_v,
                          float scale, const void *K, const void *V, int64_t n_kv, int64_t ld_k,
                          int64_t ld_v, const int32_t *pos, const int32_t *n_cells,
                          int64_t max_cells, float *out, float *lse, float *part, int S,
                          cudaStream_t st)
{
    auto k = sparse_attn_kernel<T, G>;
    const size_t smem = attn_smem_bytes(G, d_k, d_v, (int)sizeof(T));
    cudaError_t ea = ensure_kernel_attrs<sparse_attn_kernel<T, G>>(smem);
    if (ea != cudaSuccess) return ea;
    const dim3 grid((unsigned)S, (unsigned)H_kv, (unsigned)n_q);
    cudaError_t e = launch(k, grid, dim3(kAttnThreads), smem, st, 1, q, H_q, H_kv, d_k, d_v,
                           scale * kLog2e, (const T *)K, (const T *)V, n_kv, ld_k, ld_v, pos,
                           n_cells, max_cells, out, lse, part);
    if (e != cudaSuccess || S == 1) return e;
    const size_t csmem = sizeof(float) * (2 * (size_t)S + 8);
    return launch(attn_combine_kernel, dim3((unsigned)H_q, (unsigned)n_q), dim3(128), csmem, st,
                  1, (const float *)part, S, H_q, H_kv, d_v, n_cells, max_cells, out, lse);
}

}  // namespace

size_t attn_smem_bytes_host(int G, int d_k, int d_v, int esize)
{
    return attn_smem_bytes(G, d_k, d_v, esize);
}

int attn_num_splits(int64_t n_q, int H_kv, int64_t max_cells)
{
    const int64_t groups = n_q * (int64_t)H_kv;
    if (groups <= 0) return 1;
    int64_t S = (2 * kTargetSMs + groups - 1) / groups;
    const int64_t max_by_tiles = (max_cells + 63) / 64;  // at least ~64 cells per split
    if (S > max_by_tiles) S = max_by_tiles;
    if (S < 1) S = 1;
    return (int)S;
}

bool attn_uses_mma(qsa_dtype dt, int d_k, int d_v, int G)
{
    return dt == QSA_BF16 && d_k == 128 && d_v == 128 && G == 8;
}

size_t attn_workspace_bytes(int64_t n_q, int H_q, int H_kv, int d_v, int64_t max_cells)
{
    const int S = attn_num_splits(n_q, H_kv, max_cells);
    if (S <= 1 || H_kv <= 0) return 0;
    const int G = H_q / H_kv;
    return sizeof(float) * (size_t)n_q * H_kv * S * G * (size_t)(d_v + 4);
}

size_t attn_partials_bytes(qsa_dtype dt, int64_t n_q, int H_q, int H_kv, int d_k, int d_v,
                           const void *K, const void *V, int64_t ld_k, int64_t ld_v,
                           const int32_t *pos, int64_t max_cells)
{
    if (n_q <= 0 || H_kv <= 0 || H_q % H_kv) return 0;
    const int G = H_q / H_kv;
    // the same order of choices as launch_sparse_attn
    if (attn_uses_rows4(dt, n_q, H_q, H_kv, d_k, d_v, K, V, ld_k, ld_v, pos, max_cells)) return 0;
    if (H_kv == 1 && attn_uses_wide(dt, d_k, d_v, G, K, V, ld_k, ld_v)) return 0;
    if (attn_uses_mma(dt, d_k, d_v, G)) return 0;
    return attn_workspace_bytes(n_q, H_q, H_kv, d_v, max_cells);
}

bool attn_writes_host(qsa_dtype dt, int64_t n_q, int H_q, int H_kv, int d_k, int d_v,
                      const void *K, const void *V, int64_t ld_k, int64_t ld_v,
                      const int32_t *pos, int64_t max_cells)
{
    if (H_kv <= 0 || H_q % H_kv) return false;
    // the same order of choices as launch_sparse_attn
    return !attn_uses_rows4(dt, n_q, H_q, H_kv, d_k, d_v, K, V, ld_k, ld_v, pos, max_cells) &&
           !(H_kv == 1 && attn_uses_wide(dt, d_k, d_v, H_q / H_kv, K, V, ld_k, ld_v)) &&
           attn_uses_mma(dt, d_k, d_v, H_q / H_kv);
}

cudaError_t launch_sparse_attn(const float *q, int64_t n_q, int H_q, int H_kv, int d_k, int d_v,
                               float scale, const void *K, const void *V, qsa_dtype dt,
                               int64_t n_kv, int64_t ld_k, int64_t ld_v, const int32_t *pos,
                               const int32_t *n_cells, int64_t max_cells, float *out,
                               float *lse, float *partials, cudaStream_t st, bool early_q,
                               float *out_host, float *lse_host)
{
    if (n_q == 0) return cudaSuccess;
    const int S = attn_num_splits(n_q, H_kv, max_cells);
    const int G = H_q / H_kv;
    if (attn_uses_rows4(dt, n_q, H_q, H_kv, d_k, d_v, K, V, ld_k, ld_v, pos, max_cells))
        return launch_attn_rows4(q, n_q, H_q, scale, K, V, n_kv, ld_k, ld_v, pos, n_cells,
                                 max_cells, out, lse, st);
    if (H_kv == 1 && attn_uses_wide(dt, d_k, d_v, G, K, V, ld_k, ld_v))  // one latent KV head
        return launch_attn_wide(q, n_q, H_q, H_kv, scale, K, n_kv, ld_k, pos, n_cells, max_cells,
                                out, lse, st);
    if (attn_uses_mma(dt, d_k, d_v, G))
        return launch_attn_mma(q, n_q, H_q, H_kv, scale, K, V, n_kv, ld_k, ld_v, pos, n_cells,
                               max_cells, out, lse, st, early_q, out_host, lse_host);
    if (out_host || lse_host) return cudaErrorNotSupported;  // only the form above writes them
    if (d_k == 128 && d_v == 128 && G <= 8) {
#define QSA_ATTN128_CASE(GG)                                                                   \
    case GG:                                                                                   \
        return dt == QSA_BF16                                                                  \
                   ? launch_attn128_t<__nv_bfloat16, GG>(q, n_q, H_q, H_kv, scale, K, V, n_kv, \
                                                         ld_k, ld_v, pos, n_cells, max_cells,  \
                                                         out, lse, partials, S, st)            \
                   : launch_attn128_t<float, GG>(q, n_q, H_q, H_kv, scale, K, V, n_kv, ld_k,   \
                                                 ld_v, pos, n_cells, max_cells, out, lse,      \
                                                 partials, S, st);
        switch (G) {
            QSA_ATTN128_CASE(1)
            QSA_ATTN128_CASE(2)
            QSA_ATTN128_CASE(4)
            QSA_ATTN128_CASE(8)
            default: break;
        }
#undef QSA_ATTN128_CASE
    }
#define QSA_ATTN_CASE(GG)                                                                   \
    case GG:                                                                                \
        return dt == QSA_BF16                                                               \
                   ? launch_attn_t<__nv_bfloat16, GG>(q, n_q, H_q, H_kv, d_k, d_v, scale, K, \
                                                      V, n_kv, ld_k, ld_v, pos, n_cells,    \
                                                      max_cells, out, lse, partials, S, st) \
                   : launch_attn_t<float, GG>(q, n_q, H_q, H_kv, d_k, d_v, scale, K, V,      \
                                              n_kv, ld_k, ld_v, pos, n_cells, max_cells,    \
                                              out, lse, partials, S, st);
    switch (G) {
        QSA_ATTN_CASE(1)
        QSA_ATTN_CASE(2)
        QSA_ATTN_CASE(4)
        QSA_ATTN_CASE(8)
        QSA_ATTN_CASE(16)
        default: return cudaErrorInvalidValue;
    }
#undef QSA_ATTN_CASE
}

}  // namespace qsa
