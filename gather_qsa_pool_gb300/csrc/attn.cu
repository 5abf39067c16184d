// attn.cu -- attention of each query token over its listed KV cells only (split-K flash
// decoding with an online softmax per split and a log-sum-exp combine).
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "selected K/V gather (COMMON-005)" (attention over the ~2051 selected rows instead of
// the full KV: 2.939 ms -> 42 us per layer at 256k on the pages' GPU) and devotd.net,
// "llama.cpp CDNA sparse attention", sections 2-3 (attention over the listed key
// positions; DKQ 576 with 16 query heads per KV head).
//
// Grid (split, kv head, query).  Each CTA stages 32 listed rows of K and V at a time from
// the full cache into shared memory with 16-byte cp.async (the gather happens on the way
// in: no compact copy round-trips through HBM), double-buffered so the next tile's loads
// overlap this tile's math.  Logits: one warp per cell, lanes split the head dim, one
// warp reduction per query head of the group.  Softmax: one warp per head, one lane per
// cell.  P.V: each thread owns G*d_v/128 output entries.  fp32 throughout.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kAttnThreads = 128;
constexpr int kTile = 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

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

// Combine the S split partials of one (query, head): log-sum-exp weighting.
__global__ void __launch_bounds__(128)
attn_combine_kernel(const float *__restrict__ part, int S, int H_q, int H_kv, int d_v,
                    const int32_t *__restrict__ n_cells, int64_t max_cells,
                    float *__restrict__ out, float *__restrict__ lse)
{
    extern __shared__ float wsm[];  // [S] weights, then [32] reduction scratch
    const int h = blockIdx.x;
    const int64_t qi = blockIdx.y;
    const int G = H_q / H_kv;
    const int g = h / G, hh = h - g * G;
    const int rec = d_v + 4;
    pdl_wait();
    pdl_trigger();
    float *o = out + (qi * H_q + h) * (int64_t)d_v;
    if ((int64_t)n_cells[qi] > max_cells) {
        for (int c = threadIdx.x; c < d_v; c += blockDim.x) o[c] = __int_as_float(0x7fc00000);
        if (lse && threadIdx.x == 0) lse[qi * H_q + h] = __int_as_float(0x7fc00000);
        return;
    }
    const float *pr = part + ((qi * H_kv + g) * (int64_t)S * G + hh) * rec;  // split s at + s*G*rec
    float *red = wsm + S;
    float mx = -INFINITY;
    for (int s = threadIdx.x; s < S; s += blockDim.x) mx = fmaxf(mx, pr[(int64_t)s * G * rec]);
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) mx = fmaxf(mx, red[w]);
    __syncthreads();
    float lsum = 0.0f;
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
        const float m = pr[(int64_t)s * G * rec];
        const float w = (m == -INFINITY) ? 0.0f : exp2f(m - mx);
        wsm[s] = w;
        lsum += w * pr[(int64_t)s * G * rec + 1];
    }
    lsum = warp_sum(lsum);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = lsum;
    __syncthreads();
    float L = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) L += red[w];
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    for (int c = threadIdx.x; c < d_v; c += blockDim.x) {
        float acc0 = 0.0f, acc1 = 0.0f, acc2 = 0.0f, acc3 = 0.0f;
        const float *pc = pr + 4 + c;
        const int64_t stride = (int64_t)G * rec;
        int s = 0;
#pragma unroll 2
        for (; s + 4 <= S; s += 4) {
            acc0 = fmaf(wsm[s], pc[s * stride], acc0);
            acc1 = fmaf(wsm[s + 1], pc[(s + 1) * stride], acc1);
            acc2 = fmaf(wsm[s + 2], pc[(s + 2) * stride], acc2);
            acc3 = fmaf(wsm[s + 3], pc[(s + 3) * stride], acc3);
        }
        for (; s < S; ++s) acc0 = fmaf(wsm[s], pc[s * stride], acc0);
        o[c] = ((acc0 + acc1) + (acc2 + acc3)) * inv;
    }
    if (lse && threadIdx.x == 0) lse[qi * H_q + h] = L > 0.0f ? (mx + log2f(L)) * kLn2 : -INFINITY;
}

template <typename T, int G>
cudaError_t launch_attn128_t(const float *q, int64_t n_q, int H_q, int H_kv, float scale,
                             const void *K, const void *V, int64_t n_kv, int64_t ld_k, int64_t ld_v,
                             const int32_t *pos, const int32_t *n_cells, int64_t max_cells,
                             float *out, float *lse, float *part, int S, cudaStream_t st)
{
    auto k = attn128_kernel<T, G>;
    const size_t smem = attn128_smem<T, G>();
    static bool set = false;
    if (!set) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        set = true;
    }
    const dim3 grid((unsigned)S, (unsigned)H_kv, (unsigned)n_q);
    cudaError_t e = launch(k, grid, dim3(128), smem, st, 1, q, H_q, H_kv, scale * kLog2e,
                           (const T *)K, (const T *)V, n_kv, ld_k, ld_v, pos, n_cells, max_cells,
                           out, lse, part);
    if (e != cudaSuccess || S == 1) return e;
    const size_t csmem = sizeof(float) * ((size_t)S + 32);
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
    static size_t set_bytes = 0;
    if (smem > 48 * 1024 && set_bytes < smem) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        set_bytes = smem;
    }
    const dim3 grid((unsigned)S, (unsigned)H_kv, (unsigned)n_q);
    cudaError_t e = launch(k, grid, dim3(kAttnThreads), smem, st, 1, q, H_q, H_kv, d_k, d_v,
                           scale * kLog2e, (const T *)K, (const T *)V, n_kv, ld_k, ld_v, pos,
                           n_cells, max_cells, out, lse, part);
    if (e != cudaSuccess || S == 1) return e;
    const size_t csmem = sizeof(float) * ((size_t)S + 32);
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
    const int64_t max_by_tiles = (max_cells + kTile - 1) / kTile;
    if (S > max_by_tiles) S = max_by_tiles;
    if (S < 1) S = 1;
    return (int)S;
}

size_t attn_workspace_bytes(int64_t n_q, int H_q, int H_kv, int d_v, int64_t max_cells)
{
    const int S = attn_num_splits(n_q, H_kv, max_cells);
    if (S <= 1 || H_kv <= 0) return 0;
    const int G = H_q / H_kv;
    return sizeof(float) * (size_t)n_q * H_kv * S * G * (size_t)(d_v + 4);
}

cudaError_t launch_sparse_attn(const float *q, int64_t n_q, int H_q, int H_kv, int d_k, int d_v,
                               float scale, const void *K, const void *V, qsa_dtype dt,
                               int64_t n_kv, int64_t ld_k, int64_t ld_v, const int32_t *pos,
                               const int32_t *n_cells, int64_t max_cells, float *out,
                               float *lse, float *partials, cudaStream_t st)
{
    if (n_q == 0) return cudaSuccess;
    const int S = attn_num_splits(n_q, H_kv, max_cells);
    const int G = H_q / H_kv;
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
