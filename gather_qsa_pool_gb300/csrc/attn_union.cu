// attn_union.cu -- grouped-union sparse attention for many consecutive queries (a prefill
// chunk): every group of 16 consecutive queries attends over one dense sequence of K / V
// tiles, the union of the 4-cell blocks its queries selected, on the tcgen05 tensor cores;
// each query's rows are masked to that query's own cells.
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section on
// profiling the Vulkan build (its r2 / r3 table: "QSA union" OFF 221.44 -> ON 263.28 tok/s
// of prompt processing, token generation unchanged) and the COMMON-004 results section (r2's
// grouped-union keeps 128k / 256k prompt processing far ahead of r3, which lacks it).  The
// pages name grouped-union but do not describe it; the form below is this library's reading:
// queries of a chunk that share selected blocks read each shared block once.
//
// Result: for query i and head h, exactly the attention qsa_sparse_attn computes over the
// query's own list (softmax over its cells only), up to rounding.
//
// Kernel 1, union_build_kernel (one CTA per group): a bitmap over the cache's 4-cell blocks
// collects every block a listed cell of the group falls in; a block scan of its words ranks
// the blocks; the union block list is written in ascending order, and for every query one
// bit per union cell (4 per block) says whether the cell is in that query's list.
//
// Kernel 2, attn_union_kernel (one CTA per group and KV head; M = 16 queries x 8 heads =
// 128 rows): warps 0 and 10 stage the union's blocks 16 at a time (a 64-cell tile of K and
// one of V, each cell's 256-byte head row as sixteen 16-byte asynchronous copies written
// straight into the 128-byte-swizzled layout the tensor cores read) into a ring of five
// stages; a stage's barrier completes when the copies of both warps have landed.  (One TMA
// box per block and dim half, 512 bytes each, ran at about 70 cycles a box: the box count,
// not the bytes, bounded the kernel.)  Two softmax groups (warps 2-5 and 6-9, one thread per
// row and group) take alternate tiles, each with its own S, P and O in tensor memory and its
// own online maximum and sum, merged at the end.  Lane 0 of warp 1 issues S = Q K^T (N 64
// cells, K 128 dims; A is the query's bf16 high and low halves, pre-scaled by scale * log2 e,
// in shared memory) into the tile's group's S; lane 0 of warp 11 issues O_g += P V (N 128
// dims, K 64 cells; A is P's high and low halves in tensor memory, V read MN-major).  A
// group's thread reads S, masks it with the row's membership bits, moves its maximum (and
// rescales its O in tensor memory) only when it grows by more than 2^8, and writes P.  While
// one group computes, the other's MMAs run; with the S and P V issued by two threads, one
// issues while the other waits.  Every mbarrier wait is bounded: on a timeout the rows of the
// CTA become NaN, nothing new is issued, what was issued is waited for (bounded) and the
// tensor memory is returned.
#include "attn_union.cuh"

namespace qsa {
namespace {

constexpr int kUG = kUnionGroup;        // queries per group
constexpr int kUHeads = 8;              // query heads per KV head
constexpr int kUM = kUG * kUHeads;      // 128 rows
constexpr int kUD = 128;                // head dim
constexpr int kUTB = 16;                // union blocks per tile
constexpr int kUTC = 4 * kUTB;          // 64 cells per tile
constexpr int kUStages = 5;
constexpr int kUThreads = 384;          // warps 0 and 10 copy, 1 and 11 MMA, 2-9 softmax
constexpr int kUCopyThreads = 64;       // the two copy warps
constexpr int kUGroupWarps = 4;         // softmax warps of a group: one per 32 rows
constexpr float kURescale = 8.0f;       // move the running maximum past 2^8 growth
constexpr int kUMaxBlockWords = 8192;   // bitmap words: 2^18 blocks = 2^20 cells

constexpr uint32_t kTileHalf = kUTC * 128;          // 8 KB: 64 cells x 64 dims bf16
constexpr uint32_t kTileBytes = 2 * kTileHalf;      // 16 KB: one tensor's 64-cell tile
constexpr uint32_t kStageBytes = 2 * kTileBytes;    // K and V
// Tensor memory (512 columns, one row per lane), per softmax group A / B: S fp32 (64
// columns), O fp32 (128), P as bf16 high and low halves (32 each: two cells per column).
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_s(int gi) { return gi ? 64u : 0u; }
__host__ __device__ constexpr uint32_t col_o(int gi) { return gi ? 256u : 128u; }
__host__ __device__ constexpr uint32_t col_p(int gi) { return gi ? 448u : 384u; }
// Q in shared memory: its bf16 high and low halves, each two 64-dim blocks of 128 rows x 128
// bytes (128-byte swizzle), the A operand of S = Q K^T
constexpr uint32_t kQTile = kUM * 128;              // 16 KB
constexpr uint32_t kQBytes = 4 * kQTile;

__host__ __device__ constexpr size_t union_smem_bytes()
{
    return 1024 + (size_t)kUStages * kStageBytes + kQBytes + 256;
}

// Union capacity in blocks for lists of up to max_cells cells: a list of whole blocks plus
// one partial block spans at most ceil(max_cells / 4) + 1 blocks.  Whole tiles.
__host__ __device__ inline int64_t union_cap_blocks(int64_t max_cells)
{
    const int64_t per_q = (max_cells + 3) / 4 + 1;
    return ((kUG * per_q + kUTB - 1) / kUTB) * kUTB;
}

// Per-group workspace: [count, pad] int32 x 4 | blocks [cap] int32 | membership
// [cap / 16 tiles][16 queries][2 words].
__host__ __device__ inline int64_t union_group_words(int64_t max_cells)
{
    const int64_t cap = union_cap_blocks(max_cells);
    return 4 + cap + (cap / kUTB) * kUG * 2;
}

// ------------------------------------------------------------------ kernel 1: the unions

__global__ void __launch_bounds__(1024)
union_build_kernel(const int32_t *__restrict__ pos, const int32_t *__restrict__ n_cells,
                   int64_t max_cells, int64_t n_q, int64_t n_kv, uint32_t *__restrict__ ws)
{
    extern __shared__ __align__(16) uint32_t ush[];
    const int64_t cap = union_cap_blocks(max_cells);
    const int mwords = (int)(cap / 8);                 // membership words per query
    const int nblk = (int)((n_kv + 3) / 4);
    const int nwords = (nblk + 31) / 32;
    uint32_t *bits = ush;                              // [nwords]
    uint32_t *base = bits + nwords;                    // [nwords] exclusive prefix of popcounts
    uint32_t *mem = base + nwords;                     // [16][mwords]
    __shared__ uint32_t warp_tot[32];

    pdl_wait();
    QSA_AFTER_WAIT(pos);
    QSA_AFTER_WAIT(n_cells);
    pdl_trigger();

    const int64_t g = blockIdx.x, q0 = g * kUG;
    const int nq = (int)min((int64_t)kUG, n_q - q0);
    uint32_t *gw = ws + g * union_group_words(max_cells);
    const int tid = threadIdx.x, nt = blockDim.x;
    __shared__ int32_t len_s[kUG];  // cells of each list (0 for a truncated one)
    if (tid < kUG) {
        int64_t n = tid < nq ? (int64_t)n_cells[q0 + tid] : 0;
        if (n < 0 || n > max_cells) n = 0;
        len_s[tid] = (int32_t)n;
    }
    for (int w = tid; w < nwords; w += nt) bits[w] = 0u;
    for (int w = tid; w < kUG * mwords; w += nt) mem[w] = 0u;
    __syncthreads();
    // Each list's cells by two warps (16 lists x 2 = the CTA's 32 warps), 32 consecutive cells
    // per warp load (lane = cell), eight such loads in flight per lane.  A list's cells
    // ascend, so the lanes' bitmap words never decrease along the warp.
    constexpr int kU = 8;
    const int warp = tid >> 5, lane = tid & 31;
    const int li_w = warp >> 1;
    const int len_w = li_w < nq ? len_s[li_w] : 0;
    const int32_t *lp = pos + (q0 + li_w) * max_cells;
    auto or_lanes = [&](uint32_t *dst, bool valid, uint32_t word, uint32_t bit) {
        // a block's four cells sit in four consecutive lanes and set bits of one word: within
        // each quad of lanes, the first lane of every run of one word collects the run's bits
        // (the words never decrease along the warp) and alone issues the atomic
        const uint32_t wk = valid ? word : 0xffffffffu - (uint32_t)lane;  // invalid: own run
        uint32_t acc = valid ? bit : 0u;
        uint32_t wo = __shfl_xor_sync(0xffffffffu, wk, 1);
        uint32_t ao = __shfl_xor_sync(0xffffffffu, acc, 1);
        if (wo == wk) acc |= ao;
        wo = __shfl_xor_sync(0xffffffffu, wk, 2);
        ao = __shfl_xor_sync(0xffffffffu, acc, 2);
        if (wo == wk) acc |= ao;
        const uint32_t wp = __shfl_up_sync(0xffffffffu, wk, 1);
        if (valid && ((lane & 3) == 0 || wp != wk)) atomicOr(&dst[word], acc);
    };
    auto for_each_chunk = [&](auto &&f) {
        for (int e0 = (warp & 1) * 32; e0 < len_w; e0 += 64 * kU) {  // warp-uniform
            int32_t c[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int e = e0 + 64 * u + lane;
                c[u] = e < len_w ? lp[e] : -1;
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) f(c[u]);
        }
    };

    // every valid cell of every (non-truncated) list marks its block
    for_each_chunk([&](int32_t c) {
        const bool valid = c >= 0 && c < n_kv;
        const int b = valid ? c >> 2 : 0;
        or_lanes(bits, valid, (uint32_t)(b >> 5), 1u << (b & 31));
    });
    __syncthreads();

    // exclusive scan of the words' popcounts: each thread a contiguous run of words
    const int per = (nwords + nt - 1) / nt;
    const int w0 = tid * per, w1 = min(nwords, w0 + per);
    uint32_t run = 0;
    for (int w = w0; w < w1; ++w) run += __popc(bits[w]);
    uint32_t incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        uint32_t t = lane < (nt >> 5) ? warp_tot[lane] : 0u;
        uint32_t ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += v;
        }
        warp_tot[lane] = ti - t;  // exclusive prefix of the warps' totals
    }
    __syncthreads();
    uint32_t acc = warp_tot[warp] + incl - run;
    for (int w = w0; w < w1; ++w) {
        base[w] = acc;
        acc += __popc(bits[w]);
    }
    __syncthreads();
    const uint32_t total = nwords ? base[nwords - 1] + __popc(bits[nwords - 1]) : 0u;
    if ((int64_t)total > cap) {
        // lists spanning more blocks than the workspace holds: the group's rows become NaN
        if (tid == 0) gw[0] = 0xffffffffu;
        return;
    }
    // the union's blocks, ascending
    int32_t *ublk = reinterpret_cast<int32_t *>(gw + 4);
    for (int w = w0; w < w1; ++w) {
        uint32_t m = bits[w];
        uint32_t r = base[w];
        while (m) {
            const int bit = __ffs(m) - 1;
            m &= m - 1;
            ublk[r++] = w * 32 + bit;
        }
    }
    // membership: bit 4j + (c & 3) of query li's words for cell c of union block j
    for_each_chunk([&](int32_t c) {
        const bool valid = c >= 0 && c < n_kv;
        const int b = valid ? c >> 2 : 0;
        const uint32_t j = base[b >> 5] + __popc(bits[b >> 5] & ((1u << (b & 31)) - 1u));
        const uint32_t k = 4 * j + (uint32_t)(c & 3);
        or_lanes(mem, valid, (uint32_t)(li_w * mwords) + (k >> 5), 1u << (k & 31));
    });
    __syncthreads();
    // out in tile-major order: [tile][query][2 words], 64 cells per tile
    uint32_t *gm = gw + 4 + cap;
    const int n_tiles = (int)((total + kUTB - 1) / kUTB);
    for (int e = tid; e < n_tiles * kUG * 2; e += nt) {
        const int t = e / (kUG * 2), li = (e / 2) % kUG, k = e & 1;
        gm[e] = li < nq ? mem[li * mwords + 2 * t + k] : 0u;
    }
    if (tid == 0) gw[0] = total;
}

// ------------------------------------------------------------------ tcgen05 helpers

// K-major operand, 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(16u >> 4) << 16;       // leading byte offset: unused here
    d |= (uint64_t)(1024u >> 4) << 32;     // stride byte offset: next 8 rows
    d |= (uint64_t)1 << 46;                // descriptor version
    d |= (uint64_t)2 << 61;                // 128-byte swizzle
    return d;
}

// MN-major operand, 128-byte swizzle: each 128-byte row holds 64 consecutive N elements of
// one k; the next 64 N elements start `mn_stride` bytes on (leading byte offset); the next
// 8 k rows 1024 bytes on (stride byte offset).
__device__ __forceinline__ uint64_t desc_mnmajor_sw128(uint32_t saddr, uint32_t mn_stride)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((mn_stride >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, M 128, the given N,
// B MN-major when b_mn.
__host__ __device__ constexpr uint32_t idesc_m128(int n, bool b_mn)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn ? (1u << 16) : 0u) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kUM >> 4) << 24);
}

// One M128 MMA of this CTA with A read from tensor memory (row i in lane i, two bf16 per
// 32-bit column, k-contiguous) and B from shared memory.
__device__ __forceinline__ void umma_m128_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One M128 MMA of this CTA with A and B both from shared memory.
__device__ __forceinline__ void umma_m128_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the barrier once every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 16 bytes from global to shared memory, or zeros when src_bytes is 0 (src is then not read).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// Arrive on the barrier once every cp.async this thread issued so far has landed (the arrival
// is counted in the barrier's initial count).
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v)
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *v)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *v)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
}

// 2^x by the hardware's approximate exponential (2^-inf = +0).
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Barrier of the eight softmax warps (named barrier 1) that also returns the AND of `v` over
// their 256 threads.
__device__ __forceinline__ bool softmax_and(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, c;\n\t"
        "setp.ne.u32 c, %1, 0;\n\t"
        "bar.red.and.pred p, 1, 256, c;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// A bounded mbarrier wait of a whole warp: lane 0 polls, the warp learns the outcome from it
// and is ordered after the completed phase by the warp barrier.  (Thirty-two lanes polling
// the same barrier load the shared-memory pipe that the MMA issue and the tensor-memory
// accesses of the other warps go through.)
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, limit_ns);
    ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
    __syncwarp();
    return ok;
}

// ------------------------------------------------------------------ kernel 2: attention

__global__ void __launch_bounds__(kUThreads, 1)
attn_union_kernel(const __nv_bfloat16 *__restrict__ K, const __nv_bfloat16 *__restrict__ V,
                  int64_t n_kv, int64_t ld_k, int64_t ld_v, const float *__restrict__ q, int64_t n_q, int H_q, float scale_log2,
                  const int32_t *__restrict__ n_cells, int64_t max_cells,
                  const uint32_t *__restrict__ ws, float *__restrict__ out,
                  float *__restrict__ lse, const WaitCtl wc)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char *sKV = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    // [stage][K, V][2 dim halves][64 cells][128 B], 128-byte swizzle; then Q
    unsigned char *sQ = sKV + kUStages * kStageBytes;  // [hi, lo][dim block][128 rows][128 B]
    uint64_t *kv_full = reinterpret_cast<uint64_t *>(sQ + kQBytes);
    uint64_t *kv_empty = kv_full + kUStages;
    uint64_t *s_full = kv_empty + kUStages;          // [group] S(t) in the group's buffer
    uint64_t *s_empty = s_full + 2;                  // [group] the group read S(t)
    uint64_t *p_full = s_empty + 2;                  // [group] P(t) in the group's buffer
    uint64_t *o_done = p_full + 2;                   // [group] the group's last P V done
    uint64_t *q_ready = o_done + 2;
    uint64_t *drain = q_ready + 1;                   // [2] each issuing thread's MMAs done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 2);
    // each group's row maxima and sums ([2][2][128] floats) for the final merge, over Q's
    // tiles once every MMA has completed
    float *xch = reinterpret_cast<float *>(sQ);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t g = blockIdx.x;
    const int kvh = blockIdx.y;
    const int64_t gwords = union_group_words(max_cells);
    const int64_t cap = union_cap_blocks(max_cells);

    if (tid == 0) {
        for (int s = 0; s < kUStages; ++s) {
            mbar_init(&kv_full[s], kUCopyThreads);
            mbar_init(&kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&s_empty[b], kUGroupWarps);
            mbar_init(&p_full[b], kUGroupWarps);
            mbar_init(&o_done[b], 1);
        }
        mbar_init(q_ready, 2 * kUGroupWarps);
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    pdl_wait();
    QSA_AFTER_WAIT(q);
    QSA_AFTER_WAIT(n_cells);
    QSA_AFTER_WAIT(ws);
    pdl_trigger();
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    const uint32_t *gw = ws + g * gwords;
    const uint32_t ucount = gw[0];
    const bool bad_group = ucount == 0xffffffffu;
    const int n_tiles = bad_group ? 0 : (int)((ucount + kUTB - 1) / kUTB);
    const int32_t *ublk = reinterpret_cast<const int32_t *>(gw + 4);
    const uint32_t *gmem = gw + 4 + cap;
    bool ok = true;

    if (warp == 0 || warp == 10) {
        // ---- copies: warp p fills rows 32p .. 32p + 31 (blocks 8p .. 8p + 7) of the tile's
        // K and V; lane = 16 * (row parity) + 16-byte chunk of the 256-byte head row
        const int p = warp == 0 ? 0 : 1;
        const int c = lane & 15, sub = lane >> 4;
        const uint32_t half_off = (uint32_t)(c >> 3) * kTileHalf;
        const unsigned char *Kc =
            reinterpret_cast<const unsigned char *>(K) + (int64_t)kvh * kUD * 2 + c * 16;
        const unsigned char *Vc =
            reinterpret_cast<const unsigned char *>(V) + (int64_t)kvh * kUD * 2 + c * 16;
        const int64_t ldk_b = ld_k * 2, ldv_b = ld_v * 2;
        int armed = 0;
        // lanes 0-7 hold the block indices of this warp's eight blocks, one tile ahead
        auto blk_of = [&](int t) -> int32_t {
            const int64_t u = (int64_t)t * kUTB + 8 * p + (lane & 7);
            return u < ucount ? ublk[u] : ublk[0];
        };
        int32_t blk_next = n_tiles > 0 ? blk_of(0) : 0;
        for (int t = 0; t < n_tiles; ++t, ++armed) {
            const int s = t % kUStages;
            const int32_t blk = blk_next;
            if (t + 1 < n_tiles) blk_next = blk_of(t + 1);
            if (t >= kUStages &&
                !warp_wait(&kv_empty[s], (uint32_t)((t / kUStages) - 1) & 1u, wc.limit_ns)) {
                ok = false;
                break;
            }
            const uint32_t st = smem_u32(sKV + s * kStageBytes) + half_off;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int rr = 2 * i + sub;                 // row within this warp's 32
                const int r = 32 * p + rr;                  // row (cell) of the tile
                const int32_t b = __shfl_sync(0xffffffffu, blk, i >> 1);
                const int64_t cell = 4 * (int64_t)b + (rr & 3);
                const bool in = cell < n_kv;
                const int64_t row = in ? cell : 0;
                const uint32_t dst = st + (uint32_t)r * 128 + ((uint32_t)((c & 7) ^ (r & 7)) << 4);
                cp_async16(dst, Kc + row * ldk_b, in ? 16u : 0u);
                cp_async16(dst + kTileBytes, Vc + row * ldv_b, in ? 16u : 0u);
            }
            cp_async_arrive(&kv_full[s]);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        // every armed stage has completed its barrier before the CTA may leave
        for (int s = 0; s < kUStages && lane == 0; ++s) {
            const int uses = armed / kUStages + (s < armed % kUStages ? 1 : 0);
            if (uses > 0 && !mbar_wait(&kv_full[s], (uint32_t)(uses - 1) & 1u)) ok = false;
        }
    } else if (warp == 1 || warp == 11) {
        // ---- MMA issuers: lane 0 of warp 1 issues every S, lane 0 of warp 11 every P V, so
        // that one issues while the other waits (a wait or commit costs its thread over a
        // hundred cycles, and the tensor queue would drain meanwhile).  Tile t belongs to
        // softmax group t & 1: S(t) = Q K(t)^T into the group's S once K / V(t) landed and the
        // group read S(t - 2); O_g += P(t) V(t) once the group wrote P(t), which it does only
        // after reading S(t), so the stage is free when this P V completes.  The descriptors
        // of stage 0 and of Q are built once: a stage, dim block or k step moves only their
        // start-address field (bits 0-13, 16-byte units; shared addresses stay below 256 KB,
        // so the add never carries out of it).
        const bool is_s = warp == 1;
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_m128(kUTC, false);
            constexpr uint32_t id_o = idesc_m128(kUD, true);
            const uint64_t dk0 = desc_kmajor_sw128(smem_u32(sKV));
            const uint64_t dv0 = desc_mnmajor_sw128(smem_u32(sKV + kTileBytes), kTileHalf);
            const uint64_t dq0 = desc_kmajor_sw128(smem_u32(sQ));
            const uint32_t dk_lo = (uint32_t)dk0, dk_hi = (uint32_t)(dk0 >> 32);
            const uint32_t dv_lo = (uint32_t)dv0, dv_hi = (uint32_t)(dv0 >> 32);
            const uint32_t dq_lo = (uint32_t)dq0, dq_hi = (uint32_t)(dq0 >> 32);
            if (is_s && n_tiles > 0 && !mbar_wait(q_ready, 0, wc.limit_ns)) ok = false;
            for (int t = 0; ok && t < n_tiles; ++t) {
                const int s = t % kUStages, b = t & 1;
                if (is_s) {
                    if (!mbar_wait(&kv_full[s], (uint32_t)(t / kUStages) & 1u, wc.limit_ns)) {
                        ok = false;
                        break;
                    }
                    // the stage was written by ordinary (generic-proxy) copies; the tensor
                    // cores read it through the async proxy
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    if (t >= 2 &&
                        !mbar_wait(&s_empty[b], (uint32_t)((t - 2) >> 1) & 1u, wc.limit_ns)) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t ks = dk_lo + (uint32_t)s * (kStageBytes >> 4);
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
#pragma unroll
                        for (int k16 = 0; k16 < kUD / 16; ++k16) {
                            const uint32_t kb = (uint32_t)(k16 >> 2), ko = (uint32_t)(k16 & 3) * 32;
                            const uint32_t qa = dq_lo + (((uint32_t)part * 2 + kb) * kQTile + ko) / 16;
                            const uint32_t kd = ks + (kb * kTileHalf + ko) / 16;
                            umma_m128_ss(tmem + col_s(b), ((uint64_t)dq_hi << 32) | qa,
                                         ((uint64_t)dk_hi << 32) | kd, id_s,
                                         (part | k16) ? 1u : 0u);
                        }
                    }
                    umma_commit(&s_full[b]);
                } else {
                    if (!mbar_wait(&p_full[b], (uint32_t)(t >> 1) & 1u, wc.limit_ns)) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t vs = dv_lo + (uint32_t)s * (kStageBytes >> 4);
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
#pragma unroll
                        for (int k16 = 0; k16 < kUTC / 16; ++k16)
                            umma_m128_ta(tmem + col_o(b),
                                         tmem + col_p(b) + (uint32_t)(part * 32 + k16 * 8),
                                         ((uint64_t)dv_hi << 32) | (vs + (uint32_t)k16 * (2048 / 16)),
                                         id_o, (t >= 2 || part || k16) ? 1u : 0u);
                    }
                    umma_commit(&o_done[b]);
                    umma_commit(&kv_empty[s]);
                }
            }
            // every MMA this thread issued has completed before the tensor memory is freed
            umma_commit(&drain[is_s ? 0 : 1]);
            if (!mbar_wait(&drain[is_s ? 0 : 1], 0)) ok = false;
        }
    } else {
        // ---- softmax, in two groups that take alternate tiles (group gi: warps 2-5 or 6-9,
        // tiles gi, gi + 2, ...), one thread per row (row = 8 * query + head) and group, all
        // 64 columns of the group's tiles; each group keeps its own online maximum, sum and O
        const int quarter = warp & 3;
        const int gi = (warp - 2) >> 2;
        const int r = quarter * 32 + lane;
        const int li = r >> 3;
        const int64_t qi = g * kUG + li;
        const int h = kvh * kUHeads + (r & 7);
        const bool live = qi < n_q;
        const int64_t n = live ? (int64_t)n_cells[qi] : 0;
        const bool trunc = n > max_cells;
        const uint32_t lrow = (uint32_t)(quarter * 32) << 16;
        const uint32_t colS = tmem + lrow + col_s(gi), colP = tmem + lrow + col_p(gi);
        const uint32_t colO = tmem + lrow + col_o(gi);
        // dims 64*gi .. of the row's query, pre-scaled, as bf16 high and low halves into Q's
        // shared-memory tiles (128-byte swizzle: chunk c of row r at chunk c ^ (r % 8))
        {
            const float *qr = q + (qi * H_q + h) * (int64_t)kUD + gi * 64;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float x[8];
                if (live) {
                    const float4 a = *reinterpret_cast<const float4 *>(qr + 8 * c);
                    const float4 b = *reinterpret_cast<const float4 *>(qr + 8 * c + 4);
                    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
                    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = 0.0f;
                }
                uint32_t wh[4], wl[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float x0 = x[e] * scale_log2, x1 = x[e + 1] * scale_log2;
                    const float h0 = __bfloat162float(__float2bfloat16_rn(x0));
                    const float h1 = __bfloat162float(__float2bfloat16_rn(x1));
                    wh[e / 2] = pack_bf16(h0, h1);
                    wl[e / 2] = pack_bf16(x0 - h0, x1 - h1);
                }
                const uint32_t off = (uint32_t)r * 128 + ((uint32_t)(c ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(sQ + (uint32_t)gi * kQTile + off) =
                    make_uint4(wh[0], wh[1], wh[2], wh[3]);
                *reinterpret_cast<uint4 *>(sQ + (uint32_t)(2 + gi) * kQTile + off) =
                    make_uint4(wl[0], wl[1], wl[2], wl[3]);
            }
            // written by this thread (generic proxy), read by the tensor cores (async proxy)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(q_ready);
        }
        float m_ref = -INFINITY, l = 0.0f;
        const int n_mine = n_tiles > gi ? (n_tiles - gi + 1) / 2 : 0;
        uint2 mw = make_uint2(0u, 0u);
        if (n_mine > 0) mw = *reinterpret_cast<const uint2 *>(gmem + ((int64_t)gi * kUG + li) * 2);
        for (int j = 0; j < n_mine; ++j) {
            const int t = gi + 2 * j;
            const uint2 w = (live && !trunc) ? mw : make_uint2(0u, 0u);
            if (j + 1 < n_mine)  // the next tile's membership words, ahead
                mw = *reinterpret_cast<const uint2 *>(gmem + ((int64_t)(t + 2) * kUG + li) * 2);
            // waits are warp-uniform: the tensor-memory accesses below need the whole warp
            if (!(ok && warp_wait(&s_full[gi], (uint32_t)j & 1u, wc.limit_ns))) {
                ok = false;
                break;
            }
            float x[64];
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            tmem_ld32(colS, x);
            tmem_ld32(colS + 32, x + 32);
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[gi]);
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                x[e] = ((w.x >> e) & 1u) ? x[e] : -INFINITY;
                x[32 + e] = ((w.y >> e) & 1u) ? x[32 + e] : -INFINITY;
                mx[e & 3] = fmaxf(mx[e & 3], fmaxf(x[e], x[32 + e]));
            }
            const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            float alpha = 1.0f;
            bool move = false;
            if (mt > m_ref + kURescale) {  // also the first finite maximum (m_ref = -inf)
                move = true;
                alpha = m_ref == -INFINITY ? 0.0f : ex2_approx(m_ref - mt);
            }
            const bool rescale = __any_sync(0xffffffffu, move && m_ref != -INFINITY);
            if (move) {
                l *= alpha;
                m_ref = mt;
            }
            const float mu = m_ref == -INFINITY ? 0.0f : m_ref;
            // the group's P buffer and O are free once its P V(t - 2) is done
            if (j >= 1 && !warp_wait(&o_done[gi], (uint32_t)(j - 1) & 1u, wc.limit_ns)) {
                ok = false;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (rescale) {
#pragma unroll 1
                for (int c = 0; c < (int)kUD; c += 32) {
                    float o[32];
                    tmem_ld32(colO + (uint32_t)c, o);
                    uint32_t ou[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) ou[e] = __float_as_uint(o[e] * alpha);
                    tmem_st32(colO + (uint32_t)c, ou);
                }
            }
            // P(t) relative to the (possibly moved) maximum: high halves in columns 0-31 of
            // the group's P, low halves in 32-63, two cells per column; in two halves of 32
            // cells
            float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t ph[16], pl[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float p0 = ex2_approx(x[32 * hf + e] - mu);
                    const float p1 = ex2_approx(x[32 * hf + e + 1] - mu);
                    ls[(e >> 1) & 3] += p0 + p1;
                    const uint32_t hb = pack_bf16(p0, p1);
                    const float h0 = __uint_as_float(hb << 16), h1 = __uint_as_float(hb & 0xffff0000u);
                    ph[e / 2] = hb;
                    pl[e / 2] = pack_bf16(p0 - h0, p1 - h1);
                }
                tmem_st16(colP + (uint32_t)(16 * hf), ph);
                tmem_st16(colP + 32 + (uint32_t)(16 * hf), pl);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            tmem_wait_st();
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[gi]);
        }
        // the group's O is final once its last P V is done
        if (ok && n_mine > 0 &&
            !warp_wait(&o_done[gi], (uint32_t)(n_mine - 1) & 1u, wc.limit_ns))
            ok = false;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        // merge the two groups' states: m = max(m_A, m_B), each O and sum scaled by 2^(m_g - m).
        // Every softmax warp arrives at each of these barriers once, after its loop; past the
        // first, both groups saw their last P V done (so every S, which precedes the P V of
        // its tile, too), or gave up waiting and the rows are NaN
        ok = softmax_and(ok);
        if (ok) {
            xch[(2 * gi) * kUM + r] = m_ref;
            xch[(2 * gi + 1) * kUM + r] = l;
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        const float mA = ok ? xch[r] : 0.0f, lA = ok ? xch[kUM + r] : 0.0f;
        const float mB = ok ? xch[2 * kUM + r] : 0.0f, lB = ok ? xch[3 * kUM + r] : 0.0f;
        const float mm = fmaxf(mA, mB);
        const float sA = mA == -INFINITY ? 0.0f : ex2_approx(mA - mm);
        const float sB = mB == -INFINITY ? 0.0f : ex2_approx(mB - mm);
        const float lt = lA * sA + lB * sB;
        const bool nan_rows = !ok || bad_group || trunc;
        const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
        // a group that took no tile has no O (tensor memory never written)
        const bool has_a = ok && n_tiles > 0, has_b = ok && n_tiles > 1;
#pragma unroll 1
        for (int c = 64 * gi; c < 64 * gi + 64; c += 32) {
            float oa[32], ob[32];
            if (has_a) {
                tmem_ld32(tmem + lrow + col_o(0) + (uint32_t)c, oa);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) oa[e] = 0.0f;
            }
            if (has_b) {
                tmem_ld32(tmem + lrow + col_o(1) + (uint32_t)c, ob);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) ob[e] = 0.0f;
            }
            if (live) {
                float *dst = out + (qi * H_q + h) * (int64_t)kUD + c;
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    float4 v;
                    v.x = (oa[e] * sA + ob[e] * sB) * inv;
                    v.y = (oa[e + 1] * sA + ob[e + 1] * sB) * inv;
                    v.z = (oa[e + 2] * sA + ob[e + 2] * sB) * inv;
                    v.w = (oa[e + 3] * sA + ob[e + 3] * sB) * inv;
                    *reinterpret_cast<float4 *>(dst + e) =
                        nan_rows ? make_float4(NAN, NAN, NAN, NAN) : v;
                }
            }
        }
        if (live && lse && gi == 0)
            lse[qi * H_q + h] = nan_rows ? NAN
                                         : (lt > 0.0f ? (mm + log2f(lt)) * 0.6931471805599453f
                                                      : -INFINITY);
    }

    if (!ok) report_timeout(wc);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

}  // namespace

int64_t attn_union_max_kv() { return (int64_t)kUMaxBlockWords * 32 * 4; }

size_t attn_union_workspace_bytes(int64_t n_q, int64_t max_cells)
{
    if (n_q <= 0 || max_cells < 0) return 0;
    const int64_t groups = (n_q + kUG - 1) / kUG;
    return (size_t)groups * (size_t)union_group_words(max_cells) * 4;
}

bool attn_union_shape_ok(qsa_dtype dt, int H_q, int H_kv, int d_k, int d_v, const void *K,
                         const void *V, int64_t ld_k, int64_t ld_v)
{
    return dt == QSA_BF16 && H_kv >= 1 && H_q == kUHeads * H_kv && d_k == kUD && d_v == kUD &&
           ld_k % 8 == 0 && ld_v % 8 == 0 && ld_k >= (int64_t)H_kv * kUD &&
           ld_v >= (int64_t)H_kv * kUD &&
           ((reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V)) & 15) == 0;
}

qsa_status launch_attn_union(const float *q, int64_t n_q, int H_q, int H_kv, float scale,
                             const void *K, const void *V, int64_t n_kv, int64_t ld_k,
                             int64_t ld_v, const int32_t *pos, const int32_t *n_cells,
                             int64_t max_cells, float *out, float *lse, void *workspace,
                             cudaStream_t st)
{
    if (n_q == 0) return QSA_OK;
    const int64_t groups = (n_q + kUG - 1) / kUG;
    const int64_t cap = union_cap_blocks(max_cells);
    const int nblk = (int)((n_kv + 3) / 4);
    const int nwords = (nblk + 31) / 32;
    const size_t bsmem = sizeof(uint32_t) * (2 * (size_t)nwords + (size_t)kUG * (cap / 8));
    if (bsmem > 227 * 1024) return QSA_ERR_UNSUPPORTED;
    uint32_t *ws = static_cast<uint32_t *>(workspace);
    if (ensure_kernel_attrs<union_build_kernel>(bsmem) != cudaSuccess) return QSA_ERR_CUDA;
    cudaError_t e = launch(union_build_kernel, dim3((unsigned)groups), dim3(1024), bsmem, st, 1, pos,
                           n_cells, max_cells, n_q, n_kv, ws);
    if (e != cudaSuccess) return QSA_ERR_CUDA;
    if (ensure_kernel_attrs<attn_union_kernel>(union_smem_bytes()) != cudaSuccess)
        return QSA_ERR_CUDA;
    e = launch(attn_union_kernel, dim3((unsigned)groups, (unsigned)H_kv), dim3(kUThreads),
               union_smem_bytes(), st, 1, static_cast<const __nv_bfloat16 *>(K),
               static_cast<const __nv_bfloat16 *>(V), n_kv, ld_k, ld_v, q, n_q, H_q, scale * 1.4426950408889634f,
               n_cells, max_cells, (const uint32_t *)ws, out, lse, current_wait_ctl());
    return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}

}  // namespace qsa
