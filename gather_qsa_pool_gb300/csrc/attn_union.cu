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
// straight into the 128-byte-swizzled layout the tensor cores read) into a ring of six
// stages; a stage's barrier completes when the copies of both warps have landed.  (One TMA
// box per block and dim half, 512 bytes each, ran at about 70 cycles a box: the box count,
// not the bytes, bounded the kernel.)  Warp 1 issues the MMAs -- S = Q K^T (N 64 cells, K
// 128 dims; A is the query's bf16 high and low halves, pre-scaled by scale * log2 e, held in
// tensor memory) into one of two tensor-memory buffers, and O += P V (N 128 dims, K 64 cells,
// V read MN-major; A is P's high and low halves, in one of two tensor-memory buffers) into a
// third, two tiles behind the S it follows.  Warps 2-9 (two threads per row, one per half of
// the tile's columns) read S, mask it with the row's membership bits, keep an online maximum
// that is moved (and O rescaled in tensor memory) only when it grows by more than 2^8, write
// P into tensor memory, and at the end divide O by the row sum.  Every mbarrier wait is
// bounded: on a timeout the rows of the CTA become NaN, nothing new is issued, what was
// issued is waited for (bounded) and the tensor memory is returned.
#include "attn_union.cuh"

namespace qsa {
namespace {

constexpr int kUG = kUnionGroup;        // queries per group
constexpr int kUHeads = 8;              // query heads per KV head
constexpr int kUM = kUG * kUHeads;      // 128 rows
constexpr int kUD = 128;                // head dim
constexpr int kUTB = 16;                // union blocks per tile
constexpr int kUTC = 4 * kUTB;          // 64 cells per tile
constexpr int kUStages = 6;
constexpr int kUThreads = 352;          // warps 0 and 10 copy, warp 1 MMA, warps 2-9 softmax
constexpr int kUCopyThreads = 64;       // the two copy warps
constexpr int kUEpiWarps = 8;           // two per row: one per half of the tile's columns
constexpr float kURescale = 8.0f;       // move the running maximum past 2^8 growth
constexpr int kUMaxBlockWords = 8192;   // bitmap words: 2^18 blocks = 2^20 cells

constexpr uint32_t kTileHalf = kUTC * 128;          // 8 KB: 64 cells x 64 dims bf16
constexpr uint32_t kTileBytes = 2 * kTileHalf;      // 16 KB: one tensor's 64-cell tile
constexpr uint32_t kStageBytes = 2 * kTileBytes;    // K and V
// Tensor memory (512 columns, one row per lane): S[0], S[1] fp32 (64 each), O fp32 (128),
// Q's bf16 high and low halves (64 each: two dims per column), P[0], P[1] as bf16 high and
// low halves (32 each: two cells per column).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 128, kColQh = 256, kColQl = 320, kColP = 384;

__host__ __device__ constexpr size_t union_smem_bytes()
{
    return 1024 + (size_t)kUStages * kStageBytes + 256 + 6 * kUM * sizeof(float);
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
    // ascend, so the lanes' bitmap words never decrease along the warp: a segmented OR scan
    // over the lanes leaves each word's bits in the last lane holding that word, which alone
    // issues the shared atomic.
    constexpr int kU = 8;
    const int warp = tid >> 5, lane = tid & 31;
    const int li_w = warp >> 1;
    const int len_w = li_w < nq ? len_s[li_w] : 0;
    const int32_t *lp = pos + (q0 + li_w) * max_cells;
    auto or_lanes = [&](uint32_t *dst, bool valid, int64_t word, uint32_t bit) {
        const int64_t wk = valid ? word : -1 - (int64_t)lane;  // invalid lanes: own segment
        uint32_t acc = valid ? bit : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, acc, o);
            const int64_t w2 = __shfl_up_sync(0xffffffffu, wk, o);
            if (lane >= o && w2 == wk) acc |= v;
        }
        const int64_t wn = __shfl_down_sync(0xffffffffu, wk, 1);
        if (valid && (lane == 31 || wn != wk)) atomicOr(&dst[word], acc);
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
        or_lanes(bits, valid, b >> 5, 1u << (b & 31));
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
        or_lanes(mem, valid, (int64_t)li_w * mwords + (k >> 5), 1u << (k & 31));
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

// Barrier of the two softmax warps that own the same 32 rows (named barrier 1 + quarter)
// that also returns the AND of `v` over their 64 threads: both warps take every decision that
// follows it the same way (neither may leave a loop the other stays in).
__device__ __forceinline__ bool pair_and(int quarter, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, c;\n\t"
        "setp.ne.u32 c, %1, 0;\n\t"
        "bar.red.and.pred p, %2, 64, c;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(1 + quarter)
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
    // [stage][K, V][2 dim halves][64 cells][128 B], 128-byte swizzle
    uint64_t *kv_full = reinterpret_cast<uint64_t *>(sKV + kUStages * kStageBytes);
    uint64_t *kv_empty = kv_full + kUStages;
    uint64_t *s_full = kv_empty + kUStages;          // [2] S(t) in its buffer
    uint64_t *p_full = s_full + 2;                   // [2] P(t) in its buffer (S(t) read)
    uint64_t *o_done = p_full + 2;                   // [2] the P V of a tile using P buffer b done
    uint64_t *q_ready = o_done + 2;
    uint64_t *drain = q_ready + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    // row maxima of the two halves of each row, double-buffered by tile parity ([2][2][128]
    // floats), then the halves' row sums ([2][128]), at 256 bytes past the stage ring
    float *xch = reinterpret_cast<float *>(sKV + kUStages * kStageBytes + 256);

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
            mbar_init(&p_full[b], kUEpiWarps);
            mbar_init(&o_done[b], 1);
        }
        mbar_init(q_ready, kUEpiWarps);
        mbar_init(drain, 1);
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

    if (warp == 0 || warp == kUThreads / 32 - 1) {
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
    } else if (warp == 1) {
        // ---- MMA issuer (one thread): per tile t one burst, S(t) = Q K(t)^T and then
        // O += P(t-2) V(t-2), after two waits: K / V(t) landed, and P(t-2) written (so the
        // softmax warps also read S(t-2), whose buffer S(t) takes).  P V runs two tiles behind
        // so that S(t + 1) is issued while the softmax of t - 1 still runs.  Each wait or commit
        // costs this thread over a hundred cycles with the tensor queue draining meanwhile, so a
        // tile has two waits and three commits.  The issuing thread shares its sub-partition
        // with two softmax warps, so each MMA costs it one 32-bit add: the descriptors of stage
        // 0 are built once, and a stage, dim half or k step moves only the start-address field
        // (bits 0-13, 16-byte units; shared addresses stay below 256 KB, so the add never
        // carries out of it).
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_m128(kUTC, false);
            constexpr uint32_t id_o = idesc_m128(kUD, true);
            const uint64_t dk0 = desc_kmajor_sw128(smem_u32(sKV));
            const uint64_t dv0 = desc_mnmajor_sw128(smem_u32(sKV + kTileBytes), kTileHalf);
            const uint32_t dk_lo = (uint32_t)dk0, dk_hi = (uint32_t)(dk0 >> 32);
            const uint32_t dv_lo = (uint32_t)dv0, dv_hi = (uint32_t)(dv0 >> 32);
            if (n_tiles > 0 && !mbar_wait(q_ready, 0, wc.limit_ns)) ok = false;
            for (int t = 0; ok && t < n_tiles + 2; ++t) {
                const int tp = t - 2;
                if (t < n_tiles) {
                    if (!mbar_wait(&kv_full[t % kUStages], (uint32_t)(t / kUStages) & 1u, wc.limit_ns)) {
                        ok = false;
                        break;
                    }
                    // the stage was written by ordinary (generic-proxy) copies; the tensor
                    // cores read it through the async proxy
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                if (tp >= 0 && !mbar_wait(&p_full[tp & 1], (uint32_t)(tp >> 1) & 1u, wc.limit_ns)) {
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (t < n_tiles) {
                    const int s = t % kUStages, b = t & 1;
                    const uint32_t ks = dk_lo + (uint32_t)s * (kStageBytes >> 4);
                    const uint32_t d_s = tmem + kColS + (uint32_t)(b * kUTC);
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
#pragma unroll
                        for (int k16 = 0; k16 < kUD / 16; ++k16) {
                            const uint32_t off = ((uint32_t)(k16 >> 2) * kTileHalf + (uint32_t)(k16 & 3) * 32) >> 4;
                            umma_m128_ta(d_s, tmem + (part ? kColQl : kColQh) + (uint32_t)k16 * 8,
                                         ((uint64_t)dk_hi << 32) | (ks + off), id_s,
                                         (part | k16) ? 1u : 0u);
                        }
                    }
                    umma_commit(&s_full[b]);
                }
                if (tp >= 0) {
                    const int sp = tp % kUStages, pb = tp & 1;
                    const uint32_t vs = dv_lo + (uint32_t)sp * (kStageBytes >> 4);
                    const uint32_t pcol = tmem + kColP + (uint32_t)pb * 64;
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
#pragma unroll
                        for (int k16 = 0; k16 < kUTC / 16; ++k16)
                            umma_m128_ta(tmem + kColO, pcol + (uint32_t)(part * 32 + k16 * 8),
                                         ((uint64_t)dv_hi << 32) | (vs + (uint32_t)k16 * (2048 >> 4)),
                                         id_o, (tp | part | k16) ? 1u : 0u);
                    }
                    umma_commit(&o_done[pb]);
                    umma_commit(&kv_empty[sp]);
                }
            }
            // every MMA issued has completed before the tensor memory is freed
            umma_commit(drain);
            if (!mbar_wait(drain, 0)) ok = false;
        }
    } else {
        // ---- softmax / epilogue: two threads per row (row = 8 * query + head), one per half
        // of the tile's 64 columns (and of O's 128 dims)
        const int quarter = warp & 3;
        const int ch = (warp - 2) >> 2;              // column half: warps 2-5 -> 0, 6-9 -> 1
        const int r = quarter * 32 + lane;
        const int li = r >> 3;
        const int64_t qi = g * kUG + li;
        const int h = kvh * kUHeads + (r & 7);
        const bool live = qi < n_q;
        const int64_t n = live ? (int64_t)n_cells[qi] : 0;
        const bool trunc = n > max_cells;
        const uint32_t lrow = (uint32_t)(quarter * 32) << 16;
        // this half of the row's query (dims 64*ch ..), pre-scaled, as bf16 high and low
        // halves into tensor memory
        {
            const float *qr = q + (qi * H_q + h) * (int64_t)kUD + ch * 64;
            uint32_t wh[32], wl[32];
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
                float x0 = 0.0f, x1 = 0.0f;
                if (live) {
                    const float2 v = *reinterpret_cast<const float2 *>(qr + e);
                    x0 = v.x * scale_log2;
                    x1 = v.y * scale_log2;
                }
                const float h0 = __bfloat162float(__float2bfloat16_rn(x0));
                const float h1 = __bfloat162float(__float2bfloat16_rn(x1));
                wh[e / 2] = pack_bf16(h0, h1);
                wl[e / 2] = pack_bf16(x0 - h0, x1 - h1);
            }
            tmem_st32(tmem + lrow + kColQh + (uint32_t)(ch * 32), wh);
            tmem_st32(tmem + lrow + kColQl + (uint32_t)(ch * 32), wl);
            tmem_wait_st();
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(q_ready);
        }
        float m_ref = -INFINITY, l = 0.0f;
        uint32_t mw = 0;
        if (n_tiles > 0) mw = gmem[li * 2 + ch];
        // Every iteration passes exactly one pair barrier, which also decides (for both warps
        // of the pair alike) whether to stop: a warp whose wait gave up skips its tensor-memory
        // work and stops at the next pair barrier together with its partner.
        for (int t = 0; t < n_tiles; ++t) {
            const int b = t & 1;
            const uint32_t w = (live && !trunc) ? mw : 0u;
            if (t + 1 < n_tiles) mw = gmem[((int64_t)(t + 1) * kUG + li) * 2 + ch];  // ahead
            // waits are warp-uniform: the tensor-memory accesses below need the whole warp
            bool good = ok && warp_wait(&s_full[b], (uint32_t)(t >> 1) & 1u, wc.limit_ns);
            float x[32];
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (good) {
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                tmem_ld32(tmem + lrow + kColS + (uint32_t)(b * kUTC + ch * 32), x);
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    x[e] = ((w >> e) & 1u) ? x[e] : -INFINITY;
                    mx[e & 3] = fmaxf(mx[e & 3], x[e]);
                }
            }
            // the row's maximum over both halves
            float *slot = xch + (b * 2) * kUM;
            slot[ch * kUM + r] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            if (!pair_and(quarter, good)) {
                ok = false;
                break;
            }
            const float mt = fmaxf(slot[r], slot[kUM + r]);
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
            // P(t) relative to the (possibly moved) maximum, before any wait on the MMAs
            const float mu = m_ref == -INFINITY ? 0.0f : m_ref;
            uint32_t pw[32];
            float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                const float p0 = ex2_approx(x[e] - mu);
                const float p1 = ex2_approx(x[e + 1] - mu);
                ls[(e >> 1) & 3] += p0 + p1;
                const uint32_t hb = pack_bf16(p0, p1);
                const float h0 = __uint_as_float(hb << 16), h1 = __uint_as_float(hb & 0xffff0000u);
                pw[e / 2] = hb;
                pw[16 + e / 2] = pack_bf16(p0 - h0, p1 - h1);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // P buffer b was last read by P V(t - 2); O is touched only when rescaling, after
            // P V(t - 1)
            const bool w2 = t < 2 || warp_wait(&o_done[b], (uint32_t)((t - 2) >> 1) & 1u,
                                               wc.limit_ns);
            const bool w3 = !(rescale && t >= 1) ||
                            warp_wait(&o_done[b ^ 1], (uint32_t)((t - 1) >> 1) & 1u, wc.limit_ns);
            if (!(w2 && w3)) {
                ok = false;  // stops at the next pair barrier (or the one after the loop)
                continue;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (rescale) {
#pragma unroll 1
                for (int c = ch * 64; c < ch * 64 + 64; c += 32) {
                    float o[32];
                    tmem_ld32(tmem + lrow + kColO + (uint32_t)c, o);
                    uint32_t ou[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) ou[e] = __float_as_uint(o[e] * alpha);
                    tmem_st32(tmem + lrow + kColO + (uint32_t)c, ou);
                }
            }
            // P(t): high halves in columns 0-31 of the buffer, low halves in 32-63; this
            // thread's 32 cells are 16 columns of each
            const uint32_t pcol = tmem + lrow + kColP + (uint32_t)b * 64 + (uint32_t)(ch * 16);
            tmem_st16(pcol, pw);
            tmem_st16(pcol + 32, pw + 16);
            tmem_wait_st();
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[b]);
        }
        if (ok && n_tiles > 0 &&
            !warp_wait(&o_done[(n_tiles - 1) & 1], (uint32_t)((n_tiles - 1) >> 1) & 1u, wc.limit_ns))
            ok = false;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        // the row sum over both halves, and whether both warps of the pair finished (every
        // warp of a pair arrives here after the same number of pair barriers)
        float *lsum = xch + 4 * kUM;
        lsum[ch * kUM + r] = l;
        ok = pair_and(quarter, ok);
        const float lt = lsum[r] + lsum[kUM + r];
        const bool nan_rows = !ok || bad_group || trunc;
        const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
#pragma unroll 1
        for (int c = ch * 64; c < ch * 64 + 64; c += 32) {
            float o[32];
            if (n_tiles > 0 && ok) {
                tmem_ld32(tmem + lrow + kColO + (uint32_t)c, o);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = 0.0f;
            }
            if (live) {
                float *dst = out + (qi * H_q + h) * (int64_t)kUD + c;
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4 *>(dst + e) =
                        nan_rows ? make_float4(NAN, NAN, NAN, NAN)
                                 : make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv,
                                               o[e + 3] * inv);
            }
        }
        if (live && lse && ch == 0)
            lse[qi * H_q + h] = nan_rows ? NAN
                                         : (lt > 0.0f ? (m_ref + log2f(lt)) * 0.6931471805599453f
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
