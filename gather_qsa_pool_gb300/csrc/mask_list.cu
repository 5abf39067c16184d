// mask_list.cu -- mask row -> 64-bit ballot words -> ascending list of attendable keys.
//
// Source: devotd.net, "llama.cpp CDNA sparse attention", section 2: the attendable key
// positions are collected from the mask into a list before the sparse kernel runs, the
// per-lane selection is stored as a 64-bit mask (one bit per lane of a 64-wide wave) and
// the count is taken from the same words.
//
// On 32-lane warps each 64-bit word is two ballots: lanes read positions 64w + lane and
// 64w + 32 + lane; when the row is whole 64-byte words, 16-byte aligned, each thread
// instead reads its word's 64 bytes with four 16-byte loads and packs the nonzero flags
// itself (the same word).  One CTA per mask row walks the row in chunks of 64 * 1024
// positions:
//   1. the words of the chunk go to shared memory;
//   2. one block-wide exclusive scan of the word counts gives each word's list offset;
//   3. the thread owning a word writes its set positions (lowest bit first).
// The list is capped at max_list; the count written is the true count.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kMaskThreads = 1024;

constexpr int kWordsPerChunk = kMaskThreads;  // one word per thread per chunk

__global__ void __launch_bounds__(kMaskThreads)
mask_to_list_kernel(const uint8_t *__restrict__ mask, int64_t n_kv, int64_t ld_mask,
                    int64_t max_list, int32_t *__restrict__ pos_out,
                    int32_t *__restrict__ counts_out, uint64_t *__restrict__ bits_out)
{
    __shared__ unsigned long long words[kWordsPerChunk];
    __shared__ uint32_t warp_tot[kMaskThreads / 32];
    __shared__ uint32_t carry_s;
    pdl_wait();
    QSA_AFTER_WAIT(mask);
    pdl_trigger();

    const int64_t r = blockIdx.x;
    const uint8_t *row = mask + r * ld_mask;
    int32_t *plist = pos_out + r * max_list;
    const int64_t n_words = (n_kv + 63) / 64;
    uint64_t *brow = bits_out ? bits_out + r * n_words : nullptr;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int NW = kMaskThreads / 32;
    if (threadIdx.x == 0) carry_s = 0;
    __syncthreads();

    // rows whose words are all whole and 16-byte aligned: thread t builds word w0 + t from its
    // 64 mask bytes, four 16-byte loads issued together
    const bool vec = n_kv % 64 == 0 && (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    for (int64_t w0 = 0; w0 < n_words; w0 += kWordsPerChunk) {
        if (vec) {
            const int64_t w = w0 + threadIdx.x;
            unsigned long long word = 0ull;
            if (w < n_words) {
                const uint4 *src = reinterpret_cast<const uint4 *>(row + 64 * w);
                uint4 v[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) v[k] = src[k];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t u[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        word |= (unsigned long long)nonzero_byte_bits(u[m]) << (16 * k + 4 * m);
                }
            }
            words[threadIdx.x] = word;
        }
        // 1. ballots: warp `warp` builds words w0 + warp, w0 + warp + NW, ...
        for (int wi = warp; !vec && wi < kWordsPerChunk; wi += NW) {
            const int64_t w = w0 + wi;
            unsigned long long word = 0ull;
            if (w < n_words) {
                const int64_t p_lo = 64 * w + lane, p_hi = p_lo + 32;
                const bool b_lo = p_lo < n_kv && row[p_lo] != 0;
                const bool b_hi = p_hi < n_kv && row[p_hi] != 0;
                const unsigned lo = __ballot_sync(0xffffffffu, b_lo);
                const unsigned hi = __ballot_sync(0xffffffffu, b_hi);
                word = (unsigned long long)lo | ((unsigned long long)hi << 32);
            }
            if (lane == 0) words[wi] = word;
        }
        __syncthreads();
        // 2. exclusive scan of popcounts (thread t owns word w0 + t)
        const int64_t w = w0 + threadIdx.x;
        const unsigned long long word = words[threadIdx.x];
        const uint32_t c = (uint32_t)__popcll(word);
        uint32_t x = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            uint32_t t = warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, t, o);
                if (lane >= o) t += y;
            }
            warp_tot[lane] = t;
        }
        __syncthreads();
        const uint32_t carry = carry_s;
        const int64_t off = (int64_t)carry + (warp ? warp_tot[warp - 1] : 0u) + (x - c);
        // 3. positions of this word
        if (w < n_words) {
            if (brow) brow[w] = word;
            unsigned long long rest = word;
            int64_t o = off;
            while (rest && o < max_list) {
                const int bit = __ffsll((long long)rest) - 1;
                plist[o++] = (int32_t)(64 * w + bit);
                rest &= rest - 1ull;
            }
        }
        __syncthreads();  // everyone has read carry_s and words[]
        if (threadIdx.x == 0) carry_s = carry + warp_tot[NW - 1];
        __syncthreads();
    }
    if (threadIdx.x == 0) counts_out[r] = (int32_t)carry_s;
}

}  // namespace

cudaError_t launch_mask_to_list(const uint8_t *mask, int64_t n_rows, int64_t n_kv,
                                int64_t ld_mask, int64_t max_list, int32_t *pos_out,
                                int32_t *counts_out, uint64_t *bits_out, cudaStream_t st)
{
    if (n_rows == 0) return cudaSuccess;
    return launch(mask_to_list_kernel, dim3((unsigned)n_rows), dim3(kMaskThreads), 0, st, 1,
                  mask, n_kv, ld_mask, max_list, pos_out, counts_out, bits_out);
}

}  // namespace qsa
