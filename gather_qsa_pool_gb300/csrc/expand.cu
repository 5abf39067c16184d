// expand.cu -- the pages' earlier selection input: every full block's score copied to its
// four cells.  Kept for A/B measurement against the block-domain top-k.
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "block-domain top-k (COMMON-006)" (before it, each block score was copied to its cells by
// a get_rows over a cell -> block map, 0.45 ms per layer at 128k and 0.91 ms at 256k on the
// pages' GPU, and the top-k ran over the 4x longer cell list).
//
// HBM-bound: 4 bytes read and 16 written per block.  Each thread writes the four cells of
// one block as a single 16-byte store when the row start allows it.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kExpandThreads = 256;

__global__ void __launch_bounds__(kExpandThreads)
expand_scores_kernel(const float *__restrict__ scores, int64_t ld_s, int64_t n_full,
                     float *__restrict__ cells, int64_t ld_c, bool vec)
{
    pdl_wait();
    QSA_AFTER_WAIT(scores);
    pdl_trigger();
    const int64_t qi = blockIdx.y;
    const float *s = scores + qi * ld_s;
    float *c = cells + qi * ld_c;
    for (int64_t b = (int64_t)blockIdx.x * kExpandThreads + threadIdx.x; b < n_full;
         b += (int64_t)gridDim.x * kExpandThreads) {
        const float v = s[b];
        if (vec) {
            *reinterpret_cast<float4 *>(c + 4 * b) = make_float4(v, v, v, v);
        } else {
            c[4 * b] = v;
            c[4 * b + 1] = v;
            c[4 * b + 2] = v;
            c[4 * b + 3] = v;
        }
    }
}

}  // namespace

cudaError_t launch_expand_scores(const float *scores, int64_t n_q, int64_t ld_s, int64_t n_full,
                                 float *cells, int64_t ld_c, cudaStream_t st)
{
    if (n_q == 0 || n_full == 0) return cudaSuccess;
    const bool vec = (reinterpret_cast<uintptr_t>(cells) % 16 == 0) && ld_c % 4 == 0;
    int64_t gx = (n_full + kExpandThreads - 1) / kExpandThreads;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (gx > cap) gx = cap;
    return launch(expand_scores_kernel, dim3((unsigned)gx, (unsigned)n_q), dim3(kExpandThreads), 0,
                  st, 1, scores, ld_s, n_full, cells, ld_c, vec);
}

}  // namespace qsa
