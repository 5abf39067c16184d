// host_step.cu -- the new tokens' cache rows of a decode step fed from host memory: one
// host-to-device copy brings the step's packed inputs into a staging area, and this kernel
// writes the new raw indexer-key, K and V rows into their caches at the tokens' positions
// (the queries are read from the staging area in place).
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "incremental pooled-key cache (COMMON-004)" (each decode step appends the new token to
// the caches before the indexer runs).
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kScatterThreads = 256;

// Up to three row blocks, each copied from the staging area to its cache: block j holds
// rows[j] rows of row_bytes[j] bytes, contiguous in the source, dst_ld[j] bytes apart in the
// destination.  w16: every address and size is a multiple of 16 bytes (else of 4).
struct ScatterJob {
    const char *src[3];
    char *dst[3];
    int64_t row_bytes[3];
    int64_t dst_ld[3];
    int rows[3];
    bool w16;
};

__global__ void __launch_bounds__(kScatterThreads) scatter_rows_kernel(const ScatterJob job)
{
    pdl_wait();
    pdl_trigger();
    const int j = blockIdx.y;
    const char *src = job.src[j];
    char *dst = job.dst[j];
    QSA_AFTER_WAIT(src);
    const int64_t rb = job.row_bytes[j];
    const int unit = job.w16 ? 16 : 4;
    const int64_t per_row = rb / unit;
    const int64_t total = per_row * job.rows[j];
    for (int64_t e = (int64_t)blockIdx.x * kScatterThreads + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * kScatterThreads) {
        const int64_t r = e / per_row, c = e - r * per_row;
        const char *s = src + r * rb + c * unit;
        char *d = dst + r * job.dst_ld[j] + c * unit;
        if (job.w16) *reinterpret_cast<uint4 *>(d) = *reinterpret_cast<const uint4 *>(s);
        else *reinterpret_cast<uint32_t *>(d) = *reinterpret_cast<const uint32_t *>(s);
    }
}

}  // namespace

cudaError_t launch_scatter_rows(const void *const src[3], void *const dst[3],
                                const int64_t row_bytes[3], const int64_t dst_ld[3],
                                const int rows[3], cudaStream_t st)
{
    ScatterJob job;
    bool w16 = true;
    for (int j = 0; j < 3; ++j) {
        job.src[j] = static_cast<const char *>(src[j]);
        job.dst[j] = static_cast<char *>(dst[j]);
        job.row_bytes[j] = row_bytes[j];
        job.dst_ld[j] = dst_ld[j];
        job.rows[j] = rows[j];
        w16 = w16 && (reinterpret_cast<uintptr_t>(src[j]) % 16 == 0) &&
              (reinterpret_cast<uintptr_t>(dst[j]) % 16 == 0) && row_bytes[j] % 16 == 0 &&
              dst_ld[j] % 16 == 0;
    }
    job.w16 = w16;
    return launch(scatter_rows_kernel, dim3(2, 3), dim3(kScatterThreads), 0, st, 1, job);
}

}  // namespace qsa
