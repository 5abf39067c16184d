// host_step.cu -- the host transfers of a decode step fed from host memory.  On the way in,
// the new tokens' raw indexer-key, K and V rows go to their caches at the tokens' positions
// and the queries to a staging area; on the way out, the attention output (and its
// log-sum-exp) goes back to host memory.  Both are row-block copies: when the host buffer
// is page-locked and mapped into the GPU's address space the copy kernel reads or writes it
// in place over the host link, so no copy-engine transfer sits between the kernels.
//
// Source: Qiita, ariera, EVO-X2 + Qwen3.8-Flash-Next llama.cpp series part 10, section
// "incremental pooled-key cache (COMMON-004)" (each decode step appends the new token to
// the caches before the indexer runs).
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kCopyThreads = 256;

struct CopyJobs {
    RowCopy job[kMaxCopyJobs];
    bool w16;  // every address, row size and stride a multiple of 16 bytes (else of 4)
};

__global__ void __launch_bounds__(kCopyThreads) copy_rows_kernel(const CopyJobs jobs)
{
    pdl_wait();
    pdl_trigger();
    const RowCopy &jb = jobs.job[blockIdx.y];
    const char *src = static_cast<const char *>(jb.src);
    char *dst = static_cast<char *>(jb.dst);
    QSA_AFTER_WAIT(src);
    const int64_t rb = jb.row_bytes;
    const int unit = jobs.w16 ? 16 : 4;
    const int64_t per_row = rb / unit;
    const int64_t total = per_row * jb.rows;
    for (int64_t e = (int64_t)blockIdx.x * kCopyThreads + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * kCopyThreads) {
        const int64_t r = e / per_row, c = e - r * per_row;
        const char *s = src + r * rb + c * unit;
        char *d = dst + r * jb.dst_ld + c * unit;
        if (jobs.w16) *reinterpret_cast<uint4 *>(d) = *reinterpret_cast<const uint4 *>(s);
        else *reinterpret_cast<uint32_t *>(d) = *reinterpret_cast<const uint32_t *>(s);
    }
}

bool mult16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

}  // namespace

cudaError_t launch_copy_rows(const RowCopy *job, int n_jobs, cudaStream_t st)
{
    if (n_jobs < 1 || n_jobs > kMaxCopyJobs) return cudaErrorInvalidValue;
    CopyJobs jobs = {};
    bool w16 = true;
    int64_t most = 0;
    for (int j = 0; j < n_jobs; ++j) {
        jobs.job[j] = job[j];
        w16 = w16 && mult16(job[j].src) && mult16(job[j].dst) && job[j].row_bytes % 16 == 0 &&
              job[j].dst_ld % 16 == 0;
        const int64_t bytes = job[j].row_bytes * job[j].rows;
        if (bytes > most) most = bytes;
    }
    jobs.w16 = w16;
    // one 16-byte unit per thread of the largest job (a few KB per step), at most 8 CTAs
    const int64_t per_cta = (int64_t)kCopyThreads * 16;
    int64_t ctas = (most + per_cta - 1) / per_cta;
    if (ctas < 1) ctas = 1;
    if (ctas > 8) ctas = 8;
    return launch(copy_rows_kernel, dim3((unsigned)ctas, (unsigned)n_jobs), dim3(kCopyThreads), 0,
                  st, 1, jobs);
}

void *mapped_host_view(const void *h)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

}  // namespace qsa
