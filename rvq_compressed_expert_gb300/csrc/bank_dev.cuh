// Device side of the tiered expert bank shared by the fetch kernels (bank.cu) and the
// persistent step kernel's copy lanes (fused.cu): records move from the host tier into the
// HBM cache in chunks of 64 KiB, each copied by one 512-thread CTA with all of its loads in
// flight before the stores.  Twelve such CTAs keep the CPU-GPU link at its measured copy
// rate (the rate of the copy engines), so the copy lanes leave the other SMs to compute.
#pragma once

#include "common.cuh"

namespace wm {
namespace bank {

constexpr int kCopyThreads = 512;
constexpr int kCopyLoads = 8;   // 16-byte loads in flight per thread
constexpr size_t kChunkBytes = (size_t)kCopyThreads * kCopyLoads * 16;
constexpr int kCopyLanes = 12;  // CTAs that copy

__host__ __device__ __forceinline__ size_t chunks_per_record(size_t stride) {
    return (stride + kChunkBytes - 1) / kChunkBytes;
}

// Piece `piece` (chunk-sized, the last one of a record short) of copy job `j` by the calling
// CTA of kCopyThreads threads; stride is a multiple of 16.
__device__ __forceinline__ void copy_chunk(const BankDevice &D, const uint8_t *__restrict__ host, size_t stride,
                                           int j, int piece) {
    const int2 job = D.jobs[j];
    const size_t off = (size_t)piece * kChunkBytes;
    const uint4 *__restrict__ src = reinterpret_cast<const uint4 *>(host + (size_t)job.y * stride + off);
    uint4 *__restrict__ dst = reinterpret_cast<uint4 *>(D.slots + (size_t)job.x * stride + off);
    const int lim = (int)min((stride - off) / 16, (size_t)kCopyLoads * kCopyThreads);
    uint4 v[kCopyLoads];
#pragma unroll
    for (int u = 0; u < kCopyLoads; ++u) {
        const int k = u * kCopyThreads + (int)threadIdx.x;
        if (k < lim) v[u] = src[k];
    }
#pragma unroll
    for (int u = 0; u < kCopyLoads; ++u) {
        const int k = u * kCopyThreads + (int)threadIdx.x;
        if (k < lim) dst[k] = v[u];
    }
}

// Chunks first, first + step, ... of the n_jobs jobs (chunk c = piece c % per of job c / per),
// so CTAs with first = 0..step-1 finish the jobs in order.  done(j) follows the calling CTA's
// last chunk of job j: each job is signalled once by each of the min(per, step) CTAs that
// copy a part of it.
template <typename Done>
__device__ __forceinline__ void copy_jobs(const BankDevice &D, const uint8_t *__restrict__ host, size_t stride,
                                          int n_jobs, int first, int step, Done done) {
    const int per = (int)chunks_per_record(stride);
    int j = first / per, piece = first % per;
    while (j < n_jobs) {
        copy_chunk(D, host, stride, j, piece);
        piece += step;
        int next = j;
        while (piece >= per) {
            piece -= per;
            ++next;
        }
        if (next != j) done(j);
        j = next;
    }
}

__host__ __device__ __forceinline__ int copiers_per_job(size_t stride, int step) {
    const size_t per = chunks_per_record(stride);
    return per < (size_t)step ? (int)per : step;
}

} // namespace bank
} // namespace wm
