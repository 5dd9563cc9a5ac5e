// pkv_stage.cu -- the input copy of a serving step (pkv_decode_plan_step)
// when the step's staged inputs are in mapped page-locked host memory.
//
// A copy engine moves a region of one or two MB with a fixed cost that
// dominates (16-17 us for the 7B-class step's 1.6 MB, ~100 GB/s).  Here
// every thread of a one-wave grid loads 16-byte vectors of the region
// directly over the CPU-GPU link through the host memory's device mapping
// and stores them to device memory: all loads are in flight at once.  The
// kernel is launched without programmatic dependent launch and never lets
// dependents start early, so it begins after everything before it on the
// stream and the decode launch after it sees every byte it wrote.
#include <cuda_runtime.h>

#include "../../include/pkv.h"

namespace pkv {

namespace {

constexpr int kStageThreads = 256;

__global__ void __launch_bounds__(kStageThreads)
    stage_copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * kStageThreads + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * kStageThreads)
        dst[i] = src[i];
}

}  // namespace

// Copies `bytes` from host_src to dev_dst on `stream` with stage_copy_kernel
// when host_src is page-locked host memory the current device can reach and
// both addresses and the size are multiples of 16 bytes; returns false
// (nothing enqueued) when it cannot, so that the caller copies instead.
bool stage_in_by_kernel(void *dev_dst, const void *host_src, size_t bytes, cudaStream_t stream) {
    if (bytes == 0 || bytes % 16 || (reinterpret_cast<uintptr_t>(dev_dst) & 15u) ||
        (reinterpret_cast<uintptr_t>(host_src) & 15u))
        return false;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, host_src) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr ||
        (reinterpret_cast<uintptr_t>(attr.devicePointer) & 15u))
        return false;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    const int64_t n = (int64_t)(bytes / 16);
    const int64_t need = (n + kStageThreads - 1) / kStageThreads;
    const int grid = (int)(need < (int64_t)sms * 8 ? need : (int64_t)sms * 8);
    stage_copy_kernel<<<grid, kStageThreads, 0, stream>>>(static_cast<const uint4 *>(attr.devicePointer),
                                                          static_cast<uint4 *>(dev_dst), n);
    if (cudaGetLastError() != cudaSuccess) return false;
    return true;
}

}  // namespace pkv
