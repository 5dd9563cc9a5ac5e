// pkv_swap.cu -- block copies between two pools, one of them normally in
// page-locked host memory: the data movement of swapping.
//
// [P2] "Why it matters for KV cache", "Swapping and preemption": blocks are
// evicted to CPU memory when GPU memory runs short and fetched back when the
// request resumes.  [P1] "Common misconceptions": a technique separate from
// paging itself.  The block manager (pkv_alloc.cpp) decides which blocks move
// where; this file moves them.
//
// One launch moves any number of scattered blocks of any number of layers:
// SMs load 16-byte vectors from the source pool and store them to the
// destination pool, the host side reached directly over the CPU-GPU link
// (zero-copy through the page-locked mapping).  A copy engine would need one
// memcpy per contiguous run, i.e. per block per cache per layer.  The work is
// cut into 16 KiB tiles (256 threads x 4 vectors), tile-major within a block
// so that consecutive CTAs stream consecutive bytes of one block.
#include <cuda_runtime.h>

#include <algorithm>

#include "../../include/pkv.h"
#include "pkv_device.cuh"
#include "pkv_launch.h"

namespace pkv {

namespace {

constexpr int kSwapThreads = 256;
constexpr int kSwapVecsPerThread = 4;
constexpr int kSwapTileVecs = kSwapThreads * kSwapVecsPerThread;  // 16 KiB

// Per-layer pool pointers, passed by value as a kernel parameter
// (2 x 2 x PKV_MAX_LAYERS pointers = 4 KB).  Index 2 * layer + (K: 0, V: 1).
struct SwapPointers {
    const uint4 *src[2 * PKV_MAX_LAYERS];
    uint4 *dst[2 * PKV_MAX_LAYERS];
};

__global__ void __launch_bounds__(kSwapThreads)
    swap_blocks_kernel(const __grid_constant__ SwapPointers sp, const int64_t *__restrict__ pairs, int num_pairs,
                       int64_t vecs_per_block, int tiles_per_block, int64_t num_tiles, int64_t src_num_blocks,
                       int64_t dst_num_blocks, int32_t *status) {
    grid_dependency_wait();
    launch_dependents();
    const int64_t tiles_per_cache = (int64_t)num_pairs * tiles_per_block;
    for (int64_t tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        const int c = (int)(tile / tiles_per_cache);
        const int64_t r = tile - (int64_t)c * tiles_per_cache;
        const int pi = (int)(r / tiles_per_block);
        const int t = (int)(r - (int64_t)pi * tiles_per_block);
        const int64_t src = __ldg(pairs + 2 * (int64_t)pi);
        const int64_t dst = __ldg(pairs + 2 * (int64_t)pi + 1);
        if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) {
            if (threadIdx.x == 0 && t == 0 && c == 0) report(status, PKV_ERR_OUT_OF_RANGE);
            continue;
        }
        const uint4 *s = sp.src[c] + src * vecs_per_block;
        uint4 *d = sp.dst[c] + dst * vecs_per_block;
        const int64_t base = (int64_t)t * kSwapTileVecs + threadIdx.x;
        uint4 v[kSwapVecsPerThread];
#pragma unroll
        for (int j = 0; j < kSwapVecsPerThread; ++j) {
            const int64_t i = base + j * kSwapThreads;
            if (i < vecs_per_block) v[j] = s[i];
        }
#pragma unroll
        for (int j = 0; j < kSwapVecsPerThread; ++j) {
            const int64_t i = base + j * kSwapThreads;
            if (i < vecs_per_block) d[i] = v[j];
        }
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The address through which the current device reaches p: device memory of
// this device, managed memory, or page-locked host memory mapped into the
// device's address space.  Pageable host memory and other devices' memory
// are refused.
int device_view(const void *p, int device, const void **out) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    switch (attr.type) {
        case cudaMemoryTypeDevice:
            if (attr.device != device) return PKV_ERR_INVALID_ARG;
            *out = p;
            return PKV_OK;
        case cudaMemoryTypeManaged:
            *out = p;
            return PKV_OK;
        case cudaMemoryTypeHost:
            if (!attr.devicePointer) return PKV_ERR_INVALID_ARG;
            *out = attr.devicePointer;
            return PKV_OK;
        default:
            return PKV_ERR_INVALID_ARG;
    }
}

int swap_impl(const void *const *src_keys, const void *const *src_values, const void *const *dst_keys,
              const void *const *dst_values, int num_layers, const int64_t *block_pairs, int num_pairs,
              size_t block_bytes, int src_num_blocks, int dst_num_blocks, int32_t *dev_status,
              pkv_stream_t stream) {
    if (num_pairs == 0) return PKV_OK;
    if (num_layers < 1 || num_layers > PKV_MAX_LAYERS || !src_keys || !src_values || !dst_keys || !dst_values)
        return PKV_ERR_INVALID_ARG;
    if (num_pairs < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0 || block_bytes == 0 || block_bytes % 16 ||
        !block_pairs)
        return PKV_ERR_INVALID_ARG;
    for (int l = 0; l < num_layers; ++l) {
        const void *ps[4] = {src_keys[l], src_values[l], dst_keys[l], dst_values[l]};
        for (const void *q : ps)
            if (!q || !aligned16(q)) return PKV_ERR_INVALID_ARG;
    }
    const int64_t vpb = (int64_t)(block_bytes / 16);
    const int64_t tpb = (vpb + kSwapTileVecs - 1) / kSwapTileVecs;
    if (tpb > (1 << 30)) return PKV_ERR_INVALID_ARG;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    SwapPointers sp;
    for (int l = 0; l < num_layers; ++l) {
        const void *v;
        int rc;
        if ((rc = device_view(src_keys[l], device, &v)) != PKV_OK) return rc;
        sp.src[2 * l] = static_cast<const uint4 *>(v);
        if ((rc = device_view(src_values[l], device, &v)) != PKV_OK) return rc;
        sp.src[2 * l + 1] = static_cast<const uint4 *>(v);
        if ((rc = device_view(dst_keys[l], device, &v)) != PKV_OK) return rc;
        sp.dst[2 * l] = const_cast<uint4 *>(static_cast<const uint4 *>(v));
        if ((rc = device_view(dst_values[l], device, &v)) != PKV_OK) return rc;
        sp.dst[2 * l + 1] = const_cast<uint4 *>(static_cast<const uint4 *>(v));
    }
    const void *pv;
    int rc = device_view(block_pairs, device, &pv);
    if (rc != PKV_OK) return rc;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    int64_t num_tiles = 2 * (int64_t)num_layers * num_pairs * tpb;
    // 8 CTAs of 256 threads fill an SM; each CTA walks tiles grid-stride
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(num_tiles, (int64_t)sms * 8));
    const int64_t *pairs = static_cast<const int64_t *>(pv);
    int np = num_pairs, tiles_pb = (int)tpb;
    int64_t vpb_arg = vpb, snb = src_num_blocks, dnb = dst_num_blocks;
    int32_t *st = dev_status;
    void *args[] = {&sp, &pairs, &np, &vpb_arg, &tiles_pb, &num_tiles, &snb, &dnb, &st};
    if (launch_pdl(reinterpret_cast<const void *>(&swap_blocks_kernel), dim3((unsigned)grid), dim3(kSwapThreads), 0,
                   stream, args) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

}  // namespace

}  // namespace pkv

using namespace pkv;

extern "C" int pkv_swap_blocks(const void *src_key, const void *src_value, void *dst_key, void *dst_value,
                               const int64_t *block_pairs, int num_pairs, size_t block_bytes, int src_num_blocks,
                               int dst_num_blocks, int32_t *dev_status, pkv_stream_t stream) {
    const void *sk[1] = {src_key}, *sv[1] = {src_value}, *dk[1] = {dst_key}, *dv[1] = {dst_value};
    return swap_impl(sk, sv, dk, dv, 1, block_pairs, num_pairs, block_bytes, src_num_blocks, dst_num_blocks,
                     dev_status, stream);
}

extern "C" int pkv_swap_blocks_layers(const void *const *src_keys, const void *const *src_values,
                                      void *const *dst_keys, void *const *dst_values, int num_layers,
                                      const int64_t *block_pairs, int num_pairs, size_t block_bytes,
                                      int src_num_blocks, int dst_num_blocks, int32_t *dev_status,
                                      pkv_stream_t stream) {
    return swap_impl(src_keys, src_values, dst_keys, dst_values, num_layers, block_pairs, num_pairs, block_bytes,
                     src_num_blocks, dst_num_blocks, dev_status, stream);
}
