// pkv_cache_ops.cu -- slot-mapped cache write, copy-on-write block copy,
// status strings and the bounded-wait self-test.
//
// Both cache ops are plain bit copies bound by HBM bandwidth (or, for the
// handful of tokens of one decode step, by launch latency): 16-byte vector
// accesses, grid-stride loops, several loads in flight per thread.
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "../../include/pkv.h"
#include "pkv_device.cuh"
#include "pkv_launch.h"

namespace pkv {

// [P1] "How PagedAttention works", steps 2-3: token t's key/value rows go to
// slot slot_mapping[t] = block * block_size + offset.
__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                             uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache,
                             const int64_t *__restrict__ slot_mapping, int64_t num_vecs, int heads_x_vecs,
                             int vecs_per_row, int block_size, int64_t num_slots, int32_t *status) {
    grid_dependency_wait();
    launch_dependents();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < num_vecs; i += stride) {
        const int64_t t = i / heads_x_vecs;
        const int rem = (int)(i - t * heads_x_vecs);
        const int h = rem / vecs_per_row;
        const int v = rem - h * vecs_per_row;
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (rem == 0) report(status, PKV_ERR_OUT_OF_RANGE);
            continue;
        }
        const int64_t blk = slot / block_size;
        const int off = (int)(slot - blk * block_size);
        const int64_t num_heads = heads_x_vecs / vecs_per_row;
        const int64_t dst = ((blk * num_heads + h) * block_size + off) * vecs_per_row + v;
        key_cache[dst] = __ldg(key + i);
        value_cache[dst] = __ldg(value + i);
    }
}

// [P1] "Memory sharing across requests": copy-on-write copies the shared
// block to a fresh one.  grid.y walks the pairs, grid.z picks K (0) or V (1).
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache,
                       const int64_t *__restrict__ pairs, int num_pairs, int64_t vecs_per_block,
                       int num_blocks, int32_t *status) {
    grid_dependency_wait();
    launch_dependents();
    uint4 *cache = blockIdx.z ? value_cache : key_cache;
    for (int pi = blockIdx.y; pi < num_pairs; pi += gridDim.y) {
        const int64_t src = __ldg(pairs + 2 * (int64_t)pi);
        const int64_t dst = __ldg(pairs + 2 * (int64_t)pi + 1);
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0) report(status, PKV_ERR_OUT_OF_RANGE);
            continue;
        }
        const uint4 *s = cache + src * vecs_per_block;
        uint4 *d = cache + dst * vecs_per_block;
        const int64_t stride = (int64_t)gridDim.x * blockDim.x;
        int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
        for (; i + 3 * stride < vecs_per_block; i += 4 * stride) {
            const uint4 a = __ldg(s + i), b = __ldg(s + i + stride);
            const uint4 c = __ldg(s + i + 2 * stride), e = __ldg(s + i + 3 * stride);
            d[i] = a;
            d[i + stride] = b;
            d[i + 2 * stride] = c;
            d[i + 3 * stride] = e;
        }
        for (; i < vecs_per_block; i += stride) d[i] = __ldg(s + i);
    }
}

// Per-layer pointers of the multi-layer ops, passed by value as a kernel
// parameter (PKV_MAX_LAYERS x 4 pointers = 4 KB, well inside the parameter
// space).
struct LayerPointers {
    const uint4 *key[PKV_MAX_LAYERS];
    const uint4 *value[PKV_MAX_LAYERS];
    uint4 *key_cache[PKV_MAX_LAYERS];
    uint4 *value_cache[PKV_MAX_LAYERS];
};

// reshape_and_cache for every layer: grid.y = layer.
__global__ void __launch_bounds__(256)
    reshape_and_cache_layers_kernel(const __grid_constant__ LayerPointers lp,
                                    const int64_t *__restrict__ slot_mapping, int64_t num_vecs, int heads_x_vecs,
                                    int vecs_per_row, int block_size, int64_t num_slots, int32_t *status) {
    grid_dependency_wait();
    launch_dependents();
    const int layer = blockIdx.y;
    const uint4 *key = lp.key[layer];
    const uint4 *value = lp.value[layer];
    uint4 *key_cache = lp.key_cache[layer];
    uint4 *value_cache = lp.value_cache[layer];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < num_vecs; i += stride) {
        const int64_t t = i / heads_x_vecs;
        const int rem = (int)(i - t * heads_x_vecs);
        const int h = rem / vecs_per_row;
        const int v = rem - h * vecs_per_row;
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (rem == 0 && layer == 0) report(status, PKV_ERR_OUT_OF_RANGE);
            continue;
        }
        const int64_t blk = slot / block_size;
        const int off = (int)(slot - blk * block_size);
        const int64_t num_heads = heads_x_vecs / vecs_per_row;
        const int64_t dst = ((blk * num_heads + h) * block_size + off) * vecs_per_row + v;
        key_cache[dst] = __ldg(key + i);
        value_cache[dst] = __ldg(value + i);
    }
}

// copy_blocks for every layer: grid.y walks the pairs, grid.z = 2 * layer + (K: 0, V: 1).
__global__ void __launch_bounds__(256)
    copy_blocks_layers_kernel(const __grid_constant__ LayerPointers lp, const int64_t *__restrict__ pairs,
                              int num_pairs, int64_t vecs_per_block, int num_blocks, int32_t *status) {
    grid_dependency_wait();
    launch_dependents();
    const int layer = blockIdx.z >> 1;
    uint4 *cache = (blockIdx.z & 1) ? lp.value_cache[layer] : lp.key_cache[layer];
    for (int pi = blockIdx.y; pi < num_pairs; pi += gridDim.y) {
        const int64_t src = __ldg(pairs + 2 * (int64_t)pi);
        const int64_t dst = __ldg(pairs + 2 * (int64_t)pi + 1);
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0) report(status, PKV_ERR_OUT_OF_RANGE);
            continue;
        }
        const uint4 *s = cache + src * vecs_per_block;
        uint4 *d = cache + dst * vecs_per_block;
        const int64_t stride = (int64_t)gridDim.x * blockDim.x;
        int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
        for (; i + 3 * stride < vecs_per_block; i += 4 * stride) {
            const uint4 a = __ldg(s + i), b = __ldg(s + i + stride);
            const uint4 c = __ldg(s + i + 2 * stride), e = __ldg(s + i + 3 * stride);
            d[i] = a;
            d[i + stride] = b;
            d[i + 2 * stride] = c;
            d[i + 3 * stride] = e;
        }
        for (; i < vecs_per_block; i += stride) d[i] = __ldg(s + i);
    }
}

// Waits on a barrier that nothing completes; must give up and report.
__global__ void wait_timeout_selftest_kernel(int32_t *status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        fence_barrier_init();
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(smem_addr(&bar), 0, limit_ns);
    if (!__all_sync(kFullMask, ok) && threadIdx.x == 0) report(status, PKV_ERR_DEVICE_TIMEOUT);
}

namespace {
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

}  // namespace pkv

using namespace pkv;

extern "C" const char *pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
        case PKV_ERR_OUT_OF_BLOCKS: return "PKV_ERR_OUT_OF_BLOCKS";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
        case PKV_ERR_DEVICE_TIMEOUT: return "PKV_ERR_DEVICE_TIMEOUT";
        case PKV_ERR_OUT_OF_RANGE: return "PKV_ERR_OUT_OF_RANGE";
        case PKV_ERR_NOT_FOUND: return "PKV_ERR_NOT_FOUND";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        default: return "PKV_UNKNOWN_STATUS";
    }
}

extern "C" int pkv_version(void) { return 100; }

extern "C" int pkv_reshape_and_cache(const void *key, const void *value, void *key_cache, void *value_cache,
                                     const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                                     int head_dim, int block_size, int num_blocks, int32_t *dev_status,
                                     pkv_stream_t stream) {
    if (num_tokens == 0) return PKV_OK;
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 8 || block_size <= 0 ||
        num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache))
        return PKV_ERR_INVALID_ARG;
    const int vpr = head_dim / 8;
    const int64_t heads_x_vecs = (int64_t)num_kv_heads * vpr;
    if (heads_x_vecs > (1 << 30)) return PKV_ERR_INVALID_ARG;
    const int64_t num_vecs = (int64_t)num_tokens * heads_x_vecs;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>((num_vecs + threads - 1) / threads, 65536);
    // kernel arguments (non-const locals: launch_pdl takes their addresses)
    const uint4 *k4 = static_cast<const uint4 *>(key), *v4 = static_cast<const uint4 *>(value);
    uint4 *kc4 = static_cast<uint4 *>(key_cache), *vc4 = static_cast<uint4 *>(value_cache);
    const int64_t *slots = slot_mapping;
    int64_t nv = num_vecs, num_slots = (int64_t)num_blocks * block_size;
    int hxv = (int)heads_x_vecs, vr = vpr, bsz = block_size;
    int32_t *st = dev_status;
    void *args[] = {&k4, &v4, &kc4, &vc4, &slots, &nv, &hxv, &vr, &bsz, &num_slots, &st};
    if (launch_pdl(reinterpret_cast<const void *>(&reshape_and_cache_kernel), dim3((unsigned)blocks), dim3(threads),
                   0, stream, args) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

extern "C" int pkv_copy_blocks(void *key_cache, void *value_cache, const int64_t *block_pairs, int num_pairs,
                               size_t block_bytes, int num_blocks, int32_t *dev_status, pkv_stream_t stream) {
    if (num_pairs == 0) return PKV_OK;
    if (num_pairs < 0 || num_blocks <= 0 || block_bytes == 0 || block_bytes % 16) return PKV_ERR_INVALID_ARG;
    if (!key_cache || !value_cache || !block_pairs) return PKV_ERR_INVALID_ARG;
    if (!aligned16(key_cache) || !aligned16(value_cache)) return PKV_ERR_INVALID_ARG;
    const int64_t vpb = (int64_t)(block_bytes / 16);
    const int threads = 256;
    // about 4 vectors per thread per pair, at most 64 CTAs per block
    const int64_t gx = std::max<int64_t>(1, std::min<int64_t>(64, (vpb + 4 * threads - 1) / (4 * threads)));
    const int gy = std::min(num_pairs, 65535);
    uint4 *kc4 = static_cast<uint4 *>(key_cache), *vc4 = static_cast<uint4 *>(value_cache);
    const int64_t *pairs = block_pairs;
    int64_t vpb_arg = vpb;
    int np = num_pairs, nb = num_blocks;
    int32_t *st = dev_status;
    void *args[] = {&kc4, &vc4, &pairs, &np, &vpb_arg, &nb, &st};
    if (launch_pdl(reinterpret_cast<const void *>(&copy_blocks_kernel), dim3((unsigned)gx, (unsigned)gy, 2),
                   dim3(threads), 0, stream, args) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

extern "C" int pkv_validate_block_pairs(const int64_t *host_pairs, int num_pairs, int num_blocks) {
    if (num_pairs < 0 || num_blocks <= 0 || (num_pairs > 0 && !host_pairs)) return PKV_ERR_INVALID_ARG;
    std::vector<char> is_dst(num_blocks, 0), is_src(num_blocks, 0);
    for (int i = 0; i < num_pairs; ++i) {
        const int64_t s = host_pairs[2 * i], d = host_pairs[2 * i + 1];
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) return PKV_ERR_INVALID_ARG;
        if (is_dst[d]) return PKV_ERR_INVALID_ARG;
        is_dst[d] = 1;
        is_src[s] = 1;
    }
    for (int b = 0; b < num_blocks; ++b)
        if (is_dst[b] && is_src[b]) return PKV_ERR_INVALID_ARG;
    return PKV_OK;
}

extern "C" int pkv_selftest_wait_timeout(int32_t *dev_status, uint64_t limit_ns, pkv_stream_t stream) {
    if (!dev_status || limit_ns < 1000ull || limit_ns > 1000000000ull) return PKV_ERR_INVALID_ARG;
    wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(dev_status, limit_ns);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    return PKV_OK;
}

extern "C" int pkv_reshape_and_cache_layers(const void *const *keys, const void *const *values,
                                            void *const *key_caches, void *const *value_caches, int num_layers,
                                            const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                                            int head_dim, int block_size, int num_blocks, int32_t *dev_status,
                                            pkv_stream_t stream) {
    if (num_tokens == 0) return PKV_OK;
    if (num_layers < 1 || num_layers > PKV_MAX_LAYERS || !keys || !values || !key_caches || !value_caches)
        return PKV_ERR_INVALID_ARG;
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 8 || block_size <= 0 ||
        num_blocks <= 0 || !slot_mapping)
        return PKV_ERR_INVALID_ARG;
    LayerPointers lp;
    for (int l = 0; l < num_layers; ++l) {
        if (!keys[l] || !values[l] || !key_caches[l] || !value_caches[l] || !aligned16(keys[l]) ||
            !aligned16(values[l]) || !aligned16(key_caches[l]) || !aligned16(value_caches[l]))
            return PKV_ERR_INVALID_ARG;
        lp.key[l] = static_cast<const uint4 *>(keys[l]);
        lp.value[l] = static_cast<const uint4 *>(values[l]);
        lp.key_cache[l] = static_cast<uint4 *>(key_caches[l]);
        lp.value_cache[l] = static_cast<uint4 *>(value_caches[l]);
    }
    const int vpr = head_dim / 8;
    const int64_t heads_x_vecs = (int64_t)num_kv_heads * vpr;
    if (heads_x_vecs > (1 << 30)) return PKV_ERR_INVALID_ARG;
    int64_t nv = (int64_t)num_tokens * heads_x_vecs, num_slots = (int64_t)num_blocks * block_size;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>((nv + threads - 1) / threads, 4096);
    const int64_t *slots = slot_mapping;
    int hxv = (int)heads_x_vecs, vr = vpr, bsz = block_size;
    int32_t *st = dev_status;
    void *args[] = {&lp, &slots, &nv, &hxv, &vr, &bsz, &num_slots, &st};
    if (launch_pdl(reinterpret_cast<const void *>(&reshape_and_cache_layers_kernel),
                   dim3((unsigned)blocks, (unsigned)num_layers), dim3(threads), 0, stream, args) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

extern "C" int pkv_copy_blocks_layers(void *const *key_caches, void *const *value_caches, int num_layers,
                                      const int64_t *block_pairs, int num_pairs, size_t block_bytes,
                                      int num_blocks, int32_t *dev_status, pkv_stream_t stream) {
    if (num_pairs == 0) return PKV_OK;
    if (num_layers < 1 || num_layers > PKV_MAX_LAYERS || !key_caches || !value_caches) return PKV_ERR_INVALID_ARG;
    if (num_pairs < 0 || num_blocks <= 0 || block_bytes == 0 || block_bytes % 16 || !block_pairs)
        return PKV_ERR_INVALID_ARG;
    LayerPointers lp;
    for (int l = 0; l < num_layers; ++l) {
        if (!key_caches[l] || !value_caches[l] || !aligned16(key_caches[l]) || !aligned16(value_caches[l]))
            return PKV_ERR_INVALID_ARG;
        lp.key[l] = nullptr;
        lp.value[l] = nullptr;
        lp.key_cache[l] = static_cast<uint4 *>(key_caches[l]);
        lp.value_cache[l] = static_cast<uint4 *>(value_caches[l]);
    }
    const int64_t vpb = (int64_t)(block_bytes / 16);
    const int threads = 256;
    const int64_t gx = std::max<int64_t>(1, std::min<int64_t>(64, (vpb + 4 * threads - 1) / (4 * threads)));
    const int gy = std::min(num_pairs, 65535);
    const int64_t *pairs = block_pairs;
    int64_t vpb_arg = vpb;
    int np = num_pairs, nb = num_blocks;
    int32_t *st = dev_status;
    void *args[] = {&lp, &pairs, &np, &vpb_arg, &nb, &st};
    if (launch_pdl(reinterpret_cast<const void *>(&copy_blocks_layers_kernel),
                   dim3((unsigned)gx, (unsigned)gy, 2u * (unsigned)num_layers), dim3(threads), 0, stream,
                   args) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}
