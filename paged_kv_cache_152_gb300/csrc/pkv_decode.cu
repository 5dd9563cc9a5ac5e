// pkv_decode.cu -- host entry points of decode attention.
//
// pkv_paged_attention_decode validates its arguments on the host, picks the
// compiled instantiation for (head_dim, group, block_size), sizes the
// persistent grid (one full wave unless the caller fixes it), tags the call
// with a fresh generation number and launches the decode kernel on the
// caller's stream.
#include <cuda_runtime.h>

#include <atomic>
#include <math.h>
#include <mutex>

#include "../../include/pkv.h"
#include "pkv_decode_impl.cuh"

namespace pkv {

#define PKV_DECLARE_INFO(d, g) bool decode_kernel_info_d##d##_g##g(int, DecodeKernelInfo *);
PKV_DECLARE_INFO(64, 1)
PKV_DECLARE_INFO(64, 2)
PKV_DECLARE_INFO(64, 4)
PKV_DECLARE_INFO(64, 8)
PKV_DECLARE_INFO(128, 1)
PKV_DECLARE_INFO(128, 2)
PKV_DECLARE_INFO(128, 4)
PKV_DECLARE_INFO(128, 8)
#undef PKV_DECLARE_INFO

bool decode_kernel_info(int head_dim, int group, int block_size, DecodeKernelInfo *info) {
#define PKV_CASE(d, g) \
    if (head_dim == d && group == g) return decode_kernel_info_d##d##_g##g(block_size, info);
    PKV_CASE(64, 1)
    PKV_CASE(64, 2)
    PKV_CASE(64, 4)
    PKV_CASE(64, 8)
    PKV_CASE(128, 1)
    PKV_CASE(128, 2)
    PKV_CASE(128, 4)
    PKV_CASE(128, 8)
#undef PKV_CASE
    return false;
}

namespace {

constexpr int kMaxSeqs = 4096;

struct Resolved {
    DecodeKernelInfo info;
    size_t smem;
    int ctas;
    int64_t workers;
};

bool shape_supported(int num_heads, int num_kv_heads, int head_dim, int block_size) {
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return false;
    DecodeKernelInfo info;
    return decode_kernel_info(head_dim, num_heads / num_kv_heads, block_size, &info);
}

// Raises the kernel's dynamic shared-memory limit to `smem` if needed.
int ensure_smem_attr(const void *fn, size_t smem) {
    static std::mutex mu;
    static const void *fns[128];
    static size_t set[128];
    static int nfns = 0;
    std::lock_guard<std::mutex> lock(mu);
    int k = 0;
    while (k < nfns && fns[k] != fn) ++k;
    if (k < nfns && set[k] >= smem) return PKV_OK;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    if (k == nfns && nfns < 128) fns[nfns++] = fn;
    if (k < 128) set[k] = smem;
    return PKV_OK;
}

int resolve(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size, int num_ctas,
            Resolved *r) {
    if (!decode_kernel_info(head_dim, num_heads / num_kv_heads, block_size, &r->info))
        return PKV_ERR_UNSUPPORTED;
    r->smem = r->info.smem_fixed + r->info.smem_per_seq * (size_t)num_seqs + 4;
    int dev = 0, sms = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    if (r->smem + 2 * 1024 > (size_t)optin) return PKV_ERR_INVALID_ARG;  // + static shared memory
    const int rc = ensure_smem_attr(r->info.fn, r->smem);
    if (rc != PKV_OK) return rc;
    if (num_ctas <= 0) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, r->info.fn, r->info.threads, r->smem) !=
                cudaSuccess ||
            per_sm < 1) {
            cudaGetLastError();
            return PKV_ERR_CUDA;
        }
        num_ctas = sms * per_sm;
    }
    r->ctas = num_ctas;
    r->workers = (int64_t)num_ctas * r->info.warps;
    return PKV_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Distinct nonzero tag per call (wraps after 2^32 - 1 calls).
uint32_t next_generation() {
    static std::atomic<uint32_t> counter{0};
    uint32_t g;
    do { g = counter.fetch_add(1, std::memory_order_relaxed) + 1; } while (g == 0);
    return g;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" size_t pkv_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                            int block_size, int num_ctas) {
    if (num_seqs < 1 || num_seqs > kMaxSeqs) return 0;
    if (!shape_supported(num_heads, num_kv_heads, head_dim, block_size)) return 0;
    Resolved r;
    if (resolve(num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_ctas, &r) != PKV_OK) return 0;
    return DecodeWorkspace::plan(num_seqs, num_kv_heads, r.workers, num_heads / num_kv_heads, head_dim).total;
}

extern "C" int pkv_decode_default_ctas(int num_heads, int num_kv_heads, int head_dim, int block_size) {
    if (!shape_supported(num_heads, num_kv_heads, head_dim, block_size)) return 0;
    Resolved r;
    if (resolve(1, num_heads, num_kv_heads, head_dim, block_size, 0, &r) != PKV_OK) return 0;
    return r.ctas;
}

extern "C" int pkv_paged_attention_decode(void *out, const void *query, const void *key_cache,
                                          const void *value_cache, const int32_t *block_tables,
                                          int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                          int num_heads, int num_kv_heads, int head_dim, int block_size,
                                          int num_blocks, float scale, int num_ctas, void *workspace,
                                          size_t workspace_bytes, int32_t *dev_status, pkv_stream_t stream) {
    if (num_seqs == 0) return PKV_OK;
    if (num_seqs < 0 || num_seqs > kMaxSeqs || max_blocks_per_seq < 1 || num_blocks < 1 || num_ctas < 0)
        return PKV_ERR_INVALID_ARG;
    if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens || !workspace)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return PKV_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return PKV_ERR_INVALID_ARG;
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return PKV_ERR_INVALID_ARG;
    if ((int64_t)max_blocks_per_seq * block_size > (1 << 30)) return PKV_ERR_INVALID_ARG;
    if (!shape_supported(num_heads, num_kv_heads, head_dim, block_size)) return PKV_ERR_UNSUPPORTED;

    Resolved r;
    int rc = resolve(num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_ctas, &r);
    if (rc != PKV_OK) return rc;
    const int group = num_heads / num_kv_heads;
    const DecodeWorkspace ws = DecodeWorkspace::plan(num_seqs, num_kv_heads, r.workers, group, head_dim);
    if (workspace_bytes < ws.total) return PKV_ERR_INVALID_ARG;
    unsigned char *wsb = static_cast<unsigned char *>(workspace);

    DecodeParams p;
    p.out = static_cast<__half *>(out);
    p.query = static_cast<const __half *>(query);
    p.key_cache = static_cast<const __half *>(key_cache);
    p.value_cache = static_cast<const __half *>(value_cache);
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.ws_ml = reinterpret_cast<float *>(wsb + ws.ml);
    p.ws_acc = reinterpret_cast<float *>(wsb + ws.acc);
    p.ws_count = reinterpret_cast<unsigned long long *>(wsb + ws.count);
    p.status = dev_status;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
    p.generation = next_generation();
    p.wait_limit_ns = kWaitLimitNs;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    void *args[] = {&p};
    if (cudaLaunchKernel(r.info.fn, dim3(r.ctas), dim3(r.info.threads), args, r.smem, st) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }

    return PKV_OK;
}
