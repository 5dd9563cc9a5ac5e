// pkv_decode_noalloc.cu -- decode attention for callers that cannot allocate
// device memory (see pkv_paged_attention_decode_noalloc in include/pkv.h).
//
// The scratch that pkv_paged_attention_decode takes from its caller lives here
// in a fixed static device array instead.  Host code cannot use the array's
// name as a device address (on the host it names a stand-in object), so the
// first call on each device asks the runtime for the real address with that
// device current, keeps it, and hands it to the regular entry point as its
// workspace.  Nothing here allocates.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pkv.h"

namespace {

__device__ __align__(256) unsigned char g_decode_scratch[PKV_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];

// Device address of g_decode_scratch on the current device (looked up once).
int scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    if (dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;  // a limit of this table, not a CUDA failure
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return PKV_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_paged_attention_decode_noalloc(void *out, const void *query, const void *key_cache,
                                                  const void *value_cache, const int32_t *block_tables,
                                                  int max_blocks_per_seq, const int32_t *context_lens,
                                                  int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                                  int block_size, int num_blocks, float scale, int num_ctas,
                                                  int32_t *dev_status, pkv_stream_t stream) {
    if (num_seqs == 0) return PKV_OK;
    // 0 means the regular entry point will reject the shape itself
    const size_t need = pkv_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                  num_ctas);
    if (need > PKV_DECODE_NOALLOC_SCRATCH_BYTES) return PKV_ERR_INVALID_ARG;
    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != PKV_OK) return rc;
    return pkv_paged_attention_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                      context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                      num_blocks, scale, num_ctas, scratch, PKV_DECODE_NOALLOC_SCRATCH_BYTES,
                                      dev_status, stream);
}
