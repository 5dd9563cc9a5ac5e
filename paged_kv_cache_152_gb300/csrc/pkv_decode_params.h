// pkv_decode_params.h -- kernel parameter blocks of the decode path.
#ifndef PKV_DECODE_PARAMS_H
#define PKV_DECODE_PARAMS_H

#include <cuda.h>
#include <cuda_fp16.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

struct DecodeParams {
    // The caches viewed as 3-D tensors (64 dims, NB*Hkv*BS rows, D/64 halves;
    // row stride D*2 bytes, half stride 128 bytes) read with the 128-byte
    // swizzle, so that a box lands as [half][row][64 dims]:
    CUtensorMap tmap_k;           // box: all halves of one chunk's rows
    CUtensorMap tmap_v;
    CUtensorMap tmap_k8;          // box: one half of 8 rows (short last chunks)
    CUtensorMap tmap_v8;
    __half *out;                  // [N][H][D]
    const __half *query;          // [N][H][D]
    const __half *key_cache;      // [NB][Hkv][BS][D]
    const __half *value_cache;    // [NB][Hkv][BS][D]
    const __half *new_key;        // [N][Hkv][D] new token per sequence (NULL: no append)
    const __half *new_value;      // [N][Hkv][D]
    __half *key_cache_w;          // the caches, for writing the new tokens' rows
    __half *value_cache_w;
    const int32_t *block_tables;  // [N][MB]
    const int32_t *context_lens;  // [N]
    float *ws_ml;                 // [W][2][G][2] partial (max, sum) of a worker's piece
    float *ws_acc;                // [W][2][G][D] partial unnormalised outputs
    float *ws_cml;                // [C][2][G][2] a CTA's part of a segment that spans CTAs
    float *ws_cacc;               // [C][2][G][D]
    // Completion counters, each (epoch << 32 | arrivals): ws_sync[0] is the
    // epoch word, ws_sync[1 + parity] the per-call exit counters, and ws_count
    // two arrays (by epoch parity) of N*Hkv per-segment counters.
    unsigned long long *ws_sync;  // [3]
    unsigned long long *ws_count; // [2][N*Hkv]
    int32_t *status;              // nullable
    // grouped (prefix-sharing) kernel only, else NULL: the leading blocks
    // sequence s shares with s - 1 (the caller's hint), [N]
    const int32_t *shared_blocks;
    int num_seqs;
    int num_heads;
    int num_kv_heads;
    int max_blocks_per_seq;
    int num_blocks;
    float scale_log2;             // scale * log2(e)
    uint64_t wait_limit_ns;
    // 1: partials of segments cut between workers of one CTA are kept in the
    // CTA's shared memory (after the CTA bounds); 0: in ws_ml / ws_acc
    int smem_partials;
};

// Workspace carve-up (byte offsets), shared by the size query and the launch.
// group = query rows per segment (8 for the grouped kernel, whose segments'
// owners -- groups and lone sequences -- are at most num_seqs).
struct DecodeWorkspace {
    size_t sync, count, ml, acc, cml, cacc, total;
    static DecodeWorkspace plan(int num_seqs, int num_kv_heads, int64_t workers, int64_t ctas, int group,
                                int head_dim) {
        auto up = [](size_t x) { return (x + 255) / 256 * 256; };
        DecodeWorkspace w;
        w.sync = 0;
        w.count = 256;
        w.ml = w.count + up(2 * 8 * (size_t)num_seqs * num_kv_heads);
        w.acc = w.ml + up(4 * (size_t)workers * 2 * group * 2);
        w.cml = w.acc + up(4 * (size_t)workers * 2 * group * head_dim);
        w.cacc = w.cml + up(4 * (size_t)ctas * 2 * group * 2);
        w.total = w.cacc + up(4 * (size_t)ctas * 2 * group * head_dim);
        return w;
    }
};

// Host-side description of one compiled decode instantiation.
struct DecodeKernelInfo {
    const void *fn;        // __global__ function
    // the same shape's instantiation that reads query, new_key and new_value
    // with the lanes' 16-byte copies, so that they may be page-locked host
    // memory (pkv_decode_plan_step_mapped); same shared memory and grid
    const void *fn_mapped;
    int threads;           // threads per CTA
    int warps;             // workers per CTA
    int rows_per_chunk;
    size_t smem_fixed;     // dynamic shared memory without the per-sequence arrays
    size_t smem_per_seq;   // bytes per sequence (+ one extra int)
    size_t smem_per_cta;   // bytes per CTA of the grid (+ one extra)
    size_t smem_partials;  // bytes of the optional shared-memory partial slots
};

// Defined in pkv_decode_d{64,128}_g{1,2,4,8}.cu (fn) and ..._mapped.cu
// (fn_mapped); false if not compiled.
bool decode_kernel_info(int head_dim, int group, int block_size, DecodeKernelInfo *info);
// The grouped (prefix-sharing) kernel of group 1: pkv_decode_d{64,128}_grp.cu.
bool decode_kernel_info_grouped(int head_dim, int block_size, DecodeKernelInfo *info);

}  // namespace pkv

#endif  // PKV_DECODE_PARAMS_H
