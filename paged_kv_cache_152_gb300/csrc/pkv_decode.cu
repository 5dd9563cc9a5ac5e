// pkv_decode.cu -- host entry points of decode attention.
//
// pkv_paged_attention_decode validates its arguments on the host, picks the
// compiled instantiation for (head_dim, group, block_size), sizes the
// persistent grid (one full wave unless the caller fixes it), encodes the
// caches' tensor maps and launches the decode kernel on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <math.h>
#include <mutex>
#include <new>

#include <type_traits>

#include "../../include/pkv.h"
#include "pkv_decode_impl.cuh"
#include "pkv_launch.h"

// A validated decode call, ready to launch again and again (pkv_decode_plan_*).
struct pkv_decode_plan {
    pkv::DecodeParams params;
    const void *fn = nullptr;
    const void *fn_mapped = nullptr;  // the same launch reading its inputs with the lanes' copies
    int ctas = 0;
    int threads = 0;
    size_t smem = 0;
    size_t out_bytes = 0;  // fp16 [num_seqs][num_heads][head_dim]
    // bytes of each input the kernel reads (query, new key, new value, block
    // tables, context lengths, shared-prefix hints): a mapped step checks
    // that an input starting inside its host region also ends there
    size_t in_extent[6] = {0, 0, 0, 0, 0, 0};
    bool empty = true;
};

namespace pkv {

bool stage_in_by_kernel(void *dev_dst, const void *host_src, size_t bytes, cudaStream_t stream);  // pkv_stage.cu

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
bool decode_kernel_info_d64_grp(int, DecodeKernelInfo *);
bool decode_kernel_info_d128_grp(int, DecodeKernelInfo *);
#define PKV_DECLARE_MAPPED(d, g) const void *decode_kernel_fn_mapped_d##d##_g##g(int);
PKV_DECLARE_MAPPED(64, 1)
PKV_DECLARE_MAPPED(64, 2)
PKV_DECLARE_MAPPED(64, 4)
PKV_DECLARE_MAPPED(64, 8)
PKV_DECLARE_MAPPED(128, 1)
PKV_DECLARE_MAPPED(128, 2)
PKV_DECLARE_MAPPED(128, 4)
PKV_DECLARE_MAPPED(128, 8)
#undef PKV_DECLARE_MAPPED
const void *decode_kernel_fn_mapped_d64_grp(int);
const void *decode_kernel_fn_mapped_d128_grp(int);

bool decode_kernel_info_grouped(int head_dim, int block_size, DecodeKernelInfo *info) {
    if (head_dim == 64 && decode_kernel_info_d64_grp(block_size, info)) {
        info->fn_mapped = decode_kernel_fn_mapped_d64_grp(block_size);
        return true;
    }
    if (head_dim == 128 && decode_kernel_info_d128_grp(block_size, info)) {
        info->fn_mapped = decode_kernel_fn_mapped_d128_grp(block_size);
        return true;
    }
    return false;
}

bool decode_kernel_info(int head_dim, int group, int block_size, DecodeKernelInfo *info) {
#define PKV_CASE(d, g)                                                              \
    if (head_dim == d && group == g) {                                              \
        if (!decode_kernel_info_d##d##_g##g(block_size, info)) return false;        \
        info->fn_mapped = decode_kernel_fn_mapped_d##d##_g##g(block_size);          \
        return true;                                                                \
    }
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
constexpr int kMaxSeqsGrouped = 1024;  // the grouped kernel's per-sequence shared memory (32 bytes each)
constexpr int kGroupRows = 8;          // query rows of a grouped item: up to 8 sequences of group 1
constexpr int kMaxCtas = 4096;

struct Resolved {
    DecodeKernelInfo info;
    size_t smem;
    int ctas;
    int64_t workers;
    bool smem_partials;  // the grid's shared memory includes the partial slots
};

bool shape_supported(int num_heads, int num_kv_heads, int head_dim, int block_size) {
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return false;
    DecodeKernelInfo info;
    return decode_kernel_info(head_dim, num_heads / num_kv_heads, block_size, &info);
}

// Raises the kernel's dynamic shared-memory limit to `smem` on the current
// device if needed.  The attribute is held per device, so what was raised is
// remembered per (device, kernel).
int ensure_smem_attr(const void *fn, size_t smem) {
    constexpr int kSlots = 512;
    static std::mutex mu;
    static const void *fns[kSlots];
    static int devs[kSlots];
    static size_t set[kSlots];
    static int n = 0;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(mu);
    int k = 0;
    while (k < n && !(fns[k] == fn && devs[k] == dev)) ++k;
    if (k < n && set[k] >= smem) return PKV_OK;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    if (k == n && n < kSlots) {
        fns[n] = fn;
        devs[n] = dev;
        ++n;
    }
    if (k < kSlots) set[k] = smem;
    return PKV_OK;
}

// Whether a call with prefix-sharing hints runs the grouped kernel: group 1,
// whole-block chunks (block size 16 or more), a batch whose per-sequence
// arrays fit; other calls run the plain kernel and the hints are not needed.
bool use_grouped(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size) {
    DecodeKernelInfo info;
    return num_heads == num_kv_heads && block_size >= 16 && num_seqs <= kMaxSeqsGrouped &&
           decode_kernel_info_grouped(head_dim, block_size, &info);
}

int resolve(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size, int num_ctas,
            Resolved *r, bool grouped = false) {
    if (grouped ? !decode_kernel_info_grouped(head_dim, block_size, &r->info)
                : !decode_kernel_info(head_dim, num_heads / num_kv_heads, block_size, &r->info))
        return PKV_ERR_UNSUPPORTED;
    // [cum (N+1)][ctx (N)] padded to 8 bytes, then [bounds (C+1)]
    const size_t seq_bytes = ((r->info.smem_per_seq * (size_t)num_seqs + 4) + 7) & ~(size_t)7;
    auto smem_for = [&](int ctas) { return r->info.smem_fixed + seq_bytes + r->info.smem_per_cta * (size_t)(ctas + 1); };
    if (num_ctas > kMaxCtas) return PKV_ERR_INVALID_ARG;
    r->smem = smem_for(num_ctas > 0 ? num_ctas : 1);
    int dev = 0, sms = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    if (num_ctas <= 0) {
        // one full wave; the bounds array grows with the grid, so settle the
        // grid and the shared memory together
        // (the occupancy is taken with the partial slots included when they fit)
        const size_t part = r->info.smem_partials;
        size_t smem = smem_for(sms * 4) + part;
        if (smem + 2 * 1024 > (size_t)optin) smem = smem_for(sms) + part;
        if (smem + 2 * 1024 > (size_t)optin) smem = smem_for(sms);
        if (smem + 2 * 1024 > (size_t)optin) return PKV_ERR_INVALID_ARG;
        int rc0 = ensure_smem_attr(r->info.fn, smem);
        if (rc0 != PKV_OK) return rc0;
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, r->info.fn, r->info.threads, smem) !=
                cudaSuccess ||
            per_sm < 1) {
            cudaGetLastError();
            return PKV_ERR_CUDA;
        }
        num_ctas = sms * (per_sm < 4 ? per_sm : 4);
        r->smem = smem_for(num_ctas);
    }
    if (r->smem + 2 * 1024 > (size_t)optin) return PKV_ERR_INVALID_ARG;  // + static shared memory
    // partials of CTA-local merges in shared memory when they fit (else the
    // workspace holds them; same arithmetic either way)
    r->smem_partials = r->smem + r->info.smem_partials + 2 * 1024 <= (size_t)optin;
    if (r->smem_partials) r->smem += r->info.smem_partials;
    int rc = ensure_smem_attr(r->info.fn, r->smem);
    if (rc == PKV_OK && r->info.fn_mapped) rc = ensure_smem_attr(r->info.fn_mapped, r->smem);
    if (rc != PKV_OK) return rc;
    r->ctas = num_ctas;
    r->workers = (int64_t)num_ctas * r->info.warps;
    return PKV_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuTensorMapEncodeTiled from the driver (looked up once, no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            cudaGetLastError();
    });
    return fn;
}

// The cache as a 3-D tensor: 64 dims (innermost), num_blocks * Hkv *
// block_size rows (stride head_dim * 2 bytes), head_dim / 64 halves (stride
// 128 bytes), read with the 128-byte swizzle in boxes of {64, box_rows,
// box_halves}: a box lands in shared memory as [half][row][64 dims].  No L2
// promotion: a box is one contiguous run of whole 128-byte lines already,
// and widening the requests measured ~1% slower (7b 96.1 against 94.8 us).
int encode_cache_map(CUtensorMap *map, const void *cache, int num_blocks, int num_kv_heads, int block_size,
                     int head_dim, int box_rows, int box_halves) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return PKV_ERR_CUDA;
    const cuuint64_t dims[3] = {64, (cuuint64_t)num_blocks * num_kv_heads * block_size,
                                (cuuint64_t)(head_dim / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_halves};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(cache), dims, strides,
                              box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

namespace {

size_t workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size, int num_ctas,
                      bool shared) {
    if (num_seqs < 1 || num_seqs > kMaxSeqs) return 0;
    if (!shape_supported(num_heads, num_kv_heads, head_dim, block_size)) return 0;
    const bool grouped = shared && use_grouped(num_seqs, num_heads, num_kv_heads, head_dim, block_size);
    Resolved r;
    if (resolve(num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_ctas, &r, grouped) != PKV_OK)
        return 0;
    return DecodeWorkspace::plan(num_seqs, num_kv_heads, r.workers, r.ctas,
                                 grouped ? kGroupRows : num_heads / num_kv_heads, head_dim)
        .total;
}

}  // namespace

extern "C" size_t pkv_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                            int block_size, int num_ctas) {
    return workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_ctas, false);
}

extern "C" size_t pkv_decode_workspace_size_shared(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                                   int block_size, int num_ctas) {
    return workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_ctas, true);
}

extern "C" int pkv_decode_default_ctas(int num_heads, int num_kv_heads, int head_dim, int block_size) {
    if (!shape_supported(num_heads, num_kv_heads, head_dim, block_size)) return 0;
    Resolved r;
    if (resolve(1, num_heads, num_kv_heads, head_dim, block_size, 0, &r) != PKV_OK) return 0;
    return r.ctas;
}

namespace {

// Validates one decode call and fills a launch plan (kernel, grid, shared
// memory, parameter block with the encoded tensor maps).  plan->empty marks a
// call with no sequences (nothing to launch).
int build_plan(void *out, const void *query, const void *new_key, const void *new_value, const void *key_cache,
               const void *value_cache, const int32_t *block_tables, int max_blocks_per_seq,
               const int32_t *context_lens, const int32_t *shared_blocks, int num_seqs, int num_heads,
               int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale, int num_ctas,
               void *workspace, size_t workspace_bytes, int32_t *dev_status, pkv_decode_plan *plan) {
    plan->empty = num_seqs == 0;
    if (num_seqs == 0) return PKV_OK;
    if ((new_key == nullptr) != (new_value == nullptr)) return PKV_ERR_INVALID_ARG;
    if (new_key && (!aligned16(new_key) || !aligned16(new_value))) return PKV_ERR_INVALID_ARG;
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
    if ((int64_t)num_blocks * num_kv_heads * block_size >= (INT64_C(1) << 31)) return PKV_ERR_INVALID_ARG;
    if (!shape_supported(num_heads, num_kv_heads, head_dim, block_size)) return PKV_ERR_UNSUPPORTED;

    const bool grouped = shared_blocks != nullptr &&
                         use_grouped(num_seqs, num_heads, num_kv_heads, head_dim, block_size);
    Resolved r;
    int rc = resolve(num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_ctas, &r, grouped);
    if (rc != PKV_OK) return rc;
    const int group = num_heads / num_kv_heads;
    const DecodeWorkspace ws = DecodeWorkspace::plan(num_seqs, num_kv_heads, r.workers, r.ctas,
                                                     grouped ? kGroupRows : group, head_dim);
    if (workspace_bytes < ws.total) return PKV_ERR_INVALID_ARG;
    unsigned char *wsb = static_cast<unsigned char *>(workspace);

    DecodeParams &p = plan->params;
    {
        const int chunk_rows = block_size < 16 ? block_size : 16;
        const int halves = head_dim / 64;
        rc = encode_cache_map(&p.tmap_k, key_cache, num_blocks, num_kv_heads, block_size, head_dim, chunk_rows,
                              halves);
        if (rc == PKV_OK)
            rc = encode_cache_map(&p.tmap_v, value_cache, num_blocks, num_kv_heads, block_size, head_dim,
                                  chunk_rows, halves);
        if (rc == PKV_OK)
            rc = encode_cache_map(&p.tmap_k8, key_cache, num_blocks, num_kv_heads, block_size, head_dim, 8, 1);
        if (rc == PKV_OK)
            rc = encode_cache_map(&p.tmap_v8, value_cache, num_blocks, num_kv_heads, block_size, head_dim, 8, 1);
        if (rc != PKV_OK) return rc;
    }
    p.out = static_cast<__half *>(out);
    p.query = static_cast<const __half *>(query);
    p.key_cache = static_cast<const __half *>(key_cache);
    p.value_cache = static_cast<const __half *>(value_cache);
    p.new_key = static_cast<const __half *>(new_key);
    p.new_value = static_cast<const __half *>(new_value);
    p.key_cache_w = static_cast<__half *>(const_cast<void *>(key_cache));
    p.value_cache_w = static_cast<__half *>(const_cast<void *>(value_cache));
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.ws_ml = reinterpret_cast<float *>(wsb + ws.ml);
    p.ws_acc = reinterpret_cast<float *>(wsb + ws.acc);
    p.ws_cml = reinterpret_cast<float *>(wsb + ws.cml);
    p.ws_cacc = reinterpret_cast<float *>(wsb + ws.cacc);
    p.ws_sync = reinterpret_cast<unsigned long long *>(wsb + ws.sync);
    p.ws_count = reinterpret_cast<unsigned long long *>(wsb + ws.count);
    p.status = dev_status;
    p.shared_blocks = grouped ? shared_blocks : nullptr;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
    p.wait_limit_ns = kWaitLimitNs;
    p.smem_partials = r.smem_partials ? 1 : 0;

    plan->out_bytes = (size_t)num_seqs * num_heads * head_dim * 2;
    plan->in_extent[0] = (size_t)num_seqs * num_heads * head_dim * 2;
    plan->in_extent[1] = plan->in_extent[2] = (size_t)num_seqs * num_kv_heads * head_dim * 2;
    plan->in_extent[3] = (size_t)num_seqs * max_blocks_per_seq * 4;
    plan->in_extent[4] = plan->in_extent[5] = (size_t)num_seqs * 4;
    plan->fn = r.info.fn;
    plan->fn_mapped = r.info.fn_mapped;
    plan->ctas = r.ctas;
    plan->threads = r.info.threads;
    plan->smem = r.smem;
    return PKV_OK;
}

int launch_plan(const pkv_decode_plan &plan, pkv_stream_t stream) {
    if (plan.empty) return PKV_OK;
    void *args[] = {const_cast<DecodeParams *>(&plan.params)};
    if (launch_pdl(plan.fn, dim3(plan.ctas), dim3(plan.threads), plan.smem, stream, args) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

int decode_impl(void *out, const void *query, const void *new_key, const void *new_value, const void *key_cache,
                const void *value_cache, const int32_t *block_tables, int max_blocks_per_seq,
                const int32_t *context_lens, const int32_t *shared_blocks, int num_seqs, int num_heads,
                int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale, int num_ctas,
                void *workspace, size_t workspace_bytes, int32_t *dev_status, pkv_stream_t stream) {
    pkv_decode_plan plan;
    const int rc = build_plan(out, query, new_key, new_value, key_cache, value_cache, block_tables,
                              max_blocks_per_seq, context_lens, shared_blocks, num_seqs, num_heads, num_kv_heads,
                              head_dim, block_size, num_blocks, scale, num_ctas, workspace, workspace_bytes,
                              dev_status, &plan);
    if (rc != PKV_OK) return rc;
    return launch_plan(plan, stream);
}

}  // namespace

extern "C" int pkv_paged_attention_decode(void *out, const void *query, const void *key_cache,
                                          const void *value_cache, const int32_t *block_tables,
                                          int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                          int num_heads, int num_kv_heads, int head_dim, int block_size,
                                          int num_blocks, float scale, int num_ctas, void *workspace,
                                          size_t workspace_bytes, int32_t *dev_status, pkv_stream_t stream) {
    return decode_impl(out, query, nullptr, nullptr, key_cache, value_cache, block_tables, max_blocks_per_seq,
                       context_lens, nullptr, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       scale, num_ctas, workspace, workspace_bytes, dev_status, stream);
}

extern "C" int pkv_paged_attention_decode_append(void *out, const void *query, const void *key,
                                                 const void *value, void *key_cache, void *value_cache,
                                                 const int32_t *block_tables, int max_blocks_per_seq,
                                                 const int32_t *context_lens, int num_seqs, int num_heads,
                                                 int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                                 float scale, int num_ctas, void *workspace,
                                                 size_t workspace_bytes, int32_t *dev_status,
                                                 pkv_stream_t stream) {
    if (num_seqs > 0 && (!key || !value)) return PKV_ERR_INVALID_ARG;
    return decode_impl(out, query, key, value, key_cache, value_cache, block_tables, max_blocks_per_seq,
                       context_lens, nullptr, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       scale, num_ctas, workspace, workspace_bytes, dev_status, stream);
}

extern "C" int pkv_paged_attention_decode_shared(void *out, const void *query, const void *key, const void *value,
                                                 void *key_cache, void *value_cache, const int32_t *block_tables,
                                                 int max_blocks_per_seq, const int32_t *context_lens,
                                                 const int32_t *shared_blocks, int num_seqs, int num_heads,
                                                 int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                                 float scale, int num_ctas, void *workspace,
                                                 size_t workspace_bytes, int32_t *dev_status,
                                                 pkv_stream_t stream) {
    if ((key == nullptr) != (value == nullptr)) return PKV_ERR_INVALID_ARG;
    if (num_seqs > 0 && !shared_blocks) return PKV_ERR_INVALID_ARG;
    return decode_impl(out, query, key, value, key_cache, value_cache, block_tables, max_blocks_per_seq,
                       context_lens, shared_blocks, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, scale, num_ctas, workspace, workspace_bytes, dev_status, stream);
}

namespace {

// Where a plan's kernel writes its output: device memory of the current
// device, managed memory, or page-locked host memory mapped into the
// device's address space (then through its device address: the output goes
// straight over the CPU-GPU link as segments finish, and a serving step
// needs no copy back).  Pageable host memory and other devices' memory are
// refused.
int plan_output(void *out, pkv_decode_plan *plan) {
    cudaPointerAttributes attr;
    int dev = -1;
    if (cudaPointerGetAttributes(&attr, out) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    switch (attr.type) {
        case cudaMemoryTypeDevice:
            return attr.device == dev ? PKV_OK : PKV_ERR_INVALID_ARG;
        case cudaMemoryTypeManaged:
            return PKV_OK;
        case cudaMemoryTypeHost:
            if (attr.devicePointer == nullptr || !aligned16(attr.devicePointer)) return PKV_ERR_INVALID_ARG;
            plan->params.out = static_cast<__half *>(attr.devicePointer);
            return PKV_OK;
        default:
            return PKV_ERR_INVALID_ARG;
    }
}

}  // namespace

namespace {

int plan_create(void *out, const void *query, const void *key, const void *value, void *key_cache,
                void *value_cache, const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                const int32_t *shared_blocks, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                int block_size, int num_blocks, float scale, int num_ctas, void *workspace, size_t workspace_bytes,
                int32_t *dev_status, pkv_decode_plan_t **plan_out) {
    if (!plan_out) return PKV_ERR_INVALID_ARG;
    *plan_out = nullptr;
    if ((key == nullptr) != (value == nullptr)) return PKV_ERR_INVALID_ARG;
    pkv_decode_plan *plan = new (std::nothrow) pkv_decode_plan;
    if (!plan) return PKV_ERR_INVALID_ARG;
    int rc = build_plan(out, query, key, value, key_cache, value_cache, block_tables, max_blocks_per_seq,
                        context_lens, shared_blocks, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                        num_blocks, scale, num_ctas, workspace, workspace_bytes, dev_status, plan);
    if (rc == PKV_OK && !plan->empty) rc = plan_output(out, plan);
    if (rc != PKV_OK) {
        delete plan;
        return rc;
    }
    *plan_out = plan;
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_decode_plan_create(void *out, const void *query, const void *key, const void *value,
                                      void *key_cache, void *value_cache, const int32_t *block_tables,
                                      int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                      int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                      float scale, int num_ctas, void *workspace, size_t workspace_bytes,
                                      int32_t *dev_status, pkv_decode_plan_t **plan_out) {
    return plan_create(out, query, key, value, key_cache, value_cache, block_tables, max_blocks_per_seq,
                       context_lens, nullptr, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       scale, num_ctas, workspace, workspace_bytes, dev_status, plan_out);
}

extern "C" int pkv_decode_plan_create_shared(void *out, const void *query, const void *key, const void *value,
                                             void *key_cache, void *value_cache, const int32_t *block_tables,
                                             int max_blocks_per_seq, const int32_t *context_lens,
                                             const int32_t *shared_blocks, int num_seqs, int num_heads,
                                             int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                             float scale, int num_ctas, void *workspace, size_t workspace_bytes,
                                             int32_t *dev_status, pkv_decode_plan_t **plan_out) {
    if (plan_out) *plan_out = nullptr;
    if (num_seqs > 0 && !shared_blocks) return PKV_ERR_INVALID_ARG;
    return plan_create(out, query, key, value, key_cache, value_cache, block_tables, max_blocks_per_seq,
                       context_lens, shared_blocks, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, scale, num_ctas, workspace, workspace_bytes, dev_status, plan_out);
}

extern "C" int pkv_decode_plan_launch(const pkv_decode_plan_t *plan, pkv_stream_t stream) {
    if (!plan) return PKV_ERR_INVALID_ARG;
    return launch_plan(*plan, stream);
}

extern "C" int pkv_decode_plan_step(const pkv_decode_plan_t *plan, void *dev_in, const void *host_in,
                                    size_t in_bytes, void *host_out, pkv_stream_t stream) {
    if (!plan || (in_bytes && (!dev_in || !host_in))) return PKV_ERR_INVALID_ARG;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // mapped page-locked input: copied by a kernel reading it over the link
    // (one wave of 16-byte loads), else by a copy engine
    if (in_bytes && !stage_in_by_kernel(dev_in, host_in, in_bytes, s) &&
        cudaMemcpyAsync(dev_in, host_in, in_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    const int rc = launch_plan(*plan, stream);
    if (rc != PKV_OK) return rc;
    if (host_out && plan->out_bytes &&
        cudaMemcpyAsync(host_out, plan->params.out, plan->out_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

extern "C" int pkv_decode_plan_step_mapped(const pkv_decode_plan_t *plan, const void *dev_base, const void *host_in,
                                           size_t in_bytes, void *host_out, pkv_stream_t stream) {
    if (!plan || !dev_base || !host_in || in_bytes == 0) return PKV_ERR_INVALID_ARG;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, host_in) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_INVALID_ARG;
    }
    if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return PKV_ERR_INVALID_ARG;
    // every input inside the region moves to the same offset of the mapping
    const uintptr_t lo = reinterpret_cast<uintptr_t>(dev_base), hi = lo + in_bytes;
    const intptr_t delta = reinterpret_cast<intptr_t>(attr.devicePointer) - static_cast<intptr_t>(lo);
    DecodeParams prm = plan->params;
    bool inside = true;  // every moved input lies wholly inside the region
    auto move = [&](auto &ptr, size_t extent) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(ptr);
        if (!ptr || a < lo || a >= hi) return;
        if (extent > hi - a) inside = false;
        ptr = reinterpret_cast<std::remove_reference_t<decltype(ptr)>>(a + delta);
    };
    move(prm.query, plan->in_extent[0]);
    move(prm.new_key, plan->in_extent[1]);
    move(prm.new_value, plan->in_extent[2]);
    move(prm.block_tables, plan->in_extent[3]);
    move(prm.context_lens, plan->in_extent[4]);
    move(prm.shared_blocks, plan->in_extent[5]);
    if (!inside) return PKV_ERR_INVALID_ARG;
    auto aligned = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    if (!aligned(prm.query) || (prm.new_key && (!aligned(prm.new_key) || !aligned(prm.new_value))))
        return PKV_ERR_INVALID_ARG;
    if (!plan->empty) {
        if (!plan->fn_mapped) return PKV_ERR_UNSUPPORTED;
        void *args[] = {&prm};
        if (launch_pdl(plan->fn_mapped, dim3(plan->ctas), dim3(plan->threads), plan->smem, stream, args) !=
            cudaSuccess) {
            cudaGetLastError();
            return PKV_ERR_CUDA;
        }
    }
    if (host_out && plan->out_bytes &&
        cudaMemcpyAsync(host_out, plan->params.out, plan->out_bytes, cudaMemcpyDeviceToHost,
                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

extern "C" void pkv_decode_plan_destroy(pkv_decode_plan_t *plan) { delete plan; }
