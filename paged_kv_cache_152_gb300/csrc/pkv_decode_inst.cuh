// pkv_decode_inst.cuh -- instantiates the decode kernel for one (head_dim,
// group) pair and every supported block size.  Each pkv_decode_d*_g*.cu
// includes it once, so the 8 instantiation sets compile in parallel; each
// pkv_decode_d*_*_mapped.cu (PKV_MAPPED) instantiates the same shapes with
// host inputs (the mapped plan step) and defines only their look-up.
#include "pkv_decode_impl.cuh"

#ifndef PKV_D
#error "define PKV_D and PKV_G"
#endif

#define PKV_CAT2(a, b, c) a##b##_g##c
#define PKV_CAT(a, b, c) PKV_CAT2(a, b, c)
#ifdef PKV_GRP
#define PKV_CATG2(a, b) a##b##_grp
#define PKV_CATG(a, b) PKV_CATG2(a, b)
#define PKV_INFO_FN PKV_CATG(decode_kernel_info_d, PKV_D)
#define PKV_MAPPED_FN PKV_CATG(decode_kernel_fn_mapped_d, PKV_D)
#else
#define PKV_INFO_FN PKV_CAT(decode_kernel_info_d, PKV_D, PKV_G)
#define PKV_MAPPED_FN PKV_CAT(decode_kernel_fn_mapped_d, PKV_D, PKV_G)
#endif

namespace pkv {
namespace {

// Warps (workers) per CTA and ring stages per warp.  A stage holds one K
// chunk and one V chunk (4 KB each at head_dim 128) plus the group's query
// rows.  One CTA of 8 workers x 2 stages per SM measured fastest on GB300
// (more warps per SM hide the per-chunk math; deeper rings did not help).
#ifdef PKV_DECODE_WARPS
constexpr int kWarps = PKV_DECODE_WARPS;
#else
constexpr int kWarps = 8;
#endif
#ifdef PKV_DECODE_STAGES
constexpr int kStages = PKV_DECODE_STAGES;
#else
constexpr int kStages = (PKV_D == 64) ? 4 : 2;
#endif

#ifdef PKV_GRP
constexpr bool kGrouped = true;   // the grouped (prefix-sharing) kernel: 8 query rows per item
#else
constexpr bool kGrouped = false;
#endif

#ifdef PKV_MAPPED
template <int BS>
const void *mapped_of() {
    return reinterpret_cast<const void *>(&paged_decode_kernel<PKV_D, BS, PKV_G, kWarps, kStages, kGrouped, true>);
}
#else
template <int BS>
DecodeKernelInfo info_of() {
    using Geo = DecodeGeometry<PKV_D, BS, PKV_G>;
    using Smem = DecodeSmem<kWarps, kStages, PKV_D, BS, PKV_G, kGrouped>;
    DecodeKernelInfo i;
    i.fn = reinterpret_cast<const void *>(&paged_decode_kernel<PKV_D, BS, PKV_G, kWarps, kStages, kGrouped>);
    i.threads = kWarps * 32;
    i.warps = kWarps;
    i.rows_per_chunk = Geo::kRows;
    i.smem_fixed = Smem::kFixed;
    i.smem_per_seq = Smem::kPerSeq;
    i.smem_per_cta = 8;
    i.smem_partials = Smem::kPartials;
    i.fn_mapped = nullptr;  // decode_kernel_info fills it in
    return i;
}
#endif

}  // namespace

#ifdef PKV_MAPPED
const void *PKV_MAPPED_FN(int block_size) {
    switch (block_size) {
#ifndef PKV_GRP
        case 8: return mapped_of<8>();
#endif
        case 16: return mapped_of<16>();
        case 32: return mapped_of<32>();
        case 64: return mapped_of<64>();
        case 128: return mapped_of<128>();
        default: return nullptr;
    }
}
#else

bool PKV_INFO_FN(int block_size, DecodeKernelInfo *info) {
    switch (block_size) {
#ifndef PKV_GRP
        case 8: *info = info_of<8>(); return true;
#endif
        case 16: *info = info_of<16>(); return true;
        case 32: *info = info_of<32>(); return true;
        case 64: *info = info_of<64>(); return true;
        case 128: *info = info_of<128>(); return true;
        default: return false;
    }
}
#endif

}  // namespace pkv
