// pkv_decode_impl.cuh -- the persistent paged decode-attention kernel.
//
// What it computes: [P1] "Paged Attention: OS-Inspired Memory Management for
// KV Caches" (modernaiengineering.com), "How PagedAttention works" step 4 --
// walk each sequence's block table, load every block's keys and values and
// compute attention exactly as if they were contiguous:
//     out[s][h] = softmax_t(scale * q[s][h] . K_t[h/G]) . V_t[h/G].
// [P2] "What is PagedAttention..." (n4n.ai), "How PagedAttention works" and
// "Common misconceptions": tokens are contiguous inside a block and the block
// table lookup is fused into the attention kernel (no separate gather pass).
//
// Design (GB300, HBM-bound: each K/V byte is read once):
//  * The batch's work is cut into chunks of 16 rows of one (sequence, KV head)
//    -- a "segment" -- (pkv_schedule.h; at block size 8 a chunk spans two
//    blocks) and split among the CTAs of a persistent grid, with CTA
//    boundaries moved to a segment boundary within one chunk per warp, then
//    into contiguous shares, one per WARP: equal, except that a warp whose
//    piece is cut across a CTA boundary (it also counts that piece in
//    device-wide, and may merge the CTAs' parts) gives up a few chunks to the
//    CTA's other warps.  A small batch uses fewer
//    CTAs (at least 4 chunks per warp; while segments are short, at most one
//    CTA per segment).  Every warp is an independent worker; there is no
//    CTA-wide synchronisation after the prologue.  A worker walks the cut
//    pieces at the two ends of its share first, so segments cut between
//    workers complete early, under the rest of the stream, not at the tail.
//  * Each warp owns a ring of ST stages in shared memory.  Lane 0 issues, ST
//    chunks ahead, one TMA tensor copy (cp.async.bulk.tensor.3d, 128-byte
//    swizzle) per cache of the chunk's K and V rows -- the cache is viewed as
//    [halves][rows][64 dims] so one box lands the whole 16-row chunk in the
//    swizzled [half][row][128 B] tile; a short last chunk (<= 8 rows) takes
//    one 8-row box per half, and at block size 8 every block one 8-row box
//    per half; boxes never leave a block -- plus, at
//    the first chunk of each piece, a bulk copy of the KV group's query rows,
//    all completing on the stage's mbarrier.
//    Block-table entries are prefetched one per lane a window of 32 chunks
//    ahead; when a window starts, each lane turns its entry into the chunk's
//    copy descriptor (rows, flags, cache rows), so issuing a chunk is a few
//    shuffles and the copies.
//  * Math on the tensor cores, one warp per chunk (mma.sync m16n8k16, fp32
//    accumulate):
//        S^T[16 x rows] = Q[16 x D] . K^T     query heads on M (G of 16 used),
//                                               rows on N, head_dim on K
//        O^T[D x 8]    += V^T[D x rows] . P^T  head_dim on M, heads on N (G of
//                                               8 used), rows on K; P as fp16
//                                               hi + lo parts
//    K and V^T fragments come from the swizzled tiles through ldmatrix
//    (.trans for V) without bank conflicts; the S accumulator layout is P^T's
//    B-operand layout, so P never leaves registers, and the transposed P.V
//    takes half the mma of P.V with heads on M.  Scores are in log2 units and the
//    softmax is online, per warp, in fp32.  Products of fp16 inputs are exact
//    in fp32, and splitting P into two fp16 terms keeps P.V at fp32 accuracy.
//  * A piece that covers a whole segment is normalised and written as fp16
//    by the warp.  A cut piece stores (max, sum, unnormalised output) and adds
//    its chunk count to a counter; merges go in two levels (count_piece,
//    merge_part): the pieces in one CTA's range meet in shared memory, and
//    the CTA's part, once complete, is merged -- right away by the completing
//    warp when shares are short, else through a per-CTA queue by a warp that
//    has finished its own share (so no warp ends late for having merged); a
//    segment that spans CTAs then counts the CTAs' parts in device-wide, and
//    the CTA completing it merges the parts.  Fixed order throughout (deterministic, no float atomics, no
//    second kernel).  The device-wide counters are tagged with an epoch kept
//    in the workspace (see count_in_tagged): each call prepares the next
//    call's counters and the last CTA out advances the epoch, so counting in
//    is one atomic, a fresh or half-used workspace is tolerated, and a launch
//    captured once and replayed works.
//  * With new K/V rows given (pkv_paged_attention_decode_append), the last
//    chunk of each segment also brings the row of the decode step's token:
//    the warp patches it into the tile before the math and stores it to the
//    cache.
//  * Rows past the context never reach the output: their scores are masked to
//    -inf, and in a ragged chunk the warp zeroes those V rows in shared memory
//    before P.V (whatever the cache holds there, 0 * it stays 0).
//  * HOSTIN instantiations (the mapped plan step, whose query, new_key and
//    new_value may be page-locked host memory) copy a piece's query and the
//    new rows with the lanes' 16-byte cp.async instead of bulk copies, each
//    stage barrier then counting lane 0's arrival and every lane's; the
//    other instantiations' code is unchanged.
//  * Every mbarrier wait gives up after wait_limit_ns, reports
//    PKV_ERR_DEVICE_TIMEOUT, waits (again bounded) for the warp's copies in
//    flight and returns.
#ifndef PKV_DECODE_IMPL_CUH
#define PKV_DECODE_IMPL_CUH

#include <math_constants.h>

#include "pkv_decode_params.h"
#include "pkv_device.cuh"
#include "pkv_schedule.h"

namespace pkv {

template <int D, int BS, int G>
struct DecodeGeometry {
    static constexpr int kRows = 16;                  // rows per chunk
    static constexpr int kBPC = BS < 16 ? 16 / BS : 1; // blocks per chunk (2 at block size 8)
    static constexpr int kNT = kRows / 8;             // 8-row groups per chunk (mma N tiles)
    static constexpr int kHalves = D / 64;            // 64-dim (128-byte) swizzle columns
    static constexpr int kHalfBytes = kRows * 128;    // one column of a tile
    static constexpr int kTileBytes = kHalves * kHalfBytes;  // K (or V) rows of a chunk
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kQBytes = G * D * 2;         // query rows of a KV group
    static constexpr int kRowBytes = D * 2;           // one K (or V) row
    static constexpr int kSlotBytes = kQBytes + 2 * kRowBytes;  // + the new token's K and V rows
    static constexpr int kKSteps = D / 16;            // mma K steps of Q.K^T
    static constexpr int kBoxBytes = 8 * 128;         // one TMA box: 8 rows x 64 fp16
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert((BS % kRows == 0 || BS == 8) && kRows % 8 == 0,
                  "a chunk is whole 8-row boxes, inside one block (or one box per block at block size 8)");
    static_assert(G >= 1 && G <= 8, "query heads per KV head");
    static_assert(kHalfBytes % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
};

// Dynamic shared memory (from a 1024-byte aligned base):
// [stages][query + new-row slots][barriers][chunk meta][cum (N+1)][ctx (N)][bounds (C+1)]
// [partial slots (optional): NW workers x 2 (first / last piece) x G x (2 + D) fp32].
// (grouped kernel: [ctx (N)][shared (N)][cum over items] padded to 8 bytes,
// then [items int2][bounds (C+1)]; items are at most N, the arrays have room
// for 2N -- 32 bytes per sequence)
template <int NW, int ST, int D, int BS, int G, bool GRP = false>
struct DecodeSmem {
    using Geo = DecodeGeometry<D, BS, G>;
    static constexpr size_t kQ = (size_t)NW * ST * Geo::kStageBytes;
    static constexpr size_t kBars = kQ + (size_t)NW * ST * Geo::kSlotBytes;
    static constexpr size_t kMeta = kBars + (size_t)NW * ST * 8;
    static constexpr size_t kCum = kMeta + (size_t)NW * ST * 32;  // two int4 per stage
    static constexpr size_t kAlign = 1024;              // slack for aligning the base
    static constexpr size_t kFixed = kCum + kAlign;
    static constexpr size_t kPerSeq = GRP ? 32 : 8;
    static constexpr size_t kSlotFloats = (size_t)G * (2 + D);  // (m, l) per head, then the outputs
    static constexpr size_t kPartials = (size_t)NW * 2 * kSlotFloats * 4 + 16;  // + alignment slack
};

// Zeroes V rows [R, kRows) of a ragged chunk's tile (every byte of those rows,
// so the swizzle does not matter).
template <int D, int BS, int G>
__device__ __forceinline__ void zero_tail_rows(unsigned char *vt, int R, int lane) {
    using Geo = DecodeGeometry<D, BS, G>;
    constexpr int kVecs = 8 * Geo::kHalves;  // 16-byte vectors per row
    const int n = (Geo::kRows - R) * kVecs;
    for (int i = lane; i < n; i += 32) {
        const int r = R + i / kVecs;
        const int v = i % kVecs;
        *reinterpret_cast<uint4 *>(vt + (v >> 3) * Geo::kHalfBytes + r * 128 + (v & 7) * 16) =
            make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
}

// One chunk of R valid rows: tiles at kt / vt (shared-memory addresses).
// Lane (g, t) = (lane / 4, lane % 4) owns query head g (valid if g < G) and
// rows 2t, 2t+1 (+8) of the scores; the output is kept transposed, O^T
// [dims x heads]: o[i] holds dims 16i + g and 16i + g + 8 of heads 2t and
// 2t + 1 (o[i][0] / o[i][2] head 2t, o[i][1] / o[i][3] head 2t + 1).
// MASK (the grouped kernel): when live >= 0 only query row `live` sees this
// chunk -- the other rows' scores are masked, and a row that has seen no key
// of its piece yet keeps its empty state (max -inf, sum 0, output 0).
template <int D, int BS, int G, bool MASK = false>
__device__ __forceinline__ void consume_chunk(uint32_t kt, uint32_t vt, int R, const uint32_t (&qa)[D / 16][2],
                                              float scale_log2, float &m, float &l, float (&o)[D / 16][4],
                                              int lane, int live = -1) {
    using Geo = DecodeGeometry<D, BS, G>;
    const int t = lane & 3;
    const int mi = lane >> 3;   // which 8x8 matrix this lane addresses in ldmatrix
    const int rr = lane & 7;    // which row of it

    // ---- S^T = Q . K^T ------------------------------------------------------
    // (even and odd K steps accumulate separately: two dependent mma chains of
    // half the length, summed at the end -- when K/V come from L2 the warp's
    // latency per chunk is what bounds it)
    float s[Geo::kNT][4], s2[Geo::kNT][4];
#pragma unroll
    for (int nt = 0; nt < Geo::kNT; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
        s2[nt][0] = s2[nt][1] = s2[nt][2] = s2[nt][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < Geo::kKSteps; ++kk) {
        float(*acc)[4] = (kk & 1) ? s2 : s;
        // matrices: (n-tile mi>>1, dims 16kk + 8(mi&1)); the row's 16-byte chunk
        // c sits at c ^ (row & 7) in the swizzled tile
        const int nt = (Geo::kNT == 2) ? (mi >> 1) : 0;
        const int row = 8 * nt + rr;
        const int c = (2 * kk + (mi & 1)) & 7;
        const uint32_t addr = kt + (kk >> 2) * Geo::kHalfBytes + row * 128 + ((c ^ rr) << 4);
        if (Geo::kNT == 2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(addr, b0, b1, b2, b3);
            mma_16816(acc[0], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
            mma_16816(acc[Geo::kNT - 1], qa[kk][0], 0u, qa[kk][1], 0u, b2, b3);
        } else {
            uint32_t b0, b1;
            ldsm_x2(addr, b0, b1);
            mma_16816(acc[0], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
        }
    }
#pragma unroll
    for (int nt = 0; nt < Geo::kNT; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[nt][j] += s2[nt][j];

    // ---- online softmax (per query head; rows past R masked) ----------------
    float x[Geo::kNT][2];
    float mx = -CUDART_INF_F;
    const bool row_live = !MASK || live < 0 || (lane >> 2) == live;  // this lane's query row
#pragma unroll
    for (int nt = 0; nt < Geo::kNT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int row = 8 * nt + 2 * t + j;
            x[nt][j] = row < R && row_live ? s[nt][j] * scale_log2 : -CUDART_INF_F;
            mx = fmaxf(mx, x[nt][j]);
        }
    mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 2));
    const float mn = fmaxf(m, mx);          // row 0 is valid: finite (MASK: a masked row may stay -inf)
    // the exponents' reference: mn, or 0 while the row is still empty (MASK)
    const float mref = MASK ? (mn == -CUDART_INF_F ? 0.f : mn) : mn;
    const float corr = exp2f(m - mref);     // m = -inf at a piece's start -> 0
    m = mn;
    l *= corr;
    // the output columns are heads 2t and 2t + 1: their factors come from
    // the lanes that own those heads' rows
    const float corr_e = __shfl_sync(kFullMask, corr, 8 * t);
    const float corr_o = __shfl_sync(kFullMask, corr, 8 * t + 4);
    // Inside a piece the running max seldom moves after its first chunks:
    // when no head's factor differs from 1 the rescale (an exact no-op) is
    // skipped, and P.V follows the softmax at once.
    if (__any_sync(kFullMask, corr_e != 1.f || corr_o != 1.f)) {
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
            o[i][0] *= corr_e;
            o[i][1] *= corr_o;
            o[i][2] *= corr_e;
            o[i][3] *= corr_o;
        }
    }
    float pr[Geo::kNT][2];
#pragma unroll
    for (int nt = 0; nt < Geo::kNT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            pr[nt][j] = exp2f(x[nt][j] - mref);  // masked rows: exp2(-inf) = 0
            l += pr[nt][j];
        }
    // P as A fragments: hi = fp16(p), lo = fp16(p - hi)
    const uint32_t h0 = pack_half2(pr[0][0], pr[0][1]);
    const float2 f0 = unpack_half2(h0);
    const uint32_t lo0 = pack_half2(pr[0][0] - f0.x, pr[0][1] - f0.y);
    uint32_t h2 = 0u, lo2 = 0u;
    if (Geo::kNT == 2) {
        h2 = pack_half2(pr[Geo::kNT - 1][0], pr[Geo::kNT - 1][1]);
        const float2 f2 = unpack_half2(h2);
        lo2 = pack_half2(pr[Geo::kNT - 1][0] - f2.x, pr[Geo::kNT - 1][1] - f2.y);
    }

    // ---- O^T += V^T . P^T -----------------------------------------------------
    // M = 16 dims per tile, N = 8 heads, K = the chunk's 16 rows.  P's score
    // layout (head g, rows 2t, 2t+1 and 2t+8, 2t+9) is exactly the B operand
    // of P^T, and V^T comes from the V tile through ldmatrix.trans: matrices
    // (rows 8(mi>>1).., dims 16i + 8(mi&1)).
    static_assert(Geo::kNT == 2, "16-row chunks");
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
        const int row = rr + 8 * (mi >> 1);
        const int c = (2 * i + (mi & 1)) & 7;
        const uint32_t addr = vt + (i >> 2) * Geo::kHalfBytes + row * 128 + ((c ^ rr) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(addr, a0, a1, a2, a3);
        mma_16816(o[i], a0, a1, a2, a3, h0, h2);
        mma_16816(o[i], a0, a1, a2, a3, lo0, lo2);
    }
}

// ---- the CUDA-core form of one chunk, group 1 only (built with
// PKV_DECODE_G1_CUDACORE=1; the tensor-core form above is the default) ----
// Lane (h, r) = (lane >> 4, lane & 15) owns row r of the chunk and the dims
// [h * D/2, (h + 1) * D/2) of the one query head: q . K_r over its dims is
// D/2 fp32 FMAs, one shuffle adds the two halves, the online softmax takes
// 8 more, and o keeps that lane's row's share of P.V for its dims (summed
// over the 16 rows only when the piece ends, in finish_piece_cc).
template <int D>
struct CudaCoreLayout {
    static constexpr int kDH = D / 2;     // dims per lane
    static constexpr int kNV = kDH / 8;   // 16-byte vectors per lane and row
    // byte offset, in a swizzled [half][row][64 dims] tile, of vector v of
    // the lane's row and dims
    __device__ __forceinline__ static int off(int lane, int v) {
        const int r = lane & 15, h = lane >> 4;
        if (D == 128) return h * DecodeGeometry<128, 16, 1>::kHalfBytes + r * 128 + ((v ^ (r & 7)) << 4);
        return r * 128 + (((h * 4 + v) ^ (r & 7)) << 4);
    }
};

template <int D>
__device__ __forceinline__ void consume_chunk_cc(const unsigned char *kt, const unsigned char *vt, int R,
                                                 const float (&q)[D / 2], float scale_log2, float &m, float &l,
                                                 float (&o)[D / 2], int lane) {
    using L = CudaCoreLayout<D>;
    const int r = lane & 15;
    float s0 = 0.f, s1 = 0.f;  // two chains
#pragma unroll
    for (int v = 0; v < L::kNV; ++v) {
        float f[8];
        unpack8(*reinterpret_cast<const uint4 *>(kt + L::off(lane, v)), f);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            s0 = fmaf(q[8 * v + e], f[e], s0);
            s1 = fmaf(q[8 * v + e + 1], f[e + 1], s1);
        }
    }
    float sc = s0 + s1;
    sc += __shfl_xor_sync(kFullMask, sc, 16);
    const float x = r < R ? sc * scale_log2 : -CUDART_INF_F;  // rows past R: masked (their K may be anything)
    float mx = x;
#pragma unroll
    for (int k = 1; k < 16; k <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, k));
    const float mn = fmaxf(m, mx);  // row 0 is valid: finite
    const float corr = exp2f(m - mn);
    m = mn;
    const float pr = exp2f(x - mn);
    float ps = pr;
#pragma unroll
    for (int k = 1; k < 16; k <<= 1) ps += __shfl_xor_sync(kFullMask, ps, k);
    l = l * corr + ps;
    if (corr != 1.f) {  // the same on every lane
#pragma unroll
        for (int j = 0; j < D / 2; ++j) o[j] *= corr;
    }
#pragma unroll
    for (int v = 0; v < L::kNV; ++v) {
        float f[8];
        unpack8(*reinterpret_cast<const uint4 *>(vt + L::off(lane, v)), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[8 * v + e] = fmaf(pr, f[e], o[8 * v + e]);
    }
}

// The query dims of lane (h, r) as fp32, from the group's query row in the
// stage's slot (plain [D] fp16).
template <int D>
__device__ __forceinline__ void load_query_cc(const unsigned char *sq, float (&q)[D / 2], int lane) {
    const int h = lane >> 4;
#pragma unroll
    for (int v = 0; v < D / 16; ++v) {
        float f[8];
        unpack8(*reinterpret_cast<const uint4 *>(sq + (h * (D / 2) + 8 * v) * 2), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) q[8 * v + e] = f[e];
    }
}

// Sums o over the 16 lanes that share h (rows 0..15): afterwards lane L holds
// the piece's output dims [L * D/32, (L + 1) * D/32) (halving exchanges: at
// each step a lane keeps the half of its values that its bit selects and
// adds its partner's copy of that half).
template <int D>
__device__ __forceinline__ void reduce_rows_cc(float (&o)[D / 2], int lane) {
    constexpr int N0 = D / 2;
#pragma unroll
    for (int step = 0; step < 4; ++step) {
        const int bit = 8 >> step;           // lane mask of this step
        const int n = N0 >> (step + 1);      // values kept after it
        const bool upper = (lane & bit) != 0;
#pragma unroll
        for (int j = 0; j < n; ++j) {
            const float keep = upper ? o[n + j] : o[j];
            const float send = upper ? o[j] : o[n + j];
            o[j] = keep + __shfl_xor_sync(kFullMask, send, bit);
        }
    }
}

// Completion counters hold (epoch << 32 | count).  Every call prepares the
// counters of the NEXT call (the other parity) as (epoch + 1, 0), so counting
// in is normally a single atomic add.  A counter in any other state (a fresh
// workspace, or one left by a call that gave up) is swung to (epoch, amount)
// by the first arrival that sees it.  Adds `amount` (> 0) towards `total` and
// returns the count after this arrival: the arrival that returns `total` is
// the last.
__device__ __forceinline__ int count_in_tagged(unsigned long long *cnt, uint32_t epoch, int total, int amount) {
    const unsigned long long tag = (unsigned long long)epoch << 32;
    const unsigned long long kLow = 0xffffffffull;
    const unsigned long long add = (unsigned long long)amount;
    auto valid = [&](unsigned long long v) { return (v & ~kLow) == tag && (v & kLow) < (unsigned long long)total; };
    unsigned long long old = atomicAdd(cnt, add);
    if (valid(old)) return (int)(old & kLow) + amount;
    unsigned long long cur = old + add;
#pragma unroll 1
    while (true) {
        if (valid(cur)) {
            old = atomicAdd(cnt, add);
            if (valid(old)) return (int)(old & kLow) + amount;
            cur = old + add;
            continue;
        }
        const unsigned long long prev = atomicCAS(cnt, cur, tag | add);
        if (prev == cur) return amount;
        cur = prev;
    }
}

// Where a worker warp is: what finish_piece needs besides the piece itself.
// NW (workers per CTA) is a compile-time constant, so the share arithmetic
// divides by a constant.
template <int NW>
struct WorkerCtx {
    static constexpr int nw = NW;
    const int *cum;          // chunk prefix sums (shared memory)
    const int64_t *bounds;   // CTA ranges, [C + 1] (shared memory)
    int C;                   // CTAs in the grid
    int64_t wid;             // this worker
    int64_t gb, ge;          // its share
    uint32_t epoch;          // this call's epoch
    unsigned long long *count;  // this call's per-segment counters (global)
    int *cta_count;          // per-worker-slot counters of this CTA (shared)
    int *cta_cross;          // counter of the segment that reaches in from before this CTA (shared)
    float *part;             // partial slots of this CTA's workers (shared), or NULL
    const int64_t *starts;   // this CTA's NW + 1 worker starts (shared; the last is its range's end)
    // grouped kernel only (else NULL): the items (groups and lone sequences)
    const int2 *info;

    // first chunk of worker w, one of this CTA's workers or the next CTA's first
    __device__ __forceinline__ int64_t start(int64_t w) const {
        return starts[w - (int64_t)blockIdx.x * NW];
    }
    // this CTA's worker whose share holds chunk g (inside the CTA's range)
    __device__ __forceinline__ int64_t worker_of(int64_t g) const {
        return (int64_t)blockIdx.x * NW + worker_in_starts<NW>(starts, g);
    }
};

// Where segment (s, kvh) lies, and whether it lies inside this CTA's range
// (then all its pieces are this CTA's, and they meet in shared memory).
struct SegInfo {
    int64_t g0;          // first chunk of the segment
    int nch;             // its chunks
    bool local;          // inside this CTA's range
    int64_t p_lo, p_hi;  // the part of it in this CTA's range
    int mine;            // chunks of it in this worker's share
    int xw;              // 1 if it reaches in from before this CTA's range, else 0
};

template <int NW>
__device__ __forceinline__ SegInfo segment_info(const DecodeParams &p, const WorkerCtx<NW> &wc, int s, int kvh) {
    SegInfo si;
    si.nch = (wc.cum[s + 1] - wc.cum[s]) / p.num_kv_heads;
    si.g0 = wc.cum[s] + (int64_t)kvh * si.nch;
    const int64_t g1 = si.g0 + si.nch;
    const int64_t c_lo = wc.bounds[blockIdx.x], c_hi = wc.bounds[blockIdx.x + 1];
    si.local = si.g0 >= c_lo && g1 <= c_hi;
    si.p_lo = si.g0 > c_lo ? si.g0 : c_lo;
    si.p_hi = g1 < c_hi ? g1 : c_hi;
    si.mine = (int)((g1 < wc.ge ? g1 : wc.ge) - (si.g0 > wc.gb ? si.g0 : wc.gb));
    si.xw = si.g0 < c_lo ? 1 : 0;
    return si;
}

// A piece's partial: (max, sum) of head g at ml[2g], ml[2g + 1] and its
// unnormalised outputs at acc[g * D ...]; in shared memory or in the workspace.
struct PieceRef {
    float *ml;
    float *acc;
    bool smem;
    bool exists;
};

// Worker w's piece (which: 0 = the first piece of its share, 1 = the last):
// in this CTA's shared slots when they are enabled (w is then one of this
// CTA's workers), else in the workspace's worker slots.
template <int D, int G, int NW>
__device__ __forceinline__ PieceRef worker_piece(const DecodeParams &p, const WorkerCtx<NW> &wc, int64_t w,
                                                 int which) {
    if (wc.part != nullptr) {
        float *base = wc.part + ((w % NW) * 2 + which) * (G * (2 + D));
        return {base, base + 2 * G, true, true};
    }
    const int64_t b = (w * 2 + which) * G;
    return {p.ws_ml + b * 2, p.ws_acc + b * D, false, true};
}

// CTA c's part of a segment that spans CTAs (which: 1 if the segment started
// before the CTA's range, else 0 -- a CTA meets at most one of each).
template <int D, int G>
__device__ __forceinline__ PieceRef cta_piece(const DecodeParams &p, int64_t c, int which) {
    const int64_t b = (c * 2 + which) * G;
    return {p.ws_cml + b * 2, p.ws_cacc + b * D, false, true};
}

// A merge in progress, combining (max, sum, output) online:
//     M' = max(M, m_p),  X' = X 2^(M - M') + x_p 2^(m_p - M')  for X = L, O.
// Lane j holds output dims j*PER .. j*PER + PER - 1 of every head; M and L
// are the same on all lanes.
// SAFE (the grouped kernel): a row may be empty (max -inf) in both the state
// and the piece; the exponents are then taken against 0 and nothing changes.
template <int D, int G, bool SAFE = false>
struct MergeState {
    static constexpr int PER = D / 32;
    float M[G], L[G], O[G][PER];

    __device__ __forceinline__ void init() {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            M[g] = -CUDART_INF_F;
            L[g] = 0.f;
#pragma unroll
            for (int k = 0; k < PER; ++k) O[g][k] = 0.f;
        }
    }

    // Folds in one piece; its (m, l) and output slice are loaded together.
    __device__ __forceinline__ void add(const PieceRef &r, int lane) {
        float2 ml[G];
        float a[G][PER];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float2 *mp = reinterpret_cast<const float2 *>(r.ml) + g;
            ml[g] = r.smem ? *mp : __ldcg(mp);
            const float *src = r.acc + g * D + lane * PER;
#pragma unroll
            for (int k = 0; k < PER; ++k) a[g][k] = r.smem ? src[k] : __ldcg(src + k);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float mn = fmaxf(M[g], ml[g].x);
            const float mref = SAFE ? (mn == -CUDART_INF_F ? 0.f : mn) : mn;
            const float f_old = exp2f(M[g] - mref);
            const float f_new = exp2f(ml[g].x - mref);
            L[g] = L[g] * f_old + ml[g].y * f_new;
#pragma unroll
            for (int k = 0; k < PER; ++k) O[g][k] = O[g][k] * f_old + a[g][k] * f_new;
            M[g] = mn;
        }
    }

    // Normalised fp16 output rows of the KV group (s, kvh).
    __device__ __forceinline__ void write_out(const DecodeParams &p, int s, int kvh, int lane) const {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            __half *dst = p.out + ((int64_t)s * p.num_heads + kvh * G + g) * D + lane * PER;
            const float inv = 1.f / L[g];
#pragma unroll
            for (int k = 0; k < PER; ++k) dst[k] = __float2half_rn(O[g][k] * inv);
        }
    }

    // Stored as a partial, for the next level of the merge.
    __device__ __forceinline__ void store(const PieceRef &r, int lane) const {
        if (lane == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g) reinterpret_cast<float2 *>(r.ml)[g] = make_float2(M[g], L[g]);
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int k = 0; k < PER; ++k) r.acc[g * D + lane * PER + k] = O[g][k];
    }
};

// Folds pieces 0 .. cnt-1 (ref(i) -> PieceRef) into st, in order, one round
// trip per piece: for a few pieces, or for pieces in shared memory.
template <int D, int G, bool SAFE, class Ref>
__device__ __forceinline__ void merge_seq(MergeState<D, G, SAFE> &st, int cnt, Ref ref, int lane) {
#pragma unroll 1
    for (int i = 0; i < cnt; ++i) {
        const PieceRef r = ref(i);
        if (r.exists) st.add(r, lane);
    }
}

// The same for many pieces, in the same order: up
// to 32 pieces at a time, lane j fetches piece j's (m, l) -- one round trip
// for all of them -- the warp reduces M and L with shuffles, then sums the
// output slices in piece order with the loads of several pieces in flight.
template <int D, int G, bool SAFE, class Ref>
__device__ __forceinline__ void merge_wide(MergeState<D, G, SAFE> &st, int cnt, Ref ref, int lane) {
    constexpr int PER = D / 32;
    constexpr int U = G >= 8 ? 1 : (G >= 4 ? 2 : 4 / G);  // pieces whose slices are loaded together
#pragma unroll 1
    for (int i0 = 0; i0 < cnt; i0 += 32) {
        const int n = cnt - i0 < 32 ? cnt - i0 : 32;
        PieceRef mine{nullptr, nullptr, false, false};
        if (lane < n) mine = ref(i0 + lane);
        float wgt[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float2 ml = make_float2(-CUDART_INF_F, 0.f);
            if (mine.exists) {
                const float2 *mp = reinterpret_cast<const float2 *>(mine.ml) + g;
                ml = mine.smem ? *mp : __ldcg(mp);
            }
            float mx = ml.x;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, o));
            const float mn = fmaxf(st.M[g], mx);  // some piece exists: finite (SAFE: maybe -inf)
            const float mref = SAFE ? (mn == -CUDART_INF_F ? 0.f : mn) : mn;
            const float f_old = exp2f(st.M[g] - mref);
            wgt[g] = mine.exists ? exp2f(ml.x - mref) : 0.f;
            float ls = ml.y * wgt[g];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(kFullMask, ls, o);
            st.L[g] = st.L[g] * f_old + ls;
            st.M[g] = mn;
#pragma unroll
            for (int k = 0; k < PER; ++k) st.O[g][k] *= f_old;
        }
#pragma unroll 1
        for (int j0 = 0; j0 < n; j0 += U) {
            float a[U][G][PER], f[U][G];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = j0 + u < n ? j0 + u : n - 1;
                const PieceRef r = ref(i0 + j);
                const bool use = j0 + u < n && r.exists;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    f[u][g] = __shfl_sync(kFullMask, wgt[g], j);
                    const float *src = r.acc + g * D + lane * PER;
#pragma unroll
                    for (int k = 0; k < PER; ++k) a[u][g][k] = use ? (r.smem ? src[k] : __ldcg(src + k)) : 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int k = 0; k < PER; ++k) st.O[g][k] += a[u][g][k] * f[u][g];
        }
    }
}

// ---- the grouped (prefix-sharing) kernel ----------------------------------
// The caller tells, per sequence, how many leading blocks its table shares
// with the previous sequence's.  Up to 8 consecutive sequences that share
// blocks form a GROUP, and a group is one segment owner (an item) instead of
// its sequences: for each KV head its chunks are the group's shared full
// blocks, read once with every member's query as a row of the tile, then each
// member's own chunks in member order, during which only that member's row
// is live (the others' scores are masked, their softmax state untouched).
// Row g of the segment is then exactly member g's decode over its whole
// context, and it completes, splits across workers and merges like a head of
// a group-8 segment.  A sequence outside every group is an item of its own.
constexpr int kOwn = 32;         // chunk flag: a member's own chunk (one live row)
constexpr int kMemberShift = 6;  // ... and which member, in the next 3 flag bits

struct ItemInfo {
    int s0;  // first (or only) sequence
    int ns;  // sequences (members)
    int sc;  // shared chunks at the start of every KV head's segment
};
__device__ __forceinline__ ItemInfo item_info(const int2 *info, int it) {
    const int2 v = info[it];
    return {v.x & 0xffff, v.x >> 16, v.y};
}

// Output rows g < ns of item `it`'s segment for KV head kvh, from a merge
// (lane j holds dims j*D/32 ... of every row): row g is member g's output.
template <int D, int G, bool SAFE>
__device__ __forceinline__ void write_rows_grp(const DecodeParams &p, const ItemInfo &ii, int kvh,
                                               const MergeState<D, G, SAFE> &ms, int lane) {
    constexpr int PER = D / 32;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        if (g < ii.ns) {
            __half *dst = p.out + ((int64_t)(ii.s0 + g) * p.num_heads + kvh) * D + lane * PER;
            const float inv = 1.f / ms.L[g];
#pragma unroll
            for (int k = 0; k < PER; ++k) dst[k] = __float2half_rn(ms.O[g][k] * inv);
        }
    }
}

// Finish a piece: sum l over the 4 lanes of each head, then write the output
// row (whole segment) or store the partial (cut segment).  Returns true for a
// stored partial; the caller counts it in (count_piece).  The output is held
// transposed (see consume_chunk): each lane pairs its values with lane ^ 4's
// so that it stores two neighbouring dims of one head, hh = 2t + (g & 1).
template <int D, int G, int NW, bool GRP = false>
__device__ __forceinline__ bool finish_piece(const DecodeParams &p, const WorkerCtx<NW> &wc, const int4 md, float m,
                                             float l, const float (&o)[D / 16][4], SegInfo &si, int lane) {
    const int g = lane >> 2;
    const int t = lane & 3;
    l += __shfl_xor_sync(kFullMask, l, 1);
    l += __shfl_xor_sync(kFullMask, l, 2);
    const int s = md.x, kvh = md.y, flags = md.w;
    const int hh = 2 * t + (g & 1);  // the head this lane stores
    const int d0 = g & ~1;           // its first dim in each 8-dim group
    // (even g: its own head-2t value and lane ^ 4's; odd g: lane ^ 4's
    // head-(2t+1) value and its own)
    auto pair = [&](float own_e, float own_o) -> float2 {
        const float y = __shfl_xor_sync(kFullMask, (g & 1) ? own_e : own_o, 4);
        return (g & 1) ? make_float2(y, own_o) : make_float2(own_e, y);
    };
    if constexpr (GRP) {
        if (flags & kWhole) {
            // a whole segment of a group (or of a lone sequence): row hh is
            // member hh's output row
            const ItemInfo ii = item_info(wc.info, s);
            const float inv = 1.f / __shfl_sync(kFullMask, l, 4 * hh);  // l of row hh
            __half *dst = p.out + ((int64_t)(ii.s0 + (hh < ii.ns ? hh : 0)) * p.num_heads + kvh) * D + d0;
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
                const float2 a = pair(o[i][0], o[i][1]);
                const float2 b = pair(o[i][2], o[i][3]);
                if (hh < ii.ns) {
                    *reinterpret_cast<uint32_t *>(dst + 16 * i) = pack_half2(a.x * inv, a.y * inv);
                    *reinterpret_cast<uint32_t *>(dst + 16 * i + 8) = pack_half2(b.x * inv, b.y * inv);
                }
            }
            return false;
        }
    }
    if (!GRP && (flags & kWhole)) {
        const float inv = 1.f / __shfl_sync(kFullMask, l, 4 * hh);  // l of head hh
        __half *dst = p.out + ((int64_t)s * p.num_heads + kvh * G + hh) * D + d0;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
            const float2 a = pair(o[i][0], o[i][1]);
            const float2 b = pair(o[i][2], o[i][3]);
            if (hh < G) {
                *reinterpret_cast<uint32_t *>(dst + 16 * i) = pack_half2(a.x * inv, a.y * inv);
                *reinterpret_cast<uint32_t *>(dst + 16 * i + 8) = pack_half2(b.x * inv, b.y * inv);
            }
        }
        return false;
    }
    si = segment_info(p, wc, s, kvh);
    const PieceRef at = worker_piece<D, G, NW>(p, wc, wc.wid, (flags & kSlot1) ? 1 : 0);
    float *dst = at.acc + hh * D + d0;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
        const float2 a = pair(o[i][0], o[i][1]);
        const float2 b = pair(o[i][2], o[i][3]);
        if (hh < G) {
            *reinterpret_cast<float2 *>(dst + 16 * i) = a;
            *reinterpret_cast<float2 *>(dst + 16 * i + 8) = b;
        }
    }
    if (t == 0 && g < G) reinterpret_cast<float2 *>(at.ml)[g] = make_float2(m, l);
    return true;
}

// finish_piece for the CUDA-core form (group 1): the rows are summed first
// (reduce_rows_cc), then lane L writes its D/32 dims of the output row or of
// the partial; l and m are the same on every lane.
template <int D, int NW>
__device__ __forceinline__ bool finish_piece_cc(const DecodeParams &p, const WorkerCtx<NW> &wc, const int4 md,
                                                float m, float l, float (&o)[D / 2], SegInfo &si, int lane) {
    constexpr int PER = D / 32;
    reduce_rows_cc<D>(o, lane);
    const int s = md.x, kvh = md.y, flags = md.w;
    if (flags & kWhole) {
        const float inv = 1.f / l;
        __half *dst = p.out + ((int64_t)s * p.num_heads + kvh) * D + lane * PER;
        if (PER == 4) {
            uint2 w;
            w.x = pack_half2(o[0] * inv, o[1] * inv);
            w.y = pack_half2(o[2] * inv, o[3] * inv);
            *reinterpret_cast<uint2 *>(dst) = w;
        } else {
            *reinterpret_cast<uint32_t *>(dst) = pack_half2(o[0] * inv, o[1] * inv);
        }
        return false;
    }
    si = segment_info(p, wc, s, kvh);
    const PieceRef at = worker_piece<D, 1, NW>(p, wc, wc.wid, (flags & kSlot1) ? 1 : 0);
#pragma unroll
    for (int k = 0; k < PER; ++k) at.acc[lane * PER + k] = o[k];
    if (lane == 0) reinterpret_cast<float2 *>(at.ml)[0] = make_float2(m, l);
    return true;
}

// Counts a stored partial of segment (s, kvh) in, in two levels.
//  1. The pieces in this CTA's range (the whole segment, if it stays in the
//     CTA) count their chunks in on a shared-memory counter (count_piece);
//     the piece that completes the CTA's part queues the segment for merging
//     in the CTA's merge queue (it does not merge: see merge_part).
//  2. merge_part, run by a warp of the CTA that has finished its own share,
//     merges the CTA's part from shared memory.  A segment that spans CTAs:
//     the part goes to the CTA's slot in the workspace and its chunks count
//     in on the segment's device-wide counter; the CTA completing the segment
//     merges the parts, in CTA order.
// A segment cut into many pieces thus merges at most a CTA's pieces from
// shared memory plus one part per CTA from L2, and the merges fall to warps
// with nothing else to do instead of delaying a warp's own chunks.
// Returns true when this warp completed the CTA's part of the segment.
template <int D, int G, int NW>
__device__ __forceinline__ bool count_piece(const WorkerCtx<NW> &wc, const SegInfo &si, int lane) {
    const int part = (int)(si.p_hi - si.p_lo);
    const int mine = si.mine;
    if (part != mine) {
        fence_acq_rel_cta();  // the partial is visible to this CTA before it is counted
        __syncwarp();
        int done = 0;
        if (lane == 0) {
            // a worker starts at most one cut segment inside its CTA, and a CTA
            // meets at most one segment from before its range
            int *ctr = si.xw ? wc.cta_cross : wc.cta_count + (wc.worker_of(si.p_lo) % NW);
            done = atomicAdd(ctr, mine) + mine;
        }
        done = __shfl_sync(kFullMask, done, 0);
        if (done != part) return false;
        fence_acq_rel_cta();
    }
    return true;
}

// Merges this CTA's part of cut segment (s, kvh) (see count_piece); si is
// its segment_info (only the CTA-level fields are used).
template <int D, int G, int NW, bool GRP = false>
__device__ __forceinline__ void merge_part(const DecodeParams &p, const WorkerCtx<NW> &wc, int s, int kvh,
                                           const SegInfo &si, int lane) {
    const int64_t g1 = si.g0 + si.nch;
    const int part = (int)(si.p_hi - si.p_lo);
    const int64_t wa = wc.worker_of(si.p_lo);
    const int64_t wb = wc.worker_of(si.p_hi - 1);
    auto wref = [&](int i) -> PieceRef {
        const int64_t w = wa + i;
        const int64_t st = wc.start(w);
        PieceRef r = worker_piece<D, G, NW>(p, wc, w, partial_slot(st, si.g0));
        r.exists = st < wc.start(w + 1);
        return r;
    };
    MergeState<D, G, GRP> ms;
    ms.init();
    const int cnt = (int)(wb - wa + 1);
    if (cnt <= 4 || wc.part != nullptr)
        merge_seq(ms, cnt, wref, lane);
    else
        merge_wide(ms, cnt, wref, lane);
    if (si.local) {
        if constexpr (GRP)
            write_rows_grp(p, item_info(wc.info, s), kvh, ms, lane);
        else
            ms.write_out(p, s, kvh, lane);
        return;
    }
    ms.store(cta_piece<D, G>(p, blockIdx.x, si.xw), lane);
    fence_acq_rel_gpu();  // the part is visible device-wide before it is counted
    __syncwarp();
    int done = 0;
    if (lane == 0) done = count_in_tagged(wc.count + (int64_t)s * p.num_kv_heads + kvh, wc.epoch, si.nch, part);
    done = __shfl_sync(kFullMask, done, 0);
    if (done != si.nch) return;
    fence_acq_rel_gpu();
    const int ca = cta_of(wc.bounds, wc.C, si.g0, blockIdx.x);
    const int cb = cta_of(wc.bounds, wc.C, g1 - 1, blockIdx.x);
    auto cref = [&](int i) -> PieceRef {
        const int64_t c = ca + i;
        PieceRef r = cta_piece<D, G>(p, c, si.g0 < wc.bounds[c] ? 1 : 0);
        r.exists = wc.bounds[c] < wc.bounds[c + 1];
        return r;
    };
    MergeState<D, G, GRP> ms2;
    ms2.init();
    if (cb - ca < 4)
        merge_seq(ms2, cb - ca + 1, cref, lane);
    else
        merge_wide(ms2, cb - ca + 1, cref, lane);
    if constexpr (GRP)
        write_rows_grp(p, item_info(wc.info, s), kvh, ms2, lane);
    else
        ms2.write_out(p, s, kvh, lane);
}

// Inputs in page-locked host memory (a mapped plan step): the lanes copy a
// piece's query rows (first chunk) and the new token's K and V rows into the
// stage's slot 16 bytes each, so that the link's latency is paid once per
// chunk under the copies already in flight, then every lane arrives on the
// stage barrier when its copies have landed.  Only the HOSTIN instantiations
// of the kernel (a mapped plan step) contain it.
template <int D, int G, bool GRP>
__device__ __forceinline__ void copy_host_inputs(const DecodeParams &p, uint32_t slot, uint32_t bar, bool first,
                                              bool new_row, int s, int nq, int snew, int kvh, int lane) {
    using Geo = DecodeGeometry<D, 16, G>;
    constexpr int kVec = D / 8;  // 16-byte vectors per row
    if (first) {
        for (int v = lane; v < nq * kVec; v += 32) {
            const int r = v / kVec, c = v - r * kVec;
            const int64_t row = GRP ? (int64_t)(s + r) * p.num_heads + kvh : (int64_t)s * p.num_heads + kvh * G + r;
            cp_async_16(slot + (r * D + c * 8) * 2, p.query + row * D + c * 8);
        }
    }
    if (new_row) {
        const int64_t src = ((int64_t)snew * p.num_kv_heads + kvh) * D;
        for (int v = lane; v < 2 * kVec; v += 32) {
            const bool is_v = v >= kVec;
            const int c = is_v ? v - kVec : v;
            cp_async_16(slot + Geo::kQBytes + (is_v ? Geo::kRowBytes : 0) + c * 16,
                        (is_v ? p.new_value : p.new_key) + src + c * 8);
        }
    }
    cp_async_mbar_arrive_noinc(bar);
}

// The CTA's merge queue (shared memory): segments whose CTA part is complete
// and waits for merge_part.  At most NW + 1 parts complete in a CTA (a cut
// segment holds a warp or CTA boundary of the range), so kMergeQueue entries
// never run out; a push that would still overflow merges at once.
constexpr int kMergeQueue = 32;
struct MergeQueue {
    int entry[kMergeQueue];  // sequence | KV head << 16, -1 until written
    int tail;                // entries claimed by producers
    int head;                // entries taken by consumers
};

template <int D, int BS, int G, int NW, int ST, bool GRP = false, bool HOSTIN = false>
__global__ void __launch_bounds__(NW * 32, 1) paged_decode_kernel(const __grid_constant__ DecodeParams p) {
#ifdef PKV_DECODE_SNAP_CAP
    constexpr int kSnapCap = PKV_DECODE_SNAP_CAP;
#else
    constexpr int kSnapCap = NW;  // one chunk per warp of the CTA
#endif
#ifdef PKV_DECODE_MIN_SHARE
    constexpr int kMinShare = PKV_DECODE_MIN_SHARE;
#else
    constexpr int kMinShare = 4;
#endif
#ifdef PKV_DECODE_RELIEF
    constexpr int kRelief = PKV_DECODE_RELIEF;
#else
    constexpr int kRelief = 4;  // chunks a worker with a piece cut across CTAs gives up
#endif
#ifdef PKV_DECODE_DEFER_MIN
    constexpr int kDeferMin = PKV_DECODE_DEFER_MIN;
#else
    constexpr int kDeferMin = 24;  // CTAs whose warps' shares are shorter merge at once
#endif
#ifdef PKV_DECODE_RELIEF_DIV
    constexpr int kReliefDiv = PKV_DECODE_RELIEF_DIV;
#else
    constexpr int kReliefDiv = 16;  // ... at most 1/16 of a nominal share
#endif
#ifdef PKV_DECODE_G1_CUDACORE
    constexpr bool kCudaCore = PKV_DECODE_G1_CUDACORE != 0 && G == 1;
#else
    constexpr bool kCudaCore = false;  // group 1 on the tensor cores too (see consume_chunk_cc)
#endif
    using Geo = DecodeGeometry<D, BS, G>;
    using Smem = DecodeSmem<NW, ST, D, BS, G, GRP>;
    static_assert(!GRP || (G == 8 && BS >= 16), "the grouped kernel: 8 query rows per item, whole-block chunks");
    extern __shared__ unsigned char smem_raw[];
    __shared__ int warp_sums[32];
    __shared__ int warp_sums2[32];
    // 1024-byte aligned base: the 128-byte swizzle pattern is tied to address bits
    unsigned char *smem =
        smem_raw + ((Smem::kAlign - (smem_addr(smem_raw) & (Smem::kAlign - 1))) & (Smem::kAlign - 1));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Smem::kBars);
    int4 *meta = reinterpret_cast<int4 *>(smem + Smem::kMeta);
    const int N = p.num_seqs;
    // per-sequence arrays: [cum (N+1)][ctx (N)] | grouped: [ctx (N)][shared (N)]
    // [cum over items (2N+1)] [items (2N)]; then the CTA bounds
    int *cum, *ctx, *shv = nullptr;
    int2 *info = nullptr;
    int64_t *bounds;
    if constexpr (GRP) {
        ctx = reinterpret_cast<int *>(smem + Smem::kCum);
        shv = ctx + N;
        cum = shv + N;
        info = reinterpret_cast<int2 *>(smem + Smem::kCum + (((size_t)(4 * N + 1) * 4 + 7) & ~(size_t)7));
        bounds = reinterpret_cast<int64_t *>(info + 2 * N);
    } else {
        cum = reinterpret_cast<int *>(smem + Smem::kCum);
        ctx = cum + N + 1;
        bounds = reinterpret_cast<int64_t *>(smem + Smem::kCum + (((size_t)(2 * N + 1) * 4 + 7) & ~(size_t)7));
    }
    __shared__ int cta_count[NW];
    __shared__ int64_t worker_starts[NW + 1];
    __shared__ int exit_count;
    __shared__ int cta_cross;
    __shared__ MergeQueue mq;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int Hkv = p.num_kv_heads;
    const int max_ctx = p.max_blocks_per_seq * BS;

    if (tid == 0) {
        prefetch_tensormap(&p.tmap_k);
        prefetch_tensormap(&p.tmap_v);
        prefetch_tensormap(&p.tmap_k8);
        prefetch_tensormap(&p.tmap_v8);
    }
    if constexpr (HOSTIN) {
        // block tables in host memory: the CTAs bring them into L2 together
        // (one line each in turn) while the lengths load and the scan run, so
        // that the first table reads after the scan do not cross the link
        const int64_t lines = ((int64_t)p.num_seqs * p.max_blocks_per_seq * 4 + 127) / 128;
        for (int64_t l = (int64_t)blockIdx.x + (int64_t)tid * gridDim.x; l < lines;
             l += (int64_t)gridDim.x * blockDim.x)
            prefetch_l2(reinterpret_cast<const char *>(p.block_tables) + l * 128);
    }
    // Up to the grid-dependency wait below, the kernel reads only the context
    // lengths and the block tables (inputs of the call, never written by the
    // library's kernels): with programmatic dependent launch, the prologue,
    // the shares and the first table loads overlap the tail of the preceding
    // kernel in the stream.

    // ---- prologue: chunk counts per sequence and their prefix sums ----------
    const int per = (N + NW * 32 - 1) / (NW * 32);
    const int s_lo = min(N, tid * per);
    const int s_hi = min(N, s_lo + per);
    int local = 0;
    int last_start = -1;  // grouped: the last sequence of this thread's range that starts a chain
    for (int s = s_lo; s < s_hi; ++s) {
        int c = p.context_lens[s];
        if (c < 0 || c > max_ctx) {
            report(p.status, PKV_ERR_OUT_OF_RANGE);
            c = c < 0 ? 0 : max_ctx;
        }
        ctx[s] = c;
        local += Hkv * chunks_for(c, Geo::kRows);
        if constexpr (GRP) {
            const int h = s == 0 ? 0 : max(0, (int)p.shared_blocks[s]);
            shv[s] = h;
            if (h == 0) last_start = s;
        }
    }
    if constexpr (GRP) local = last_start;  // the first scan is a max over chain starts
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl = GRP ? max(incl, y) : incl + y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    if (tid == 0) {
        // lane 0's arrival (with the copies' byte count); with host inputs
        // also every lane's, after its 16-byte copies
        for (int i = 0; i < NW * ST; ++i) mbar_init(smem_addr(bars + i), HOSTIN ? 33 : 1);
        fence_barrier_init();
    }
    if (tid < NW) cta_count[tid] = 0;
    if (tid < kMergeQueue) mq.entry[tid] = -1;
    if (tid == 0) {
        exit_count = 0;
        cta_cross = 0;
        mq.tail = mq.head = 0;
    }
    __syncthreads();
    int NI = N;  // segments' owners: sequences, or the grouped kernel's items
    if constexpr (!GRP) {
        // every warp scans the warps' sums itself (no second barrier)
        const int v = lane < NW ? warp_sums[lane] : 0;
        int vi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFullMask, vi, o);
            if (lane >= o) vi += y;
        }
        int run = __shfl_sync(kFullMask, vi - v, warp) + incl - local;
        const int total = __shfl_sync(kFullMask, vi, 31);
        for (int s = s_lo; s < s_hi; ++s) {
            cum[s] = run;
            run += Hkv * chunks_for(ctx[s], Geo::kRows);
        }
        if (tid == 0) cum[N] = total;
    } else {
        // The chain start before this thread's range: the max over the
        // threads before it (each warp scans the warps' maxima itself).
        int chain;
        {
            const int v = lane < NW ? warp_sums[lane] : -1;
            int vi = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFullMask, vi, o);
                if (lane >= o) vi = max(vi, y);
            }
            const int before_warp = warp > 0 ? __shfl_sync(kFullMask, vi, warp - 1) : -1;
            const int before_lane = __shfl_up_sync(kFullMask, incl, 1);
            chain = max(before_warp, lane > 0 ? before_lane : -1);
        }
        // Each sequence's group (the leader and its members, up to 8
        // consecutive sequences of one chain) and the shared full blocks P:
        // at most the blocks every member shares with its predecessor, and
        // never the block of a member's last token.  A group (P >= 1) is one
        // item; its chunks per KV head: the P shared blocks', then every
        // member's own.
        auto group_of = [&](int s, int cs, int &lead, int &ns, int &shared_chunks) {
            lead = cs + ((s - cs) & ~7);
            ns = 1;
            int pb = ctx[lead] >= 1 ? (ctx[lead] - 1) / BS : -1;
            for (int j = 1; j < 8; ++j) {
                const int m = lead + j;
                if (m >= N || shv[m] == 0) break;
                ++ns;
                pb = min(pb, min(shv[m], ctx[m] >= 1 ? (ctx[m] - 1) / BS : -1));
            }
            shared_chunks = (ns >= 2 && pb >= 1) ? pb * (BS / Geo::kRows) : 0;
        };
        int nitems = 0, nchunks = 0;
        {
            int cs = chain;
            for (int s = s_lo; s < s_hi; ++s) {
                if (shv[s] == 0) cs = s;
                int lead, ns, sc;
                group_of(s, cs, lead, ns, sc);
                nitems += sc > 0 ? (s == lead ? 1 : 0) : 1;
                nchunks += Hkv * (chunks_for(ctx[s], Geo::kRows) - (sc > 0 && s != lead ? sc : 0));
            }
        }
        // exclusive scans of (items, chunks) over the threads
        int ii = nitems, ic = nchunks;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int yi = __shfl_up_sync(kFullMask, ii, o);
            const int yc = __shfl_up_sync(kFullMask, ic, o);
            if (lane >= o) {
                ii += yi;
                ic += yc;
            }
        }
        __syncthreads();  // every warp has read warp_sums
        if (lane == 31) {
            warp_sums[warp] = ii;
            warp_sums2[warp] = ic;
        }
        __syncthreads();
        int vi = lane < NW ? warp_sums[lane] : 0, vc = lane < NW ? warp_sums2[lane] : 0;
        const int v0 = vi, c0 = vc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int yi = __shfl_up_sync(kFullMask, vi, o);
            const int yc = __shfl_up_sync(kFullMask, vc, o);
            if (lane >= o) {
                vi += yi;
                vc += yc;
            }
        }
        int item = __shfl_sync(kFullMask, vi - v0, warp) + ii - nitems;
        int run = __shfl_sync(kFullMask, vc - c0, warp) + ic - nchunks;
        NI = __shfl_sync(kFullMask, vi, 31);
        const int total = __shfl_sync(kFullMask, vc, 31);
        {
            int cs = chain;
            for (int s = s_lo; s < s_hi; ++s) {
                if (shv[s] == 0) cs = s;
                int lead, ns, sc;
                group_of(s, cs, lead, ns, sc);
                // a group's leader opens its item (its members' own chunks follow
                // inside it); a lone sequence is an item of its own
                if (sc == 0 || s == lead) {
                    info[item] = sc > 0 ? make_int2(lead | (ns << 16), sc) : make_int2(s | (1 << 16), 0);
                    cum[item++] = run;
                }
                run += Hkv * (chunks_for(ctx[s], Geo::kRows) - (sc > 0 && s != lead ? sc : 0));
            }
        }
        if (tid == 0) cum[NI] = total;
    }
    __syncthreads();

    // ---- this warp's share: CTA ranges snapped to segment boundaries, each
    // divided among the CTA's warps (cta_share_start).  A warp works out its own CTA's
    // range itself and starts its block-table loads; the CTA-wide array of
    // ranges (for the merges) is filled after that. ----
    const int64_t T = cum[NI];
    // A small batch uses only as many CTAs as give every worker at least
    // kMinShare chunks (a segment split into one-chunk pieces costs more to
    // merge than the extra workers save), and, while segments are short (up to
    // 2 kMinShare chunks per worker), no more CTAs than segments: equal
    // segments then fall one per CTA and merge in shared memory.  The other
    // CTAs have nothing to do.
    const int64_t seg_cap = max((int64_t)NI * Hkv, (T + NW * 2 * kMinShare - 1) / (NW * 2 * kMinShare));
    const int C = (int)min(min((int64_t)gridDim.x, seg_cap),
                           max((int64_t)1, (T + NW * kMinShare - 1) / (NW * kMinShare)));
    if ((int)blockIdx.x >= C) return;
    const int64_t wid = (int64_t)blockIdx.x * NW + warp;
    int64_t gb, ge, c_lo, c_len;
    {
        // lane 0: the CTA range's start, lane 1: its end (and whether each
        // cuts a segment)
        const int c = (int)blockIdx.x + (lane & 1);
        bool cuts = false;
        const int64_t v = c == C ? T : snapped_cta_start(cum, NI, Hkv, c, C, T, kSnapCap, &cuts);
        c_lo = __shfl_sync(kFullMask, v, 0);
        c_len = __shfl_sync(kFullMask, v, 1) - c_lo;
        const int r = cut_relief_for(cuts, c_len, NW, kRelief, kReliefDiv);
        const int r0 = __shfl_sync(kFullMask, r, 0);
        const int r1 = __shfl_sync(kFullMask, r, 1);
        // lane 0 this warp's start, lane 1 its end
        const int64_t st = cta_share_start(c_lo, c_len, NW, warp + (lane & 1), r0, r1);
        gb = __shfl_sync(kFullMask, st, 0);
        ge = __shfl_sync(kFullMask, st, 1);
        // the CTA's worker starts, looked up by the merges (after the barrier
        // that follows the first copies)
        if (lane == 0) worker_starts[warp] = gb;
        if (lane == 0 && warp == NW - 1) worker_starts[NW] = ge;
    }
    const int n = gb < ge ? (int)(ge - gb) : 0;

    // the walk: cut pieces first (see share_order); lane 0 locates the
    // share's first chunk, lane 1 its last
    ShareOrder order = share_order(cum, NI, Hkv, gb, gb);  // empty
    if (n > 0) {
        const ChunkPos e = locate_chunk(cum, NI, Hkv, (lane & 1) ? ge - 1 : gb);
        ChunkPos first, last;
        first.c = __shfl_sync(kFullMask, e.c, 0);
        first.nch = __shfl_sync(kFullMask, e.nch, 0);
        last.c = __shfl_sync(kFullMask, e.c, 1);
        last.nch = __shfl_sync(kFullMask, e.nch, 1);
        order = share_order_at(first, last, gb, ge);
    }

    // block-table entry of the chunk at walk position i (raw; validated when
    // its descriptor is built), 0 past the share
    // (at block size 8 a chunk spans two blocks: the second entry comes in the
    // high half, 0 when the chunk does not reach it)
    // Where chunk c (of nch) of a segment owned by `it` lies: its sequence,
    // the chunk within that sequence, whether it is the sequence's last, and
    // (grouped) the member whose own chunk it is (-1: all rows see it).
    struct Where {
        int seq, lc, member;
        bool last;
    };
    auto where = [&](int it, int c, int nch) -> Where {
        if constexpr (!GRP) {
            return {it, c, -1, c == nch - 1};
        } else {
            const ItemInfo ii = item_info(info, it);
            if (c < ii.sc) return {ii.s0, c, -1, false};
            int r = c - ii.sc, j = 0;
            int own = chunks_for(ctx[ii.s0], Geo::kRows) - ii.sc;
            while (j < ii.ns - 1 && r >= own) {
                r -= own;
                ++j;
                own = chunks_for(ctx[ii.s0 + j], Geo::kRows) - ii.sc;
            }
            return {ii.s0 + j, ii.sc + r, ii.ns > 1 ? j : -1, r == own - 1};
        }
    };
    auto table_entry_at = [&](const ChunkPos &q) -> int2 {
        const Where w = where(q.s, q.c, q.nch);
        const int lb = chunk_block(w.lc, BS, Geo::kRows);
        const int32_t *row = p.block_tables + (int64_t)w.seq * p.max_blocks_per_seq;
        int second = 0;
        if (Geo::kBPC == 2 && (lb + 1) * BS < ctx[w.seq]) second = __ldg(row + lb + 1);
        return make_int2(__ldg(row + lb), second);
    };
    auto table_entry = [&](int i) -> int2 {
        if (i >= n) return make_int2(0, 0);
        return table_entry_at(locate_chunk(cum, NI, Hkv, order.at(i)));
    };
    const bool append = p.new_key != nullptr;
    // Descriptor of the chunk at walk position i, built by one lane for a
    // window of 32 positions at a time (lane j: position win + j) from its
    // table entry `tab`: x = segment owner | KV head << 16, y = rows | flags << 8,
    // z / w = the cache row of its box (of each block's box at block size 8).
    // Issuing a chunk is then a few shuffles and the copies.
    auto chunk_desc_at = [&](int64_t g, const ChunkPos &q, int2 tab) -> int4 {
        int phys = tab.x, phys2 = tab.y;
        if (phys < 0 || phys >= p.num_blocks) {
            report(p.status, PKV_ERR_OUT_OF_RANGE);
            phys = 0;
        }
        if (phys2 < 0 || phys2 >= p.num_blocks) {
            report(p.status, PKV_ERR_OUT_OF_RANGE);
            phys2 = 0;
        }
        const Where w = where(q.s, q.c, q.nch);
        const int rows = chunk_rows(w.lc, ctx[w.seq], Geo::kRows);
        // the decode step's new token is the last row of its sequence's last
        // chunk (never in a group's shared blocks: they stop before it)
        const bool new_row = append && w.last;
        const int flags = chunk_flags(q, g, gb, ge) | (new_row ? kAppendRow : 0) |
                          (w.member >= 0 ? kOwn | (w.member << kMemberShift) : 0);
        // row of the cache viewed as [num_blocks * Hkv * BS rows]
        const int y = (int)(((int64_t)phys * Hkv + q.kvh) * BS + (w.lc * Geo::kRows) % BS);
        const int y2 = (int)(((int64_t)phys2 * Hkv + q.kvh) * BS);
        return make_int4(q.s | (q.kvh << 16), rows | (flags << 8), y, y2);
    };
    auto chunk_desc = [&](int i, int2 tab) -> int4 {
        if (i >= n) return make_int4(0, 0, 0, 0);
        const int64_t g = order.at(i);
        return chunk_desc_at(g, locate_chunk(cum, NI, Hkv, g), tab);
    };
    // windows 0 and 1: each lane locates its two positions in one search and
    // starts their table loads; window 0's descriptors follow as soon as the
    // entries arrive (the CTA-wide ranges, which only the merges need, come
    // after the first copies are out)
    int win = 0;
    int4 desc = make_int4(0, 0, 0, 0);  // descriptors of window win
    int2 tab_nxt = make_int2(0, 0);     // table entries of window win + 1
    {
        ChunkPos q0, q1;
        int2 tab0 = make_int2(0, 0);
        if (n > 0) {
            locate_chunk2(cum, NI, Hkv, lane < n ? order.at(lane) : gb, 32 + lane < n ? order.at(32 + lane) : gb,
                          q0, q1);
            if (lane < n) tab0 = table_entry_at(q0);
            if (32 + lane < n) tab_nxt = table_entry_at(q1);
        }
        if (lane < n) desc = chunk_desc_at(order.at(lane), q0, tab0);
    }

    unsigned char *wst = smem + (size_t)warp * ST * Geo::kStageBytes;
    const uint32_t wst_a = smem_addr(wst);
    const unsigned char *wq = smem + Smem::kQ + (size_t)warp * ST * Geo::kSlotBytes;
    const uint32_t wq_a = smem_addr(wq);
    const uint32_t bar_a = smem_addr(bars + warp * ST);
    int4 *wmeta = meta + 2 * warp * ST;

    auto issue = [&](int i) {
        if (i == win + 32) {
            // next window: its descriptors from the entries loaded one window
            // ago, then the loads for the window after it
            win += 32;
            desc = chunk_desc(win + lane, tab_nxt);
            tab_nxt = table_entry(win + 32 + lane);
        }
        const int j = i - win;
        const int sk = __shfl_sync(kFullMask, desc.x, j);
        const int rf = __shfl_sync(kFullMask, desc.y, j);
        const int y = __shfl_sync(kFullMask, desc.z, j);
        const int y2 = Geo::kBPC == 2 ? __shfl_sync(kFullMask, desc.w, j) : 0;
        if (lane == 0) {
            const int it = sk & 0xffff, kvh = sk >> 16;
            const int rows = rf & 0xff, flags = rf >> 8;
            // the query rows' first sequence and count (grouped: the members,
            // one row each), and the sequence whose new token a chunk carries
            int s = it, nq = G, snew = it;
            if constexpr (GRP) {
                const ItemInfo ii = item_info(info, it);
                s = ii.s0;
                nq = ii.ns;
                snew = ii.s0 + ((flags & kOwn) ? (flags >> kMemberShift) & 7 : 0);
            }
            const bool new_row = (flags & kAppendRow) != 0;
            const int stage = i % ST;
            const uint32_t bar = bar_a + stage * 8;
            const uint32_t kdst = wst_a + stage * Geo::kStageBytes;
            const uint32_t vdst = kdst + Geo::kTileBytes;
            // a whole chunk inside one block is one box per cache; a last chunk
            // of at most 8 rows takes one 8-row box per half instead, and at
            // block size 8 each block of the chunk is one 8-row box per half
            // (the second lands 8 rows down, at +1 KB in each half)
            const bool short_box = Geo::kBPC == 2 || rows <= 8;
            const bool second = Geo::kBPC == 2 && rows > 8;
            wmeta[2 * stage] = make_int4(it, kvh, rows, flags);  // x: the segment's owner
            wmeta[2 * stage + 1] = make_int4(y, y2, 0, 0);
            // (with host inputs the lanes' arrivals, not bytes, cover the query and new rows)
            const uint32_t side = HOSTIN ? 0u
                                         : ((flags & kFirst) ? (GRP ? nq * D * 2 : Geo::kQBytes) : 0) +
                                               (new_row ? 2 * Geo::kRowBytes : 0);
            mbar_arrive_expect_tx(bar, (short_box ? (second ? 4 : 2) * Geo::kHalves * Geo::kBoxBytes
                                                  : 2 * Geo::kTileBytes) + side);
            if (!short_box) {
                tma_load_3d(kdst, &p.tmap_k, 0, y, 0, bar);
                tma_load_3d(vdst, &p.tmap_v, 0, y, 0, bar);
            } else {
#pragma unroll
                for (int h = 0; h < Geo::kHalves; ++h) {
                    tma_load_3d(kdst + h * Geo::kHalfBytes, &p.tmap_k8, 0, y, h, bar);
                    tma_load_3d(vdst + h * Geo::kHalfBytes, &p.tmap_v8, 0, y, h, bar);
                    if (second) {
                        tma_load_3d(kdst + h * Geo::kHalfBytes + Geo::kBoxBytes, &p.tmap_k8, 0, y2, h, bar);
                        tma_load_3d(vdst + h * Geo::kHalfBytes + Geo::kBoxBytes, &p.tmap_v8, 0, y2, h, bar);
                    }
                }
            }
            if constexpr (!HOSTIN) {
                const uint32_t slot = wq_a + stage * Geo::kSlotBytes;
                if (flags & kFirst) {
                    if constexpr (GRP) {
                        for (int j = 0; j < nq; ++j)
                            bulk_g2s(slot + j * D * 2, p.query + ((int64_t)(s + j) * p.num_heads + kvh) * D, D * 2,
                                     bar);
                    } else {
                        bulk_g2s(slot, p.query + ((int64_t)s * p.num_heads + kvh * G) * D, Geo::kQBytes, bar);
                    }
                }
                if (new_row) {
                    const int64_t src = ((int64_t)snew * Hkv + kvh) * D;
                    bulk_g2s(slot + Geo::kQBytes, p.new_key + src, Geo::kRowBytes, bar);
                    bulk_g2s(slot + Geo::kQBytes + Geo::kRowBytes, p.new_value + src, Geo::kRowBytes, bar);
                }
            }
        }
        if constexpr (HOSTIN) {
            // inputs in host memory: every lane takes part (copy_host_inputs)
            const int it = sk & 0xffff, kvh = sk >> 16, flags = rf >> 8;
            int s = it, nq = G, snew = it;
            if constexpr (GRP) {
                const ItemInfo ii = item_info(info, it);
                s = ii.s0;
                nq = ii.ns;
                snew = ii.s0 + ((flags & kOwn) ? (flags >> kMemberShift) & 7 : 0);
            }
            const int stage = i % ST;
            copy_host_inputs<D, G, GRP>(p, wq_a + stage * Geo::kSlotBytes, bar_a + stage * 8, (flags & kFirst) != 0,
                                        (flags & kAppendRow) != 0, s, nq, snew, kvh, lane);
        }
    };

    int issued = 0;

    // ---- from here on the kernel reads and writes what the preceding kernel
    // may write: the caches, the workspace, the output ----
    grid_dependency_wait();
    launch_dependents();
    // this call counts on the counters of its epoch's parity, and prepares the
    // other parity's counters for the next call (the epoch only changes when
    // every CTA of a call is out, so every warp of this call reads the same);
    // the load goes out before the first copies, its value is used after them
    uint32_t epoch = 0;
    if (lane == 0) epoch = (uint32_t)__ldcg(p.ws_sync);
    for (; issued < min(ST, n); ++issued) issue(issued);
    // the CTA-wide ranges (needed only by the merges)
    for (int c = tid; c <= C; c += NW * 32)
        bounds[c] = c == C ? T : snapped_cta_start(cum, NI, Hkv, c, C, T, kSnapCap);
    __syncthreads();  // the ranges are visible to every warp's merges
    epoch = __shfl_sync(kFullMask, epoch, 0);
    const int parity = epoch & 1;
    unsigned long long *count_now = p.ws_count + (int64_t)parity * N * Hkv;
    {
        unsigned long long *count_next = p.ws_count + (int64_t)(parity ^ 1) * N * Hkv;
        const unsigned long long next_tag = (unsigned long long)(epoch + 1) << 32;
        for (int64_t i = (int64_t)blockIdx.x * NW * 32 + tid; i < (int64_t)N * Hkv; i += (int64_t)C * NW * 32)
            count_next[i] = next_tag;
        if (blockIdx.x == 0 && tid == 0) p.ws_sync[1 + (parity ^ 1)] = next_tag;
    }
    // rows of empty contexts are zero; no worker visits them
    for (int s = blockIdx.x; s < N; s += C) {
        if (ctx[s] != 0) continue;
        uint4 *row = reinterpret_cast<uint4 *>(p.out + (int64_t)s * p.num_heads * D);
        for (int i = tid; i < p.num_heads * D / 8; i += NW * 32) row[i] = make_uint4(0, 0, 0, 0);
    }
    // every warp counts itself out at the end
    // (the CTA's warps count out in shared memory; the last of them counts the
    // CTA out of the grid, and the last CTA out advances the epoch)
    auto exit_warp = [&]() {
        if (lane == 0 && atomicAdd(&exit_count, 1) == NW - 1 &&
            count_in_tagged(p.ws_sync + 1 + parity, epoch, C, 1) == C)
            atomicExch(p.ws_sync, (unsigned long long)(epoch + 1));
    };
    // shared partial slots: 16-byte aligned, after the bounds
    float *part = nullptr;
    if (p.smem_partials)
        part = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(bounds + C + 1) + 15) & ~(uintptr_t)15);
    const WorkerCtx<NW> wc{cum, bounds, C, wid, gb, ge, epoch, count_now, cta_count, &cta_cross, part,
                           worker_starts, info};

    // the CTA's merge queue (count_piece / merge_part)
    auto vload = [](const int *a) { return *reinterpret_cast<const volatile int *>(a); };
    auto push = [&](int s, int kvh) {  // (an overflowing push merges at once: see MergeQueue)
        int idx = 0;
        if (lane == 0) {
            idx = atomicAdd(&mq.tail, 1);
            if (idx < kMergeQueue) *reinterpret_cast<volatile int *>(&mq.entry[idx]) = s | (kvh << 16);
        }
        idx = __shfl_sync(kFullMask, idx, 0);
        if (idx >= kMergeQueue) merge_part<D, G, NW, GRP>(p, wc, s, kvh, segment_info(p, wc, s, kvh), lane);
    };
    // After its own share a warp merges queued parts until the queue is empty.
    // No entry is left behind: a warp pushes only during its own share and
    // drains after it, so whatever it pushed is either taken by another warp
    // or by itself.  Warps that finish early thus take the parts queued early
    // (the cut pieces come first in every share).
    auto drain = [&]() {
        const uint64_t t0 = global_ns();
        while (true) {
            int e = -1;
            if (lane == 0) {
                int h = vload(&mq.head);
                while (h < vload(&mq.tail)) {
                    const int prev = atomicCAS(&mq.head, h, h + 1);
                    if (prev == h) {
                        e = h;
                        break;
                    }
                    h = prev;
                }
            }
            e = __shfl_sync(kFullMask, e, 0);
            if (e < 0) return;               // empty
            if (e >= kMergeQueue) continue;  // merged by its producer
            int v = -1;
            if (lane == 0)  // written by its producer right after the claim
                while ((v = vload(&mq.entry[e])) < 0 && global_ns() - t0 < p.wait_limit_ns) {
                }
            v = __shfl_sync(kFullMask, v, 0);
            if (v < 0) {
                if (lane == 0) report(p.status, PKV_ERR_DEVICE_TIMEOUT);
                return;
            }
            fence_acq_rel_cta();
            merge_part<D, G, NW, GRP>(p, wc, v & 0xffff, v >> 16, segment_info(p, wc, v & 0xffff, v >> 16), lane);
        }
    };
    // whether this CTA queues its merges (the same for all its warps): when
    // its warps' shares are long enough for the merging warp to end late
    const bool defer = c_len >= (int64_t)kDeferMin * NW;
    if (n == 0) {
        if (defer) drain();
        exit_warp();
        return;
    }

    const int gq = lane >> 2;
    const int tq = lane & 3;
    uint32_t qa[D / 16][2];
    float m = -CUDART_INF_F, l = 0.f;
    float o[D / 16][4];  // O^T: dims 16i + g (+8) of heads 2t, 2t + 1
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) qa[kk][0] = qa[kk][1] = 0u;
#pragma unroll
    for (int j = 0; j < D / 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    // the CUDA-core form (group 1, opt-in build): the lane's query dims and
    // its row's share of the output (consume_chunk_cc)
    float qc[kCudaCore ? D / 2 : 1], oc[kCudaCore ? D / 2 : 1];
#pragma unroll
    for (int j = 0; j < (kCudaCore ? D / 2 : 1); ++j) qc[j] = oc[j] = 0.f;

    for (int i = 0; i < n; ++i) {
        const int stage = i % ST;
        const uint32_t parity = (uint32_t)(i / ST) & 1u;
        const bool ok = mbar_wait_bounded(bar_a + stage * 8, parity, p.wait_limit_ns);
        if (!__all_sync(kFullMask, ok)) {
            // give up: report, then wait (bounded) for this warp's copies still
            // in flight so that none lands after the CTA has exited
            if (lane == 0) report(p.status, PKV_ERR_DEVICE_TIMEOUT);
            for (int j = i; j < issued; ++j)
                mbar_wait_bounded(bar_a + (j % ST) * 8, (uint32_t)(j / ST) & 1u, p.wait_limit_ns);
            exit_warp();
            return;
        }
        const int4 md = wmeta[2 * stage];
        if (md.w & kFirst) {
            const unsigned char *sq = wq + stage * Geo::kSlotBytes;
            if constexpr (kCudaCore) {
                load_query_cc<D>(sq, qc, lane);
#pragma unroll
                for (int j = 0; j < D / 2; ++j) oc[j] = 0.f;
            } else {
                // query rows of the group as mma A fragments (rows g >= G stay 0;
                // grouped: rows past the item's sequences too)
                int nq = G;
                if constexpr (GRP) nq = item_info(info, md.x).ns;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    qa[kk][0] =
                        gq < nq ? *reinterpret_cast<const uint32_t *>(sq + (gq * D + 16 * kk + 2 * tq) * 2) : 0u;
                    qa[kk][1] =
                        gq < nq ? *reinterpret_cast<const uint32_t *>(sq + (gq * D + 16 * kk + 8 + 2 * tq) * 2) : 0u;
                }
#pragma unroll
                for (int j = 0; j < D / 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
            }
            m = -CUDART_INF_F;
            l = 0.f;
        }
        if (md.z < Geo::kRows) zero_tail_rows<D, BS, G>(wst + stage * Geo::kStageBytes + Geo::kTileBytes, md.z, lane);
        if (md.w & kAppendRow) {
            // the new token (row md.z - 1): into the swizzled tiles for this
            // step, and into the cache for the steps after it
            constexpr int kVecs = D / 8;  // 16-byte pieces of a row
            const int r = md.z - 1;
            if (lane < 2 * kVecs) {
                const int v = lane % kVecs;
                const bool is_v = lane >= kVecs;
                const uint4 val = *reinterpret_cast<const uint4 *>(wq + stage * Geo::kSlotBytes + Geo::kQBytes +
                                                                   (is_v ? Geo::kRowBytes : 0) + v * 16);
                unsigned char *tile = wst + stage * Geo::kStageBytes + (is_v ? Geo::kTileBytes : 0);
                *reinterpret_cast<uint4 *>(tile + (v >> 3) * Geo::kHalfBytes + r * 128 + (((v & 7) ^ (r & 7)) << 4)) =
                    val;
                __half *cache = is_v ? p.value_cache_w : p.key_cache_w;
                const int4 yy = wmeta[2 * stage + 1];
                const int64_t crow = (Geo::kBPC == 2 && r >= 8) ? (int64_t)yy.y + (r - 8) : (int64_t)yy.x + r;
                *reinterpret_cast<uint4 *>(cache + crow * D + v * 8) = val;
            }
            __syncwarp();
        }
        // The stage's tiles were written through the generic proxy (zeroed tail
        // rows, the new row): order those writes before the TMA copy that
        // refills this stage (issued after the __syncwarp below).  Reads need
        // no fence: every ldmatrix has delivered before the mma that uses it.
        if (md.z < Geo::kRows || (md.w & kAppendRow)) fence_proxy_async_smem();
        const uint32_t kt = wst_a + stage * Geo::kStageBytes;
        if constexpr (kCudaCore)
            consume_chunk_cc<D>(wst + stage * Geo::kStageBytes, wst + stage * Geo::kStageBytes + Geo::kTileBytes,
                                md.z, qc, p.scale_log2, m, l, oc, lane);
        else
            consume_chunk<D, BS, G, GRP>(kt, kt + Geo::kTileBytes, md.z, qa, p.scale_log2, m, l, o, lane,
                                         (GRP && (md.w & kOwn)) ? (md.w >> kMemberShift) & 7 : -1);
        // refill the stage first: a piece's finish (and a cut piece's count and
        // merge) then overlaps the copies in flight instead of draining the ring
        __syncwarp();
        if (issued < n) issue(issued++);
        SegInfo si;
        bool stored = false;
        if (md.w & kLast) {
            if constexpr (kCudaCore)
                stored = finish_piece_cc<D, NW>(p, wc, md, m, l, oc, si, lane);
            else
                stored = finish_piece<D, G, NW, GRP>(p, wc, md, m, l, o, si, lane);
        }
        if (stored &&
            count_piece<D, G, NW>(wc, si, lane)) {
            // with long shares the merge goes to a warp that is done with its
            // own (the merging warp would otherwise end late); with short ones
            // every warp ends at about the same time, and merging at once
            // overlaps the copies still in flight
            if (defer) {
                fence_acq_rel_cta();  // the part's pieces are visible to whoever merges it
                push(md.x, md.y);
            } else {
                merge_part<D, G, NW, GRP>(p, wc, md.x, md.y, si, lane);
            }
        }
    }
    if (defer) drain();
    exit_warp();
}

}  // namespace pkv

#endif  // PKV_DECODE_IMPL_CUH
