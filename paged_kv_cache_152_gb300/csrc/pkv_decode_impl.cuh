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
// Design (GB300, HBM-bound: each K/V byte is read exactly once):
//  * The batch's work is cut into 4 KB chunks (pkv_schedule.h) and split into
//    equal contiguous shares, one per WARP of a persistent grid.  Every warp
//    is an independent worker; no CTA-wide synchronisation after the prologue.
//  * Each warp owns a ring of ST stages in shared memory.  Lane 0 issues, ST
//    chunks ahead, one cp.async.bulk (TMA engine) per K chunk and per V chunk
//    -- the chunk is one contiguous run of rows*head_dim fp16 in the
//    [block][kv_head][slot][dim] layout -- plus the query rows of the KV group
//    at the first chunk of each piece, all completing on the stage's
//    mbarrier.  Block-table entries for the next 32 chunks are prefetched one
//    per lane into registers, 32 chunks ahead of use.
//  * Compute: a lane covers 8 consecutive head-dim elements of one row (16-B
//    shared loads, conflict-free).  q.k partial sums are reduced with xor
//    shuffles inside the D/8 lanes of a row; each lane then holds the full
//    score of the rows it loads, so P.V needs no shuffle.  All G query heads
//    of a KV group use each loaded K/V element (K/V read once per group).
//    Scores are in log2 units (scale*log2(e) folded into q) and the softmax is
//    online, per warp, in fp32.
//  * A piece that covers a whole (sequence, KV head) is normalised and written
//    as fp16 by the warp.  A cut piece stores (max, sum, unnormalised output)
//    in the workspace and counts itself in on the segment's counter; the warp
//    that brings the count to the number of pieces merges them, in worker
//    order (deterministic, no float atomics, no second kernel).  Counters hold
//    (call tag << 32 | count) and the merging warp zeroes its counter again:
//    garbage in a fresh workspace, or a count left by a failed call, carries
//    another call's tag and is ignored, and a replayed launch (same tag) finds
//    every counter it uses back at zero.
//  * Rows past the context are never used: the bulk copy of a ragged last
//    chunk moves only its valid rows, masked scores become -inf, and V rows
//    past the context are not loaded.
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
    static constexpr int kRowBytes = D * 2;
    // rows per chunk: a whole block, or 4 KB of it when the block is larger
    static constexpr int kRows = (BS * kRowBytes <= 4096) ? BS : 4096 / kRowBytes;
    static constexpr int kChunkBytes = kRows * kRowBytes;
    static constexpr int kQBytes = G * D * 2;
    static constexpr int kQSlot = (kQBytes + 127) / 128 * 128;
    static constexpr int kStageBytes = 2 * kChunkBytes + kQSlot;
    static constexpr int kLanesPerRow = D / 8;
    static constexpr int kRowsPerLoad = 32 / kLanesPerRow;
    static constexpr int kLoads = kRows / kRowsPerLoad;               // 16-B loads per lane per chunk
    static constexpr int kSub = (kLoads * G <= 32) ? kLoads : 32 / G; // loads per softmax sub-step
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(kRows % kRowsPerLoad == 0, "rows per chunk");
    static_assert(kLoads % kSub == 0, "sub-steps");
    static_assert(BS % kRows == 0, "a chunk never crosses a block");
    static_assert(kChunkBytes % 128 == 0, "stage alignment");
};

// Dynamic shared memory: [stages][barriers][chunk meta][cum (N+1)][ctx (N)].
template <int NW, int ST, int STAGE>
struct DecodeSmem {
    static constexpr size_t kBars = (size_t)NW * ST * STAGE;
    static constexpr size_t kMeta = kBars + (size_t)NW * ST * 8;
    static constexpr size_t kCum = kMeta + (size_t)NW * ST * 16;
    static constexpr size_t kFixed = kCum;
    static constexpr size_t kPerSeq = 8;
    __host__ __device__ static size_t bytes(int n) { return kCum + 4 * (size_t)(n + 1) + 4 * (size_t)n; }
};

// One chunk: rows [0, rows) of the K and V tiles in shared memory.
template <int D, int BS, int G>
__device__ __forceinline__ void process_chunk(const unsigned char *sk, const unsigned char *sv, int rows,
                                              const float (&q)[G][8], float (&m)[G], float (&l)[G],
                                              float (&acc)[G][8], int lane) {
    using Geo = DecodeGeometry<D, BS, G>;
    constexpr int LPR = Geo::kLanesPerRow;
    constexpr int RPI = Geo::kRowsPerLoad;
    const int rg = lane / LPR;
    const int cl = lane % LPR;
#pragma unroll
    for (int c0 = 0; c0 < Geo::kLoads; c0 += Geo::kSub) {
        if (c0 * RPI >= rows) break;  // warp-uniform: the rest of the chunk is past the context
        float sc[Geo::kSub][G];
#pragma unroll
        for (int i = 0; i < Geo::kSub; ++i) {
            const int row = (c0 + i) * RPI + rg;
            const uint4 raw = *reinterpret_cast<const uint4 *>(sk + row * Geo::kRowBytes + cl * 16);
            float kf[8];
            unpack8(raw, kf);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) d = fmaf(q[g][e], kf[e], d);
                sc[i][g] = d;
            }
        }
#pragma unroll
        for (int i = 0; i < Geo::kSub; ++i)
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int o = LPR / 2; o >= 1; o >>= 1) sc[i][g] += __shfl_xor_sync(kFullMask, sc[i][g], o);

        float mx[G];
#pragma unroll
        for (int g = 0; g < G; ++g) mx[g] = -CUDART_INF_F;
#pragma unroll
        for (int i = 0; i < Geo::kSub; ++i) {
            const bool valid = (c0 + i) * RPI + rg < rows;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                sc[i][g] = valid ? sc[i][g] : -CUDART_INF_F;
                mx[g] = fmaxf(mx[g], sc[i][g]);
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int o = LPR; o < 32; o <<= 1) mx[g] = fmaxf(mx[g], __shfl_xor_sync(kFullMask, mx[g], o));
            // row 0 of this sub-step is valid, so mx and the new max are finite
            const float mn = fmaxf(m[g], mx[g]);
            const float corr = exp2f(m[g] - mn);  // m = -inf at a piece's start -> 0
            m[g] = mn;
            l[g] *= corr;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[g][e] *= corr;
        }
#pragma unroll
        for (int i = 0; i < Geo::kSub; ++i) {
            const int row = (c0 + i) * RPI + rg;
            float pr[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                pr[g] = exp2f(sc[i][g] - m[g]);  // masked rows: exp2(-inf) = 0
                l[g] += pr[g];
            }
            if (row < rows) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(sv + row * Geo::kRowBytes + cl * 16);
                float vf[8];
                unpack8(raw, vf);
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[g][e] = fmaf(pr[g], vf[e], acc[g][e]);
            }
        }
    }
}

// Counts one more piece of a segment in for this call; returns the count.
__device__ __forceinline__ int count_piece(unsigned long long *cnt, uint32_t generation) {
    unsigned long long cur = atomicAdd(cnt, 0ull);
#pragma unroll 1
    while (true) {
        const unsigned long long want =
            ((uint32_t)(cur >> 32) == generation) ? cur + 1 : (((unsigned long long)generation << 32) | 1ull);
        const unsigned long long prev = atomicCAS(cnt, cur, want);
        if (prev == cur) return (int)(want & 0xffffffffull);
        cur = prev;
    }
}

// Where a worker warp is: what finish_piece needs besides the piece itself.
struct WorkerCtx {
    const int *cum;   // chunk prefix sums (shared memory)
    int64_t W;        // workers in the grid
    int64_t T;        // chunks in the batch
    int64_t wid;      // this worker
    int rows_per_chunk;
};

// One warp merges the pieces of a cut segment:
// M = max_p m_p;  out = sum_p acc_p 2^(m_p - M) / sum_p l_p 2^(m_p - M).
template <int D, int G>
__device__ __forceinline__ void merge_segment(const DecodeParams &p, int s, int kvh, int64_t g0, int64_t wa,
                                           int64_t wb, int64_t W, int64_t T, int lane) {
    constexpr int PER = D / 32;  // output elements per lane and head
#pragma unroll 1
    for (int g = 0; g < G; ++g) {
        float M = -CUDART_INF_F;
        for (int64_t w = wa; w <= wb; ++w) {
            const int64_t st = worker_start(w, W, T);
            if (st == worker_start(w + 1, W, T)) continue;
            const int64_t b = (w * 2 + partial_slot(st, g0)) * G + g;
            M = fmaxf(M, __ldcg(p.ws_ml + b * 2));
        }
        float L = 0.f, O[PER];
#pragma unroll
        for (int k = 0; k < PER; ++k) O[k] = 0.f;
        for (int64_t w = wa; w <= wb; ++w) {
            const int64_t st = worker_start(w, W, T);
            if (st == worker_start(w + 1, W, T)) continue;
            const int64_t b = (w * 2 + partial_slot(st, g0)) * G + g;
            const float f = exp2f(__ldcg(p.ws_ml + b * 2) - M);
            L = fmaf(__ldcg(p.ws_ml + b * 2 + 1), f, L);
            const float *src = p.ws_acc + b * D + lane * PER;
#pragma unroll
            for (int k = 0; k < PER; ++k) O[k] = fmaf(__ldcg(src + k), f, O[k]);
        }
        __half *dst = p.out + ((int64_t)s * p.num_heads + kvh * G + g) * D + lane * PER;
#pragma unroll
        for (int k = 0; k < PER; ++k) dst[k] = __float2half_rn(O[k] / L);
    }
}

// Finish a piece: fold the row groups of the warp together, then write the
// output row (whole segment) or the partial (cut segment); the last piece of
// a cut segment to arrive merges the segment.
template <int D, int G>
__device__ __forceinline__ void finish_piece(const DecodeParams &p, const WorkerCtx &wc, const int4 md,
                                             const float (&m)[G], float (&l)[G], float (&acc)[G][8],
                                             int lane) {
    constexpr int LPR = D / 8;
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            l[g] += __shfl_xor_sync(kFullMask, l[g], o);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[g][e] += __shfl_xor_sync(kFullMask, acc[g][e], o);
        }
    }
    const int s = md.x, kvh = md.y, flags = md.w;
    if (flags & kWhole) {
        if (lane < LPR) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float o8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = acc[g][e] / l[g];
                __half *dst = p.out + ((int64_t)s * p.num_heads + kvh * G + g) * D + lane * 8;
                *reinterpret_cast<uint4 *>(dst) = pack8(o8);
            }
        }
        return;
    }
    const int64_t base = (wc.wid * 2 + ((flags & kSlot1) ? 1 : 0)) * G;
    if (lane < LPR) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float4 *dst = reinterpret_cast<float4 *>(p.ws_acc + (base + g) * D + lane * 8);
            dst[0] = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
            dst[1] = make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            p.ws_ml[(base + g) * 2] = m[g];
            p.ws_ml[(base + g) * 2 + 1] = l[g];
        }
    }
    // make the partial visible device-wide, then count it in
    __threadfence();
    __syncwarp();
    const int nch = (wc.cum[s + 1] - wc.cum[s]) / p.num_kv_heads;
    const int64_t g0 = wc.cum[s] + (int64_t)kvh * nch;
    const int64_t wa = worker_of(g0, wc.W, wc.T);
    const int64_t wb = worker_of(g0 + nch - 1, wc.W, wc.T);
    int pieces = 0;
    for (int64_t w = wa; w <= wb; ++w) pieces += worker_start(w, wc.W, wc.T) < worker_start(w + 1, wc.W, wc.T);
    int arrived = 0;
    if (lane == 0) arrived = count_piece(p.ws_count + (int64_t)s * p.num_kv_heads + kvh, p.generation);
    arrived = __shfl_sync(kFullMask, arrived, 0);
    if (arrived == pieces) {
        __threadfence();
        merge_segment<D, G>(p, s, kvh, g0, wa, wb, wc.W, wc.T, lane);
        // every piece of this call has arrived: leave the counter at zero, so
        // that a replay of the same launch (same tag) starts from a clean count
        if (lane == 0) atomicExch(p.ws_count + (int64_t)s * p.num_kv_heads + kvh, 0ull);
    }
}

template <int D, int BS, int G, int NW, int ST>
__global__ void __launch_bounds__(NW * 32) paged_decode_kernel(const DecodeParams p) {
    using Geo = DecodeGeometry<D, BS, G>;
    using Smem = DecodeSmem<NW, ST, Geo::kStageBytes>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int warp_sums[32];
    __shared__ int grand_total;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Smem::kBars);
    int4 *meta = reinterpret_cast<int4 *>(smem + Smem::kMeta);
    int *cum = reinterpret_cast<int *>(smem + Smem::kCum);
    const int N = p.num_seqs;
    int *ctx = cum + N + 1;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int Hkv = p.num_kv_heads;
    const int max_ctx = p.max_blocks_per_seq * BS;

    // ---- prologue: chunk counts per sequence and their prefix sums ----------
    const int per = (N + NW * 32 - 1) / (NW * 32);
    const int s_lo = min(N, tid * per);
    const int s_hi = min(N, s_lo + per);
    int local = 0;
    for (int s = s_lo; s < s_hi; ++s) {
        int c = p.context_lens[s];
        if (c < 0 || c > max_ctx) {
            report(p.status, PKV_ERR_OUT_OF_RANGE);
            c = c < 0 ? 0 : max_ctx;
        }
        ctx[s] = c;
        local += Hkv * chunks_for(c, Geo::kRows);
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    if (tid == 0) {
        for (int i = 0; i < NW * ST; ++i) mbar_init(smem_addr(bars + i), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (warp == 0) {
        const int v = lane < NW ? warp_sums[lane] : 0;
        int vi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFullMask, vi, o);
            if (lane >= o) vi += y;
        }
        warp_sums[lane] = vi - v;
        if (lane == 31) grand_total = vi;
    }
    __syncthreads();
    {
        int run = warp_sums[warp] + incl - local;
        for (int s = s_lo; s < s_hi; ++s) {
            cum[s] = run;
            run += Hkv * chunks_for(ctx[s], Geo::kRows);
        }
        if (tid == 0) cum[N] = grand_total;
    }
    __syncthreads();
    // rows of empty contexts are zero; no worker visits them
    for (int s = blockIdx.x; s < N; s += gridDim.x) {
        if (ctx[s] != 0) continue;
        uint4 *row = reinterpret_cast<uint4 *>(p.out + (int64_t)s * p.num_heads * D);
        for (int i = tid; i < p.num_heads * D / 8; i += NW * 32) row[i] = make_uint4(0, 0, 0, 0);
    }

    // ---- this warp's share of the chunks -----------------------------------
    const int64_t T = cum[N];
    const int64_t W = (int64_t)gridDim.x * NW;
    const int64_t wid = (int64_t)blockIdx.x * NW + warp;
    const int64_t gb = worker_start(wid, W, T);
    const int64_t ge = worker_start(wid + 1, W, T);
    if (gb >= ge) return;
    const int n = (int)(ge - gb);
    const WorkerCtx wc{cum, W, T, wid, Geo::kRows};

    unsigned char *wst = smem + (size_t)warp * ST * Geo::kStageBytes;
    const uint32_t wst_a = smem_addr(wst);
    const uint32_t bar_a = smem_addr(bars + warp * ST);
    int4 *wmeta = meta + warp * ST;

    // block-table entry of chunk g (raw; validated when used), 0 past the share
    auto table_entry = [&](int64_t g) -> int {
        if (g >= ge) return 0;
        const ChunkPos q = locate_chunk(cum, N, Hkv, g);
        const int lb = chunk_block(q.c, BS, Geo::kRows);
        return __ldg(p.block_tables + (int64_t)q.s * p.max_blocks_per_seq + lb);
    };
    int64_t win = gb;
    int tab_cur = table_entry(gb + lane);
    int tab_nxt = table_entry(gb + 32 + lane);
    ChunkPos pos = locate_chunk(cum, N, Hkv, gb);  // next chunk to issue

    auto issue = [&](int i) {
        const int64_t g = gb + i;
        if (g - win >= 32) {
            win += 32;
            tab_cur = tab_nxt;
            tab_nxt = table_entry(win + 32 + lane);
        }
        int phys = __shfl_sync(kFullMask, tab_cur, (int)(g - win));
        if (lane == 0) {
            if (phys < 0 || phys >= p.num_blocks) {
                report(p.status, PKV_ERR_OUT_OF_RANGE);
                phys = 0;
            }
            const int stage = i % ST;
            const int rows = chunk_rows(pos.c, ctx[pos.s], Geo::kRows);
            const int flags = chunk_flags(pos, g, gb, ge);
            wmeta[stage] = make_int4(pos.s, pos.kvh, rows, flags);
            const uint32_t bar = bar_a + stage * 8;
            const uint32_t dst = wst_a + stage * Geo::kStageBytes;
            const uint32_t kv_bytes = (uint32_t)rows * Geo::kRowBytes;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, 2 * kv_bytes + ((flags & kFirst) ? Geo::kQBytes : 0));
            const int64_t off = chunk_src_offset(phys, pos.kvh, pos.c, Hkv, BS, Geo::kRows, D);
            bulk_g2s(dst, p.key_cache + off, kv_bytes, bar);
            bulk_g2s(dst + Geo::kChunkBytes, p.value_cache + off, kv_bytes, bar);
            if (flags & kFirst)
                bulk_g2s(dst + 2 * Geo::kChunkBytes,
                         p.query + ((int64_t)pos.s * p.num_heads + pos.kvh * G) * D, Geo::kQBytes, bar);
        }
    };

    int issued = 0;
    for (; issued < min(ST, n); ++issued) {
        issue(issued);
        if (issued + 1 < n) next_chunk(pos, cum, N, Hkv);
    }

    float q[G][8], m[G], l[G], acc[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -CUDART_INF_F;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) q[g][e] = acc[g][e] = 0.f;
    }
    const int cl = lane % Geo::kLanesPerRow;

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
            return;
        }
        const int4 md = wmeta[stage];
        const unsigned char *sk = wst + stage * Geo::kStageBytes;
        if (md.w & kFirst) {
            const unsigned char *sq = sk + 2 * Geo::kChunkBytes;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(sq + g * D * 2 + cl * 16);
                float f[8];
                unpack8(raw, f);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    q[g][e] = f[e] * p.scale_log2;
                    acc[g][e] = 0.f;
                }
                m[g] = -CUDART_INF_F;
                l[g] = 0.f;
            }
        }
        process_chunk<D, BS, G>(sk, sk + Geo::kChunkBytes, md.z, q, m, l, acc, lane);
        if (md.w & kLast) finish_piece<D, G>(p, wc, md, m, l, acc, lane);
        __syncwarp();
        if (issued < n) {
            issue(issued);
            if (issued + 1 < n) next_chunk(pos, cum, N, Hkv);
            ++issued;
        }
    }
}

}  // namespace pkv

#endif  // PKV_DECODE_IMPL_CUH
