// pkv_schedule.h -- work split of the persistent decode kernel.
//
// Host and device share these functions, so the host test binary
// (tests/cpp/test_schedule.cpp) can check them exhaustively on the CPU.
//
// The decode work is cut into CHUNKS: up to `rows_per_chunk` consecutive
// tokens of one (sequence, KV head) SEGMENT.  A chunk never crosses a block
// boundary (rows_per_chunk divides block_size), so one chunk is one
// contiguous run of rows * head_dim fp16 values in each cache -- one bulk copy.
// Chunks are numbered sequence-major, then KV head, then position:
//
//   g = cum[s] + kvh * nch[s] + c,   nch[s] = ceil(ctx[s] / rows_per_chunk),
//   cum[0] = 0, cum[s+1] = cum[s] + num_kv_heads * nch[s],  T = cum[N].
//
// W workers (one per warp) each take one contiguous, equal share:
// worker w owns chunks [worker_start(w), worker_start(w+1)).  A worker walks
// its chunks in order; each maximal run of its chunks inside one segment is a
// PIECE.  A piece that is a whole segment is finished by the worker itself.
// Otherwise the worker stores a partial (running max, sum, unnormalised
// output) in slot 0 if the piece holds the worker's first chunk, else in slot
// 1 (only the first and the last piece of a worker can be partial); the
// last piece of a cut segment to finish merges the segment's pieces.
#ifndef PKV_SCHEDULE_H
#define PKV_SCHEDULE_H

#include <stdint.h>

#if defined(__CUDACC__)
#define PKV_HD __host__ __device__ __forceinline__
#else
#define PKV_HD inline
#endif

namespace pkv {

enum ChunkFlags {
    kFirst = 1,   // first chunk of a piece: reset the softmax state, q arrives
    kLast = 2,    // last chunk of a piece: finish it
    kWhole = 4,   // the piece is a whole segment: write the output row directly
    kSlot1 = 8    // partial goes to slot 1 (else slot 0)
};

PKV_HD int chunks_for(int ctx, int rows_per_chunk) {
    return ctx <= 0 ? 0 : (ctx + rows_per_chunk - 1) / rows_per_chunk;
}

PKV_HD int64_t worker_start(int64_t w, int64_t W, int64_t T) {
    return (w * T) / W;
}

// Largest w with worker_start(w) <= g, for 0 <= g < T.
PKV_HD int64_t worker_of(int64_t g, int64_t W, int64_t T) {
    return ((g + 1) * W + T - 1) / T - 1;
}

// Largest s in [0, n) with cum[s] <= g, given cum[n] > g (cum non-decreasing).
// Lands on the sequence that owns chunk g even when empty sequences share
// the same cum value.
PKV_HD int find_seq(const int *cum, int n, int64_t g) {
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cum[mid] <= g) lo = mid; else hi = mid;
    }
    return lo;
}

struct ChunkPos {
    int s;      // sequence
    int kvh;    // KV head
    int c;      // chunk index inside the segment
    int nch;    // chunks in the segment
};

PKV_HD ChunkPos locate_chunk(const int *cum, int n, int num_kv_heads, int64_t g) {
    ChunkPos p;
    p.s = find_seq(cum, n, g);
    p.nch = (cum[p.s + 1] - cum[p.s]) / num_kv_heads;
    const int off = (int)(g - cum[p.s]);
    p.kvh = off / p.nch;
    p.c = off - p.kvh * p.nch;
    return p;
}

// Step to chunk g+1 (which must exist).
PKV_HD void next_chunk(ChunkPos &p, const int *cum, int n, int num_kv_heads) {
    if (++p.c < p.nch) return;
    p.c = 0;
    if (++p.kvh < num_kv_heads) return;
    p.kvh = 0;
    do { ++p.s; } while (p.s < n - 1 && cum[p.s + 1] == cum[p.s]);
    p.nch = (cum[p.s + 1] - cum[p.s]) / num_kv_heads;
}

// Flags of chunk g (at position p) for the worker owning [gb, ge).
PKV_HD int chunk_flags(const ChunkPos &p, int64_t g, int64_t gb, int64_t ge) {
    const int64_t g0 = g - p.c;          // segment's first chunk
    const int64_t g1 = g0 + p.nch;       // one past its last
    int f = 0;
    if (p.c == 0 || g == gb) f |= kFirst;
    if (p.c == p.nch - 1 || g == ge - 1) f |= kLast;
    if (g0 >= gb && g1 <= ge) f |= kWhole;
    if (g0 > gb) f |= kSlot1;
    return f;
}

// Slot in which worker w (owning [st, en), non-empty) stored its partial for
// a cut segment starting at chunk g0.
PKV_HD int partial_slot(int64_t st, int64_t g0) {
    return st < g0 ? 1 : 0;
}

// Element offset, in either cache, of the first row of chunk c of KV head kvh
// whose block is physical block phys.
PKV_HD int64_t chunk_src_offset(int phys, int kvh, int c, int num_kv_heads,
                                int block_size, int rows_per_chunk, int head_dim) {
    const int row0 = (c * rows_per_chunk) % block_size;
    return (((int64_t)phys * num_kv_heads + kvh) * block_size + row0) * head_dim;
}

// Logical block of chunk c.
PKV_HD int chunk_block(int c, int block_size, int rows_per_chunk) {
    return (c * rows_per_chunk) / block_size;
}

// Rows of chunk c that hold tokens of a context of ctx tokens.
PKV_HD int chunk_rows(int c, int ctx, int rows_per_chunk) {
    const int left = ctx - c * rows_per_chunk;
    return left < rows_per_chunk ? left : rows_per_chunk;
}

}  // namespace pkv

#endif  // PKV_SCHEDULE_H
