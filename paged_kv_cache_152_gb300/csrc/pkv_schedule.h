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
    kSlot1 = 8,   // partial goes to slot 1 (else slot 0)
    kAppendRow = 16  // (set by the kernel) the chunk's last row is the decode step's new token
};

// a / b for 0 <= a, 0 < b: a 32-bit unsigned division when both fit (the
// usual case; a 64-bit division is a long instruction sequence on the GPU).
PKV_HD int64_t div_nonneg(int64_t a, int64_t b) {
    if (((uint64_t)a | (uint64_t)b) >> 32 == 0) return (int64_t)((uint32_t)a / (uint32_t)b);
    return a / b;
}

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
    p.nch = (int)((unsigned)(cum[p.s + 1] - cum[p.s]) / (unsigned)num_kv_heads);
    const int off = (int)(g - cum[p.s]);
    p.kvh = (int)((unsigned)off / (unsigned)p.nch);
    p.c = off - p.kvh * p.nch;
    return p;
}

// locate_chunk for two chunks at once: the two binary searches run in one
// loop, so their dependent loads overlap.
PKV_HD void locate_chunk2(const int *cum, int n, int num_kv_heads, int64_t g0, int64_t g1, ChunkPos &p0,
                          ChunkPos &p1) {
    int lo0 = 0, hi0 = n, lo1 = 0, hi1 = n;
    while (hi0 - lo0 > 1 || hi1 - lo1 > 1) {
        const int m0 = (lo0 + hi0) >> 1, m1 = (lo1 + hi1) >> 1;
        const bool d0 = hi0 - lo0 > 1, d1 = hi1 - lo1 > 1;
        const int c0 = cum[m0], c1 = cum[m1];
        if (d0) { if (c0 <= g0) lo0 = m0; else hi0 = m0; }
        if (d1) { if (c1 <= g1) lo1 = m1; else hi1 = m1; }
    }
    p0.s = lo0;
    p1.s = lo1;
    p0.nch = (int)((unsigned)(cum[lo0 + 1] - cum[lo0]) / (unsigned)num_kv_heads);
    p1.nch = (int)((unsigned)(cum[lo1 + 1] - cum[lo1]) / (unsigned)num_kv_heads);
    const int off0 = (int)(g0 - cum[lo0]), off1 = (int)(g1 - cum[lo1]);
    p0.kvh = (int)((unsigned)off0 / (unsigned)p0.nch);
    p1.kvh = (int)((unsigned)off1 / (unsigned)p1.nch);
    p0.c = off0 - p0.kvh * p0.nch;
    p1.c = off1 - p1.kvh * p1.nch;
}

// Step to chunk g+1 (which must exist).
PKV_HD void next_chunk(ChunkPos &p, const int *cum, int n, int num_kv_heads) {
    if (++p.c < p.nch) return;
    p.c = 0;
    if (++p.kvh < num_kv_heads) return;
    p.kvh = 0;
    do { ++p.s; } while (p.s < n - 1 && cum[p.s + 1] == cum[p.s]);
    p.nch = (int)((unsigned)(cum[p.s + 1] - cum[p.s]) / (unsigned)num_kv_heads);
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

// Two-level split.  The T chunks are first divided among C CTAs: CTA c's
// nominal start c*T/C moves to the nearest segment boundary when one lies
// within snap = min(T/(4C), snap_cap) chunks, so that fewer segments are read
// by two CTAs (moving a boundary by d chunks costs the CTA's warps d/NW
// chunks each; a segment cut across CTAs costs a device-wide count and a
// merge of the CTAs' parts, worth about a chunk per warp -- hence a small
// absolute cap, one chunk per warp in the decode kernel).  Each
// CTA's range is then divided equally among its NW warps: worker w = c*NW + k.
// *cuts (if given) tells whether the start lies inside a segment.
PKV_HD int64_t snapped_cta_start(const int *cum, int n, int num_kv_heads, int64_t c, int64_t C, int64_t T,
                                 int64_t snap_cap, bool *cuts = nullptr) {
    if (cuts) *cuts = false;
    const int64_t nominal = div_nonneg(c * T, C);
    if (c == 0 || nominal >= T) return nominal >= T ? T : 0;
    const ChunkPos p = locate_chunk(cum, n, num_kv_heads, nominal);
    const int64_t g0 = nominal - p.c;          // segment's first chunk
    const int64_t g1 = g0 + p.nch;             // one past its last
    const int64_t quarter = div_nonneg(T, 4 * C);
    const int64_t snap = quarter < snap_cap ? quarter : snap_cap;
    const int64_t left = nominal - g0, right = g1 - nominal;
    if (left == 0) return nominal;
    if (left <= right && left <= snap) return g0;
    if (right < left && right <= snap) return g1;
    if (cuts) *cuts = true;
    return nominal;
}

// Start of worker k (0 <= k <= nw) of a CTA whose range is [a, a + len):
// equal shares, except that the first worker gives up r0 chunks and the last
// r1, spread evenly over the workers between them (nw >= 3).  A worker whose
// piece is cut across a CTA boundary also counts that piece in device-wide
// and may merge the CTAs' parts -- a few round trips to L2 that its share
// makes up for.  Callers pass r0, r1 <= len / (2 nw) (cut_relief), so starts
// never decrease.
PKV_HD int64_t cta_share_start(int64_t a, int64_t len, int nw, int k, int r0, int r1) {
    const int64_t st = a + ((int64_t)k * len) / nw;
    if (k == 0 || k == nw || nw < 3) return st;
    return st - r0 + ((int64_t)(k - 1) * (r0 + r1)) / (nw - 2);
}

// Relief for one end of a CTA range of len chunks when the CTA boundary at
// chunk b (0 < b < T) lies inside a segment: `relief` chunks, but at most
// 1/div of a nominal share (the cut costs a fixed time, so short shares give
// up less); else 0.  div >= 2.
// The same, given whether the boundary cuts a segment (snapped_cta_start
// tells).
PKV_HD int cut_relief_for(bool cuts, int64_t len, int nw, int relief, int div) {
    if (!cuts || relief <= 0 || nw < 3) return 0;
    const int64_t cap = len / ((int64_t)div * nw);
    return cap < relief ? (int)cap : relief;
}

PKV_HD int cut_relief(const int *cum, int n, int num_kv_heads, int64_t b, int64_t T, int64_t len, int nw,
                      int relief, int div) {
    if (relief <= 0 || nw < 3 || b <= 0 || b >= T) return 0;
    return cut_relief_for(locate_chunk(cum, n, num_kv_heads, b).c != 0, len, nw, relief, div);
}

// The worker k of a CTA (0 <= k < NW) whose share holds chunk g, given the
// CTA's NW + 1 worker starts (the last one when empty shares start at g).
template <int NW>
PKV_HD int worker_in_starts(const int64_t *starts, int64_t g) {
    int k = 0;
    for (int j = 1; j < NW; ++j) k += starts[j] <= g ? 1 : 0;
    return k;
}

// The CTA whose range holds chunk g (0 <= g < T): `hint` when it does, else
// the largest c with bounds[c] <= g.
PKV_HD int cta_of(const int64_t *bounds, int C, int64_t g, int hint) {
    if (bounds[hint] <= g && g < bounds[hint + 1]) return hint;
    int lo = 0, hi = C;  // bounds[lo] <= g < bounds[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (bounds[mid] <= g) lo = mid; else hi = mid;
    }
    return lo;
}

// The order in which a worker walks its share [gb, ge): its cut pieces first
// -- the last piece (when it runs past ge), then the first piece (when it
// starts before gb) -- then everything between them in chunk order.  The
// other pieces of a cut segment sit at the starts and ends of neighbouring
// shares, so with every worker doing the same, cut segments complete early
// and their merges are ready long before the tail.  Pieces stay contiguous runs
// of the walk, so chunk_flags is unchanged.
struct ShareOrder {
    int64_t a0, a1;   // range 1: the cut last piece (empty if none)
    int64_t b0, b1;   // range 2: the cut first piece (empty if none)
    int64_t c0, c1;   // range 3: the rest, in order

    PKV_HD int64_t size() const { return (a1 - a0) + (b1 - b0) + (c1 - c0); }

    // chunk at position i of the walk (0 <= i < size())
    PKV_HD int64_t at(int64_t i) const {
        const int64_t na = a1 - a0, nb = b1 - b0;
        if (i < na) return a0 + i;
        if (i < na + nb) return b0 + (i - na);
        return c0 + (i - na - nb);
    }

    // true if position i starts a range (the walk jumps there)
    PKV_HD bool jumps_at(int64_t i) const {
        const int64_t na = a1 - a0, nb = b1 - b0;
        return i == 0 || i == na || i == na + nb;
    }
};

// The walk of a non-empty share [gb, ge) given where its first chunk (gb)
// and its last (ge - 1) lie (only c and nch of each are used).
PKV_HD ShareOrder share_order_at(const ChunkPos &first, const ChunkPos &last, int64_t gb, int64_t ge) {
    ShareOrder o;
    o.a0 = o.a1 = o.b0 = o.b1 = gb;
    o.c0 = gb;
    o.c1 = ge;
    const int64_t first_seg_end = gb + (first.nch - first.c);   // one past the first segment
    const int64_t last_seg_start = (ge - 1) - last.c;           // the last segment's first chunk
    if (first_seg_end >= ge) return o;  // the share lies inside one segment: one piece
    const bool last_cut = last.c < last.nch - 1;
    const bool first_cut = first.c > 0;
    if (last_cut) {
        o.a0 = last_seg_start;
        o.a1 = ge;
        o.c1 = last_seg_start;
    }
    if (first_cut) {
        o.b0 = gb;
        o.b1 = first_seg_end;
        o.c0 = first_seg_end;
    }
    if (o.c0 > o.c1) o.c0 = o.c1;
    return o;
}

PKV_HD ShareOrder share_order(const int *cum, int n, int num_kv_heads, int64_t gb, int64_t ge) {
    if (gb >= ge) {
        ShareOrder o;
        o.a0 = o.a1 = o.b0 = o.b1 = gb;
        o.c0 = gb;
        o.c1 = ge;
        return o;
    }
    return share_order_at(locate_chunk(cum, n, num_kv_heads, gb), locate_chunk(cum, n, num_kv_heads, ge - 1), gb,
                          ge);
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
