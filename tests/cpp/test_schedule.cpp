// Exhaustive CPU check of the decode kernel's work split (pkv_schedule.h).
// Built and run by tests/test_native_host.py.  Exits non-zero on the first
// violation, printing it.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <vector>
#include <random>
#include <map>
#include <set>

#include "pkv_schedule.h"

using namespace pkv;

static int fails = 0;
static long relieved = 0;  // CTA ends where a relief applied (the test must exercise it)
#define CHECK(c, ...) do { if (!(c)) { std::printf("FAIL %s:%d: ", __FILE__, __LINE__); \
    std::printf(__VA_ARGS__); std::printf("\n"); if (++fails > 5) std::exit(1); } } while (0)

// split 0: equal shares over all W workers; split 1: snapped CTA ranges of
// nw workers each (W = C * nw), divided equally (relief 0) or with the first
// and last worker giving up `relief` chunks where their CTA boundary cuts a
// segment.
static void run_case_split(const std::vector<int> &ctx, int hkv, int bs, int sr, int mb, int64_t W, int split,
                           int nw, int relief = 0);

static void run_case(const std::vector<int> &ctx, int hkv, int bs, int sr, int mb, int64_t W) {
    run_case_split(ctx, hkv, bs, sr, mb, W, 0, 1);
    for (int nw : {1, 3, 8}) run_case_split(ctx, hkv, bs, sr, mb, ((W + nw - 1) / nw) * nw, 1, nw);
    for (int nw : {3, 8})
        for (int relief : {1, 2, 1000}) run_case_split(ctx, hkv, bs, sr, mb, ((W + nw - 1) / nw) * nw, 1, nw, relief);
}

template <int NW>
static int worker_in_starts_rt(int nw, const int64_t *starts, int64_t g) {
    CHECK(nw == NW, "nw");
    return worker_in_starts<NW>(starts, g);
}

static void run_case_split(const std::vector<int> &ctx, int hkv, int bs, int sr, int mb, int64_t W, int split,
                           int nw, int relief) {
    const int n = (int)ctx.size();
    std::vector<int> cum(n + 1, 0);
    for (int s = 0; s < n; ++s) cum[s + 1] = cum[s] + hkv * chunks_for(ctx[s], sr);
    const int64_t T = cum[n];
    // brute-force owner of each chunk: (s, kvh, c)
    std::vector<ChunkPos> truth;
    for (int s = 0; s < n; ++s)
        for (int h = 0; h < hkv; ++h)
            for (int c = 0; c < chunks_for(ctx[s], sr); ++c)
                truth.push_back({s, h, c, chunks_for(ctx[s], sr)});
    CHECK((int64_t)truth.size() == T, "T");
    if (T == 0) return;
    const int C = (int)(W / nw);
    const int64_t snap_cap = nw;  // as in the decode kernel
    std::vector<int64_t> bounds(C + 1);
    if (split == 1) {
        for (int c = 0; c <= C; ++c)
            bounds[c] = c == C ? T : snapped_cta_start(cum.data(), n, hkv, c, C, T, snap_cap);
        for (int c = 0; c < C; ++c) CHECK(bounds[c] <= bounds[c + 1], "cta bounds not monotonic");
        // the reported cut, and the relief derived from it, match a fresh look-up
        for (int c = 0; c <= C; ++c) {
            bool cuts = true;
            const int64_t b = c == C ? T : snapped_cta_start(cum.data(), n, hkv, c, C, T, snap_cap, &cuts);
            if (c == C) cuts = false;
            const bool want = b > 0 && b < T && locate_chunk(cum.data(), n, hkv, b).c != 0;
            CHECK(cuts == want, "cut flag of cta %d start %lld", c, (long long)b);
            for (int64_t len : {(int64_t)0, (int64_t)17, (int64_t)1000})
                CHECK(cut_relief_for(cuts, len, nw, 3, 4) == cut_relief(cum.data(), n, hkv, b, T, len, nw, 3, 4),
                      "cut_relief_for");
        }
        // a CTA boundary inside a segment could not snap: both ends are far
        for (int c = 1; c < C; ++c) {
            const int64_t b = bounds[c];
            if (b <= 0 || b >= T) continue;
            const ChunkPos p = locate_chunk(cum.data(), n, hkv, b);
            if (p.c == 0) continue;
            const int64_t snap = std::min<int64_t>(T / (4 * (int64_t)C), snap_cap);
            CHECK(p.c > snap && p.nch - p.c > snap, "boundary left inside a short segment");
        }
    }
    // reliefs of each CTA's first and last worker
    std::vector<int> r0(C, 0), r1(C, 0);
    if (split == 1 && relief > 0) {
        for (int c = 0; c < C; ++c) {
            const int64_t a = bounds[c], len = bounds[c + 1] - a;
            r0[c] = cut_relief(cum.data(), n, hkv, a, T, len, nw, relief, 2);
            r1[c] = cut_relief(cum.data(), n, hkv, a + len, T, len, nw, relief, 2);
            relieved += (r0[c] > 0) + (r1[c] > 0);
            for (int end = 0; end < 2; ++end) {
                const int r = end ? r1[c] : r0[c];
                const int64_t b = end ? a + len : a;
                const bool cuts = b > 0 && b < T && locate_chunk(cum.data(), n, hkv, b).c != 0;
                const int64_t cap = nw >= 3 ? std::min<int64_t>(relief, len / (2 * nw)) : 0;
                CHECK(r == (cuts ? cap : 0), "relief %d at boundary %lld", r, (long long)b);
            }
            CHECK(cta_share_start(a, len, nw, 0, r0[c], r1[c]) == a &&
                      cta_share_start(a, len, nw, nw, r0[c], r1[c]) == a + len,
                  "relief shares do not span the CTA range");
            // the first and last worker give up exactly their relief
            if (nw >= 3) {
                CHECK(cta_share_start(a, len, nw, 1, r0[c], r1[c]) == a + len / nw - r0[c], "first share");
                CHECK(cta_share_start(a, len, nw, nw - 1, r0[c], r1[c]) == a + ((nw - 1) * len) / nw + r1[c],
                      "last share");
            }
        }
    }
    // each CTA's worker starts, as the kernel's warps compute them (the
    // merges look workers up in this array)
    std::vector<int64_t> starts(split == 1 ? (size_t)C * (nw + 1) : 0);
    for (int c = 0; split == 1 && c < C; ++c) {
        const int64_t a = bounds[c], len = bounds[c + 1] - a;
        for (int k = 0; k <= nw; ++k) {
            starts[(size_t)c * (nw + 1) + k] = cta_share_start(a, len, nw, k, r0[c], r1[c]);
            if (relief == 0)  // equal shares
                CHECK(starts[(size_t)c * (nw + 1) + k] == a + (k * len) / nw, "equal share %d of cta %d", k, c);
        }
    }
    auto wstart = [&](int64_t w) -> int64_t {
        if (split == 0) return worker_start(w, W, T);
        if (w >= W) return T;
        return starts[(size_t)(w / nw) * (nw + 1) + w % nw];
    };
    auto wof = [&](int64_t g) -> int64_t {
        if (split == 0) return worker_of(g, W, T);
        const int c = cta_of(bounds.data(), C, g, 0);
        const int64_t *st = starts.data() + (size_t)c * (nw + 1);
        const int k = nw == 1 ? worker_in_starts_rt<1>(nw, st, g)
                    : nw == 3 ? worker_in_starts_rt<3>(nw, st, g) : worker_in_starts_rt<8>(nw, st, g);
        return (int64_t)c * nw + k;
    };
    // ranges partition [0, T)
    std::vector<int> owner(T, -1);
    for (int64_t w = 0; w < W; ++w) {
        const int64_t st = wstart(w), en = wstart(w + 1);
        CHECK(st <= en, "range order");
        for (int64_t g = st; g < en; ++g) { CHECK(owner[g] == -1, "overlap"); owner[g] = (int)w; }
    }
    for (int64_t g = 0; g < T; ++g) {
        CHECK(owner[g] >= 0, "uncovered chunk %lld", (long long)g);
        CHECK(wof(g) == owner[g], "worker_of(%lld)=%lld want %d (split %d)", (long long)g, (long long)wof(g),
              owner[g], split);
        if (split == 1) {
            // the CTA look-up, from several hint CTAs
            for (int hint = 0; hint < C; hint += (C > 16 ? C / 7 : 1)) {
                const int c = cta_of(bounds.data(), C, g, hint);
                CHECK(bounds[c] <= g && g < bounds[c + 1], "cta_of(%lld, hint %d)", (long long)g, hint);
            }
        }
        {
            // the two-key search agrees with two single ones
            const int64_t g2 = (g * 7919) % T;
            ChunkPos a2, b2;
            locate_chunk2(cum.data(), n, hkv, g, g2, a2, b2);
            const ChunkPos t2 = truth[g2];
            CHECK(a2.s == truth[g].s && a2.kvh == truth[g].kvh && a2.c == truth[g].c && a2.nch == truth[g].nch &&
                      b2.s == t2.s && b2.kvh == t2.kvh && b2.c == t2.c && b2.nch == t2.nch,
                  "locate_chunk2(%lld, %lld)", (long long)g, (long long)g2);
        }
        const ChunkPos p = locate_chunk(cum.data(), n, hkv, g);
        CHECK(p.s == truth[g].s && p.kvh == truth[g].kvh && p.c == truth[g].c && p.nch == truth[g].nch,
              "locate %lld", (long long)g);
        // addressing stays inside the table row and the block
        const int lb = chunk_block(p.c, bs, sr);
        CHECK(lb >= 0 && lb < mb, "logical block %d outside table of %d", lb, mb);
        const int rows = chunk_rows(p.c, ctx[p.s], sr);
        CHECK(rows >= 1 && rows <= sr, "rows %d", rows);
        CHECK(p.c * sr + rows <= ctx[p.s], "chunk past context");
        const int nb = 7;
        if (bs >= sr) {
            const int row0 = (p.c * sr) % bs;
            CHECK(row0 + rows <= bs, "chunk crosses block");
            for (int phys : {0, nb - 1}) {
                const int64_t off = chunk_src_offset(phys, p.kvh, p.c, hkv, bs, sr, 64);
                CHECK(off >= 0 && off + (int64_t)rows * 64 <= (int64_t)nb * hkv * bs * 64, "src offset");
            }
        } else {
            // small blocks: the chunk's rows fill whole blocks lb, lb+1, ... (one
            // 8-row box each), all inside the table row
            CHECK(sr % bs == 0 && (p.c * sr) % bs == 0, "chunk not block-aligned");
            const int last_lb = (p.c * sr + rows - 1) / bs;
            CHECK(last_lb < mb && last_lb - lb < sr / bs, "chunk's blocks %d..%d outside table of %d", lb,
                  last_lb, mb);
        }
    }
    // walk every worker as the kernel does; record pieces and partial slots
    std::map<std::pair<int, int>, std::vector<std::pair<int64_t, int>>> partials;  // seg -> (worker, slot)
    std::set<std::pair<int, int>> whole_done;
    for (int64_t w = 0; w < W; ++w) {
        const int64_t gb = wstart(w), ge = wstart(w + 1);
        if (gb == ge) continue;
        ChunkPos p = locate_chunk(cum.data(), n, hkv, gb);
        bool in_piece = false;
        int64_t piece_start = 0;
        int slots_used[2] = {0, 0};
        for (int64_t g = gb; g < ge; ++g) {
            const ChunkPos q = locate_chunk(cum.data(), n, hkv, g);
            CHECK(p.s == q.s && p.kvh == q.kvh && p.c == q.c && p.nch == q.nch, "walk at %lld", (long long)g);
            const int f = chunk_flags(p, g, gb, ge);
            const bool seg_start = (g == gb) || (locate_chunk(cum.data(), n, hkv, g - 1).s != p.s ||
                                                 locate_chunk(cum.data(), n, hkv, g - 1).kvh != p.kvh);
            CHECK(((f & kFirst) != 0) == seg_start, "first flag");
            if (f & kFirst) { CHECK(!in_piece, "nested piece"); in_piece = true; piece_start = g; }
            CHECK(in_piece, "chunk outside piece");
            const bool seg_end = (g == ge - 1) || (locate_chunk(cum.data(), n, hkv, g + 1).s != p.s ||
                                                   locate_chunk(cum.data(), n, hkv, g + 1).kvh != p.kvh);
            CHECK(((f & kLast) != 0) == seg_end, "last flag");
            if (f & kLast) {
                const int64_t g0 = g - p.c, g1 = g0 + p.nch;
                const bool whole = piece_start == g0 && g + 1 == g1;
                CHECK(((f & kWhole) != 0) == whole, "whole flag");
                const auto seg = std::make_pair(p.s, p.kvh);
                if (whole) {
                    CHECK(!whole_done.count(seg), "segment finished twice");
                    whole_done.insert(seg);
                } else {
                    const int slot = (f & kSlot1) ? 1 : 0;
                    CHECK(slot == (piece_start == gb ? 0 : 1), "slot rule");
                    CHECK(slot == 0 || g == ge - 1, "slot 1 only for the last piece");
                    CHECK(slots_used[slot] == 0, "slot %d used twice by worker %lld", slot, (long long)w);
                    slots_used[slot] = 1;
                    partials[seg].push_back({w, slot});
                }
                in_piece = false;
            }
            if (g + 1 < ge) next_chunk(p, cum.data(), n, hkv);
        }
        CHECK(!in_piece, "unterminated piece");
    }
    // the reordered walk visits every chunk of the share once, keeps each piece
    // a contiguous run that starts with its kFirst chunk and ends with its
    // kLast chunk, and puts cut pieces before whole ones
    for (int64_t w = 0; w < W; ++w) {
        const int64_t gb = wstart(w), ge = wstart(w + 1);
        const ShareOrder so = share_order(cum.data(), n, hkv, gb, ge);
        CHECK(so.size() == ge - gb, "order size");
        std::vector<int> seen(ge - gb + 1, 0);
        bool in_piece = false, seen_whole = false;
        for (int64_t i = 0; i < so.size(); ++i) {
            const int64_t g = so.at(i);
            CHECK(g >= gb && g < ge, "order outside share");
            if (g < gb || g >= ge) break;
            CHECK(seen[g - gb] == 0, "chunk visited twice");
            seen[g - gb] = 1;
            const ChunkPos p = locate_chunk(cum.data(), n, hkv, g);
            const int f = chunk_flags(p, g, gb, ge);
            if (i > 0 && !so.jumps_at(i)) {
                const ChunkPos q = locate_chunk(cum.data(), n, hkv, so.at(i - 1));
                ChunkPos nx = q;
                next_chunk(nx, cum.data(), n, hkv);
                CHECK(nx.s == p.s && nx.kvh == p.kvh && nx.c == p.c, "walk step");
            }
            if (f & kFirst) { CHECK(!in_piece, "piece not contiguous"); in_piece = true; }
            CHECK(in_piece, "chunk before its piece's first");
            if (f & kLast) {
                in_piece = false;
                if (f & kWhole) seen_whole = true;
                else CHECK(!seen_whole, "cut piece after a whole one");
            }
        }
        CHECK(!in_piece, "order ends inside a piece");
    }
    // the merge queue of a CTA (32 entries in the decode kernel) receives one
    // entry per cut segment whose part lies in the CTA's range: at most nw + 1
    // (a cut segment holds a worker or CTA boundary of the range)
    if (split == 1) {
        std::vector<int> queued(C, 0);
        for (int s = 0; s < n; ++s) {
            const int nch = chunks_for(ctx[s], sr);
            for (int h = 0; h < hkv && nch > 0; ++h) {
                const int64_t g0 = cum[s] + (int64_t)h * nch, g1 = g0 + nch;
                if (wof(g0) == wof(g1 - 1)) continue;  // one piece: not cut
                for (int c = 0; c < C; ++c)
                    if (g0 < bounds[c + 1] && g1 > bounds[c]) ++queued[c];
            }
        }
        for (int c = 0; c < C; ++c)
            CHECK(queued[c] <= nw + 1 && queued[c] <= 32, "cta %d queues %d merges (nw %d)", c, queued[c], nw);
    }
    // the merge kernel finds exactly the stored partials of every cut segment
    for (int s = 0; s < n; ++s) {
        const int nch = chunks_for(ctx[s], sr);
        for (int h = 0; h < hkv; ++h) {
            const auto seg = std::make_pair(s, h);
            if (nch == 0) { CHECK(!partials.count(seg) && !whole_done.count(seg), "empty seg touched"); continue; }
            const int64_t g0 = cum[s] + (int64_t)h * nch, g1 = g0 + nch;
            const int64_t wa = wof(g0), wb = wof(g1 - 1);
            if (wa == wb) { CHECK(whole_done.count(seg) && !partials.count(seg), "uncut seg %d,%d", s, h); continue; }
            CHECK(!whole_done.count(seg), "cut seg written whole");
            std::vector<std::pair<int64_t, int>> found;
            for (int64_t w = wa; w <= wb; ++w) {
                const int64_t st = wstart(w), en = wstart(w + 1);
                if (st == en) continue;
                found.push_back({w, partial_slot(st, g0)});
            }
            CHECK(found == partials[seg], "merge pieces of seg %d,%d", s, h);
        }
    }
}

int main() {
    std::mt19937_64 rng(152);
    int cases = 0;
    const int bss[] = {8, 16, 32, 64, 128};
    for (int it = 0; it < 3000; ++it) {
        const int bs = bss[rng() % 5];
        const int sr = 16;  // rows per chunk, as in the decode kernel
        const int n = 1 + (int)(rng() % 40);
        const int hkv = 1 + (int)(rng() % 4);
        const int maxctx = 1 + (int)(rng() % 600);
        const int mb = (maxctx + bs - 1) / bs;
        std::vector<int> ctx(n);
        for (auto &c : ctx) c = (rng() % 5 == 0) ? 0 : 1 + (int)(rng() % maxctx);
        const int64_t W = 1 + (int64_t)(rng() % 300);
        run_case(ctx, hkv, bs, sr, mb, W);
        ++cases;
    }
    // hand-picked edge cases
    run_case({0, 0, 0}, 2, 16, 16, 1, 4);
    run_case({1}, 1, 16, 16, 1, 1000);
    run_case({0, 5, 0, 0, 17, 0}, 3, 16, 16, 2, 3);
    run_case({4096, 256, 1000}, 8, 32, 16, 128, 1216);
    // the largest batch (4096 sequences): short contexts, some empty, one long
    for (int bs : {16, 128}) {
        std::vector<int> ctx(4096);
        for (auto &c : ctx) c = (rng() % 20 == 0) ? 0 : (int)(rng() % 25);
        ctx[1234] = 3000;
        const int mb = (3000 + bs - 1) / bs;
        run_case(ctx, 1, bs, 16, mb, 1216);
        run_case(ctx, 1, bs, 16, mb, 8);
    }
    CHECK(relieved > 1000, "relief exercised only %ld times", relieved);
    if (fails) { std::printf("%d failures\n", fails); return 1; }
    std::printf("schedule ok: %d random cases (%ld relieved CTA ends)\n", cases, relieved);
    return 0;
}
