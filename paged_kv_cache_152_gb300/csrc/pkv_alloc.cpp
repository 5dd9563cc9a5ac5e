// pkv_alloc.cpp -- the host block manager that produces block tables.
//
// [P1] "Paged Attention: OS-Inspired Memory Management for KV Caches"
// (modernaiengineering.com): "How PagedAttention works" (allocate on demand,
// free on finish), "Memory sharing across requests" (reference counts,
// copy-on-write of a shared partial block), the practice block manager and
// its exercises (fork, release).  [P2] "What is PagedAttention..." (n4n.ai),
// "How PagedAttention works": one global pool handed out block by block.
//
// Swapping: [P2] "Why it matters for KV cache", "Swapping and preemption";
// [P1] "Common misconceptions".  A second pool of host blocks; a swapped-out
// sequence's table names host blocks until it is swapped back in.
//
// Every operation first checks that it can complete (free blocks, ids,
// buffer sizes) and only then mutates, so a failed call changes nothing.
#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <vector>

#include "../../include/pkv.h"

struct pkv_alloc {
    int num_blocks = 0;
    int block_size = 0;
    std::deque<int32_t> free_list;  // FIFO: take from the front, return to the back
    std::vector<int32_t> refs;      // sequences using each block
    std::vector<int32_t> fill;      // token slots written in each block
    struct Seq {
        bool alive = false;
        bool swapped = false;        // table names host blocks
        std::vector<int32_t> table;  // logical block -> physical block
    };
    // host pool (swapped-out sequences), same bookkeeping as the device pool
    int num_host_blocks = 0;
    std::deque<int32_t> host_free_list;
    std::vector<int32_t> host_refs;
    std::vector<int32_t> host_fill;
    std::vector<Seq> seqs;  // indexed by id; ids are never reused

    Seq *find(int id) {
        if (id < 0 || id >= (int)seqs.size() || !seqs[id].alive) return nullptr;
        return &seqs[id];
    }
    const Seq *find(int id) const {
        if (id < 0 || id >= (int)seqs.size() || !seqs[id].alive) return nullptr;
        return &seqs[id];
    }

    int32_t take() {
        const int32_t b = free_list.front();
        free_list.pop_front();
        refs[b] = 1;
        fill[b] = 0;
        return b;
    }

    int64_t length(const Seq &s) const {
        if (s.table.empty()) return 0;
        const std::vector<int32_t> &f = s.swapped ? host_fill : fill;
        return (int64_t)(s.table.size() - 1) * block_size + f[s.table.back()];
    }

    // Fresh blocks that appending n tokens to s takes: a copy-on-write of a
    // shared, not yet full last block, plus new blocks for what overflows it.
    int64_t blocks_needed(const Seq &s, int64_t n) const {
        if (n <= 0) return 0;
        int64_t need = 0, room = 0;
        if (!s.table.empty()) {
            const int32_t last = s.table.back();
            room = block_size - fill[last];
            if (room > 0 && refs[last] > 1) need += 1;
        }
        const int64_t overflow = n > room ? n - room : 0;
        return need + (overflow + block_size - 1) / block_size;
    }

    // One token; the caller has checked that a block is available if needed.
    int64_t append_one(Seq &s, int32_t *cow_src, int32_t *cow_dst) {
        *cow_src = *cow_dst = -1;
        if (s.table.empty() || fill[s.table.back()] == block_size) {
            s.table.push_back(take());
        } else if (refs[s.table.back()] > 1) {
            const int32_t old = s.table.back();
            const int32_t fresh = take();
            fill[fresh] = fill[old];
            refs[old] -= 1;
            s.table.back() = fresh;
            *cow_src = old;
            *cow_dst = fresh;
        }
        const int32_t last = s.table.back();
        const int64_t slot = (int64_t)last * block_size + fill[last];
        fill[last] += 1;
        return slot;
    }
};

extern "C" int pkv_alloc_create(int num_blocks, int block_size, const int32_t *initial_free_order,
                                pkv_alloc_t **out) {
    if (!out || num_blocks <= 0 || block_size <= 0) return PKV_ERR_INVALID_ARG;
    if ((int64_t)num_blocks * block_size > INT64_C(1) << 40) return PKV_ERR_INVALID_ARG;
    if (initial_free_order) {
        std::vector<char> seen(num_blocks, 0);
        for (int i = 0; i < num_blocks; ++i) {
            const int32_t b = initial_free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) return PKV_ERR_INVALID_ARG;
            seen[b] = 1;
        }
    }
    pkv_alloc *a = new (std::nothrow) pkv_alloc;
    if (!a) return PKV_ERR_INVALID_ARG;
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->refs.assign(num_blocks, 0);
    a->fill.assign(num_blocks, 0);
    for (int i = 0; i < num_blocks; ++i) a->free_list.push_back(initial_free_order ? initial_free_order[i] : i);
    *out = a;
    return PKV_OK;
}

extern "C" void pkv_alloc_destroy(pkv_alloc_t *a) { delete a; }

extern "C" int pkv_seq_new(pkv_alloc_t *a, int *seq_id) {
    if (!a || !seq_id) return PKV_ERR_INVALID_ARG;
    a->seqs.emplace_back();
    a->seqs.back().alive = true;
    *seq_id = (int)a->seqs.size() - 1;
    return PKV_OK;
}

extern "C" int pkv_append_token(pkv_alloc_t *a, int seq, int64_t *slot_out, int32_t cow_pair_out[2]) {
    if (!a || !slot_out) return PKV_ERR_INVALID_ARG;
    pkv_alloc::Seq *s = a->find(seq);
    if (!s) return PKV_ERR_NOT_FOUND;
    if (s->swapped) return PKV_ERR_SWAPPED;
    if (a->blocks_needed(*s, 1) > (int64_t)a->free_list.size()) return PKV_ERR_OUT_OF_BLOCKS;
    int32_t src, dst;
    const bool shared_partial = !s->table.empty() && a->fill[s->table.back()] < a->block_size &&
                                a->refs[s->table.back()] > 1;
    if (shared_partial && !cow_pair_out) return PKV_ERR_INVALID_ARG;
    *slot_out = a->append_one(*s, &src, &dst);
    if (cow_pair_out) {
        cow_pair_out[0] = src;
        cow_pair_out[1] = dst;
    }
    return PKV_OK;
}

extern "C" int pkv_append_tokens(pkv_alloc_t *a, int seq, int n, int64_t *slots_out, int32_t *cow_pair_out,
                                 int *n_cow) {
    if (!a || n < 0) return PKV_ERR_INVALID_ARG;
    pkv_alloc::Seq *s = a->find(seq);
    if (!s) return PKV_ERR_NOT_FOUND;
    if (s->swapped) return PKV_ERR_SWAPPED;
    if (a->blocks_needed(*s, n) > (int64_t)a->free_list.size()) return PKV_ERR_OUT_OF_BLOCKS;
    int cows = 0;
    if (cow_pair_out) cow_pair_out[0] = cow_pair_out[1] = -1;
    for (int i = 0; i < n; ++i) {
        int32_t src, dst;
        const int64_t slot = a->append_one(*s, &src, &dst);
        if (slots_out) slots_out[i] = slot;
        if (src >= 0) {
            ++cows;
            if (cow_pair_out) {
                cow_pair_out[0] = src;
                cow_pair_out[1] = dst;
            }
        }
    }
    if (n_cow) *n_cow = cows;
    return PKV_OK;
}

extern "C" int pkv_append_batch(pkv_alloc_t *a, const int32_t *seqs, int n, int64_t *slots_out,
                                int32_t *cow_pairs_out, int *n_cow) {
    if (!a || n < 0 || (n > 0 && (!seqs || !slots_out || !cow_pairs_out))) return PKV_ERR_INVALID_ARG;
    // check ids, distinctness and the total number of fresh blocks first
    std::vector<char> seen(a->seqs.size(), 0);
    int64_t need = 0;
    std::vector<int32_t> touched;  // blocks whose count this batch lowers (copy-on-write)
    std::vector<int32_t> drop;     // ... and by how much, to simulate in order
    for (int i = 0; i < n; ++i) {
        const pkv_alloc::Seq *s = a->find(seqs[i]);
        if (!s) return PKV_ERR_NOT_FOUND;
        if (s->swapped) return PKV_ERR_SWAPPED;
        if (seen[seqs[i]]) return PKV_ERR_INVALID_ARG;
        seen[seqs[i]] = 1;
        if (s->table.empty() || a->fill[s->table.back()] == a->block_size) {
            need += 1;
            continue;
        }
        const int32_t last = s->table.back();
        int32_t lowered = 0;
        size_t k = 0;
        for (; k < touched.size(); ++k)
            if (touched[k] == last) break;
        if (k < touched.size()) lowered = drop[k];
        if (a->refs[last] - lowered > 1) {
            need += 1;
            if (k < touched.size()) {
                drop[k] += 1;
            } else {
                touched.push_back(last);
                drop.push_back(1);
            }
        }
    }
    if (need > (int64_t)a->free_list.size()) return PKV_ERR_OUT_OF_BLOCKS;
    int cows = 0;
    for (int i = 0; i < n; ++i) {
        int32_t src, dst;
        slots_out[i] = a->append_one(*a->find(seqs[i]), &src, &dst);
        if (src >= 0) {
            cow_pairs_out[2 * cows] = src;
            cow_pairs_out[2 * cows + 1] = dst;
            ++cows;
        }
    }
    if (n_cow) *n_cow = cows;
    return PKV_OK;
}

extern "C" int pkv_fork(pkv_alloc_t *a, int parent, int *child) {
    if (!a || !child) return PKV_ERR_INVALID_ARG;
    if (!a->find(parent)) return PKV_ERR_NOT_FOUND;
    if (a->find(parent)->swapped) return PKV_ERR_SWAPPED;
    a->seqs.emplace_back();
    pkv_alloc::Seq &c = a->seqs.back();
    const pkv_alloc::Seq &p = a->seqs[parent];  // after emplace_back: re-read
    c.alive = true;
    c.table = p.table;
    for (int32_t b : c.table) a->refs[b] += 1;
    *child = (int)a->seqs.size() - 1;
    return PKV_OK;
}

extern "C" int pkv_release(pkv_alloc_t *a, int seq, int *n_freed) {
    if (!a) return PKV_ERR_INVALID_ARG;
    pkv_alloc::Seq *s = a->find(seq);
    if (!s) return PKV_ERR_NOT_FOUND;
    // a swapped-out sequence gives its host blocks back to the host pool
    std::vector<int32_t> &refs = s->swapped ? a->host_refs : a->refs;
    std::vector<int32_t> &fill = s->swapped ? a->host_fill : a->fill;
    std::deque<int32_t> &free_list = s->swapped ? a->host_free_list : a->free_list;
    int freed = 0;
    for (int32_t b : s->table) {
        refs[b] -= 1;
        if (refs[b] == 0) {
            fill[b] = 0;
            free_list.push_back(b);
            ++freed;
        }
    }
    s->alive = false;
    s->swapped = false;
    std::vector<int32_t>().swap(s->table);
    if (n_freed) *n_freed = freed;
    return PKV_OK;
}

extern "C" int pkv_export_tables(const pkv_alloc_t *a, const int32_t *seqs, int n, int32_t *tables,
                                 int max_blocks_per_seq, int32_t *ctx_lens) {
    if (!a || n < 0 || max_blocks_per_seq < 0 || (n > 0 && (!seqs || !tables))) return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        const pkv_alloc::Seq *s = a->find(seqs[i]);
        if (!s) return PKV_ERR_NOT_FOUND;
        if (s->swapped) return PKV_ERR_SWAPPED;
        if ((int64_t)s->table.size() > max_blocks_per_seq) return PKV_ERR_INVALID_ARG;
        if (a->length(*s) > INT32_MAX) return PKV_ERR_INVALID_ARG;
    }
    for (int i = 0; i < n; ++i) {
        const pkv_alloc::Seq &s = *a->find(seqs[i]);
        int32_t *row = tables + (int64_t)i * max_blocks_per_seq;
        const size_t nb = s.table.size();
        if (nb) std::memcpy(row, s.table.data(), nb * sizeof(int32_t));
        for (int j = (int)nb; j < max_blocks_per_seq; ++j) row[j] = -1;
        if (ctx_lens) ctx_lens[i] = (int32_t)a->length(s);
    }
    return PKV_OK;
}

extern "C" int pkv_export_shared_prefix(const pkv_alloc_t *a, const int32_t *seqs, int n, int32_t *shared_out) {
    if (!a || n < 0 || (n > 0 && (!seqs || !shared_out))) return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        const pkv_alloc::Seq *s = a->find(seqs[i]);
        if (!s) return PKV_ERR_NOT_FOUND;
        if (s->swapped) return PKV_ERR_SWAPPED;
    }
    for (int i = 0; i < n; ++i) {
        int32_t common = 0;
        if (i > 0) {
            const std::vector<int32_t> &x = a->find(seqs[i])->table, &y = a->find(seqs[i - 1])->table;
            const size_t m = x.size() < y.size() ? x.size() : y.size();
            while ((size_t)common < m && x[common] == y[common]) ++common;
        }
        shared_out[i] = common;
    }
    return PKV_OK;
}

extern "C" int pkv_seq_length(const pkv_alloc_t *a, int seq, int *num_tokens) {
    if (!a || !num_tokens) return PKV_ERR_INVALID_ARG;
    const pkv_alloc::Seq *s = a->find(seq);
    if (!s) return PKV_ERR_NOT_FOUND;
    const int64_t len = a->length(*s);
    if (len > INT32_MAX) return PKV_ERR_INVALID_ARG;
    *num_tokens = (int)len;
    return PKV_OK;
}

extern "C" int pkv_seq_num_blocks(const pkv_alloc_t *a, int seq, int *num_blocks) {
    if (!a || !num_blocks) return PKV_ERR_INVALID_ARG;
    const pkv_alloc::Seq *s = a->find(seq);
    if (!s) return PKV_ERR_NOT_FOUND;
    *num_blocks = (int)s->table.size();
    return PKV_OK;
}

extern "C" int pkv_seq_table(const pkv_alloc_t *a, int seq, int32_t *table, int cap, int *num_blocks) {
    if (!a || cap < 0 || (cap > 0 && !table)) return PKV_ERR_INVALID_ARG;
    const pkv_alloc::Seq *s = a->find(seq);
    if (!s) return PKV_ERR_NOT_FOUND;
    if ((int64_t)s->table.size() > cap) return PKV_ERR_INVALID_ARG;
    if (!s->table.empty()) std::memcpy(table, s->table.data(), s->table.size() * sizeof(int32_t));
    if (num_blocks) *num_blocks = (int)s->table.size();
    return PKV_OK;
}

extern "C" int pkv_block_refcount(const pkv_alloc_t *a, int block, int *refs) {
    if (!a || !refs || block < 0 || block >= a->num_blocks) return PKV_ERR_INVALID_ARG;
    *refs = a->refs[block];
    return PKV_OK;
}

extern "C" int pkv_block_fill(const pkv_alloc_t *a, int block, int *fill) {
    if (!a || !fill || block < 0 || block >= a->num_blocks) return PKV_ERR_INVALID_ARG;
    *fill = a->fill[block];
    return PKV_OK;
}

extern "C" int pkv_num_free(const pkv_alloc_t *a, int *num_free) {
    if (!a || !num_free) return PKV_ERR_INVALID_ARG;
    *num_free = (int)a->free_list.size();
    return PKV_OK;
}

extern "C" int pkv_free_list(const pkv_alloc_t *a, int32_t *out, int cap, int *n) {
    if (!a || cap < 0 || (cap > 0 && !out)) return PKV_ERR_INVALID_ARG;
    if ((int64_t)a->free_list.size() > cap) return PKV_ERR_INVALID_ARG;
    int i = 0;
    for (int32_t b : a->free_list) out[i++] = b;
    if (n) *n = i;
    return PKV_OK;
}

// ---------------------------------------------------------------------------
// Swapping
// ---------------------------------------------------------------------------

extern "C" int pkv_alloc_host_pool(pkv_alloc_t *a, int num_host_blocks, const int32_t *host_free_order) {
    if (!a || num_host_blocks < 0) return PKV_ERR_INVALID_ARG;
    if ((int)a->host_free_list.size() != a->num_host_blocks) return PKV_ERR_INVALID_ARG;  // host blocks in use
    if (host_free_order) {
        std::vector<char> seen(num_host_blocks, 0);
        for (int i = 0; i < num_host_blocks; ++i) {
            const int32_t b = host_free_order[i];
            if (b < 0 || b >= num_host_blocks || seen[b]) return PKV_ERR_INVALID_ARG;
            seen[b] = 1;
        }
    }
    a->num_host_blocks = num_host_blocks;
    a->host_refs.assign(num_host_blocks, 0);
    a->host_fill.assign(num_host_blocks, 0);
    a->host_free_list.clear();
    for (int i = 0; i < num_host_blocks; ++i) a->host_free_list.push_back(host_free_order ? host_free_order[i] : i);
    return PKV_OK;
}

namespace {

// Moves the blocks of a group of sequences from one pool to the other; see
// the rules in the header.  to_host selects the direction.
int move_group(pkv_alloc *a, const int32_t *seqs, int n, bool to_host, int32_t *pairs_out, int cap,
               int *n_pairs) {
    if (!a || n < 0 || cap < 0 || (n > 0 && !seqs) || (cap > 0 && !pairs_out)) return PKV_ERR_INVALID_ARG;
    std::vector<char> seen(a->seqs.size(), 0);
    int64_t entries = 0;
    for (int i = 0; i < n; ++i) {
        const pkv_alloc::Seq *s = a->find(seqs[i]);
        if (!s) return PKV_ERR_NOT_FOUND;
        if (seen[seqs[i]]) return PKV_ERR_INVALID_ARG;
        seen[seqs[i]] = 1;
        if (s->swapped == to_host) return PKV_ERR_SWAPPED;
        entries += (int64_t)s->table.size();
    }
    if (entries > cap) return PKV_ERR_INVALID_ARG;
    std::vector<int32_t> &src_refs = to_host ? a->refs : a->host_refs;
    std::vector<int32_t> &src_fill = to_host ? a->fill : a->host_fill;
    std::deque<int32_t> &src_free = to_host ? a->free_list : a->host_free_list;
    std::vector<int32_t> &dst_refs = to_host ? a->host_refs : a->refs;
    std::vector<int32_t> &dst_fill = to_host ? a->host_fill : a->fill;
    std::deque<int32_t> &dst_free = to_host ? a->host_free_list : a->free_list;
    // distinct source blocks in order of first appearance, with their holders
    std::vector<int32_t> order, holders, slot_of(src_refs.size(), -1);
    for (int i = 0; i < n; ++i)
        for (int32_t b : a->seqs[seqs[i]].table) {
            if (slot_of[b] < 0) {
                slot_of[b] = (int32_t)order.size();
                order.push_back(b);
                holders.push_back(0);
            }
            holders[slot_of[b]] += 1;
        }
    if (order.size() > dst_free.size()) return PKV_ERR_OUT_OF_BLOCKS;
    std::vector<int32_t> moved(order.size());
    for (size_t k = 0; k < order.size(); ++k) {
        const int32_t nb = dst_free.front();
        dst_free.pop_front();
        dst_refs[nb] = holders[k];
        dst_fill[nb] = src_fill[order[k]];
        moved[k] = nb;
        pairs_out[2 * k] = order[k];
        pairs_out[2 * k + 1] = nb;
    }
    for (size_t k = 0; k < order.size(); ++k) {
        const int32_t b = order[k];
        src_refs[b] -= holders[k];
        if (src_refs[b] == 0) {
            src_fill[b] = 0;
            src_free.push_back(b);
        }
    }
    for (int i = 0; i < n; ++i) {
        pkv_alloc::Seq &s = a->seqs[seqs[i]];
        for (int32_t &b : s.table) b = moved[slot_of[b]];
        s.swapped = to_host;
    }
    if (n_pairs) *n_pairs = (int)order.size();
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_swap_out(pkv_alloc_t *a, const int32_t *seqs, int n, int32_t *pairs_out, int cap,
                            int *n_pairs) {
    return move_group(a, seqs, n, true, pairs_out, cap, n_pairs);
}

extern "C" int pkv_swap_in(pkv_alloc_t *a, const int32_t *seqs, int n, int32_t *pairs_out, int cap,
                           int *n_pairs) {
    return move_group(a, seqs, n, false, pairs_out, cap, n_pairs);
}

extern "C" int pkv_seq_swapped(const pkv_alloc_t *a, int seq, int *swapped) {
    if (!a || !swapped) return PKV_ERR_INVALID_ARG;
    const pkv_alloc::Seq *s = a->find(seq);
    if (!s) return PKV_ERR_NOT_FOUND;
    *swapped = s->swapped ? 1 : 0;
    return PKV_OK;
}

extern "C" int pkv_host_block_refcount(const pkv_alloc_t *a, int block, int *refs) {
    if (!a || !refs || block < 0 || block >= a->num_host_blocks) return PKV_ERR_INVALID_ARG;
    *refs = a->host_refs[block];
    return PKV_OK;
}

extern "C" int pkv_host_block_fill(const pkv_alloc_t *a, int block, int *fill) {
    if (!a || !fill || block < 0 || block >= a->num_host_blocks) return PKV_ERR_INVALID_ARG;
    *fill = a->host_fill[block];
    return PKV_OK;
}

extern "C" int pkv_num_free_host(const pkv_alloc_t *a, int *num_free) {
    if (!a || !num_free) return PKV_ERR_INVALID_ARG;
    *num_free = (int)a->host_free_list.size();
    return PKV_OK;
}

extern "C" int pkv_host_free_list(const pkv_alloc_t *a, int32_t *out, int cap, int *n) {
    if (!a || cap < 0 || (cap > 0 && !out)) return PKV_ERR_INVALID_ARG;
    if ((int64_t)a->host_free_list.size() > cap) return PKV_ERR_INVALID_ARG;
    int i = 0;
    for (int32_t b : a->host_free_list) out[i++] = b;
    if (n) *n = i;
    return PKV_OK;
}

// ---------------------------------------------------------------------------
// Checkpoint (format and acceptance rules in the header)
// ---------------------------------------------------------------------------

namespace {

constexpr uint32_t kBlobMagic = 0x41564B50u;  // "PKVA" as little-endian bytes
constexpr int32_t kBlobVersion = 1;

// Little-endian int32 writer; counts bytes when out is null.
struct BlobWriter {
    unsigned char *out;
    size_t n = 0;
    void i32(int32_t v) {
        const uint32_t u = (uint32_t)v;
        if (out)
            for (int k = 0; k < 4; ++k) out[n + k] = (unsigned char)(u >> (8 * k));
        n += 4;
    }
    template <class C>
    void ids(const C &c) {
        i32((int32_t)c.size());
        for (int32_t b : c) i32(b);
    }
};

// Little-endian int32 reader that fails (instead of reading past the end).
struct BlobReader {
    const unsigned char *in;
    size_t size, n = 0;
    bool ok = true;
    int32_t i32() {
        if (!ok || size - n < 4) {
            ok = false;
            return 0;
        }
        uint32_t u = 0;
        for (int k = 0; k < 4; ++k) u |= (uint32_t)in[n + k] << (8 * k);
        n += 4;
        return (int32_t)u;
    }
    // a count of int32 items that must still fit in the blob
    int32_t count(int64_t max_items) {
        const int32_t c = i32();
        if (!ok || c < 0 || c > max_items || (size_t)c > (size - n) / 4) ok = false;
        return ok ? c : 0;
    }
};

void write_state(const pkv_alloc &a, BlobWriter &w) {
    w.i32((int32_t)kBlobMagic);
    w.i32(kBlobVersion);
    w.i32(a.num_blocks);
    w.i32(a.block_size);
    w.i32(a.num_host_blocks);
    w.i32((int32_t)a.seqs.size());
    w.ids(a.free_list);
    for (int32_t f : a.fill) w.i32(f);
    w.ids(a.host_free_list);
    for (int32_t f : a.host_fill) w.i32(f);
    for (const pkv_alloc::Seq &s : a.seqs) {
        w.i32((s.alive ? 1 : 0) | (s.swapped ? 2 : 0));
        w.ids(s.table);
    }
}

// One pool's part of the acceptance check: the free list and the holders
// (counts rebuilt from the tables) partition the pool, free blocks have fill
// 0, and held blocks obey the fill rules recorded in full / last.
bool pool_consistent(int nb, int bs, const std::deque<int32_t> &free_list, const std::vector<int32_t> &refs,
                     const std::vector<int32_t> &fill, const std::vector<char> &non_last,
                     const std::vector<char> &last) {
    std::vector<char> listed(nb, 0);
    for (int32_t b : free_list) {
        if (b < 0 || b >= nb || listed[b]) return false;
        listed[b] = 1;
    }
    for (int b = 0; b < nb; ++b) {
        if (fill[b] < 0 || fill[b] > bs) return false;
        if (refs[b] == 0) {
            if (!listed[b] || fill[b] != 0) return false;
        } else {
            if (listed[b]) return false;
            if (non_last[b] && fill[b] != bs) return false;
            if (last[b] && fill[b] < 1) return false;
        }
    }
    return true;
}

}  // namespace

extern "C" int pkv_alloc_save(const pkv_alloc_t *a, void *buf, size_t cap, size_t *bytes) {
    if (!a || !bytes) return PKV_ERR_INVALID_ARG;
    BlobWriter count{nullptr};
    write_state(*a, count);
    *bytes = count.n;
    if (!buf) return PKV_OK;
    if (cap < count.n) return PKV_ERR_INVALID_ARG;
    BlobWriter w{static_cast<unsigned char *>(buf)};
    write_state(*a, w);
    return PKV_OK;
}

extern "C" int pkv_alloc_load(const void *buf, size_t bytes, pkv_alloc_t **out) {
    if (!buf || !out) return PKV_ERR_INVALID_ARG;
    BlobReader r{static_cast<const unsigned char *>(buf), bytes};
    if ((uint32_t)r.i32() != kBlobMagic || r.i32() != kBlobVersion) return PKV_ERR_INVALID_ARG;
    const int32_t nb = r.i32(), bs = r.i32(), nh = r.i32(), m = r.i32();
    if (!r.ok || nb <= 0 || bs <= 0 || nh < 0 || m < 0 || (int64_t)nb * bs > INT64_C(1) << 40)
        return PKV_ERR_INVALID_ARG;
    // every array must fit in what is left before anything is allocated
    const size_t left = bytes - r.n;
    if ((size_t)nb + (size_t)nh + 2 * (size_t)m + 2 > left / 4) return PKV_ERR_INVALID_ARG;

    std::deque<int32_t> free_list, host_free_list;
    std::vector<int32_t> fill(nb), host_fill(nh);
    for (int32_t i = 0, f = r.count(nb); i < f; ++i) free_list.push_back(r.i32());
    for (int32_t &v : fill) v = r.i32();
    for (int32_t i = 0, f = r.count(nh); i < f; ++i) host_free_list.push_back(r.i32());
    for (int32_t &v : host_fill) v = r.i32();
    std::vector<pkv_alloc::Seq> seqs(m);
    for (pkv_alloc::Seq &s : seqs) {
        const int32_t flags = r.i32();
        if (flags != 0 && flags != 1 && flags != 3) r.ok = false;
        s.alive = flags & 1;
        s.swapped = (flags & 2) != 0;
        const int32_t len = r.count(s.swapped ? nh : nb);
        if (!s.alive && len != 0) r.ok = false;
        s.table.resize(len);
        for (int32_t &b : s.table) b = r.i32();
        if (!r.ok) break;
    }
    if (!r.ok || r.n != bytes) return PKV_ERR_INVALID_ARG;

    // counts from the tables, and the rules a reachable state obeys
    std::vector<int32_t> refs(nb, 0), host_refs(nh, 0);
    std::vector<char> non_last(nb, 0), last(nb, 0), host_non_last(nh, 0), host_last(nh, 0);
    std::vector<int32_t> seen(nb, -1), host_seen(nh, -1), pos(nb, -1), host_pos(nh, -1);
    for (int32_t id = 0; id < m; ++id) {
        const pkv_alloc::Seq &s = seqs[id];
        const int32_t pool = s.swapped ? nh : nb;
        std::vector<int32_t> &cnt = s.swapped ? host_refs : refs;
        std::vector<char> &nl = s.swapped ? host_non_last : non_last;
        std::vector<char> &ls = s.swapped ? host_last : last;
        std::vector<int32_t> &sn = s.swapped ? host_seen : seen;
        std::vector<int32_t> &ps = s.swapped ? host_pos : pos;
        for (size_t i = 0; i < s.table.size(); ++i) {
            const int32_t b = s.table[i];
            if (b < 0 || b >= pool || sn[b] == id) return PKV_ERR_INVALID_ARG;  // outside, or twice in one table
            if (ps[b] >= 0 && ps[b] != (int32_t)i) return PKV_ERR_INVALID_ARG;  // a shared block moved
            sn[b] = id;
            ps[b] = (int32_t)i;
            cnt[b] += 1;
            (i + 1 < s.table.size() ? nl : ls)[b] = 1;
        }
    }
    if (!pool_consistent(nb, bs, free_list, refs, fill, non_last, last) ||
        !pool_consistent(nh, bs, host_free_list, host_refs, host_fill, host_non_last, host_last))
        return PKV_ERR_INVALID_ARG;

    pkv_alloc *a = new (std::nothrow) pkv_alloc;
    if (!a) return PKV_ERR_INVALID_ARG;
    a->num_blocks = nb;
    a->block_size = bs;
    a->free_list = std::move(free_list);
    a->refs = std::move(refs);
    a->fill = std::move(fill);
    a->num_host_blocks = nh;
    a->host_free_list = std::move(host_free_list);
    a->host_refs = std::move(host_refs);
    a->host_fill = std::move(host_fill);
    a->seqs = std::move(seqs);
    *out = a;
    return PKV_OK;
}
