// Random operations on the host block manager through its C ABI, built with
// AddressSanitizer and UndefinedBehaviorSanitizer (tests/test_native_host.py).
// After every call: blocks and references are conserved in both pools, every
// table matches its context length, and a call that fails leaves the whole
// state exactly as it was.  Every 50 calls the state is checkpointed: the
// restored object must equal the saved one (and the fuzzing goes on with it
// half of the time), and corrupted blobs must be refused or load as a state
// that keeps the invariants.  Exits non-zero on the first violation.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <random>
#include <set>
#include <vector>

#include "pkv.h"

static int fails = 0;
#define CHECK(c, ...)                                              \
    do {                                                           \
        if (!(c)) {                                                \
            std::printf("FAIL %s:%d: ", __FILE__, __LINE__);       \
            std::printf(__VA_ARGS__);                              \
            std::printf("\n");                                     \
            if (++fails > 5) std::exit(1);                         \
        }                                                          \
    } while (0)

struct Snapshot {
    std::vector<int32_t> free_dev, free_host;
    std::map<int, std::vector<int32_t>> tables;  // seq -> table
    std::map<int, int> lens, swapped;
    bool operator==(const Snapshot &o) const {
        return free_dev == o.free_dev && free_host == o.free_host && tables == o.tables && lens == o.lens &&
               swapped == o.swapped;
    }
};

struct Fuzz {
    pkv_alloc_t *a = nullptr;
    int nb = 0, nh = 0, bs = 0;
    std::set<int> live;  // sequences not released
    std::mt19937_64 rng;

    Snapshot snap() {
        Snapshot s;
        int n = 0;
        s.free_dev.resize(nb + 1);
        CHECK(pkv_free_list(a, s.free_dev.data(), nb + 1, &n) == PKV_OK, "free list");
        s.free_dev.resize(n);
        s.free_host.resize(nh + 1);
        CHECK(pkv_host_free_list(a, s.free_host.data(), nh + 1, &n) == PKV_OK, "host free list");
        s.free_host.resize(n);
        for (int q : live) {
            int len = 0, nbk = 0, sw = 0;
            CHECK(pkv_seq_length(a, q, &len) == PKV_OK, "length of %d", q);
            CHECK(pkv_seq_swapped(a, q, &sw) == PKV_OK, "swapped of %d", q);
            std::vector<int32_t> t(nb + nh + 1);
            CHECK(pkv_seq_table(a, q, t.data(), (int)t.size(), &nbk) == PKV_OK, "table of %d", q);
            t.resize(nbk);
            s.tables[q] = t;
            s.lens[q] = len;
            s.swapped[q] = sw;
        }
        return s;
    }

    // conservation: free + referenced = pool, counts = holders, tables fit lengths
    void invariants(const Snapshot &s) {
        std::map<int, int> dev_holders, host_holders;
        for (auto &kv : s.tables) {
            const int q = kv.first;
            CHECK((int)kv.second.size() == (s.lens.at(q) + bs - 1) / bs, "seq %d: %zu blocks for %d tokens", q,
                  kv.second.size(), s.lens.at(q));
            for (int b : kv.second) (s.swapped.at(q) ? host_holders : dev_holders)[b]++;
        }
        std::set<int> fd(s.free_dev.begin(), s.free_dev.end()), fh(s.free_host.begin(), s.free_host.end());
        CHECK(fd.size() == s.free_dev.size() && fh.size() == s.free_host.size(), "duplicate in a free list");
        CHECK((int)(fd.size() + dev_holders.size()) == nb, "device blocks: %zu free + %zu held != %d", fd.size(),
              dev_holders.size(), nb);
        CHECK((int)(fh.size() + host_holders.size()) == nh, "host blocks: %zu free + %zu held != %d", fh.size(),
              host_holders.size(), nh);
        for (auto &kv : dev_holders) {
            int r = -1;
            CHECK(pkv_block_refcount(a, kv.first, &r) == PKV_OK && r == kv.second, "block %d: count %d, %d holders",
                  kv.first, r, kv.second);
            CHECK(!fd.count(kv.first), "block %d held and free", kv.first);
        }
        for (auto &kv : host_holders) {
            int r = -1;
            CHECK(pkv_host_block_refcount(a, kv.first, &r) == PKV_OK && r == kv.second,
                  "host block %d: count %d, %d holders", kv.first, r, kv.second);
        }
    }

    int pick() {  // a live sequence, or an id that is not one
        if (live.empty() || rng() % 10 == 0) return (int)(rng() % 1000) - 5;
        auto it = live.begin();
        std::advance(it, rng() % live.size());
        return *it;
    }

    // one random call; returns true if the library refused it
    bool step() {
        const Snapshot before = snap();
        int rc = PKV_OK;
        const int op = (int)(rng() % 9);
        std::vector<int32_t> seqs;
        for (int i = 0, k = 1 + (int)(rng() % 4); i < k; ++i) seqs.push_back(pick());
        switch (op) {
            case 0: {
                int id = -1;
                rc = pkv_seq_new(a, &id);
                if (rc == PKV_OK) live.insert(id);
                break;
            }
            case 1: {
                int64_t slot = 0;
                int32_t pair[2];
                rc = pkv_append_token(a, seqs[0], &slot, pair);
                break;
            }
            case 2: {
                const int n = (int)(rng() % 40);
                std::vector<int64_t> slots(n + 1);
                int32_t pair[2];
                int ncow = 0;
                rc = pkv_append_tokens(a, seqs[0], n, slots.data(), pair, &ncow);
                break;
            }
            case 3: {
                std::vector<int64_t> slots(seqs.size());
                std::vector<int32_t> pairs(2 * seqs.size());
                int ncow = 0;
                rc = pkv_append_batch(a, seqs.data(), (int)seqs.size(), slots.data(), pairs.data(), &ncow);
                break;
            }
            case 4: {
                int child = -1;
                rc = pkv_fork(a, seqs[0], &child);
                if (rc == PKV_OK) live.insert(child);
                break;
            }
            case 5: {
                int freed = 0;
                rc = pkv_release(a, seqs[0], &freed);
                if (rc == PKV_OK) live.erase(seqs[0]);
                break;
            }
            case 6:
            case 7: {
                const int cap = (int)(rng() % 3 == 0 ? rng() % 4 : nb + nh);
                std::vector<int32_t> pairs(2 * (cap + 1));
                int np = 0;
                rc = op == 6 ? pkv_swap_out(a, seqs.data(), (int)seqs.size(), pairs.data(), cap, &np)
                             : pkv_swap_in(a, seqs.data(), (int)seqs.size(), pairs.data(), cap, &np);
                break;
            }
            default: {
                const int mb = 1 + (int)(rng() % 6);
                std::vector<int32_t> tables(seqs.size() * mb), lens(seqs.size());
                rc = pkv_export_tables(a, seqs.data(), (int)seqs.size(), tables.data(), mb, lens.data());
                break;
            }
        }
        const Snapshot after = snap();
        if (rc != PKV_OK) CHECK(after == before, "op %d failed with %d but changed the state", op, rc);
        invariants(after);
        return rc != PKV_OK;
    }
};

// The object a blob describes, seen through the Fuzz checks: its live ids
// are probed (the blob header says how many ids were handed out).
static Fuzz view_of(pkv_alloc_t *b, const std::vector<unsigned char> &blob) {
    Fuzz g;
    g.a = b;
    auto field = [&](int k) {
        uint32_t u = 0;
        for (int i = 0; i < 4; ++i) u |= (uint32_t)blob[4 * k + i] << (8 * i);
        return (int)u;
    };
    g.nb = field(2);
    g.bs = field(3);
    g.nh = field(4);
    for (int id = 0, m = field(5); id < m; ++id) {
        int len = 0;
        if (pkv_seq_length(b, id, &len) == PKV_OK) g.live.insert(id);
    }
    return g;
}

static std::vector<unsigned char> save(pkv_alloc_t *a) {
    size_t n = 0;
    CHECK(pkv_alloc_save(a, nullptr, 0, &n) == PKV_OK && n >= 24, "blob size");
    std::vector<unsigned char> blob(n);
    size_t n2 = 0;
    CHECK(pkv_alloc_save(a, blob.data(), n, &n2) == PKV_OK && n2 == n, "save");
    if (n > 0) {
        std::vector<unsigned char> small(n - 1);
        CHECK(pkv_alloc_save(a, small.data(), n - 1, &n2) == PKV_ERR_INVALID_ARG, "short buffer accepted");
    }
    return blob;
}

static long loads_accepted = 0, loads_refused = 0;

// Save, restore, compare; then corrupt the blob in several ways.
static void checkpoint(Fuzz &f) {
    const std::vector<unsigned char> blob = save(f.a);
    pkv_alloc_t *b = nullptr;
    CHECK(pkv_alloc_load(blob.data(), blob.size(), &b) == PKV_OK, "load of a saved state");
    if (!b) return;
    Fuzz g = view_of(b, blob);
    CHECK(g.live == f.live, "live ids differ after restore");
    CHECK(g.snap() == f.snap(), "restored state differs");
    CHECK(save(b) == blob, "re-saved blob differs");
    if (f.rng() % 2) {  // go on with the restored object
        pkv_alloc_destroy(f.a);
        f.a = b;
    } else {
        pkv_alloc_destroy(b);
    }
    for (int k = 0; k < 20; ++k) {
        std::vector<unsigned char> bad = blob;
        switch (f.rng() % 4) {
            case 0: bad[f.rng() % bad.size()] ^= (unsigned char)(1u << (f.rng() % 8)); break;
            case 1: bad.resize(f.rng() % bad.size()); break;
            case 2: bad.push_back((unsigned char)f.rng()); break;
            default: {  // a plausible small change to one int32 field
                const size_t at = 4 * (f.rng() % (bad.size() / 4));
                bad[at] = (unsigned char)(bad[at] + (f.rng() % 2 ? 1 : 255));
            }
        }
        pkv_alloc_t *c = nullptr;
        if (pkv_alloc_load(bad.data(), bad.size(), &c) != PKV_OK) {
            CHECK(c == nullptr, "refused load wrote *out");
            ++loads_refused;
            continue;
        }
        ++loads_accepted;
        Fuzz h = view_of(c, bad);
        h.invariants(h.snap());
        CHECK(save(c) == bad, "an accepted blob does not re-save to itself");
        pkv_alloc_destroy(c);
    }
}

int main() {
    long ops = 0, failed_calls = 0;
    for (int trial = 0; trial < 12; ++trial) {
        Fuzz f;
        f.rng.seed(152 + trial);
        const int sizes[] = {1, 2, 4, 16};
        f.bs = sizes[trial % 4];
        f.nb = 4 + (int)(f.rng() % 28);
        f.nh = (int)(f.rng() % 16);
        CHECK(pkv_alloc_create(f.nb, f.bs, nullptr, &f.a) == PKV_OK, "create");
        if (f.nh) CHECK(pkv_alloc_host_pool(f.a, f.nh, nullptr) == PKV_OK, "host pool");
        // argument checks that must not touch anything
        CHECK(pkv_append_batch(f.a, nullptr, 3, nullptr, nullptr, nullptr) == PKV_ERR_INVALID_ARG, "null batch");
        CHECK(pkv_export_tables(f.a, nullptr, 1, nullptr, 4, nullptr) == PKV_ERR_INVALID_ARG, "null export");
        for (int i = 0; i < 1000; ++i) {
            failed_calls += f.step();
            ++ops;
            if (i % 50 == 49) checkpoint(f);
        }
        pkv_alloc_destroy(f.a);
    }
    CHECK(loads_refused > 1000 && loads_accepted > 10, "corruptions: %ld refused, %ld accepted", loads_refused,
          loads_accepted);
    if (fails) {
        std::printf("%d failures\n", fails);
        return 1;
    }
    std::printf("alloc fuzz ok: %ld operations (%ld refused, state unchanged); checkpoints: %ld corrupt blobs "
                "refused, %ld loaded as valid states\n",
                ops, failed_calls, loads_refused, loads_accepted);
    return 0;
}
