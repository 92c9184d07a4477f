// Host block manager of the paged KV cache: free list, per-block reference
// counts, sequences as lists of physical blocks, fork (prefix sharing) and
// append with copy-on-write.
//
// Pages followed:
//  * logical blocks map to physical blocks anywhere in the pool through a
//    per-sequence table ("PagedAttention: memetakan blok KV logis ke memori
//    fisik tidak kontigu", section "Urutan logis dipisahkan dari penempatan
//    fisik");
//  * a physical block is taken only when the sequence crosses a block
//    boundary ("Melihat Lebih Dalam vLLM v0.7", section "Blueprint Arsitektur
//    2", item "Alokasi On-Demand"), so a sequence wastes less than one block
//    (nalar.dev, section "Sisa alokasi dibatasi oleh granularitas blok");
//  * several sequences may reference one block; a branch that must change a
//    shared block gets its own copy first ("Apa itu PagedAttention?", section
//    "Cara kerja PagedAttention", item 3; nalar.dev, section "Sharing blok
//    dapat menghindari duplikasi state KV").
//
// Choices the pages leave open: the free list is a stack (freed blocks are
// reused first) whose initial order is 0..n-1 or a SplitMix64-driven
// Fisher-Yates shuffle; the first branch that appends into a shared, partly
// filled last block takes the copy; a full shared block is never copied.
// Every failing call leaves the state unchanged, host allocation failures
// included: every call allocates what it needs (vector capacity, map nodes)
// before it changes anything, and no exception leaves the C ABI.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <memory>
#include <new>
#include <unordered_map>
#include <utility>
#include <vector>

#include "pa.h"

namespace pa {
int fail(int code, const char *fmt, ...);
void clear_error();
}  // namespace pa

struct pa_bm {
    int64_t num_blocks = 0;
    int bs = 0;
    std::vector<int32_t> free_stack;  // top = back
    std::vector<int32_t> ref;
    struct Seq {
        std::vector<int32_t> blocks;
        int64_t len = 0;
    };
    std::unordered_map<int64_t, Seq> seqs;

    int32_t take() {
        const int32_t b = free_stack.back();
        free_stack.pop_back();
        ref[b] = 1;
        return b;
    }
    // never allocates: the stack holds each block at most once and keeps the
    // capacity of num_blocks it was created with
    void release(int32_t b) {
        if (--ref[b] == 0) free_stack.push_back(b);
    }
    // Blocks an append of n tokens to s would take (new blocks + a CoW copy).
    int64_t needed(const Seq &s, int64_t n) const {
        const int64_t have = (s.len + bs - 1) / bs;
        const int64_t want = (s.len + n + bs - 1) / bs;
        int64_t need = want - have;
        if (n > 0 && s.len % bs != 0 && ref[s.blocks.back()] > 1) ++need;
        return need;
    }
    int64_t slot(const Seq &s, int64_t j) const {
        return int64_t(s.blocks[j / bs]) * bs + j % bs;
    }
};

namespace {

// Host fault injection for tests: the k-th allocation point from now on
// (0 = the next) throws std::bad_alloc as if host memory had run out.
std::atomic<int64_t> g_alloc_failure{-1};

// Marks a statement that may allocate host memory.
void alloc_point() {
    int64_t k = g_alloc_failure.load(std::memory_order_relaxed);
    if (k < 0) return;
    g_alloc_failure.store(k - 1, std::memory_order_relaxed);
    if (k == 0) throw std::bad_alloc();
}

// Capacity for n elements, growing geometrically (a plain reserve(size + 1)
// per append would copy the table every time).
void ensure_capacity(std::vector<int32_t> &v, size_t n) {
    if (v.capacity() >= n) return;
    alloc_point();
    v.reserve(std::max(n, 2 * v.capacity()));
}

// Runs an entry point's body; host allocation failures become PA_ERR_OOM
// (the body has changed nothing when one is thrown) and no exception crosses
// the C ABI.
template <class F>
int guarded(const char *what, F &&body) {
    try {
        return body();
    } catch (const std::bad_alloc &) {
        return pa::fail(PA_ERR_OOM, "%s: host allocation failed", what);
    } catch (...) {
        return pa::fail(PA_ERR_INVALID, "%s: unexpected host error", what);
    }
}

uint64_t splitmix64(uint64_t &state) {
    state += 0x9E3779B97F4A7C15ull;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Append one token to s; the caller has checked that a block is available
// and made room in s.blocks for a new block (nothing here allocates).
void append_one(pa_bm *bm, pa_bm::Seq &s, int64_t *slot, int64_t *cow_src, int64_t *cow_dst) {
    int64_t src = -1, dst = -1;
    if (s.len % bm->bs == 0) {
        s.blocks.push_back(bm->take());
    } else if (bm->ref[s.blocks.back()] > 1) {
        src = s.blocks.back();
        dst = bm->take();
        bm->release(static_cast<int32_t>(src));
        s.blocks.back() = static_cast<int32_t>(dst);
    }
    *slot = bm->slot(s, s.len);
    s.len += 1;
    if (cow_src) *cow_src = src;
    if (cow_dst) *cow_dst = dst;
}

}  // namespace

extern "C" {

int pa_bm_create(int64_t num_blocks, int block_size, uint64_t seed, pa_bm **out) {
    pa::clear_error();
    if (!out) return pa::fail(PA_ERR_INVALID, "bm_create: out is NULL");
    *out = nullptr;
    if (num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0)
        return pa::fail(PA_ERR_INVALID, "bm_create: bad sizes");
    return guarded("bm_create", [&] {
        alloc_point();
        std::unique_ptr<pa_bm> bm(new pa_bm());
        bm->num_blocks = num_blocks;
        bm->bs = block_size;
        alloc_point();
        std::vector<int32_t> order(num_blocks);
        for (int64_t i = 0; i < num_blocks; ++i) order[i] = static_cast<int32_t>(i);
        if (seed) {
            uint64_t st = seed;
            for (int64_t i = num_blocks - 1; i > 0; --i) {
                const uint64_t j = splitmix64(st) % uint64_t(i + 1);
                std::swap(order[i], order[j]);
            }
        }
        alloc_point();
        bm->free_stack.assign(order.rbegin(), order.rend());
        alloc_point();
        bm->ref.assign(num_blocks, 0);
        *out = bm.release();
        return int(PA_OK);
    });
}

void pa_bm_destroy(pa_bm *bm) { delete bm; }

int pa_bm_add_seq(pa_bm *bm, int64_t seq, int64_t n_tokens, int64_t *slots) {
    pa::clear_error();
    if (!bm || n_tokens < 0) return pa::fail(PA_ERR_INVALID, "bm_add_seq: bad arguments");
    if (bm->seqs.count(seq)) return pa::fail(PA_ERR_INVALID, "bm_add_seq: sequence exists");
    const int64_t nblk = (n_tokens + bm->bs - 1) / bm->bs;
    if (nblk > int64_t(bm->free_stack.size()))
        return pa::fail(PA_ERR_OOM, "bm_add_seq: %lld blocks needed, %zu free", (long long)nblk,
                        bm->free_stack.size());
    return guarded("bm_add_seq", [&] {
        pa_bm::Seq s;
        ensure_capacity(s.blocks, size_t(nblk));
        alloc_point();
        pa_bm::Seq &dst = bm->seqs.emplace(seq, pa_bm::Seq{}).first->second;
        // nothing below allocates
        for (int64_t i = 0; i < nblk; ++i) s.blocks.push_back(bm->take());
        s.len = n_tokens;
        if (slots)
            for (int64_t j = 0; j < n_tokens; ++j) slots[j] = bm->slot(s, j);
        dst = std::move(s);
        return int(PA_OK);
    });
}

int pa_bm_fork(pa_bm *bm, int64_t parent, int64_t child) {
    pa::clear_error();
    if (!bm) return pa::fail(PA_ERR_INVALID, "bm_fork: NULL manager");
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end()) return pa::fail(PA_ERR_INVALID, "bm_fork: unknown parent");
    if (bm->seqs.count(child)) return pa::fail(PA_ERR_INVALID, "bm_fork: child exists");
    return guarded("bm_fork", [&] {
        alloc_point();
        pa_bm::Seq c = it->second;
        alloc_point();
        // (the insertion may rehash: `it` is not used after it)
        const pa_bm::Seq &cs = bm->seqs.emplace(child, std::move(c)).first->second;
        for (int32_t b : cs.blocks) ++bm->ref[b];
        return int(PA_OK);
    });
}

int pa_bm_append(pa_bm *bm, int64_t seq, int64_t *slot, int64_t *cow_src, int64_t *cow_dst) {
    pa::clear_error();
    if (!bm || !slot) return pa::fail(PA_ERR_INVALID, "bm_append: bad arguments");
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return pa::fail(PA_ERR_INVALID, "bm_append: unknown sequence");
    if (bm->needed(it->second, 1) > int64_t(bm->free_stack.size()))
        return pa::fail(PA_ERR_OOM, "bm_append: no free block");
    return guarded("bm_append", [&] {
        pa_bm::Seq &s = it->second;
        ensure_capacity(s.blocks, size_t((s.len + 1 + bm->bs - 1) / bm->bs));
        append_one(bm, s, slot, cow_src, cow_dst);
        return int(PA_OK);
    });
}

int pa_bm_append_n(pa_bm *bm, int64_t seq, int64_t n, int64_t *slots, int64_t *cow_src,
                   int64_t *cow_dst) {
    pa::clear_error();
    if (!bm || n < 0 || (n > 0 && !slots))
        return pa::fail(PA_ERR_INVALID, "bm_append_n: bad arguments");
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return pa::fail(PA_ERR_INVALID, "bm_append_n: unknown sequence");
    if (bm->needed(it->second, n) > int64_t(bm->free_stack.size()))
        return pa::fail(PA_ERR_OOM, "bm_append_n: not enough free blocks");
    return guarded("bm_append_n", [&] {
        pa_bm::Seq &s = it->second;
        ensure_capacity(s.blocks, size_t((s.len + n + bm->bs - 1) / bm->bs));
        int64_t src = -1, dst = -1;
        for (int64_t i = 0; i < n; ++i) {
            int64_t a, b;
            append_one(bm, s, &slots[i], &a, &b);
            if (a >= 0) {
                src = a;
                dst = b;
            }
        }
        if (cow_src) *cow_src = src;
        if (cow_dst) *cow_dst = dst;
        return int(PA_OK);
    });
}

int pa_bm_free_seq(pa_bm *bm, int64_t seq) {
    pa::clear_error();
    if (!bm) return pa::fail(PA_ERR_INVALID, "bm_free_seq: NULL manager");
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return pa::fail(PA_ERR_INVALID, "bm_free_seq: unknown sequence");
    for (int32_t b : it->second.blocks) bm->release(b);
    bm->seqs.erase(it);
    return PA_OK;
}

int pa_bm_block_table(const pa_bm *bm, const int64_t *seqs, int n, int32_t *out,
                      int max_blocks) {
    pa::clear_error();
    if (!bm || n < 0 || max_blocks <= 0 || (n > 0 && (!seqs || !out)))
        return pa::fail(PA_ERR_INVALID, "bm_block_table: bad arguments");
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seqs[i]);
        if (it == bm->seqs.end())
            return pa::fail(PA_ERR_INVALID, "bm_block_table: unknown sequence %lld",
                            (long long)seqs[i]);
        if (int64_t(it->second.blocks.size()) > max_blocks)
            return pa::fail(PA_ERR_INVALID, "bm_block_table: sequence %lld has %zu blocks > %d",
                            (long long)seqs[i], it->second.blocks.size(), max_blocks);
    }
    for (int i = 0; i < n; ++i) {
        const auto &bl = bm->seqs.find(seqs[i])->second.blocks;
        int32_t *row = out + int64_t(i) * max_blocks;
        for (int j = 0; j < max_blocks; ++j) row[j] = j < int(bl.size()) ? bl[j] : 0;
    }
    return PA_OK;
}

int pa_bm_seq_len(const pa_bm *bm, int64_t seq, int64_t *len) {
    pa::clear_error();
    if (!bm || !len) return pa::fail(PA_ERR_INVALID, "bm_seq_len: bad arguments");
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return pa::fail(PA_ERR_INVALID, "bm_seq_len: unknown sequence");
    *len = it->second.len;
    return PA_OK;
}

int pa_bm_seq_blocks(const pa_bm *bm, int64_t seq, int32_t *out, int64_t cap, int64_t *n) {
    pa::clear_error();
    if (!bm || !n || cap < 0 || (cap > 0 && !out))
        return pa::fail(PA_ERR_INVALID, "bm_seq_blocks: bad arguments");
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return pa::fail(PA_ERR_INVALID, "bm_seq_blocks: unknown sequence");
    const auto &bl = it->second.blocks;
    *n = int64_t(bl.size());
    for (int64_t i = 0; i < *n && i < cap; ++i) out[i] = bl[i];
    return PA_OK;
}

int pa_bm_refcount(const pa_bm *bm, int64_t block, int *refcount) {
    pa::clear_error();
    if (!bm || !refcount || block < 0 || block >= bm->num_blocks)
        return pa::fail(PA_ERR_INVALID, "bm_refcount: bad arguments");
    *refcount = bm->ref[block];
    return PA_OK;
}

int64_t pa_bm_num_free(const pa_bm *bm) { return bm ? int64_t(bm->free_stack.size()) : -1; }

void pa_bm_inject_alloc_failure(int64_t k) {
    g_alloc_failure.store(k < 0 ? -1 : k, std::memory_order_relaxed);
}

}  // extern "C"
