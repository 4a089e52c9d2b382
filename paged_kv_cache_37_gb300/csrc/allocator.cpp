// allocator.cpp -- host O(1) free-list block allocator and demand paging.
//
// A LIFO stack of free block ids ("Why Naive KV-Caches Waste >60% VRAM",
// "Implementation Walkthrough": the stack starts as reversed(range(n)) so
// block 0 is handed out first; allocate pops, free appends; an empty stack is
// an out-of-memory error).  Allocation and release are O(1) per block
// (PageForge, "Five techniques", 02).  alloc(n) is all-or-nothing and a bad
// free changes nothing (PageFault README, "Test": exhaustion, double free,
// all-or-nothing).
//
// Shared blocks (PagedAttention blog, "Copy-on-Write for Parallel
// Sampling"): each block has a reference count -- 1 when allocated, one more
// per share (a forked sequence's table pointing at the parent's blocks).  A
// free drops one reference per listed id and returns a block to the stack
// when its last reference goes, in list order.  Copy-on-write gives a writer
// a fresh block for a block others still reference and patches only the
// writer's table entry; the caller copies the contents (pf_copy_blocks).
//
// shuffle_seed != 0 permutes the initial hand-out order (a pool after churn,
// PageFault README "Four stages") with Fisher-Yates driven by SplitMix64
// (Steele, Lea and Flood, OOPSLA 2014), drawing j uniform in [0, i] by
// rejecting the low 2^64 mod (i + 1) outputs.
#include <cstdint>
#include <new>
#include <vector>

#include "internal.h"

struct pf_alloc {
    int n_blocks;
    std::vector<int32_t> stack;   // free ids; back() is handed out next
    std::vector<uint32_t> refs;   // references per block; 0 = free
};

namespace {

struct SplitMix64 {
    uint64_t state;
    uint64_t next() {
        state += 0x9E3779B97F4A7C15ull;
        uint64_t z = state;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        return z ^ (z >> 31);
    }
    // Uniform in [0, n), n >= 1.
    uint64_t below(uint64_t n) {
        uint64_t threshold = (0 - n) % n;   // 2^64 mod n
        for (;;) {
            uint64_t r = next();
            if (r >= threshold) return r % n;
        }
    }
};

int64_t blocks_for(int64_t len, int block_size) {
    return (len + block_size - 1) / block_size;
}

}  // namespace

extern "C" {

int pf_alloc_create(pf_alloc **out, int n_blocks, uint64_t shuffle_seed) {
    pkv::clear_error();
    if (!out) return pkv::set_error(PF_ERR_INVALID, "pf_alloc_create: out is null");
    *out = nullptr;
    if (n_blocks <= 0)
        return pkv::set_error(PF_ERR_INVALID, "pf_alloc_create: n_blocks must be positive");
    pf_alloc *a = new (std::nothrow) pf_alloc;
    if (!a) return pkv::set_error(PF_ERR_OOM, "pf_alloc_create: host allocation failed");
    try {
        std::vector<int32_t> order(n_blocks);
        for (int i = 0; i < n_blocks; ++i) order[i] = i;
        if (shuffle_seed) {
            SplitMix64 rng{shuffle_seed};
            for (int i = n_blocks - 1; i > 0; --i) {
                int j = (int)rng.below((uint64_t)i + 1);
                int32_t tmp = order[i];
                order[i] = order[j];
                order[j] = tmp;
            }
        }
        a->n_blocks = n_blocks;
        a->stack.assign(order.rbegin(), order.rend());
        a->refs.assign(n_blocks, 0);
    } catch (...) {
        delete a;
        return pkv::set_error(PF_ERR_OOM, "pf_alloc_create: host allocation failed");
    }
    *out = a;
    return PF_OK;
}

int pf_alloc_destroy(pf_alloc *a) {
    pkv::clear_error();
    delete a;
    return PF_OK;
}

int pf_alloc_free_count(const pf_alloc *a) {
    return a ? (int)a->stack.size() : -1;
}

int pf_alloc_blocks(pf_alloc *a, int n, int32_t *ids_out) {
    pkv::clear_error();
    if (!a) return pkv::set_error(PF_ERR_INVALID, "pf_alloc_blocks: null allocator");
    if (n < 0) return pkv::set_error(PF_ERR_INVALID, "pf_alloc_blocks: negative count");
    if (n > 0 && !ids_out) return pkv::set_error(PF_ERR_INVALID, "pf_alloc_blocks: ids_out is null");
    if ((size_t)n > a->stack.size())
        return pkv::set_error(PF_ERR_OOM, "pf_alloc_blocks: need " + std::to_string(n) +
                                              " blocks, " + std::to_string(a->stack.size()) + " free");
    for (int i = 0; i < n; ++i) {
        int32_t b = a->stack.back();
        a->stack.pop_back();
        a->refs[b] = 1;
        ids_out[i] = b;
    }
    return PF_OK;
}

int pf_free_blocks(pf_alloc *a, const int32_t *ids, int n) {
    pkv::clear_error();
    if (!a) return pkv::set_error(PF_ERR_INVALID, "pf_free_blocks: null allocator");
    if (n < 0) return pkv::set_error(PF_ERR_INVALID, "pf_free_blocks: negative count");
    if (n > 0 && !ids) return pkv::set_error(PF_ERR_INVALID, "pf_free_blocks: ids is null");
    // Validate everything first (taking the references as we go, so a block
    // listed more often than it is referenced is caught), then give them back:
    // the call is all-or-nothing.
    int bad = -1;
    for (int i = 0; i < n; ++i) {
        int32_t b = ids[i];
        if (b < 0 || b >= a->n_blocks || a->refs[b] == 0) { bad = i; break; }
        --a->refs[b];
    }
    for (int i = 0; i < (bad < 0 ? n : bad); ++i) ++a->refs[ids[i]];
    if (bad >= 0)
        return pkv::set_error(PF_ERR_DOUBLE_FREE, "pf_free_blocks: block " + std::to_string(ids[bad]) +
                                                      " is not allocated (or listed more often than it is "
                                                      "referenced)");
    for (int i = 0; i < n; ++i) {
        if (--a->refs[ids[i]] == 0) a->stack.push_back(ids[i]);
    }
    return PF_OK;
}

int pf_alloc_share(pf_alloc *a, const int32_t *ids, int n) {
    pkv::clear_error();
    if (!a) return pkv::set_error(PF_ERR_INVALID, "pf_alloc_share: null allocator");
    if (n < 0) return pkv::set_error(PF_ERR_INVALID, "pf_alloc_share: negative count");
    if (n > 0 && !ids) return pkv::set_error(PF_ERR_INVALID, "pf_alloc_share: ids is null");
    for (int i = 0; i < n; ++i) {
        int32_t b = ids[i];
        if (b < 0 || b >= a->n_blocks || a->refs[b] == 0)
            return pkv::set_error(PF_ERR_INVALID, "pf_alloc_share: block " + std::to_string(b) +
                                                      " is not allocated");
        if (a->refs[b] >= 0x7fffffffu - (uint32_t)n)
            return pkv::set_error(PF_ERR_INVALID, "pf_alloc_share: reference count overflow");
    }
    for (int i = 0; i < n; ++i) ++a->refs[ids[i]];
    return PF_OK;
}

int pf_alloc_refcount(const pf_alloc *a, int32_t id) {
    if (!a || id < 0 || id >= a->n_blocks) return -1;
    return (int)a->refs[id];
}

int pf_alloc_cow(pf_alloc *a, int32_t *entry, int32_t *src_out, int32_t *dst_out) {
    pkv::clear_error();
    if (!a || !entry || !src_out || !dst_out) return pkv::set_error(PF_ERR_INVALID, "pf_alloc_cow: null argument");
    const int32_t b = *entry;
    if (b < 0 || b >= a->n_blocks || a->refs[b] == 0)
        return pkv::set_error(PF_ERR_INVALID, "pf_alloc_cow: block " + std::to_string(b) + " is not allocated");
    *src_out = b;
    *dst_out = -1;
    if (a->refs[b] == 1) return PF_OK;   // the writer's own block: write in place
    if (a->stack.empty()) return pkv::set_error(PF_ERR_OOM, "pf_alloc_cow: need 1 block, 0 free");
    const int32_t d = a->stack.back();
    a->stack.pop_back();
    a->refs[d] = 1;
    --a->refs[b];
    *entry = d;
    *dst_out = d;
    return PF_OK;
}

int pf_seq_reserve(pf_alloc *a, int block_size, int32_t *table_row, int max_blocks,
                   int cur_len, int new_len) {
    pkv::clear_error();
    if (!a || !table_row) return pkv::set_error(PF_ERR_INVALID, "pf_seq_reserve: null argument");
    if (block_size <= 0 || cur_len < 0 || new_len < cur_len || max_blocks < 0)
        return pkv::set_error(PF_ERR_INVALID, "pf_seq_reserve: bad sizes");
    int64_t have = blocks_for(cur_len, block_size);
    int64_t need = blocks_for(new_len, block_size);
    if (need > max_blocks)
        return pkv::set_error(PF_ERR_INVALID, "pf_seq_reserve: table row holds " +
                                                  std::to_string(max_blocks) + " blocks, need " +
                                                  std::to_string(need));
    if (need == have) return PF_OK;
    return pf_alloc_blocks(a, (int)(need - have), table_row + have);
}

int pf_seq_fork(pf_alloc *a, int block_size, const int32_t *parent_row, int len, int32_t *child_row,
                int max_blocks) {
    pkv::clear_error();
    if (!a || !parent_row || !child_row) return pkv::set_error(PF_ERR_INVALID, "pf_seq_fork: null argument");
    if (block_size <= 0 || len < 0 || max_blocks < 0) return pkv::set_error(PF_ERR_INVALID, "pf_seq_fork: bad sizes");
    const int64_t n = blocks_for(len, block_size);
    if (n > max_blocks)
        return pkv::set_error(PF_ERR_INVALID, "pf_seq_fork: table row holds " + std::to_string(max_blocks) +
                                                  " blocks, need " + std::to_string(n));
    int rc = pf_alloc_share(a, parent_row, (int)n);
    if (rc) return rc;
    for (int64_t i = 0; i < n; ++i) child_row[i] = parent_row[i];
    return PF_OK;
}

int pf_seq_release(pf_alloc *a, int block_size, const int32_t *table_row, int len) {
    pkv::clear_error();
    if (!a || !table_row) return pkv::set_error(PF_ERR_INVALID, "pf_seq_release: null argument");
    if (block_size <= 0 || len < 0) return pkv::set_error(PF_ERR_INVALID, "pf_seq_release: bad sizes");
    return pf_free_blocks(a, table_row, (int)blocks_for(len, block_size));
}

}  // extern "C"
