// Host block allocator: one global pool of fixed-size physical blocks, a
// free list and a reference count per physical block.
//
//  "3.3 页面级显存管理" 3.3.2 (batch allocation at prefill, one more block
//    when the token count passes num_blocks*block_size, refcounts and
//    sharing), 3.3.4 (one global pool, O(1) alloc and free)
//  "vLLM三大核心技术分页内存与共享解码", "Copy-on-Write共享解码的显存优化原理"
//    (write in place at refcount 1, else copy to a new block, repoint the
//    table and drop one reference; free at refcount 0)
//  "3.1 PagedAttention的核心原理" 3.1.5 (CoW steps 1-4)
//
// Layout: `stack` holds the free ids (top = stack[top-1]) and `rc` the
// count of every block (0 = free).  Every operation validates all of its
// inputs before changing anything, so a failure leaves the pool as it was.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>
#include <utility>
#include <vector>

#include "pagedkv.h"
#include "pkv_internal.h"

struct pkv_allocator {
    int32_t num_blocks = 0;
    int32_t top = 0;               // number of free blocks
    int32_t shared = 0;            // blocks with rc > 1
    std::vector<int32_t> stack;    // free ids, top of stack at [top-1]
    std::vector<int32_t> rc;       // refcount per block
    std::vector<int32_t> delta;    // fork scratch, all zero between calls
    std::vector<int32_t> nchild;   // fork scratch: children per row
    std::vector<int32_t> rows;     // fork scratch: the old tables
};

namespace {

void set_rc(pkv_allocator* a, int32_t id, int32_t v) {
    int32_t old = a->rc[id];
    a->shared += (v > 1) - (old > 1);
    a->rc[id] = v;
}

int32_t pop(pkv_allocator* a) {
    int32_t id = a->stack[--a->top];
    set_rc(a, id, 1);
    return id;
}

void push(pkv_allocator* a, int32_t id) {
    a->stack[a->top++] = id;
}

bool valid_id(const pkv_allocator* a, int32_t id) { return id >= 0 && id < a->num_blocks; }

}  // namespace

extern "C" {

pkv_status pkv_alloc_create(int32_t num_blocks, pkv_allocator** out) {
    PKV_TRACE("pkv_alloc_create");
    pkv::clear_error();
    if (!out || num_blocks < 0) return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_create: bad argument");
    pkv_allocator* a = new (std::nothrow) pkv_allocator();
    if (!a) return pkv::fail(PKV_ERR_HOST_MEMORY, "alloc_create: out of host memory");
    try {
        a->num_blocks = num_blocks;
        a->stack.resize(num_blocks);
        a->rc.assign(num_blocks, 0);
        a->delta.assign(num_blocks, 0);
    } catch (...) {
        delete a;
        return pkv::fail(PKV_ERR_HOST_MEMORY, "alloc_create: out of host memory");
    }
    // popping from the top hands out num_blocks-1 first
    for (int32_t i = 0; i < num_blocks; ++i) a->stack[i] = i;
    a->top = num_blocks;
    *out = a;
    return PKV_OK;
}

pkv_status pkv_alloc_create_with_order(int32_t num_blocks, const int32_t* initial_free,
                                       int32_t n_free, pkv_allocator** out) {
    PKV_TRACE("pkv_alloc_create_with_order");
    pkv::clear_error();
    if (!out || num_blocks < 0 || n_free < 0 || n_free > num_blocks || (n_free && !initial_free))
        return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_create_with_order: bad argument");
    std::vector<uint8_t> seen;
    try {
        seen.assign(num_blocks, 0);
    } catch (...) {
        return pkv::fail(PKV_ERR_HOST_MEMORY, "alloc_create_with_order: out of host memory");
    }
    for (int32_t i = 0; i < n_free; ++i) {
        int32_t id = initial_free[i];
        if (id < 0 || id >= num_blocks || seen[id])
            return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_create_with_order: id out of range or repeated");
        seen[id] = 1;
    }
    pkv_allocator* a = nullptr;
    pkv_status st = pkv_alloc_create(num_blocks, &a);
    if (st != PKV_OK) return st;
    for (int32_t i = 0; i < n_free; ++i) a->stack[i] = initial_free[i];
    a->top = n_free;
    for (int32_t id = 0; id < num_blocks; ++id)
        if (!seen[id]) a->rc[id] = 1;
    *out = a;
    return PKV_OK;
}

void pkv_alloc_destroy(pkv_allocator* a) { delete a; }

pkv_status pkv_alloc_blocks(pkv_allocator* a, int32_t n, int32_t* out_ids) {
    PKV_TRACE("pkv_alloc_blocks");
    pkv::clear_error();
    if (!a || n < 0 || (n && !out_ids)) return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_blocks: bad argument");
    if (a->top < n) return pkv::fail(PKV_ERR_OOM, "alloc_blocks: out of free blocks");
    for (int32_t i = 0; i < n; ++i) out_ids[i] = pop(a);
    return PKV_OK;
}

pkv_status pkv_alloc_incref(pkv_allocator* a, const int32_t* ids, int32_t n) {
    PKV_TRACE("pkv_alloc_incref");
    pkv::clear_error();
    if (!a || n < 0 || (n && !ids)) return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_incref: bad argument");
    for (int32_t i = 0; i < n; ++i)
        if (!valid_id(a, ids[i]) || a->rc[ids[i]] <= 0)
            return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_incref: block not held");
    for (int32_t i = 0; i < n; ++i) set_rc(a, ids[i], a->rc[ids[i]] + 1);
    return PKV_OK;
}

pkv_status pkv_alloc_decref(pkv_allocator* a, const int32_t* ids, int32_t n, int32_t* num_freed) {
    PKV_TRACE("pkv_alloc_decref");
    pkv::clear_error();
    if (!a || n < 0 || (n && !ids)) return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_decref: bad argument");
    // validate with multiplicity: a block listed k times needs rc >= k
    for (int32_t i = 0; i < n; ++i)
        if (!valid_id(a, ids[i])) return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_decref: id out of range");
    for (int32_t i = 0; i < n; ++i) a->rc[ids[i]] -= 1;
    bool ok = true;
    for (int32_t i = 0; i < n; ++i) ok = ok && a->rc[ids[i]] >= 0;
    for (int32_t i = 0; i < n; ++i) a->rc[ids[i]] += 1;  // undo the probe
    if (!ok) return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_decref: block not held");
    int32_t freed = 0;
    for (int32_t i = 0; i < n; ++i) {
        int32_t id = ids[i];
        set_rc(a, id, a->rc[id] - 1);
        if (a->rc[id] == 0) {
            push(a, id);
            ++freed;
        }
    }
    if (num_freed) *num_freed = freed;
    return PKV_OK;
}

pkv_status pkv_alloc_cow(pkv_allocator* a, int32_t id, int32_t* out_id, int32_t* needs_copy) {
    PKV_TRACE("pkv_alloc_cow");
    pkv::clear_error();
    if (!a || !out_id || !needs_copy || !valid_id(a, id) || a->rc[id] <= 0)
        return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_cow: bad argument or block not held");
    if (a->rc[id] == 1) {
        *out_id = id;
        *needs_copy = 0;
        return PKV_OK;
    }
    if (a->top < 1) return pkv::fail(PKV_ERR_OOM, "alloc_cow: out of free blocks");
    int32_t fresh = pop(a);
    set_rc(a, id, a->rc[id] - 1);
    *out_id = fresh;
    *needs_copy = 1;
    return PKV_OK;
}

pkv_status pkv_alloc_append(pkv_allocator* a, int32_t* table, int32_t* num_blocks,
                            int32_t max_blocks, int32_t ctx_before, int32_t n_new, int32_t bs,
                            int64_t* pairs, int32_t* n_pairs) {
    PKV_TRACE("pkv_alloc_append");
    pkv::clear_error();
    if (!a || !num_blocks || !n_pairs || bs <= 0 || ctx_before < 0 || n_new < 0 ||
        *num_blocks < 0 || *num_blocks > max_blocks || (max_blocks > 0 && !table))
        return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_append: bad argument");
    *n_pairs = 0;
    if (n_new == 0) return PKV_OK;
    const int64_t ctx_after = (int64_t)ctx_before + n_new;
    const int64_t first = ctx_before / bs, last = (ctx_after - 1) / bs;
    const int64_t blocks_needed = (ctx_after + bs - 1) / bs;
    const int32_t nb = *num_blocks;
    if (blocks_needed > max_blocks) return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_append: table row too short");
    if (first > nb) return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_append: table shorter than the cached tokens");
    int64_t shared = 0;
    for (int64_t lb = first; lb <= last && lb < nb; ++lb) {
        int32_t id = table[lb];
        if (!valid_id(a, id) || a->rc[id] <= 0)
            return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_append: table holds a block that is not held");
        if (!pairs && a->rc[id] > 1) return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_append: pairs is null");
        shared += a->rc[id] > 1;
    }
    const int64_t fresh = blocks_needed > nb ? blocks_needed - nb : 0;
    if (a->top < fresh + shared) return pkv::fail(PKV_ERR_OOM, "alloc_append: out of free blocks");
    int32_t k = 0;
    for (int64_t lb = first; lb <= last && lb < nb; ++lb) {
        int32_t id = table[lb];
        if (a->rc[id] > 1) {
            int32_t nid = pop(a);
            set_rc(a, id, a->rc[id] - 1);
            pairs[2 * k] = id;
            pairs[2 * k + 1] = nid;
            ++k;
            table[lb] = nid;
        }
    }
    for (int64_t i = 0; i < fresh; ++i) table[nb + i] = pop(a);
    *num_blocks = (int32_t)blocks_needed > nb ? (int32_t)blocks_needed : nb;
    *n_pairs = k;
    return PKV_OK;
}

pkv_status pkv_alloc_append_batch(pkv_allocator* a, int32_t* tables, int32_t* num_blocks,
                                  int32_t S, int32_t MB, const int32_t* ctx_before,
                                  const int32_t* n_new, int32_t bs, int64_t* pairs,
                                  int32_t max_pairs, int32_t* n_pairs, int32_t* n_done) {
    PKV_TRACE("pkv_alloc_append_batch");
    pkv::clear_error();
    if (!a || S < 0 || MB < 0 || (S > 0 && (!num_blocks || !ctx_before || !n_new)) ||
        (S > 0 && MB > 0 && !tables) || !n_pairs || !n_done || max_pairs < 0 ||
        (max_pairs > 0 && !pairs))
        return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_append_batch: bad argument");
    *n_pairs = 0;
    *n_done = 0;
    int64_t one[2 * 64];
    for (int32_t s = 0; s < S; ++s) {
        // one sequence's copies fit in ceil(n_new/bs) + 1 pairs
        const int64_t cap = (int64_t)n_new[s] / (bs > 0 ? bs : 1) + 2;
        std::vector<int64_t> big;
        int64_t* buf = one;
        if (cap > 64) {
            try {
                big.resize(2 * cap);
            } catch (...) {
                return pkv::fail(PKV_ERR_HOST_MEMORY, "alloc_append_batch: out of host memory");
            }
            buf = big.data();
        }
        // refuse before touching sequence s if its copies might not fit
        if (*n_pairs + cap > max_pairs)
            return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_append_batch: pairs buffer too small");
        int32_t np = 0;
        int32_t nb = num_blocks[s];
        pkv_status st = pkv_alloc_append(a, tables + (int64_t)s * MB, &nb, MB, ctx_before[s],
                                         n_new[s], bs, buf, &np);
        if (st != PKV_OK) return st;  // error text already set; nothing changed for s
        num_blocks[s] = nb;
        for (int32_t k = 0; k < np; ++k) {
            pairs[2 * (*n_pairs + k)] = buf[2 * k];
            pairs[2 * (*n_pairs + k) + 1] = buf[2 * k + 1];
        }
        *n_pairs += np;
        *n_done = s + 1;
    }
    return PKV_OK;
}

pkv_status pkv_alloc_fork(pkv_allocator* a, int32_t* tables, int32_t* num_blocks, int32_t S,
                          int32_t MB, const int32_t* parents) {
    PKV_TRACE("pkv_alloc_fork");
    pkv::clear_error();
    if (!a || S < 0 || MB < 0 || (S > 0 && (!num_blocks || !parents)) || (S > 0 && MB > 0 && !tables))
        return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_fork: bad argument");
    for (int32_t s = 0; s < S; ++s) {
        if (parents[s] < 0 || parents[s] >= S || num_blocks[s] < 0 || num_blocks[s] > MB)
            return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_fork: bad parent or row length");
        for (int32_t j = 0; j < num_blocks[s]; ++j) {
            const int32_t id = tables[(int64_t)s * MB + j];
            if (!valid_id(a, id) || a->rc[id] <= 0)
                return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_fork: table holds a block that is not held");
        }
    }
    // Row r of the old tables is copied into nchild[r] new rows, so each of
    // its entries changes its block's count by nchild[r] - 1: rows forked
    // once change nothing.  The counts are checked before anything changes
    // (no release may underflow), then holds are added (rows with several
    // children) before the releases (rows with none), in row order, so a
    // block that survives never reaches 0 and the freed blocks reach the
    // free list in the order the releases one by one would give.
    try {
        a->nchild.assign(S, 0);
        a->rows.assign(tables, tables + (size_t)S * MB);
    } catch (...) {
        return pkv::fail(PKV_ERR_HOST_MEMORY, "alloc_fork: out of host memory");
    }
    int32_t* nchild = a->nchild.data();
    const int32_t* old_tab = a->rows.data();
    for (int32_t s = 0; s < S; ++s) ++nchild[parents[s]];
    int32_t* delta = a->delta.data();
    for (int32_t r = 0; r < S; ++r) {
        if (nchild[r] == 1) continue;
        for (int32_t j = 0; j < num_blocks[r]; ++j) delta[old_tab[(size_t)r * MB + j]] += nchild[r] - 1;
    }
    bool ok = true;
    for (int32_t r = 0; r < S; ++r) {
        if (nchild[r] == 1) continue;
        for (int32_t j = 0; j < num_blocks[r]; ++j) {
            const int32_t id = old_tab[(size_t)r * MB + j];
            ok = ok && a->rc[id] + delta[id] >= 0;
            delta[id] = 0;
        }
    }
    if (!ok) return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_fork: release would underflow a refcount");
    for (int32_t r = 0; r < S; ++r) {
        if (nchild[r] < 2) continue;
        for (int32_t j = 0; j < num_blocks[r]; ++j) {
            const int32_t id = old_tab[(size_t)r * MB + j];
            set_rc(a, id, a->rc[id] + nchild[r] - 1);
        }
    }
    for (int32_t r = 0; r < S; ++r) {
        if (nchild[r] != 0) continue;
        for (int32_t j = 0; j < num_blocks[r]; ++j) {
            const int32_t id = old_tab[(size_t)r * MB + j];
            set_rc(a, id, a->rc[id] - 1);
            if (a->rc[id] == 0) push(a, id);
        }
    }
    std::vector<int32_t>& old_nb = a->nchild;  // children counted; reuse for the lengths
    std::copy(num_blocks, num_blocks + S, old_nb.begin());
    for (int32_t s = 0; s < S; ++s) {
        const int32_t p = parents[s];
        std::memcpy(tables + (size_t)s * MB, old_tab + (size_t)p * MB, (size_t)MB * 4);
        num_blocks[s] = old_nb[p];
    }
    return PKV_OK;
}

pkv_status pkv_alloc_refcount(const pkv_allocator* a, int32_t id, int32_t* rc) {
    pkv::clear_error();
    if (!a || !rc || !valid_id(a, id)) return pkv::fail(PKV_ERR_INVALID_ARG, "alloc_refcount: bad argument");
    *rc = a->rc[id];
    return PKV_OK;
}

pkv_status pkv_check_copy_pairs(const int64_t* pairs, int32_t P, int32_t NB) {
    PKV_TRACE("pkv_check_copy_pairs");
    pkv::clear_error();
    if (P < 0 || NB < 0 || (P > 0 && !pairs)) return pkv::fail(PKV_ERR_INVALID_ARG, "check_copy_pairs: bad argument");
    char msg[160];
    for (int32_t i = 0; i < P; ++i) {
        if (pairs[2 * i] < 0 || pairs[2 * i] >= NB || pairs[2 * i + 1] < 0 || pairs[2 * i + 1] >= NB) {
            snprintf(msg, sizeof msg, "check_copy_pairs: pair %d holds an id outside [0, %d)", i, NB);
            return pkv::fail(PKV_ERR_INVALID_ARG, msg);
        }
    }
    // (dst, pair index) sorted by dst: a repeated dst sits next to its twin,
    // and each src is looked up among the dsts by binary search
    std::vector<std::pair<int64_t, int32_t>> dst;
    try {
        dst.resize(P);
    } catch (...) {
        return pkv::fail(PKV_ERR_HOST_MEMORY, "check_copy_pairs: out of host memory");
    }
    for (int32_t i = 0; i < P; ++i) dst[i] = {pairs[2 * i + 1], i};
    std::sort(dst.begin(), dst.end());
    for (int32_t i = 1; i < P; ++i) {
        if (dst[i].first == dst[i - 1].first) {
            snprintf(msg, sizeof msg, "check_copy_pairs: pairs %d and %d copy into the same block %lld",
                     dst[i - 1].second, dst[i].second, (long long)dst[i].first);
            return pkv::fail(PKV_ERR_INVALID_ARG, msg);
        }
    }
    for (int32_t i = 0; i < P; ++i) {
        const int64_t src = pairs[2 * i];
        auto it = std::lower_bound(dst.begin(), dst.end(), std::make_pair(src, (int32_t)-1));
        if (it != dst.end() && it->first == src) {
            snprintf(msg, sizeof msg, "check_copy_pairs: block %lld is the source of pair %d and the target of pair %d",
                     (long long)src, i, it->second);
            return pkv::fail(PKV_ERR_INVALID_ARG, msg);
        }
    }
    return PKV_OK;
}

int32_t pkv_alloc_num_blocks(const pkv_allocator* a) { return a ? a->num_blocks : 0; }
int32_t pkv_alloc_num_free(const pkv_allocator* a) { return a ? a->top : 0; }
int32_t pkv_alloc_num_shared(const pkv_allocator* a) { return a ? a->shared : 0; }

}  // extern "C"
