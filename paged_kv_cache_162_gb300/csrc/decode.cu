// Single-query paged decode attention for sm_103a.
//
// What it computes ("3.1 PagedAttention的核心原理" 3.1.3; notes on "vLLM: Easy,
// Fast, and Cheap LLM Serving with PagedAttention", "疑问" 1): for every
// sequence s and head h, out = softmax(scale * q K^T) V over the sequence's
// context, each token's K/V row found through the block table (logical =
// j / bs, offset = j % bs, physical = table[logical]).
//
// How (HBM-bound GEMV: 1 FMA per 16-bit element loaded, so no tensor cores):
//  * A work item is (sequence, partition of `PT` tokens, group of 4 heads).
//    The CTA has 4 warps, one per head; a warp streams its partition in
//    16-token tiles.  Within a tile, lane (r, c) loads 16 bytes (8 dims,
//    chunk c) of rows r, r + RPI, ... so every warp-wide load reads whole
//    256-byte (D=128) or 128-byte (D=64) rows: coalesced 128-bit loads, and
//    the 4 warps of a CTA together read 4 consecutive heads = 1 KB (512 B)
//    of each token row.  Only tiles of one physical block are read together
//    ("3.3 页面级显存管理" 3.3.1: work organised per physical block, reads
//    within a block coalesced).
//  * q.k: per-lane partial dots over 8 dims with fp32-accumulating fma on
//    the 16-bit operands themselves (the products are exact in fp32), then a
//    reduce-scatter across the lanes of a row (log2(NI) halving steps + one
//    xor-1 step) leaves each lane with the full logit of one row.  Online
//    softmax in log2 units (logits scaled by scale*log2(e)); P.V
//    accumulates 8 dims per lane in fp32 and is combined across row groups
//    once at the end.
//  * The tile loop is software-pipelined on the registers it already has:
//    the V loads of tile t are in flight while q.K(t) is computed, the K
//    loads of tile t+1 while P.V(t) is accumulated.  Full tiles take no
//    per-row predicates.
//  * Block table: each warp keeps a window of 64 of its partition's table
//    entries in shared memory, filled by one coalesced load across its lanes
//    and refilled when a tile passes the window, so a tile's lookup is a
//    shared-memory read ("3.1 PagedAttention的核心原理" 3.1.3: the kernel
//    indexes a flat block_table array).  Tile t+1's lookup is made while
//    tile t is computed, so it stays off the load chain.
//  * Partitions: a context longer than PT tokens is split.  Each partition
//    writes (running max, running sum, unnormalised output) to the
//    workspace; the CTA that finishes a (sequence, head group) last -- known
//    from an atomic ticket, no waiting -- merges them.  A single-partition
//    context writes its output directly.
//  * Scheduling: one CTA plans (plan_cta): it chooses the partition size,
//    lists the (sequence, partition) items -- full partitions in sequence
//    order, with the partial (last) partitions before or after them -- and
//    resets the work counter and tickets.  The plan runs as plan_kernel, or
//    as CTA 0 of step_prologue_kernel when a whole decode step (slot
//    mapping, cache write, attention) is one call.  The decode kernel is
//    persistent (as many CTAs as fit on the SMs) and takes items from the
//    counter.  It is launched with programmatic dependent launch so its
//    CTAs are resident when the plan ends.
//  * Shared prefixes: when sequences share the blocks of a prefix, a
//    prefix kernel (mma.sync, or tcgen05 + TMA in prefix_tc.cuh) reads each
//    shared block once for all members of the group; the decode kernel then
//    covers only the members' own tokens.  The prefix kernel has completed
//    when the decode kernel begins, so a member whose own tokens are one
//    partition merges the prefix partials into it in registers; otherwise
//    the tickets merge both.
//  * Safety: a table entry outside [0, NB) or a context outside
//    [0, max_context_len] is never dereferenced; the kernel masks it and
//    sets a bit in the device error word.  No CTA ever waits on another.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "pagedkv.h"
#include "pkv_device.cuh"

namespace {

constexpr int kWarps = 4;                // heads per CTA, one warp per head
constexpr int kThreads = 32 * kWarps;
constexpr int kTile = 16;                // tokens per tile
constexpr int kMinAutoPartition = 64;    // smallest partition the automatic choice uses
constexpr int kAutoCandidates = 7;       // 64, 128, ..., 4096 tokens
constexpr int kItemsPerCta = 6;          // automatic choice: at least this many items per CTA
constexpr int kPlanThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

struct Workspace {
    unsigned* counter;  // next work item
    int* n_items;       // number of (sequence, partition) items
    int* pt;            // tokens per partition chosen by the plan kernel
    unsigned* pcounter; // next prefix item (shared-prefix decode)
    int* n_pitems;      // number of (group, partition) prefix items
    int* pitems;        // packed (group << 16 | partition)
    int* pre_parts;     // per sequence: leading partitions its group's prefix covers
    int* items;         // packed (sequence << 16 | partition)
    int* nparts;        // partitions per sequence
    unsigned* tickets;  // per (sequence, head group): partitions finished
    float* m;           // [S][H][max_parts] running max (log2 units)
    float* l;           // [S][H][max_parts] running sum
    float* acc;         // [S][H][max_parts][D] unnormalised output
};

struct Layout {
    size_t items, nparts, tickets, m, l, acc, pre_parts, pitems, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

Layout layout_of(int S, int H, int D, int max_parts) {
    const size_t HG = (size_t)(H + kWarps - 1) / kWarps;
    const size_t part_elems = (size_t)S * H * max_parts;
    Layout L;
    size_t o = 256;  // header: counter, n_items, partition size
    L.items = o;   o = align256(o + (size_t)S * max_parts * sizeof(int));
    L.nparts = o;  o = align256(o + (size_t)S * sizeof(int));
    L.tickets = o; o = align256(o + (size_t)S * HG * sizeof(unsigned));
    L.m = o;       o = align256(o + part_elems * sizeof(float));
    L.l = o;       o = align256(o + part_elems * sizeof(float));
    L.acc = o;     o = align256(o + part_elems * D * sizeof(float));
    L.pre_parts = L.pitems = 0;
    L.total = o;
    return L;
}

// The decode layout plus what shared-prefix decode needs: per-sequence
// prefix partition counts and the list of (group, partition) items.
Layout layout_shared(int S, int H, int D, int G, int max_parts) {
    Layout L = layout_of(S, H, D, max_parts);
    size_t o = L.total;
    L.pre_parts = o; o = align256(o + (size_t)S * sizeof(int));
    L.pitems = o;    o = align256(o + (size_t)(G > 0 ? G : 1) * max_parts * sizeof(int));
    L.total = o;
    return L;
}

Workspace bind(void* base, const Layout& L) {
    char* b = static_cast<char*>(base);
    Workspace w;
    w.counter = reinterpret_cast<unsigned*>(b);
    w.n_items = reinterpret_cast<int*>(b + 4);
    w.pt = reinterpret_cast<int*>(b + 8);
    w.pcounter = reinterpret_cast<unsigned*>(b + 12);
    w.n_pitems = reinterpret_cast<int*>(b + 16);
    w.pre_parts = L.pre_parts ? reinterpret_cast<int*>(b + L.pre_parts) : nullptr;
    w.pitems = L.pitems ? reinterpret_cast<int*>(b + L.pitems) : nullptr;
    w.items = reinterpret_cast<int*>(b + L.items);
    w.nparts = reinterpret_cast<int*>(b + L.nparts);
    w.tickets = reinterpret_cast<unsigned*>(b + L.tickets);
    w.m = reinterpret_cast<float*>(b + L.m);
    w.l = reinterpret_cast<float*>(b + L.l);
    w.acc = reinterpret_cast<float*>(b + L.acc);
    return w;
}

struct DecodeParams {
    void* out;
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int S, H, NB, MB, HG, max_parts, max_ctx;
    float qscale;  // scale * log2(e)
    Workspace ws;
    int* err;
};

__device__ __forceinline__ int clamp_ctx(int c, int max_ctx) {
    return c < 0 ? 0 : (c > max_ctx ? max_ctx : c);
}

// ---------------------------------------------------------------------------
// Plan: choose the partition size, list the work items, reset the counter
// and the tickets.  One CTA.
//
// Partition size when the caller leaves it to the library: the largest of
// pt_min, 2*pt_min, ... that still gives every resident CTA at least
// kItemsPerCta items (so the tail is short) and is at most 3/4 of the mean
// context (so ragged contexts split into similar pieces).
//
// Order of the items: when the partial (last) partitions are well filled --
// on average at least 3/8 of a partition -- they go first.  Their spread of
// lengths staggers the CTAs, so the full partitions that follow do not run
// in lock-step waves, and each sequence's merge follows its last full
// partition through the run instead of piling up at the end.  Nearly empty
// partial partitions go last instead, where they fill the final wave of
// full ones.  Either way the full partitions keep sequence order.
struct PlanArgs {
    const int32_t* context_lens;
    int S, pt_fixed, pt_min, max_ctx;
    int slots;      // CTAs of the decode kernel's grid
    int HG;         // head groups of 4 heads
    int n_tickets;  // S * HG
    Workspace ws;
    const int32_t* groups;  // shared-prefix groups (G of them) or nullptr
    int G;
    int* err;
};

// The plan, computed by one CTA of kPlanThreads threads.
__device__ __forceinline__ void plan_cta(const PlanArgs& pa) {
    const int32_t* __restrict__ context_lens = pa.context_lens;
    const int S = pa.S, pt_fixed = pa.pt_fixed, pt_min = pa.pt_min, max_ctx = pa.max_ctx;
    const int slots = pa.slots, HG = pa.HG, n_tickets = pa.n_tickets, G = pa.G;
    const Workspace& ws = pa.ws;
    const int32_t* __restrict__ groups = pa.groups;
    int* err = pa.err;
    constexpr int kWarpsP = kPlanThreads / 32;
    constexpr int kVals = 2 * kAutoCandidates;  // full and all partitions per candidate
    __shared__ int red[kWarpsP][kVals];
    __shared__ int tot[kVals];
    __shared__ long long red_ctx[kWarpsP];
    __shared__ long long s_ctx_sum;  // may exceed 2^31
    __shared__ int wsum[2][kWarpsP];
    __shared__ int carry[2];
    __shared__ int s_pt, s_full_total, s_items;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const bool fixed = pt_fixed > 0;
    const int ncand = fixed ? 1 : kAutoCandidates;

    // per candidate partition size: full partitions and all partitions
    int v[kVals];
    long long ctx_sum = 0;
#pragma unroll
    for (int k = 0; k < kVals; ++k) v[k] = 0;
    for (int s = tid; s < S; s += kPlanThreads) {
        int c = context_lens[s];
        if (c < 0 || c > max_ctx) {
            pkv::report(err, PKV_DEVERR_CONTEXT);
            c = clamp_ctx(c, max_ctx);
        }
        ctx_sum += c;
#pragma unroll
        for (int k = 0; k < kAutoCandidates; ++k) {
            if (k < ncand) {
                const int pt = fixed ? pt_fixed : (pt_min << k);
                const int nf = c / pt;
                v[k] += nf;
                v[kAutoCandidates + k] += nf + ((c % pt != 0 || c == 0) ? 1 : 0);
            }
        }
    }
#pragma unroll
    for (int k = 0; k < kVals; ++k) {
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) v[k] += __shfl_xor_sync(kFull, v[k], o);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ctx_sum += __shfl_xor_sync(kFull, ctx_sum, o);
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kVals; ++k) red[wid][k] = v[k];
        red_ctx[wid] = ctx_sum;
    }
    __syncthreads();
    if (tid < kVals) {
        int t = 0;
#pragma unroll
        for (int w = 0; w < kWarpsP; ++w) t += red[w][tid];
        tot[tid] = t;
    }
    if (tid == kVals) {
        long long t = 0;
#pragma unroll
        for (int w = 0; w < kWarpsP; ++w) t += red_ctx[w];
        s_ctx_sum = t;
    }
    __syncthreads();
    // shared prefixes (automatic size): partitions no longer than the
    // shortest valid group prefix, so whole partitions can be shared
    __shared__ int s_min_prefix;
    if (tid == 0) s_min_prefix = INT32_MAX;
    __syncthreads();
    if (G > 0 && !fixed) {
        for (int g = tid; g < G; g += kPlanThreads) {
            const int first = groups[3 * g], n = groups[3 * g + 1], ptok = groups[3 * g + 2];
            if (first >= 0 && n >= 1 && n <= 16 && first <= S - n && ptok >= pt_min && ptok % kTile == 0)
                atomicMin(&s_min_prefix, ptok);
        }
    }
    __syncthreads();
    if (tid == 0) {
        int pick = 0;
        if (!fixed && G > 0 && s_min_prefix != INT32_MAX) {
            bool fits = true;
#pragma unroll
            for (int k = 1; k < kAutoCandidates; ++k) {
                fits = fits && (pt_min << k) <= s_min_prefix;
                if (fits) pick = k;
            }
        } else if (!fixed) {
            const long long mean = S > 0 ? s_ctx_sum / S : 0;
            bool grow = true;
#pragma unroll
            for (int k = 1; k < kAutoCandidates; ++k) {
                const long long cand = (long long)pt_min << k;
                grow = grow && (long long)HG * tot[kAutoCandidates + k] >= (long long)kItemsPerCta * slots &&
                       4 * cand <= 3 * mean;
                if (grow) pick = k;
            }
        }
        s_pt = fixed ? pt_fixed : (pt_min << pick);
        s_full_total = tot[pick];
        s_items = tot[kAutoCandidates + pick];
        carry[0] = carry[1] = 0;
    }
    __syncthreads();
    const int PT = s_pt;

    // shared prefixes: every member of group g skips the first pp_g
    // partitions, which the prefix kernel computes for all members at once
    __shared__ int s_full_skip, s_pitems;
    if (ws.pre_parts) {  // read by the decode kernel whenever present
        for (int s = tid; s < S; s += kPlanThreads) ws.pre_parts[s] = 0;
    }
    if (G > 0) {
        if (tid == 0) { s_full_skip = 0; s_pitems = 0; }
        __syncthreads();
        for (int g = tid; g < G; g += kPlanThreads) {
            const int first = groups[3 * g], n = groups[3 * g + 1], ptok = groups[3 * g + 2];
            if (first < 0 || n < 1 || n > 16 || first > S - n || ptok < 0 || ptok % kTile) {
                pkv::report(err, PKV_DEVERR_GROUP);
                continue;
            }
            int pp = ptok / PT;
            for (int j = 0; j < n; ++j) pp = min(pp, clamp_ctx(context_lens[first + j], max_ctx) / PT);
            for (int j = 0; j < n; ++j) ws.pre_parts[first + j] = pp;
            atomicAdd(&s_full_skip, pp * n);
            // this group's prefix items; their order in the list does not
            // matter (partials are merged in partition order)
            const int off = atomicAdd(&s_pitems, pp);
            for (int part = 0; part < pp; ++part) ws.pitems[off + part] = (g << 16) | part;
        }
        __syncthreads();
        if (tid == 0) {
            s_full_total -= s_full_skip;
            s_items -= s_full_skip;
        }
        __syncthreads();
    }

    // Item order.  Partial partitions go first when they are full enough,
    // else last.  With prefix groups the items left are the members' own
    // tokens; when some of them are long (a partial of PT / 8 tokens or
    // more), full partitions go first and then the partial ones longest
    // first (64 length classes), so that no long item starts last.  The
    // class counts and positions are taken with one shared-memory atomic per
    // class present in a warp: same-address atomics from every lane would
    // serialise when the lengths fall in a class or two.
    __shared__ int s_longest_first;
    auto len_class = [&](int rem) { return 63 - (int)min(63LL, (long long)rem * 64 / PT); };
    __shared__ int s_cls[64];                // per class: count, then next position
    __shared__ long long s_fill[kWarpsP];
    __shared__ int s_partials_first;
    if (tid < 64) s_cls[tid] = 0;
    __syncthreads();
    {
        long long fill = 0;
        for (int base = 0; base < S; base += kPlanThreads) {  // the same trip count in every lane
            const int s = base + tid;
            const int c = s < S ? clamp_ctx(context_lens[s], max_ctx) : PT;
            if (s < S) fill += c % PT;
            if (G > 0) {  // one atomic per class present in the warp
                const int cls = (s < S && (c % PT != 0 || c == 0)) ? len_class(c % PT) : 64;
                const unsigned same = __match_any_sync(kFull, cls);
                if (cls != 64 && (same & ((1u << lane) - 1u)) == 0u) atomicAdd(&s_cls[cls], __popc(same));
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) fill += __shfl_xor_sync(kFull, fill, o);
        if (lane == 0) s_fill[wid] = fill;
        __syncthreads();
        if (tid == 0) {
            long long f = 0;
#pragma unroll
            for (int w = 0; w < kWarpsP; ++w) f += s_fill[w];
            s_partials_first = 8 * f >= 3 * (long long)(s_items - s_full_total) * PT;
        }
        if (G > 0 && wid == 0) {  // class counts -> first positions
            const int c0 = s_cls[2 * lane], c1 = s_cls[2 * lane + 1];
            // classes 0 .. 55: partials of PT / 8 tokens or more
            const unsigned long_ones = __ballot_sync(kFull, (2 * lane <= 55 && c0 > 0) ||
                                                               (2 * lane + 1 <= 55 && c1 > 0));
            if (lane == 0) s_longest_first = long_ones != 0u;
            int incl = c0 + c1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int x = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += x;
            }
            const int excl = incl - c0 - c1;
            s_cls[2 * lane] = excl;
            s_cls[2 * lane + 1] = excl + c0;
        }
        __syncthreads();
    }
    const int n_partial = s_items - s_full_total;
    const bool longest_first = G > 0 && s_longest_first != 0;
    const bool partials_first = s_partials_first != 0 && !longest_first;
    for (int base = 0; base < S; base += kPlanThreads) {
        const int s = base + tid;
        int nf = 0, np = 0, skip = 0;
        if (s < S) {
            const int c = clamp_ctx(context_lens[s], max_ctx);
            nf = c / PT;
            np = (c % PT != 0 || c == 0) ? 1 : 0;  // an empty context still writes zeros
            skip = G > 0 ? ws.pre_parts[s] : 0;
        }
        // longest first: this sequence's partial item goes to its class's
        // next position (one atomic per class present in the warp)
        int my_pos = 0;
        if (longest_first) {
            const int cls = np ? len_class(clamp_ctx(context_lens[s], max_ctx) % PT) : 64;
            const unsigned same = __match_any_sync(kFull, cls);
            const int rank = __popc(same & ((1u << lane) - 1u));
            int first = 0;
            if (cls != 64 && rank == 0) first = atomicAdd(&s_cls[cls], __popc(same));
            my_pos = __shfl_sync(kFull, first, __ffs(same) - 1) + rank;
        }
        int a = nf - skip, b = np;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(kFull, a, o), y = __shfl_up_sync(kFull, b, o);
            if (lane >= o) { a += x; b += y; }
        }
        if (lane == 31) { wsum[0][wid] = a; wsum[1][wid] = b; }
        __syncthreads();
        int off_f = carry[0] + a - (nf - skip), off_p = carry[1] + b - np;
        for (int w = 0; w < wid; ++w) { off_f += wsum[0][w]; off_p += wsum[1][w]; }
        if (s < S) {
            const int at_f = partials_first ? n_partial + off_f : off_f;
            const int at_p = longest_first ? s_full_total + my_pos
                                           : partials_first ? off_p : s_full_total + off_p;
            for (int k = skip; k < nf; ++k) ws.items[at_f + k - skip] = (s << 16) | k;
            if (np) ws.items[at_p] = (s << 16) | nf;
            ws.nparts[s] = nf + np;
        }
        __syncthreads();
        if (tid == kPlanThreads - 1) { carry[0] = off_f + nf - skip; carry[1] = off_p + np; }
        __syncthreads();
    }
    for (int i = tid; i < n_tickets; i += kPlanThreads) ws.tickets[i] = 0u;
    if (tid == 0) {
        *ws.counter = 0u;
        *ws.n_items = s_items;
        *ws.pt = PT;
        *ws.pcounter = 0u;
        *ws.n_pitems = G > 0 ? s_pitems : 0;
    }
}

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(PlanArgs pa) {
    // context_lens may come from the kernel before this one
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the decode kernel may become resident now; it waits for this grid
    asm volatile("griddepcontrol.launch_dependents;");
    plan_cta(pa);
}

// The new tokens of one decode step (pkv_decode_step).
struct TokenArgs {
    const uint4* key;    // [T][H*D/8]
    const uint4* value;
    uint4* k_cache;      // [NB*bs][H*D/8]
    uint4* v_cache;
    const int32_t* block_tables;  // [S][MB]
    const int32_t* seq_idx;  // [T]
    const int32_t* pos;      // [T]
    int64_t* slot_mapping;   // [T], written
    int T, MB, bs, vec_per_row;
    int64_t num_slots;       // NB * bs
};

// Prologue of a fused step: CTA 0 plans the decode while the other CTAs
// each take kPrologueTokens new tokens: their slots (address translation,
// written out to slot_mapping) and the copies of their K and V rows into
// the caches -- the work of the slot-mapping, cache-write and plan kernels
// in one launch.  The plan's registers hold this kernel to 4 CTAs per SM,
// so each thread keeps the loads of several tokens in flight.
constexpr int kPrologueTokens = 4;

__global__ void __launch_bounds__(kPlanThreads, 4) step_prologue_kernel(PlanArgs pa, TokenArgs ta) {
    // inputs may come from the kernel before this one
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the decode kernel may become resident now; it waits for this grid
    asm volatile("griddepcontrol.launch_dependents;");
    if (blockIdx.x == 0) {
        plan_cta(pa);
        return;
    }
    const int t0 = (blockIdx.x - 1) * kPrologueTokens;
    __shared__ long long s_slot[kPrologueTokens];
    if (threadIdx.x < kPrologueTokens) {
        const int t = t0 + threadIdx.x;
        int64_t slot = -1;
        if (t < ta.T) {
            slot = pkv::slot_of(ta.block_tables, ta.seq_idx[t], ta.pos[t], pa.S, ta.MB, ta.bs,
                                pa.err);
            ta.slot_mapping[t] = slot;
            if (slot >= ta.num_slots) {
                pkv::report(pa.err, PKV_DEVERR_SLOT);
                slot = -1;
            }
        }
        s_slot[threadIdx.x] = slot;
    }
    __syncthreads();
    const int vpr = ta.vec_per_row;
    const uint4* __restrict__ key = ta.key + (int64_t)t0 * vpr;
    const uint4* __restrict__ value = ta.value + (int64_t)t0 * vpr;
    uint4* __restrict__ kc = ta.k_cache;
    uint4* __restrict__ vc = ta.v_cache;
    int64_t slot[kPrologueTokens];
#pragma unroll
    for (int j = 0; j < kPrologueTokens; ++j) slot[j] = s_slot[j];
    for (int i = threadIdx.x; i < vpr; i += blockDim.x) {
        uint4 kv[kPrologueTokens], vv[kPrologueTokens];
#pragma unroll
        for (int j = 0; j < kPrologueTokens; ++j) {
            if (slot[j] >= 0) {
                kv[j] = key[(int64_t)j * vpr + i];
                vv[j] = value[(int64_t)j * vpr + i];
            }
        }
#pragma unroll
        for (int j = 0; j < kPrologueTokens; ++j) {
            if (slot[j] >= 0) {
                kc[slot[j] * vpr + i] = kv[j];
                vc[slot[j] * vpr + i] = vv[j];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// One warp: one head over one partition.
// ---------------------------------------------------------------------------

// acc + q.k over 8 dims, both operands 16-bit: f16 x f16 (or bf16 x bf16)
// products are exact in fp32 and each is added with one fp32 rounding
// (fma with .f32 result and 16-bit sources), so no operand is converted.
template <class E>
__device__ __forceinline__ float dot8(const uint4& q, const uint4& k, float acc);

template <>
__device__ __forceinline__ float dot8<pkv::F16>(const uint4& q, const uint4& k, float acc) {
    const uint32_t qw[4] = {q.x, q.y, q.z, q.w}, kw[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
        asm("{.reg .b16 ql, qh, kl, kh;\n\t"
            "mov.b32 {ql, qh}, %1;\n\t"
            "mov.b32 {kl, kh}, %2;\n\t"
            "fma.rn.f32.f16 %0, ql, kl, %0;\n\t"
            "fma.rn.f32.f16 %0, qh, kh, %0;}"
            : "+f"(acc)
            : "r"(qw[j]), "r"(kw[j]));
    return acc;
}

template <>
__device__ __forceinline__ float dot8<pkv::BF16>(const uint4& q, const uint4& k, float acc) {
    const uint32_t qw[4] = {q.x, q.y, q.z, q.w}, kw[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
        asm("{.reg .b16 ql, qh, kl, kh;\n\t"
            "mov.b32 {ql, qh}, %1;\n\t"
            "mov.b32 {kl, kh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, ql, kl, %0;\n\t"
            "fma.rn.f32.bf16 %0, qh, kh, %0;}"
            : "+f"(acc)
            : "r"(qw[j]), "r"(kw[j]));
    return acc;
}

// Loads the lane's NI rows (r, r + RPI, ...) of a 16-token tile: rows at or
// past `nvalid` are zero and not read.  A full tile takes no predicates.
// A tile covers TB = max(1, 16 / BS) blocks; base[b] points at row r of the
// tile's part in block b, and the lane's i-th row lies in block
// (RPI * i) / BS (BS is a multiple of RPI, so this does not depend on r).
template <int NI, int RPI, int BS>
__device__ __forceinline__ void load_tile(uint4 (&dst)[NI], const uint16_t* const (&base)[(BS < kTile) ? kTile / BS : 1],
                                          int64_t HD, int nvalid, int r) {
    constexpr int TB = (BS < kTile) ? kTile / BS : 1;
    constexpr int SPAN = (BS < kTile) ? BS : kTile;  // tile rows per block
    if (nvalid == kTile) {
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int b = (RPI * i) / SPAN;
            dst[i] = pkv::ld_stream(base[b < TB ? b : 0] + (RPI * i - b * SPAN) * HD);
        }
    } else {
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int b = (RPI * i) / SPAN;
            dst[i] = (RPI * i + r < nvalid)
                         ? pkv::ld_stream(base[b < TB ? b : 0] + (RPI * i - b * SPAN) * HD)
                         : make_uint4(0, 0, 0, 0);
        }
    }
}

constexpr int kWarpWindow = 64;  // table entries one warp holds in shared memory

// `wtab` is this warp's window of kWarpWindow table entries in shared
// memory, refilled (by the whole warp) when a tile's block falls outside it.
// `pre`: the leading partitions of the sequence that a prefix kernel has
// already written (it completed before this kernel began).  When this is the
// sequence's one other partition, the output is merged here (fused).
template <class E, int D, int BS>
__device__ __forceinline__ void attend_partition(const DecodeParams& a, int s, int h, int part,
                                                 int t_begin, int t_end, int np, int pre,
                                                 int lane, int* wtab) {
    constexpr int LPR = D / 8;         // lanes per row: 16 bytes each
    constexpr int RPI = 32 / LPR;      // rows per warp-wide load
    constexpr int NI = kTile / RPI;    // warp-wide loads per tile (K and V each)
    const int r = lane / LPR, c = lane % LPR;
    const int64_t HD = (int64_t)a.H * D;

    const uint4 qv = __ldg(reinterpret_cast<const uint4*>(
        static_cast<const uint16_t*>(a.q) + ((int64_t)s * a.H + h) * D + c * 8));
    // row r of (physical block 0, offset 0), this lane's 8 dims
    const uint16_t* kb = static_cast<const uint16_t*>(a.k_cache) + r * HD + (int64_t)h * D + c * 8;
    const uint16_t* vb = static_cast<const uint16_t*>(a.v_cache) + r * HD + (int64_t)h * D + c * 8;
    const int32_t* bt_row = a.block_tables + (int64_t)s * a.MB;

    float m_run = -INFINITY, l_run = 0.f;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;

    // the window covers logical blocks [win0, win0 + kWarpWindow); entries
    // past the partition's last block are not read
    const int lb_last = t_end > t_begin ? (t_end - 1) / BS : 0;
    int win0 = -kWarpWindow;
    auto entry = [&](int lb) -> int {
        if ((unsigned)(lb - win0) >= (unsigned)kWarpWindow) {  // the same in every lane
            __syncwarp();
            win0 = lb;
#pragma unroll
            for (int i = lane; i < kWarpWindow; i += 32)
                if (lb + i <= lb_last) wtab[i] = __ldg(bt_row + lb + i);
            __syncwarp();
        }
        return wtab[lb - win0];
    };

    constexpr int TB = (BS < kTile) ? kTile / BS : 1;  // blocks per tile
    // element offsets of the tile at t0 in each of its TB blocks, and its
    // valid rows (masked from the first block whose id is out of range)
    auto locate = [&](int t0, int64_t (&off)[TB], int& nvalid) {
        nvalid = min(kTile, t_end - t0);
#pragma unroll
        for (int b = 0; b < TB; ++b) {
            const int tb = t0 + b * BS;  // first token of this block's part
            int phys = 0;
            if (tb < t_end) {
                const int lb = tb / BS;
                phys = entry(lb);
                if ((unsigned)phys >= (unsigned)a.NB) {
                    if (lane == 0) pkv::report(a.err, PKV_DEVERR_BLOCK_ID);
                    nvalid = min(nvalid, b * BS);
                    phys = 0;
                }
                off[b] = ((int64_t)phys * BS + (tb - lb * BS)) * HD;
            } else {
                off[b] = 0;
            }
        }
    };
    auto bases = [&](const uint16_t* p, const int64_t (&off)[TB], const uint16_t* (&out)[TB]) {
#pragma unroll
        for (int b = 0; b < TB; ++b) out[b] = p + off[b];
    };

    if (t_begin < t_end) {
        // software pipeline: V(t) loads fly while q.K(t) is computed, K(t+1)
        // loads fly while P.V(t) is accumulated
        uint4 kr[NI], vr[NI];
        int nv;
        int64_t off[TB];
        const uint16_t* pb[TB];
        locate(t_begin, off, nv);
        bases(kb, off, pb);
        load_tile<NI, RPI, BS>(kr, pb, HD, nv, r);
        bases(vb, off, pb);
        load_tile<NI, RPI, BS>(vr, pb, HD, nv, r);
        for (int t0 = t_begin;;) {
            const int t1 = t0 + kTile;
            const bool more = t1 < t_end;
            int nv1 = 0;
            int64_t off1[TB];
            if (more) locate(t1, off1, nv1);

            // partial dots over this lane's 8 dims, one per loaded row
            float pd[NI];
#pragma unroll
            for (int i = 0; i < NI; ++i) pd[i] = dot8<E>(qv, kr[i], 0.f);
            if (more) {
                bases(kb, off1, pb);
                load_tile<NI, RPI, BS>(kr, pb, HD, nv1, r);
            }
            // reduce-scatter across the LPR lanes of a row group: after the
            // halving steps lane c holds row index c>>1 summed over half the
            // lanes, the xor-1 step completes the sum
#pragma unroll
            for (int mask = LPR / 2, n = NI; mask >= 2; mask >>= 1, n >>= 1) {
                const bool upper = (lane & mask) != 0;
#pragma unroll
                for (int j = 0; j < n / 2; ++j) {
                    const float send = upper ? pd[j] : pd[j + n / 2];
                    const float keep = upper ? pd[j + n / 2] : pd[j];
                    pd[j] = keep + __shfl_xor_sync(kFull, send, mask);
                }
            }
            const float logit = (pd[0] + __shfl_xor_sync(kFull, pd[0], 1)) * a.qscale;
            const int own_row = RPI * (c >> 1) + r;
            const float sc = own_row < nv ? logit : -INFINITY;

            float mt = sc;
#pragma unroll
            for (int mask = 16; mask >= 2; mask >>= 1) mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, mask));
            const float m_new = fmaxf(m_run, mt);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float corr = exp2f(m_run - m_use);
            const float p = exp2f(sc - m_use);
            l_run = fmaf(l_run, corr, p);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] *= corr;
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const float pi = __shfl_sync(kFull, p, r * LPR + 2 * i);
                float vf[8];
                pkv::unpack8<E>(vr[i], vf);
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = fmaf(pi, vf[j], acc[j]);
            }
            m_run = m_new;
            if (!more) break;
            bases(vb, off1, pb);
            load_tile<NI, RPI, BS>(vr, pb, HD, nv1, r);
            t0 = t1;
            nv = nv1;
        }
    }

    // combine the row groups; l over the 16 distinct rows of each tile
#pragma unroll
    for (int mask = LPR; mask < 32; mask <<= 1) {
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] += __shfl_xor_sync(kFull, acc[j], mask);
    }
#pragma unroll
    for (int mask = 16; mask >= 2; mask >>= 1) l_run += __shfl_xor_sync(kFull, l_run, mask);

    if (np == 1) {
        if (lane < LPR) {
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] *= inv;
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + ((int64_t)s * a.H + h) * D +
                                      c * 8) = pkv::pack8<E>(acc);
        }
    } else if (pre > 0 && np - pre == 1) {
        // the prefix partials 0 .. pre-1 are complete: fold each into this
        // partition's (max, sum, output), one load round per partial, and
        // write the normalised output -- no partial, no ticket
        if (lane < LPR) {
            const int64_t base = ((int64_t)s * a.H + h) * a.max_parts;
            float M = m_run, L = l_run;
            for (int p = 0; p < pre; ++p) {
                const float mp = __ldcg(a.ws.m + base + p);
                const float lp = __ldcg(a.ws.l + base + p);
                const float4* src = reinterpret_cast<const float4*>(a.ws.acc + (base + p) * D + c * 8);
                const float4 x0 = __ldcg(src), x1 = __ldcg(src + 1);
                const float Mn = fmaxf(M, mp);
                const float wo = (M == -INFINITY) ? 0.f : exp2f(M - Mn);
                const float wp = (mp == -INFINITY) ? 0.f : exp2f(mp - Mn);
                const float xp[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = fmaf(wp, xp[j], acc[j] * wo);
                L = fmaf(wp, lp, L * wo);
                M = Mn;
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] *= inv;
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + ((int64_t)s * a.H + h) * D +
                                      c * 8) = pkv::pack8<E>(acc);
        }
    } else {
        const int64_t idx = ((int64_t)s * a.H + h) * a.max_parts + part;
        if (lane < LPR) {
            float4* dst = reinterpret_cast<float4*>(a.ws.acc + idx * D + c * 8);
            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
        if (lane == 0) {
            a.ws.m[idx] = m_run;
            a.ws.l[idx] = l_run;
        }
    }
}

// Merge the partitions of one (sequence, head): with M = max_p m_p,
// out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p.
// Partitions go in chunks of 32: lane i holds the weight of the chunk's
// partition i, and the chunk's acc rows are loaded 8 at a time with no
// dependent load in between.  The sums keep partition order.
template <class E, int D>
__device__ __forceinline__ void merge_partitions(const DecodeParams& a, int s, int h, int np,
                                                 int lane) {
    constexpr int DPL = D / 32;  // dims per lane
    const int64_t base = ((int64_t)s * a.H + h) * a.max_parts;
    const float* accp = a.ws.acc + base * D + lane * DPL;
    auto load_acc = [&](int p, float (&v)[DPL]) {
        if constexpr (DPL == 4) {
            const float4 t = __ldcg(reinterpret_cast<const float4*>(accp + (int64_t)p * D));
            v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
        } else {
            const float2 t = __ldcg(reinterpret_cast<const float2*>(accp + (int64_t)p * D));
            v[0] = t.x; v[1] = t.y;
        }
    };

    float m0 = -INFINITY, l0 = 0.f;
    if (lane < np) { m0 = __ldcg(a.ws.m + base + lane); l0 = __ldcg(a.ws.l + base + lane); }
    float M = m0;
    for (int p = lane + 32; p < np; p += 32) M = fmaxf(M, __ldcg(a.ws.m + base + p));
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, mask));
    const float w0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - M);
    float L = w0 * l0;
    for (int p = lane + 32; p < np; p += 32) {
        const float mp = __ldcg(a.ws.m + base + p);
        if (mp != -INFINITY) L = fmaf(exp2f(mp - M), __ldcg(a.ws.l + base + p), L);
    }
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) L += __shfl_xor_sync(kFull, L, mask);

    float o[DPL];
#pragma unroll
    for (int j = 0; j < DPL; ++j) o[j] = 0.f;
    for (int c0 = 0; c0 < np; c0 += 32) {  // c0 and n are the same in every lane
        const int n = min(np - c0, 32);
        float wl = w0;
        if (c0 > 0) {
            wl = 0.f;
            if (lane < n) {
                const float mp = __ldcg(a.ws.m + base + c0 + lane);
                if (mp != -INFINITY) wl = exp2f(mp - M);
            }
        }
        for (int p = 0; p < n; p += 8) {
            float v[8][DPL];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (p + u < n) {
                    load_acc(c0 + p + u, v[u]);
                } else {
#pragma unroll
                    for (int j = 0; j < DPL; ++j) v[u][j] = 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float w = __shfl_sync(kFull, wl, (p + u) & 31);
                if (p + u < n) {
#pragma unroll
                    for (int j = 0; j < DPL; ++j) o[j] = fmaf(w, v[u][j], o[j]);
                }
            }
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint16_t* dst = static_cast<uint16_t*>(a.out) + ((int64_t)s * a.H + h) * D + lane * DPL;
    if constexpr (DPL == 4) {
        uint2 v;
        v.x = E::from_float2(o[0] * inv, o[1] * inv);
        v.y = E::from_float2(o[2] * inv, o[3] * inv);
        *reinterpret_cast<uint2*>(dst) = v;
    } else {
        *reinterpret_cast<uint32_t*>(dst) = E::from_float2(o[0] * inv, o[1] * inv);
    }
}

#ifndef PKV_MIN_CTAS_PER_SM
#define PKV_MIN_CTAS_PER_SM 4
#endif

template <class E, int D, int BS>
__global__ void __launch_bounds__(kThreads, PKV_MIN_CTAS_PER_SM) decode_kernel(DecodeParams a) {
    // wait for the plan kernel (programmatic dependent launch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ int s_item;
    __shared__ int s_last;
    __shared__ int s_tab[kWarps][kWarpWindow];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = *a.ws.n_items * a.HG;
    const int PT = *a.ws.pt;
    if (threadIdx.x == 0) s_item = (int)atomicAdd(a.ws.counter, 1u);
    __syncthreads();
    int item = s_item;
    while (item < total) {
        int next = 0;
        if (threadIdx.x == 0) next = (int)atomicAdd(a.ws.counter, 1u);  // used at the end
        const int hg = item % a.HG;
        const int packed = a.ws.items[item / a.HG];
        const int s = packed >> 16, part = packed & 0xffff;
        const int np = a.ws.nparts[s];
        // partitions a prefix kernel wrote before this kernel began
        const int pre = a.ws.pre_parts ? a.ws.pre_parts[s] : 0;
        const int ctx = clamp_ctx(a.context_lens[s], a.max_ctx);
        const int t_begin = part * PT;
        const int t_end = min(t_begin + PT, ctx);
        const int h = hg * kWarps + warp;
        if (h < a.H)
            attend_partition<E, D, BS>(a, s, h, part, t_begin, t_end, np, pre, lane, s_tab[warp]);
        if (np > 1 && !(pre > 0 && np - pre == 1)) {
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) {
                const unsigned done = atomicAdd(&a.ws.tickets[s * a.HG + hg], 1u);
                s_last = (done == (unsigned)(np - 1)) ? 1 : 0;
            }
            __syncthreads();
            if (s_last) {
                __threadfence();
                if (h < a.H) merge_partitions<E, D>(a, s, h, np, lane);
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) s_item = next;
        __syncthreads();
        item = s_item;
    }
}

// ---------------------------------------------------------------------------
// Shared-prefix decode: one warp computes one head of one prefix partition
// for all (up to 16) members of a group on the tensor cores.
//
// With the members' queries as the rows of Q (M = 16, unused rows zero):
//   S^T = Q K^T   m16n8k16, A = Q (registers), B = K tile (ldmatrix)
//   O  += P V     m16n8k16, A = P (the S^T accumulators, rounded to 16 bits:
//                 the accumulator layout of the first product is the A layout
//                 of the second), B = V tile (ldmatrix.trans)
// K/V tiles of 16 tokens stream through a 3-stage cp.async ring per warp in
// shared memory, 16-byte chunks XOR-swizzled by row so ldmatrix reads are
// conflict-free.  Each member's (max, sum, output) partial goes to the same
// workspace slots as the decode kernel's, and the same tickets merge them.
// ---------------------------------------------------------------------------
constexpr int kPrefixStages = 3;

template <class E>
struct Mma;
template <>
struct Mma<pkv::F16> {
    static __device__ __forceinline__ void run(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};
template <>
struct Mma<pkv::BF16> {
    static __device__ __forceinline__ void run(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct PrefixParams {
    DecodeParams d;
    const int32_t* groups;  // [G][3]: first sequence, members, prefix tokens
    int G;
};

template <class E, int D, int BS>
__device__ __forceinline__ void prefix_partition(const DecodeParams& a, const int32_t* bt_row,
                                                 int first, int n, int h, int part, int PT,
                                                 unsigned char* stage_base, int lane) {
    constexpr int NK = D / 16;           // k-steps of q.K
    constexpr int NO = D / 8;            // 8-dim column tiles of the output
    constexpr int ROWB = D * 2;          // bytes of one K or V row
    constexpr int TILEB = kTile * ROWB;  // bytes of one K (or V) tile
    constexpr int CPR = ROWB / 16;       // 16-byte chunks per row
    constexpr int CPL = kTile * CPR / 32;  // chunks per lane per tile
    const int g = lane >> 2, t = lane & 3;
    const int64_t HD = (int64_t)a.H * D;

    // Q fragments: rows = members g and g+8, dims 16k + 2t (+8)
    uint32_t qa[NK][4];
    {
        const uint16_t* q0 = static_cast<const uint16_t*>(a.q) + ((int64_t)(first + g) * a.H + h) * D;
        const uint16_t* q1 = static_cast<const uint16_t*>(a.q) + ((int64_t)(first + g + 8) * a.H + h) * D;
        const bool r0 = g < n, r1 = g + 8 < n;
#pragma unroll
        for (int k = 0; k < NK; ++k) {
            qa[k][0] = r0 ? __ldg(reinterpret_cast<const uint32_t*>(q0 + 16 * k + 2 * t)) : 0u;
            qa[k][1] = r1 ? __ldg(reinterpret_cast<const uint32_t*>(q1 + 16 * k + 2 * t)) : 0u;
            qa[k][2] = r0 ? __ldg(reinterpret_cast<const uint32_t*>(q0 + 16 * k + 8 + 2 * t)) : 0u;
            qa[k][3] = r1 ? __ldg(reinterpret_cast<const uint32_t*>(q1 + 16 * k + 8 + 2 * t)) : 0u;
        }
    }
    const uint16_t* k_head = static_cast<const uint16_t*>(a.k_cache) + (int64_t)h * D;
    const uint16_t* v_head = static_cast<const uint16_t*>(a.v_cache) + (int64_t)h * D;
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(stage_base));
    const int t_begin = part * PT, ntiles = PT / kTile;

    // issue the copies of tile i into stage i % kPrefixStages
    auto issue = [&](int i) {
        if (i < ntiles) {
            const int t0 = t_begin + i * kTile;
            const uint32_t sk = sbase + (i % kPrefixStages) * 2 * TILEB, sv = sk + TILEB;
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const int chunk = lane + 32 * j;
                const int row = chunk / CPR, c = chunk % CPR;
                const int tok = t0 + row;
                int phys = __ldg(bt_row + tok / BS);
                if ((unsigned)phys >= (unsigned)a.NB) {
                    pkv::report(a.err, PKV_DEVERR_BLOCK_ID);
                    phys = 0;
                }
                const int64_t off = ((int64_t)phys * BS + tok % BS) * HD + c * 8;
                const uint32_t dst = row * ROWB + ((c ^ (row & 7)) * 16);
                cp_async16(sk + dst, k_head + off);
                cp_async16(sv + dst, v_head + off);
            }
        }
        cp_async_commit();  // an empty group past the end keeps the counting simple
    };

    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[NO][4];
#pragma unroll
    for (int j = 0; j < NO; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

#pragma unroll
    for (int i = 0; i < kPrefixStages - 1; ++i) issue(i);
    for (int i = 0; i < ntiles; ++i) {
        issue(i + kPrefixStages - 1);
        cp_async_wait<kPrefixStages - 1>();
        __syncwarp();
        const uint32_t sk = sbase + (i % kPrefixStages) * 2 * TILEB, sv = sk + TILEB;
        // S^T = Q K^T: two 8-token column tiles
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
            const int mi = lane >> 3, ri = lane & 7;
            const int row = (mi >> 1) * 8 + ri;
#pragma unroll
            for (int k = 0; k < NK; ++k) {
                uint32_t b[4];
                const int c = 2 * k + (mi & 1);
                ldsm_x4(b, sk + row * ROWB + ((c ^ (row & 7)) * 16));
                Mma<E>::run(sc[0], qa[k], b[0], b[1]);
                Mma<E>::run(sc[1], qa[k], b[2], b[3]);
            }
        }
        // logits in log2 units, scaled before the max (the scale may be < 0)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[j][e] *= a.qscale;
        }
        // online softmax per member row (g: [0],[1]; g+8: [2],[3])
        float mt[2];
        mt[0] = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        mt[1] = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mt[r] = fmaxf(mt[r], __shfl_xor_sync(kFull, mt[r], 1));
            mt[r] = fmaxf(mt[r], __shfl_xor_sync(kFull, mt[r], 2));
        }
        float corr[2], mu[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const float m_new = fmaxf(m_run[r], mt[r]);
            corr[r] = exp2f(m_run[r] - m_new);
            mu[r] = m_new;
            m_run[r] = m_new;
        }
        float p[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            p[j][0] = exp2f(sc[j][0] - mu[0]);
            p[j][1] = exp2f(sc[j][1] - mu[0]);
            p[j][2] = exp2f(sc[j][2] - mu[1]);
            p[j][3] = exp2f(sc[j][3] - mu[1]);
        }
        l_run[0] = l_run[0] * corr[0] + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
        l_run[1] = l_run[1] * corr[1] + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
#pragma unroll
        for (int j = 0; j < NO; ++j) {
            o[j][0] *= corr[0]; o[j][1] *= corr[0];
            o[j][2] *= corr[1]; o[j][3] *= corr[1];
        }
        // P as the A operand: (row g, tokens 2t..), (row g+8, 2t..), (g, 8+2t..), (g+8, 8+2t..)
        const uint32_t pa[4] = {E::from_float2(p[0][0], p[0][1]), E::from_float2(p[0][2], p[0][3]),
                                E::from_float2(p[1][0], p[1][1]), E::from_float2(p[1][2], p[1][3])};
        {
            const int mi = lane >> 3, ri = lane & 7;
            const int row = (mi & 1) * 8 + ri;
#pragma unroll
            for (int j = 0; j < NO; j += 2) {
                uint32_t b[4];
                const int c = j + (mi >> 1);
                ldsm_x4_trans(b, sv + row * ROWB + ((c ^ (row & 7)) * 16));
                Mma<E>::run(o[j], pa, b[0], b[1]);
                Mma<E>::run(o[j + 1], pa, b[2], b[3]);
            }
        }
        __syncwarp();  // the stage may be refilled now
    }
    cp_async_wait<0>();

    // per member: sum over the quad, then the partial (or the output)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        l_run[r] += __shfl_xor_sync(kFull, l_run[r], 1);
        l_run[r] += __shfl_xor_sync(kFull, l_run[r], 2);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int member = g + 8 * r;
        if (member >= n) continue;
        const int s = first + member;
        const int np = a.ws.nparts[s];
        if (np == 1) {
            const float inv = l_run[r] > 0.f ? 1.f / l_run[r] : 0.f;
            uint16_t* dst = static_cast<uint16_t*>(a.out) + ((int64_t)s * a.H + h) * D + 2 * t;
#pragma unroll
            for (int j = 0; j < NO; ++j)
                *reinterpret_cast<uint32_t*>(dst + 8 * j) =
                    E::from_float2(o[j][2 * r] * inv, o[j][2 * r + 1] * inv);
        } else {
            const int64_t idx = ((int64_t)s * a.H + h) * a.max_parts + part;
            float* dst = a.ws.acc + idx * D + 2 * t;
#pragma unroll
            for (int j = 0; j < NO; ++j)
                *reinterpret_cast<float2*>(dst + 8 * j) = make_float2(o[j][2 * r], o[j][2 * r + 1]);
            if (t == 0) {
                a.ws.m[idx] = m_run[r];
                a.ws.l[idx] = l_run[r];
            }
        }
    }
}

template <class E, int D, int BS>
__global__ void __launch_bounds__(kThreads, 2) prefix_kernel(PrefixParams pp) {
    // wait for the plan kernel (programmatic dependent launch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    extern __shared__ __align__(128) unsigned char prefix_smem[];
    __shared__ int s_item;
    __shared__ unsigned s_last;  // bit j: member j's (sequence, head group) completes here
    const DecodeParams& a = pp.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = *a.ws.n_pitems * a.HG;
    const int PT = *a.ws.pt;
    constexpr int STAGE_BYTES = kPrefixStages * 2 * kTile * D * 2;
    unsigned char* my_stages = prefix_smem + warp * STAGE_BYTES;
    if (threadIdx.x == 0) s_item = (int)atomicAdd(a.ws.pcounter, 1u);
    __syncthreads();
    int item = s_item;
    while (item < total) {
        int next = 0;
        if (threadIdx.x == 0) next = (int)atomicAdd(a.ws.pcounter, 1u);
        const int hg = item % a.HG;
        const int packed = a.ws.pitems[item / a.HG];
        const int gi = packed >> 16, part = packed & 0xffff;
        const int first = pp.groups[3 * gi], n = pp.groups[3 * gi + 1];
        const int h = hg * kWarps + warp;
        const int32_t* bt_row = a.block_tables + (int64_t)first * a.MB;  // the shared blocks
        if (h < a.H) prefix_partition<E, D, BS>(a, bt_row, first, n, h, part, PT, my_stages, lane);
        // tickets of the members that have more than one partition
        __threadfence();
        __syncthreads();
        if (threadIdx.x < 16) {
            const int j = threadIdx.x;
            unsigned bit = 0;
            if (j < n) {
                const int s = first + j;
                const int np = a.ws.nparts[s];
                if (np > 1) {
                    const unsigned done = atomicAdd(&a.ws.tickets[s * a.HG + hg], 1u);
                    bit = (done == (unsigned)(np - 1)) ? (1u << j) : 0u;
                }
            }
            // gather the 16 bits in warp 0's first half
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) bit |= __shfl_xor_sync(0xffffu, bit, o);
            if (j == 0) s_last = bit;
        }
        __syncthreads();
        unsigned last = s_last;
        if (last) {
            __threadfence();
            while (last) {
                const int j = __ffs(last) - 1;
                last &= last - 1;
                const int s = first + j;
                if (h < a.H) merge_partitions<E, D>(a, s, h, a.ws.nparts[s], lane);
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) s_item = next;
        __syncthreads();
        item = s_item;
    }
}

#include "prefix_tc.cuh"

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
using KernelFn = void (*)(DecodeParams);

template <class E, int D>
KernelFn pick_bs(int bs) {
    switch (bs) {
        case 8: return decode_kernel<E, D, 8>;
        case 16: return decode_kernel<E, D, 16>;
        case 32: return decode_kernel<E, D, 32>;
        default: return decode_kernel<E, D, 64>;
    }
}

template <class E>
KernelFn pick_d(int D, int bs) {
    return D == 64 ? pick_bs<E, 64>(bs) : pick_bs<E, 128>(bs);
}

KernelFn pick(pkv_dtype dt, int D, int bs) {
    return dt == PKV_BF16 ? pick_d<pkv::BF16>(D, bs) : pick_d<pkv::F16>(D, bs);
}

using PrefixFn = void (*)(PrefixParams);

template <class E, int D>
PrefixFn pick_prefix_bs(int bs) {
    switch (bs) {
        case 8: return prefix_kernel<E, D, 8>;
        case 16: return prefix_kernel<E, D, 16>;
        case 32: return prefix_kernel<E, D, 32>;
        default: return prefix_kernel<E, D, 64>;
    }
}

PrefixFn pick_prefix(pkv_dtype dt, int D, int bs) {
    if (dt == PKV_BF16) return D == 64 ? pick_prefix_bs<pkv::BF16, 64>(bs) : pick_prefix_bs<pkv::BF16, 128>(bs);
    return D == 64 ? pick_prefix_bs<pkv::F16, 64>(bs) : pick_prefix_bs<pkv::F16, 128>(bs);
}

size_t prefix_smem_bytes(int D) { return (size_t)kWarps * kPrefixStages * 2 * kTile * D * 2; }

// Resident CTAs per SM of the prefix kernel (its shared memory set once).
int prefix_resident(PrefixFn fn, int D) {
    static std::mutex mu;
    static struct { PrefixFn fn; int dev; int n; } cache[64];
    static int used = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].fn == fn && cache[i].dev == dev) return cache[i].n;
    const int smem = (int)prefix_smem_bytes(D);
    int n = 0;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, smem) != cudaSuccess || n < 1) {
        cudaGetLastError();
        return 0;
    }
    if (used < 64) cache[used++] = {fn, dev, n};
    return n;
}

// ---- the tensor-core prefix kernel (head_dim 128) ----
using PrefixTcFn = void (*)(PrefixParams, const CUtensorMap, const CUtensorMap);

template <class E>
PrefixTcFn pick_prefix_tc_bs(int bs) {
    switch (bs) {
        case 8: return prefix_tc_kernel<E, 8>;
        case 16: return prefix_tc_kernel<E, 16>;
        case 32: return prefix_tc_kernel<E, 32>;
        default: return prefix_tc_kernel<E, 64>;
    }
}

PrefixTcFn pick_prefix_tc(pkv_dtype dt, int bs) {
    return dt == PKV_BF16 ? pick_prefix_tc_bs<pkv::BF16>(bs) : pick_prefix_tc_bs<pkv::F16>(bs);
}

// The cache as a 3-D tensor [NB*bs rows][H heads][128 dims] of 16-bit
// elements; a box is min(bs, 16) rows (one block holds them) x 1 head x 64
// dims (128 bytes), 128-byte swizzle.
pkv_status encode_cache_map(CUtensorMap* map, const void* cache, int H, int NB, int bs,
                            pkv_dtype dtype) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static std::mutex mu;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!encode) {
            cudaDriverEntryPointQueryResult q;
            void* f = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                                 &q) != cudaSuccess ||
                !f || q != cudaDriverEntryPointSuccess) {
                cudaGetLastError();
                return pkv::fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
            }
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        }
    }
    const cuuint64_t gdim[3] = {(cuuint64_t)kTcD, (cuuint64_t)H, (cuuint64_t)NB * bs};
    const cuuint64_t gstride[2] = {(cuuint64_t)kTcD * 2, (cuuint64_t)H * kTcD * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)(bs < 16 ? bs : 16)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (encode(map, dt, 3, const_cast<void*>(cache), gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return pkv::fail(PKV_ERR_CUDA, "tensor map encoding failed");
    return PKV_OK;
}

// The shared-prefix decode runs the mma.sync prefix kernel, which measured
// faster on this HBM-bound contraction; PKV_PREFIX_KERNEL=tcgen05 in the
// environment selects the tensor-core (tcgen05, TMA) kernel for head_dim
// 128 instead.  Read on every call.
bool prefix_tc_selected() {
    const char* e = std::getenv("PKV_PREFIX_KERNEL");
    return e && std::strcmp(e, "tcgen05") == 0;
}

// Allows the tensor-core prefix kernel its shared memory (once per device).
bool prefix_tc_ready(PrefixTcFn fn) {
    static std::mutex mu;
    static struct { PrefixTcFn fn; int dev; } done[64];
    static int used = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i)
        if (done[i].fn == fn && done[i].dev == dev) return true;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes) !=
        cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (used < 64) done[used++] = {fn, dev};
    return true;
}

int resident_ctas(KernelFn fn) {
    static std::mutex mu;
    static struct { KernelFn fn; int dev; int n; } cache[64];
    static int used = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].fn == fn && cache[i].dev == dev) return cache[i].n;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, 0) != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = 1;
    }
    if (used < 64) cache[used++] = {fn, dev, n};
    return n;
}

int max_parts_of(int max_ctx, int PT) {
    int mp = (max_ctx + PT - 1) / PT;
    return mp < 1 ? 1 : mp;
}

// Partition sizing for one call.  A fixed partition_tokens is used as is;
// 0 lets the plan kernel choose among pt_min, 2*pt_min, ... (see
// plan_kernel), and the workspace is laid out for pt_min, the smallest.
struct CallShape {
    int pt_fixed;   // > 0: the caller's partition size; 0: automatic
    int pt_min;     // smallest partition size the call may use
    int max_ctx;
    int max_parts;  // partitions of the longest context at pt_min
    Layout L;
};

// Smallest automatic partition (64 * 2^k) whose layout fits `capacity`
// bytes and gives at most 65535 partitions; 0 if none does.
int auto_pt_min(int S, int H, int D, int max_ctx, size_t capacity) {
    for (int k = 0; k < kAutoCandidates; ++k) {
        const int pt = kMinAutoPartition << k;
        const int mp = max_parts_of(max_ctx, pt);
        if (mp <= 65535 && layout_of(S, H, D, mp).total <= capacity) return pt;
    }
    return 0;
}

pkv_status check_call(const char* who, void* out, const void* q, const void* k_cache,
                      const void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
                      int S, int H, int D, int bs, int NB, int MB, int max_context_len,
                      float scale, pkv_dtype dtype, int partition_tokens, size_t capacity,
                      CallShape* cs) {
    char msg[320];
    auto bad = [&](pkv_status st, const char* what) {
        snprintf(msg, sizeof msg, "%s: %s", who, what);
        return pkv::fail(st, msg);
    };
    if (S < 0 || H <= 0 || NB <= 0 || MB <= 0 || (dtype != PKV_F16 && dtype != PKV_BF16))
        return bad(PKV_ERR_INVALID_ARG, "bad size or dtype");
    if ((D != 64 && D != 128) || (bs != 8 && bs != 16 && bs != 32 && bs != 64))
        return bad(PKV_ERR_UNSUPPORTED, "head_dim must be 64/128, block_size 8/16/32/64");
    if (S == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return bad(PKV_ERR_INVALID_ARG, "null pointer");
    if (!pkv::aligned16(out) || !pkv::aligned16(q) || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
        return bad(PKV_ERR_INVALID_ARG, "token pointers must be 16-byte aligned");
    const int64_t cap = (int64_t)MB * bs;
    const int max_ctx = max_context_len == 0 ? (int)(cap < INT32_MAX ? cap : INT32_MAX) : max_context_len;
    if (max_ctx < 0 || max_ctx > cap) return bad(PKV_ERR_INVALID_ARG, "max_context_len must be in [0, MB*bs]");
    if (partition_tokens < 0 || (partition_tokens > 0 && (partition_tokens % kTile || partition_tokens % bs)))
        return bad(PKV_ERR_INVALID_ARG, "partition_tokens must be 0 or a multiple of 16 and of block_size");
    if (!(scale == scale) || std::isinf(scale)) return bad(PKV_ERR_INVALID_ARG, "scale must be finite");
    if (S > 32767) return bad(PKV_ERR_INVALID_ARG, "at most 32767 sequences");
    cs->max_ctx = max_ctx;
    if (partition_tokens > 0) {
        cs->pt_fixed = cs->pt_min = partition_tokens;
    } else {
        cs->pt_fixed = 0;
        cs->pt_min = auto_pt_min(S, H, D, max_ctx, capacity);
        if (cs->pt_min == 0) cs->pt_min = kMinAutoPartition << (kAutoCandidates - 1);
    }
    cs->max_parts = max_parts_of(max_ctx, cs->pt_min);
    if (cs->max_parts > 65535 || (int64_t)S * cs->max_parts > INT32_MAX / 64)
        return bad(PKV_ERR_INVALID_ARG, "too many partitions: raise partition_tokens");
    cs->L = layout_of(S, H, D, cs->max_parts);
    if (cs->L.total > capacity) {
        snprintf(msg, sizeof msg, "%s: this size needs %zu bytes of workspace, %zu available", who,
                 cs->L.total, capacity);
        return pkv::fail(PKV_ERR_WORKSPACE, msg);
    }
    return PKV_OK;
}

cudaLaunchAttribute pdl_attr() {
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

// Launches the plan (or, with `tokens`, the fused step prologue), then the
// prefix kernel (with groups) or the decode kernel.
pkv_status launch_decode(const char* who, const CallShape& cs, void* out, const void* q,
                         const void* k_cache, const void* v_cache, const int32_t* block_tables,
                         const int32_t* context_lens, int S, int H, int D, int bs, int NB, int MB,
                         float scale, pkv_dtype dtype, void* workspace, cudaStream_t st,
                         const int32_t* groups = nullptr, int G = 0,
                         const TokenArgs* tokens = nullptr) {
    DecodeParams p;
    p.out = out;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.S = S;
    p.H = H;
    p.NB = NB;
    p.MB = MB;
    p.HG = (H + kWarps - 1) / kWarps;
    p.max_parts = cs.max_parts;
    p.max_ctx = cs.max_ctx;
    p.qscale = scale * 1.4426950408889634f;  // log2(e)
    p.ws = bind(workspace, cs.L);
    p.err = pkv::device_error_word();

    KernelFn fn = pick(dtype, D, bs);
    const int64_t upper = (int64_t)S * cs.max_parts * p.HG;
    const int64_t resident = (int64_t)resident_ctas(fn) * pkv::sm_count();
    const int grid = (int)(upper < resident ? upper : resident);

    char msg[160];
    cudaLaunchAttribute attr[1] = {pdl_attr()};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    PlanArgs pa;
    pa.context_lens = context_lens;
    pa.S = S;
    pa.pt_fixed = cs.pt_fixed;
    pa.pt_min = cs.pt_min;
    pa.max_ctx = cs.max_ctx;
    pa.slots = grid;
    pa.HG = p.HG;
    pa.n_tickets = S * p.HG;
    pa.ws = p.ws;
    pa.groups = groups;
    pa.G = G;
    pa.err = p.err;
    cudaError_t e;
    if (tokens) {
        cfg.gridDim = dim3(1 + (unsigned)((tokens->T + kPrologueTokens - 1) / kPrologueTokens));
        e = cudaLaunchKernelEx(&cfg, step_prologue_kernel, pa, *tokens);
    } else {
        e = cudaLaunchKernelEx(&cfg, plan_kernel, pa);
    }
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "%s plan launch", who);
        return pkv::cuda_fail(e, msg);
    }
    if (G > 0 && D == kTcD && prefix_tc_selected()) {
        PrefixTcFn tfn = pick_prefix_tc(dtype, bs);
        if (!prefix_tc_ready(tfn)) return pkv::fail(PKV_ERR_CUDA, "prefix_tc shared memory");
        CUtensorMap tmk, tmv;
        pkv_status ms = encode_cache_map(&tmk, k_cache, H, NB, bs, dtype);
        if (ms == PKV_OK) ms = encode_cache_map(&tmv, v_cache, H, NB, bs, dtype);
        if (ms != PKV_OK) return ms;
        const int64_t pupper = (int64_t)(G > 0 ? G : 1) * cs.max_parts * p.HG;
        const int64_t president = (int64_t)kTcCtasPerSm * pkv::sm_count();
        PrefixParams pp;
        pp.d = p;
        pp.groups = groups;
        pp.G = G;
        cfg.gridDim = dim3((unsigned)(pupper < president ? pupper : president));
        cfg.blockDim = dim3(kTcThreads);
        cfg.dynamicSmemBytes = kTcSmemBytes;
        e = cudaLaunchKernelEx(&cfg, tfn, pp, tmk, tmv);
        if (e != cudaSuccess) {
            snprintf(msg, sizeof msg, "%s prefix launch", who);
            return pkv::cuda_fail(e, msg);
        }
        cfg.dynamicSmemBytes = 0;
    } else if (G > 0) {
        PrefixFn pfn = pick_prefix(dtype, D, bs);
        const int per_sm = prefix_resident(pfn, D);
        if (per_sm < 1) return pkv::fail(PKV_ERR_CUDA, "prefix kernel cannot be resident");
        const int64_t pupper = (int64_t)G * cs.max_parts * p.HG;
        const int64_t president = (int64_t)per_sm * pkv::sm_count();
        PrefixParams pp;
        pp.d = p;
        pp.groups = groups;
        pp.G = G;
        cfg.gridDim = dim3((unsigned)(pupper < president ? pupper : president));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = prefix_smem_bytes(D);
        e = cudaLaunchKernelEx(&cfg, pfn, pp);
        if (e != cudaSuccess) {
            snprintf(msg, sizeof msg, "%s prefix launch", who);
            return pkv::cuda_fail(e, msg);
        }
        cfg.dynamicSmemBytes = 0;
    }
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    e = cudaLaunchKernelEx(&cfg, fn, p);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "%s launch", who);
        return pkv::cuda_fail(e, msg);
    }
    return PKV_OK;
}
}  // namespace

extern "C" {

size_t pkv_decode_workspace_size(int S, int H, int D, int max_context_len, int partition_tokens) {
    if (S < 0 || H <= 0 || (D != 64 && D != 128) || max_context_len < 0 || partition_tokens < 0 ||
        partition_tokens % kTile)
        return 0;
    int pt = partition_tokens;
    if (pt == 0) pt = auto_pt_min(S, H, D, max_context_len, SIZE_MAX);
    if (pt == 0) return 0;
    const int mp = max_parts_of(max_context_len, pt);
    if (mp > 65535) return 0;
    return layout_of(S, H, D, mp).total;
}

pkv_status pkv_paged_attention_decode(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      const int32_t* context_lens, int S, int H, int D, int bs,
                                      int NB, int MB, int max_context_len, float scale,
                                      pkv_dtype dtype, int partition_tokens, void* workspace,
                                      size_t workspace_bytes, void* stream) {
    PKV_TRACE("pkv_paged_attention_decode");
    static const char* who = "paged_attention_decode";
    pkv::clear_error();
    if (S > 0 && workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return pkv::fail(PKV_ERR_INVALID_ARG, "paged_attention_decode: workspace must be 256-byte aligned");
    CallShape cs;
    // the automatic partition size is laid out for the smallest candidate,
    // whatever the workspace holds: its size depends only on the arguments
    pkv_status st = check_call(who, out, q, k_cache, v_cache, block_tables, context_lens, S, H, D,
                               bs, NB, MB, max_context_len, scale, dtype, partition_tokens,
                               SIZE_MAX, &cs);
    if (st != PKV_OK || S == 0) return st;
    if (!workspace) return pkv::fail(PKV_ERR_INVALID_ARG, "paged_attention_decode: null workspace");
    if (workspace_bytes < cs.L.total)
        return pkv::fail(PKV_ERR_WORKSPACE, "paged_attention_decode: workspace too small");
    return launch_decode(who, cs, out, q, k_cache, v_cache, block_tables, context_lens, S, H, D, bs,
                         NB, MB, scale, dtype, workspace, pkv::as_stream(stream));
}

pkv_status pkv_decode_step(void* out, const void* q, const void* key, const void* value,
                           void* k_cache, void* v_cache, const int32_t* block_tables,
                           const int32_t* context_lens, const int32_t* seq_idx, const int32_t* pos,
                           int64_t* slot_mapping, const int32_t* prefix_groups, int G, int T,
                           int S, int H, int D, int bs, int NB, int MB, int max_context_len,
                           float scale, pkv_dtype dtype, int partition_tokens, void* workspace,
                           size_t workspace_bytes, void* stream) {
    PKV_TRACE("pkv_decode_step");
    static const char* who = "decode_step";
    pkv::clear_error();
    if (T < 0 || T == INT32_MAX) return pkv::fail(PKV_ERR_INVALID_ARG, "decode_step: bad token count");
    if (G < 0 || G > 32767 || (G > 0 && !prefix_groups))
        return pkv::fail(PKV_ERR_INVALID_ARG, "decode_step: bad groups");
    if (T > 0 && (!key || !value || !seq_idx || !pos || !slot_mapping))
        return pkv::fail(PKV_ERR_INVALID_ARG, "decode_step: null token pointer");
    if (T > 0 && (!pkv::aligned16(key) || !pkv::aligned16(value)))
        return pkv::fail(PKV_ERR_INVALID_ARG, "decode_step: key/value must be 16-byte aligned");
    if (S > 0 && workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return pkv::fail(PKV_ERR_INVALID_ARG, "decode_step: workspace must be 256-byte aligned");
    CallShape cs;
    pkv_status st = check_call(who, out, q, k_cache, v_cache, block_tables, context_lens, S, H, D,
                               bs, NB, MB, max_context_len, scale, dtype, partition_tokens,
                               SIZE_MAX, &cs);
    if (st != PKV_OK) return st;
    if (S == 0) {
        if (T == 0) return PKV_OK;
        return pkv::fail(PKV_ERR_INVALID_ARG, "decode_step: new tokens for an empty batch");
    }
    if (G > 0) cs.L = layout_shared(S, H, D, G, cs.max_parts);
    if (!workspace) return pkv::fail(PKV_ERR_INVALID_ARG, "decode_step: null workspace");
    if (workspace_bytes < cs.L.total)
        return pkv::fail(PKV_ERR_WORKSPACE, "decode_step: workspace too small");
    TokenArgs ta;
    ta.key = static_cast<const uint4*>(key);
    ta.value = static_cast<const uint4*>(value);
    ta.k_cache = static_cast<uint4*>(k_cache);
    ta.v_cache = static_cast<uint4*>(v_cache);
    ta.block_tables = block_tables;
    ta.seq_idx = seq_idx;
    ta.pos = pos;
    ta.slot_mapping = slot_mapping;
    ta.T = T;
    ta.MB = MB;
    ta.bs = bs;
    ta.vec_per_row = H * D / 8;
    ta.num_slots = (int64_t)NB * bs;
    return launch_decode(who, cs, out, q, k_cache, v_cache, block_tables, context_lens, S, H, D, bs,
                         NB, MB, scale, dtype, workspace, pkv::as_stream(stream),
                         G > 0 ? prefix_groups : nullptr, G, &ta);
}

size_t pkv_decode_shared_prefix_workspace_size(int S, int H, int D, int G, int max_context_len,
                                               int partition_tokens) {
    if (S < 0 || H <= 0 || (D != 64 && D != 128) || G < 0 || max_context_len < 0 ||
        partition_tokens < 0 || partition_tokens % kTile)
        return 0;
    int pt = partition_tokens;
    if (pt == 0) pt = auto_pt_min(S, H, D, max_context_len, SIZE_MAX);
    if (pt == 0) return 0;
    const int mp = max_parts_of(max_context_len, pt);
    if (mp > 65535) return 0;
    return layout_shared(S, H, D, G, mp).total;
}

pkv_status pkv_paged_attention_decode_shared_prefix(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, const int32_t* prefix_groups, int G,
    int S, int H, int D, int bs, int NB, int MB, int max_context_len, float scale, pkv_dtype dtype,
    int partition_tokens, void* workspace, size_t workspace_bytes, void* stream) {
    PKV_TRACE("pkv_paged_attention_decode_shared_prefix");
    static const char* who = "paged_attention_decode_shared_prefix";
    pkv::clear_error();
    if (G < 0 || G > 32767 || (G > 0 && !prefix_groups))
        return pkv::fail(PKV_ERR_INVALID_ARG, "paged_attention_decode_shared_prefix: bad groups");
    if (S > 0 && workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return pkv::fail(PKV_ERR_INVALID_ARG, "paged_attention_decode_shared_prefix: workspace must be 256-byte aligned");
    CallShape cs;
    pkv_status st = check_call(who, out, q, k_cache, v_cache, block_tables, context_lens, S, H, D,
                               bs, NB, MB, max_context_len, scale, dtype, partition_tokens,
                               SIZE_MAX, &cs);
    if (st != PKV_OK || S == 0) return st;
    cs.L = layout_shared(S, H, D, G, cs.max_parts);
    if (!workspace) return pkv::fail(PKV_ERR_INVALID_ARG, "paged_attention_decode_shared_prefix: null workspace");
    if (workspace_bytes < cs.L.total)
        return pkv::fail(PKV_ERR_WORKSPACE, "paged_attention_decode_shared_prefix: workspace too small");
    return launch_decode(who, cs, out, q, k_cache, v_cache, block_tables, context_lens, S, H, D,
                         bs, NB, MB, scale, dtype, workspace, pkv::as_stream(stream),
                         prefix_groups, G);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode for callers that cannot allocate device memory.  The split-K
// scratch is this file's static device array instead of a caller workspace.
// ---------------------------------------------------------------------------

// One copy per device that loads the library, held until the process exits.
// Host code must not use this name as a device address (on the host it is a
// stand-in): the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};
unsigned long long g_noalloc_ctx[kNoAllocMaxDevices] = {};

// Unique id of the calling thread's current context; 0 when there is none
// or the driver does not offer the lookup.  A device reset ends the
// context, and the array lives at a new address in the next one.
unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
        cudaGetLastError();
    });
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c ||
        get_id(c, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array on the current device, looked up with
// that device current once per context of the device.
pkv_status noalloc_scratch(void** addr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return pkv::cuda_fail(e, "paged_attention_decode_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kNoAllocMaxDevices)
        return pkv::fail(PKV_ERR_INVALID_ARG, "paged_attention_decode_noalloc: device ordinal above 63");
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    const unsigned long long ctx = current_context_id();
    if (!g_noalloc_addr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return pkv::cuda_fail(e, "paged_attention_decode_noalloc: cudaGetSymbolAddress of the scratch array");
        }
        g_noalloc_addr[dev] = p;
        // the lookup made the context current if it was not yet
        g_noalloc_ctx[dev] = current_context_id();
    }
    *addr = g_noalloc_addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_attention_decode_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, int S, int H, int D, int bs, int NB,
    int MB, int max_context_len, float scale, pkv_dtype dtype, int partition_tokens,
    void* stream) {
    PKV_TRACE("pkv_paged_attention_decode_noalloc");
    static const char* who = "paged_attention_decode_noalloc";
    pkv::clear_error();
    CallShape cs;
    // an automatic partition size starts from the smallest one whose
    // partials fit the built-in scratch
    pkv_status st = check_call(who, out, q, k_cache, v_cache, block_tables, context_lens, S, H, D,
                               bs, NB, MB, max_context_len, scale, dtype, partition_tokens,
                               (size_t)PKV_NOALLOC_SCRATCH_BYTES, &cs);
    if (st == PKV_ERR_WORKSPACE) {
        char msg[320];
        snprintf(msg, sizeof msg,
                 "%s: this size needs %zu bytes of scratch, more than the %u built into the "
                 "library; call pkv_paged_attention_decode with a workspace",
                 who, cs.L.total, (unsigned)PKV_NOALLOC_SCRATCH_BYTES);
        return pkv::fail(PKV_ERR_WORKSPACE, msg);
    }
    if (st != PKV_OK || S == 0) return st;
    void* scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != PKV_OK) return st;
    // The plan kernel rewrites the work counter, the item list, the
    // partition counts and the merge tickets at the start of every call;
    // each partial is written before it is read, so the previous call's
    // contents never reach the output.
    return launch_decode(who, cs, out, q, k_cache, v_cache, block_tables, context_lens, S, H, D, bs,
                         NB, MB, scale, dtype, scratch, pkv::as_stream(stream));
}
