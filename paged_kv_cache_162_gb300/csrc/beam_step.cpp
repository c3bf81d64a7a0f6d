// One beam-search step in one native call: the host allocator's fork and
// append, the upload of what the device needs, and the step's kernels.
//
//  "3.3 页面级显存管理" 3.3.2: share_blocks when a sequence forks (beam
//    search, parallel sampling), one more block when a sequence's tokens
//    pass num_blocks * block_size
//  "vLLM三大核心技术分页内存与共享解码", "Copy-on-Write共享解码的显存优化原理":
//    a write into a shared block copies it first
//  notes on "vLLM: Easy, Fast, and Cheap LLM Serving with PagedAttention",
//    "Memory Sharing与写时复制": beams share blocks until they diverge
//
// The call is the composition of public entry points -- pkv_alloc_fork,
// pkv_alloc_append_batch, pkv_copy_blocks and pkv_decode_step -- with the
// host arrays staged in one pinned buffer and uploaded by one copy, so a
// serving loop crosses the library boundary once per step.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace {

// Byte offsets of the staged inputs (the same in the pinned staging buffer
// and in the device buffer): tables [S][MB] int32, context lengths [S],
// token positions [S], sequence index [S] (int32), room for 2S copy pairs
// [2S][2] int64 (one token per sequence copies at most one block, but
// pkv_alloc_append_batch asks for room for two per sequence).  Every part
// starts on a 256-byte boundary.
struct BeamLayout {
    size_t tables, ctx, pos, seq, pairs, total;
};

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

BeamLayout beam_layout(int32_t S, int32_t MB) {
    BeamLayout L;
    L.tables = 0;
    L.ctx = up256((size_t)S * MB * 4);
    L.pos = L.ctx + up256((size_t)S * 4);
    L.seq = L.pos + up256((size_t)S * 4);
    L.pairs = L.seq + up256((size_t)S * 4);
    L.total = L.pairs + up256((size_t)S * 2 * 2 * 8);
    return L;
}

}  // namespace

extern "C" {

size_t pkv_beam_inputs_bytes(int32_t S, int32_t MB) {
    if (S <= 0 || MB <= 0) return 0;
    return beam_layout(S, MB).total;
}

pkv_status pkv_beam_step(pkv_allocator* a, int32_t* tables, int32_t* num_blocks,
                         int32_t* context_lens, const int32_t* parents, int32_t S, int32_t MB,
                         void* staging, void* dev_inputs, size_t inputs_bytes, void* out,
                         const void* q, const void* key, const void* value, void* k_cache,
                         void* v_cache, int64_t* slot_mapping, const int32_t* prefix_groups,
                         int G, int H, int D, int bs, int NB,
                         float scale, pkv_dtype dtype, int partition_tokens, void* workspace,
                         size_t workspace_bytes, int32_t* n_pairs, void* stream) {
    PKV_TRACE("pkv_beam_step");
    pkv::clear_error();
    if (!a || S <= 0 || MB <= 0 || !tables || !num_blocks || !context_lens || !parents ||
        !staging || !dev_inputs || !n_pairs || bs <= 0 || G < 0 || (G > 0 && !prefix_groups))
        return pkv::fail(PKV_ERR_INVALID_ARG, "beam_step: bad argument");
    const BeamLayout L = beam_layout(S, MB);
    if (inputs_bytes < L.total)
        return pkv::fail(PKV_ERR_INVALID_ARG, "beam_step: staging/device input buffers too small");
    if ((reinterpret_cast<uintptr_t>(staging) & 255u) || (reinterpret_cast<uintptr_t>(dev_inputs) & 255u))
        return pkv::fail(PKV_ERR_INVALID_ARG, "beam_step: input buffers must be 256-byte aligned");
    for (int32_t s = 0; s < S; ++s)
        if (parents[s] < 0 || parents[s] >= S)
            return pkv::fail(PKV_ERR_INVALID_ARG, "beam_step: parent out of range");
    *n_pairs = 0;

    unsigned char* stg = static_cast<unsigned char*>(staging);
    int32_t* pos = reinterpret_cast<int32_t*>(stg + L.pos);
    int32_t* ctx = reinterpret_cast<int32_t*>(stg + L.ctx);
    int32_t* seq = reinterpret_cast<int32_t*>(stg + L.seq);
    int64_t* pairs = reinterpret_cast<int64_t*>(stg + L.pairs);

    // the new token of sequence s sits at its parent's old length
    for (int32_t s = 0; s < S; ++s) {
        pos[s] = context_lens[parents[s]];
        if (pos[s] < 0 || (int64_t)pos[s] >= (int64_t)MB * bs)
            return pkv::fail(PKV_ERR_INVALID_ARG, "beam_step: a context would pass the table");
    }
    pkv_status st = pkv_alloc_fork(a, tables, num_blocks, S, MB, parents);
    if (st != PKV_OK) return st;
    // one token per sequence: seq doubles as the n_new array (all ones)
    for (int32_t s = 0; s < S; ++s) seq[s] = 1;
    int32_t np = 0, ndone = 0;
    st = pkv_alloc_append_batch(a, tables, num_blocks, S, MB, pos, seq, bs, pairs, 2 * S, &np,
                                &ndone);
    if (st != PKV_OK) return st;  // forked; rows [0, ndone) extended, nothing launched
    // the copies must meet pkv_copy_blocks' precondition before any of them
    // reaches the device
    st = pkv_check_copy_pairs(pairs, np, NB);
    if (st != PKV_OK) return st;
    for (int32_t s = 0; s < S; ++s) {
        context_lens[s] = pos[s] + 1;
        ctx[s] = context_lens[s];
        seq[s] = s;
    }
    std::memcpy(stg + L.tables, tables, (size_t)S * MB * 4);
    *n_pairs = np;

    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const size_t used = np ? L.pairs + (size_t)np * 16 : L.pairs;
    cudaError_t e = cudaMemcpyAsync(dev_inputs, staging, used, cudaMemcpyHostToDevice, cs);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return pkv::fail(PKV_ERR_CUDA, "beam_step: input upload failed");
    }
    unsigned char* dev = static_cast<unsigned char*>(dev_inputs);
    if (np) {
        st = pkv_copy_blocks(k_cache, v_cache, reinterpret_cast<const int64_t*>(dev + L.pairs), np,
                             H, D, bs, NB, dtype, stream);
        if (st != PKV_OK) return st;
    }
    // max_context_len 0: the workspace is sized for MB * bs, so it serves
    // every step of the search.  With prefix groups (the beams of one
    // request share their prompt's full blocks for the whole search: only
    // the ends of the contexts are ever written) each prompt is read once
    // per request.
    return pkv_decode_step(out, q, key, value, k_cache, v_cache,
                           reinterpret_cast<const int32_t*>(dev + L.tables),
                           reinterpret_cast<const int32_t*>(dev + L.ctx),
                           reinterpret_cast<const int32_t*>(dev + L.seq),
                           reinterpret_cast<const int32_t*>(dev + L.pos), slot_mapping,
                           prefix_groups, G, S, S, H, D, bs, NB, MB, 0, scale, dtype,
                           partition_tokens, workspace,
                           workspace_bytes, stream);
}

struct pkv_beam_search {
    pkv_allocator* a;
    int32_t *tables, *num_blocks, *context_lens;
    int32_t S, MB;
    void* staging[2];
    void* dev_inputs;
    size_t inputs_bytes;
    void *out, *k_cache, *v_cache;
    int64_t* slot_mapping;
    const int32_t* prefix_groups;
    int G, H, D, bs, NB;
    float scale;
    pkv_dtype dtype;
    int partition_tokens;
    void* workspace;
    size_t workspace_bytes;
    size_t pairs_offset;
    cudaEvent_t done[2];
    bool used[2];
    int turn;
};

pkv_status pkv_beam_search_create(
    pkv_allocator* a, int32_t* tables, int32_t* num_blocks, int32_t* context_lens, int32_t S,
    int32_t MB, void* staging0, void* staging1, void* dev_inputs, size_t inputs_bytes, void* out,
    void* k_cache, void* v_cache, int64_t* slot_mapping, const int32_t* prefix_groups, int G,
    int H, int D, int bs, int NB, float scale, pkv_dtype dtype, int partition_tokens,
    void* workspace, size_t workspace_bytes, pkv_beam_search** out_search) {
    PKV_TRACE("pkv_beam_search_create");
    pkv::clear_error();
    if (!out_search) return pkv::fail(PKV_ERR_INVALID_ARG, "beam_search_create: null handle pointer");
    *out_search = nullptr;
    if (!a || S <= 0 || MB <= 0 || !tables || !num_blocks || !context_lens || !staging0 ||
        !staging1 || !dev_inputs || !out || !k_cache || !v_cache || !slot_mapping || !workspace ||
        bs <= 0 || G < 0 || (G > 0 && !prefix_groups))
        return pkv::fail(PKV_ERR_INVALID_ARG, "beam_search_create: bad argument");
    const BeamLayout L = beam_layout(S, MB);
    if (inputs_bytes < L.total)
        return pkv::fail(PKV_ERR_INVALID_ARG, "beam_search_create: staging/device input buffers too small");
    for (const void* p : {staging0, staging1, dev_inputs})
        if (reinterpret_cast<uintptr_t>(p) & 255u)
            return pkv::fail(PKV_ERR_INVALID_ARG, "beam_search_create: input buffers must be 256-byte aligned");
    pkv_beam_search* b = new (std::nothrow) pkv_beam_search();
    if (!b) return pkv::fail(PKV_ERR_HOST_MEMORY, "beam_search_create: out of host memory");
    *b = pkv_beam_search{a, tables, num_blocks, context_lens, S, MB, {staging0, staging1},
                         dev_inputs, inputs_bytes, out, k_cache, v_cache, slot_mapping,
                         prefix_groups, G, H, D, bs, NB, scale, dtype, partition_tokens,
                         workspace, workspace_bytes, L.pairs, {nullptr, nullptr}, {false, false}, 0};
    for (int i = 0; i < 2; ++i) {
        const cudaError_t e = cudaEventCreateWithFlags(&b->done[i], cudaEventDisableTiming);
        if (e != cudaSuccess) {
            cudaGetLastError();
            if (i == 1) cudaEventDestroy(b->done[0]);
            delete b;
            return pkv::fail(PKV_ERR_CUDA, "beam_search_create: cudaEventCreate failed");
        }
    }
    *out_search = b;
    return PKV_OK;
}

pkv_status pkv_beam_search_step(pkv_beam_search* b, const int32_t* parents, const void* q,
                                const void* key, const void* value, void* stream,
                                int32_t* n_pairs, const int64_t** pairs) {
    PKV_TRACE("pkv_beam_search_step");
    pkv::clear_error();
    if (!b || !parents || !n_pairs || !pairs)
        return pkv::fail(PKV_ERR_INVALID_ARG, "beam_search_step: bad argument");
    const int slot = b->turn;
    b->turn ^= 1;
    if (b->used[slot]) {
        // the upload from this buffer two steps ago must be done before
        // the buffer is written again
        const cudaError_t e = cudaEventSynchronize(b->done[slot]);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return pkv::fail(PKV_ERR_CUDA, "beam_search_step: waiting for the staging buffer failed");
        }
    }
    const pkv_status st = pkv_beam_step(
        b->a, b->tables, b->num_blocks, b->context_lens, parents, b->S, b->MB, b->staging[slot],
        b->dev_inputs, b->inputs_bytes, b->out, q, key, value, b->k_cache, b->v_cache,
        b->slot_mapping, b->prefix_groups, b->G, b->H, b->D, b->bs, b->NB, b->scale, b->dtype,
        b->partition_tokens, b->workspace, b->workspace_bytes, n_pairs, stream);
    // recorded whatever the outcome: a failure after the upload was queued
    // still leaves it in flight
    const cudaError_t e = cudaEventRecord(b->done[slot], reinterpret_cast<cudaStream_t>(stream));
    b->used[slot] = true;
    *pairs = reinterpret_cast<const int64_t*>(static_cast<unsigned char*>(b->staging[slot]) +
                                              b->pairs_offset);
    if (st != PKV_OK) return st;
    if (e != cudaSuccess) {
        cudaGetLastError();
        return pkv::fail(PKV_ERR_CUDA, "beam_search_step: event record failed");
    }
    return PKV_OK;
}

void pkv_beam_search_destroy(pkv_beam_search* b) {
    if (!b) return;
    for (int i = 0; i < 2; ++i)
        if (b->done[i]) cudaEventDestroy(b->done[i]);
    delete b;
}

}  // extern "C"
