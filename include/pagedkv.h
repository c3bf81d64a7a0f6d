/*
 * pagedkv -- paged KV-cache decode attention for NVIDIA GB300 (sm_103a).
 *
 * C ABI of the library libpagedkv.so.  Every entry point is `extern "C"`,
 * takes plain pointers and sizes, and returns a pkv_status.  No exception
 * crosses this boundary.
 *
 * Sources (web pages on PagedAttention; cited by title and section):
 *  [P1] "3.3 页面级显存管理" (page-level GPU memory management)
 *  [P2] "vLLM三大核心技术分页内存与共享解码" (vLLM core techniques)
 *  [P3] "3.1 PagedAttention的核心原理" (PagedAttention core principles)
 *  [P4] notes on "vLLM: Easy, Fast, and Cheap LLM Serving with PagedAttention"
 *
 * Conventions shared by every device entry point
 *  - Device pointers are caller-owned device memory; the library allocates
 *    no device memory.  Token data (q, K, V, out, key, value) is 16-bit
 *    (pkv_dtype) and every such pointer must be 16-byte aligned.  q, key,
 *    value and out may instead point to pinned host memory (cudaHostAlloc;
 *    the GPU addresses it with the same pointer): the kernels then read the
 *    step's tokens and write its output across the host link (on GB300 the
 *    coherent NVLink-C2C link to the Grace CPU), which takes the place of
 *    copying those bytes.  The caches, tables and workspace belong in
 *    device memory: they are read many times per call.
 *  - KV cache layout ([P3] 3.1.2 "页面结构设计", 3.1.3 step 4): separate K
 *    and V caches, each [NB][bs][H][D] row-major.  Token offset o of
 *    physical block p, head h, dim d sits at ((p*bs + o)*H + h)*D + d, i.e.
 *    physical_page*page_size*kv_dim + page_offset*kv_dim with kv_dim = H*D.
 *  - Block tables ([P2] "KV Cache逻辑块物理块映射机制", [P3] 3.1.3, [P4]
 *    "关键误解"): one flat int32 row of MB entries per sequence, row-major
 *    [S][MB]; entry j is the physical block of logical block j.  Only the
 *    first ceil(context_len/bs) entries of a row are read.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Kernels run asynchronously on it; a launch error is returned
 *    at once, an error raised while a kernel runs surfaces on a later call
 *    or through pkv_sync_check().
 *  - Supported shapes: D (head_dim) in {64, 128}, bs (block size) in
 *    {8, 16, 32, 64}; anything else returns PKV_ERR_UNSUPPORTED.
 *  - Out-of-range ids (a physical block outside [0, NB), a slot outside
 *    [0, NB*bs), a context longer than MB*bs) are never dereferenced: the
 *    kernel skips the access and records PKV_DEVERR_* in a device error word
 *    that pkv_get_device_errors() returns.
 *  - pkv_last_error_string() describes the last failure of this thread.
 *
 * The host block allocator (pkv_alloc_*) is not thread-safe: the caller
 * serialises calls on one handle, as the pages' single scheduler does.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or id   */
    PKV_ERR_UNSUPPORTED = 2, /* head_dim / block_size / dtype not built   */
    PKV_ERR_OOM = 3,         /* allocator: not enough free blocks          */
    PKV_ERR_WORKSPACE = 4,   /* decode: workspace too small               */
    PKV_ERR_CUDA = 5,        /* a CUDA runtime call failed                */
    PKV_ERR_HOST_MEMORY = 6  /* the library's own host allocation failed  */
} pkv_status;

typedef enum { PKV_F16 = 0, PKV_BF16 = 1 } pkv_dtype;

/* Bits of the device error word (pkv_get_device_errors). */
#define PKV_DEVERR_BLOCK_ID 0x1  /* block table entry outside [0, NB)     */
#define PKV_DEVERR_SLOT 0x2      /* slot outside [0, NB*bs) (and >= 0)    */
#define PKV_DEVERR_CONTEXT 0x4   /* context_len < 0 or > max context      */
#define PKV_DEVERR_POSITION 0x8  /* slot mapping: position past the table */
#define PKV_DEVERR_GROUP 0x10    /* shared-prefix group out of range      */
#define PKV_DEVERR_TIMEOUT 0x20  /* a bounded wait inside a kernel ran out: the call's
                                    results are not valid */

/* Thread-local text of the last error ("" if none).  Never NULL. */
const char* pkv_last_error_string(void);

/* Library version string. */
const char* pkv_version(void);

/* ------------------------------------------------------------------ *
 * Decode attention
 * ------------------------------------------------------------------ */

/* Bytes of device workspace pkv_paged_attention_decode needs for S
 * sequences, H heads, head_dim D, contexts of at most max_context_len tokens
 * and partitions of partition_tokens tokens (0 = library default).  The
 * workspace holds the work list, per-partition softmax partials (running
 * max, running sum and the unnormalised output, fp32) and merge tickets.
 * Returns 0 for invalid arguments. */
size_t pkv_decode_workspace_size(int S, int H, int D, int max_context_len,
                                 int partition_tokens);

/* Single-query decode attention over the paged cache.
 *
 * For every sequence s and head h, with n = context_lens[s]:
 *   out[s,h,:] = sum_{j<n} softmax_j(scale * q[s,h,:] . K_j) V_j
 * where K_j, V_j are the cache rows of token j, found by address
 * translation: logical = j / bs, offset = j % bs, physical =
 * block_tables[s*MB + logical] ([P3] 3.1.3 steps 1-4; [P4] "疑问" 1).
 * n = 0 gives out = 0.  num_kv_heads = num_heads (multi-head attention).
 *
 *   out           [S][H][D] dtype, written
 *   q             [S][H][D] dtype
 *   k_cache, v_cache  [NB][bs][H][D] dtype, read only
 *   block_tables  [S][MB] int32
 *   context_lens  [S] int32, each in [0, max_context_len]
 *   max_context_len  upper bound of context_lens (0 = MB*bs); at most MB*bs
 *   scale         logit scale (usually 1/sqrt(D))
 *   partition_tokens  tokens per split-K partition, a multiple of 16 and of
 *                 bs (0 = library default).  Contexts longer than one
 *                 partition are split; each partition's (max, sum, output)
 *                 is merged by the last partition to finish.
 *   workspace     device memory of at least pkv_decode_workspace_size(S, H,
 *                 D, max_context_len, partition_tokens) bytes, 256-byte
 *                 aligned; no initial contents needed.  One call at a time
 *                 may use a workspace (calls that overlap on the GPU race).
 * Computation is fp32 with one round-to-nearest-even to dtype at the end.
 */
pkv_status pkv_paged_attention_decode(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens,
    int S, int H, int D, int bs, int NB, int MB, int max_context_len,
    float scale, pkv_dtype dtype, int partition_tokens,
    void* workspace, size_t workspace_bytes, void* stream);

/* One decode step's device work after the host has made room for the new
 * tokens (and copied any copy-on-write blocks with pkv_copy_blocks): the
 * new tokens' slots, their K/V written into the caches, then decode
 * attention over every sequence's whole context.  The result is exactly
 * that of pkv_compute_slot_mapping, pkv_reshape_and_cache and
 * pkv_paged_attention_decode called in that order with the same arguments
 * (same slots, same cache contents, bit-identical output); it runs in two
 * kernels instead of four (three with prefix groups), the slot mapping,
 * cache write and the decode's work plan in one.  This fusion is this
 * library's; the pages describe the three operations, not a combined call.
 *
 *   key, value    [T][H][D] dtype: K and V of the new tokens, 16-byte aligned
 *   seq_idx, pos  [T] int32: each new token's sequence and position
 *   slot_mapping  [T] int64, written: the slots, as pkv_compute_slot_mapping
 *                 gives them (-1: not written, see there)
 *   k_cache, v_cache  written for the new tokens, then read
 *   prefix_groups, G  G = 0 (prefix_groups may be NULL): the decode is
 *                 pkv_paged_attention_decode's.  G > 0: it is
 *                 pkv_paged_attention_decode_shared_prefix's with these
 *                 groups, and the workspace is sized by
 *                 pkv_decode_shared_prefix_workspace_size.
 *   other arguments as in pkv_paged_attention_decode; context_lens count the
 *   new tokens.  T = 0 is a plain decode; S = 0 with T > 0 is
 *   PKV_ERR_INVALID_ARG. */
pkv_status pkv_decode_step(
    void* out, const void* q, const void* key, const void* value,
    void* k_cache, void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, const int32_t* seq_idx, const int32_t* pos,
    int64_t* slot_mapping, const int32_t* prefix_groups, int G, int T, int S,
    int H, int D, int bs, int NB, int MB, int max_context_len, float scale,
    pkv_dtype dtype, int partition_tokens, void* workspace,
    size_t workspace_bytes, void* stream);

/* Decode attention where groups of sequences share a prefix (parallel
 * sampling, beam search, a common system prompt: [P1] 3.3.2 "Copy-on-Write
 * 页面共享机制", [P3] 3.1.5, [P4] "Memory Sharing与写时复制").  Computes exactly
 * what pkv_paged_attention_decode computes; the shared prefix of each group
 * is read from HBM once for all its members and its q.K and P.V run on the
 * tensor cores with the members' queries as one matrix.
 *
 *   prefix_groups  [G][3] int32, device memory: (first sequence, number of
 *                  members n in 1..16, prefix tokens).  The members are the
 *                  sequences first .. first+n-1; their block tables must hold
 *                  the same physical blocks for the first `prefix tokens`
 *                  tokens (a multiple of 16, at most each member's context).
 *                  Groups must not overlap; other sequences are decoded as
 *                  usual.
 *   other arguments as in pkv_paged_attention_decode, except that the
 *   workspace needs pkv_decode_shared_prefix_workspace_size(S, H, D, G,
 *   max_context_len, partition_tokens) bytes.
 * Only whole partitions inside a prefix are shared; a prefix shorter than a
 * partition is decoded as usual.  The prefix runs on mma.sync by default;
 * with PKV_PREFIX_KERNEL=tcgen05 in the environment (read on every call) and
 * head_dim 128 it runs on tcgen05 with TMA loads instead (same results
 * within the attention tolerance). */
size_t pkv_decode_shared_prefix_workspace_size(int S, int H, int D, int G, int max_context_len,
                                               int partition_tokens);
pkv_status pkv_paged_attention_decode_shared_prefix(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, const int32_t* prefix_groups,
    int G, int S, int H, int D, int bs, int NB, int MB, int max_context_len, float scale,
    pkv_dtype dtype, int partition_tokens, void* workspace, size_t workspace_bytes,
    void* stream);

/* Size of the scratch array built into the library for
 * pkv_paged_attention_decode_noalloc: 16 MiB per device. */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)

/* Decode attention for callers that cannot allocate device memory.
 *
 * The pages have no counterpart: this is a deployment convenience.  Some
 * callers may not call cudaMalloc at all: a plugin inside a serving runtime
 * that owns every byte of device memory and hands it out only through its
 * own pool, a latency-critical loop where a cudaMalloc could synchronise
 * the whole device, or a small C host program with no device allocator of
 * its own.  This entry point takes the same arguments as
 * pkv_paged_attention_decode except the workspace, runs the same kernels,
 * and allocates nothing (no cudaMalloc, no cudaFree).
 *
 * Its split-K scratch is a static device array of PKV_NOALLOC_SCRATCH_BYTES
 * inside the library: every GPU that loads the library holds one copy until
 * the process exits.
 *   - A fixed partition_tokens > 0 gives pkv_paged_attention_decode's
 *     result at that partition size bit for bit; a call whose need
 *     (pkv_decode_workspace_size of the same S, H, D, max_context_len,
 *     partition_tokens) exceeds the array returns PKV_ERR_WORKSPACE.
 *   - partition_tokens = 0 starts the automatic choice from the smallest of
 *     64, 128, ..., 4096 tokens whose partials fit the array, so it may run
 *     larger partitions than pkv_paged_attention_decode would: the result
 *     then agrees with it within the attention tolerance, not bit for bit.
 *     Only a size that does not fit even at 4096-token partitions returns
 *     PKV_ERR_WORKSPACE.
 * Use pkv_paged_attention_decode with a caller workspace for larger sizes.
 *
 * The first call in a device's context looks up the array's device address
 * with that device current; make that first call before any stream capture
 * begins.  The address is kept per device together with the id of the
 * context it was found in: after a device reset the next call sees a new
 * context and looks the address up again (so that call, too, should come
 * before any capture).  All calls on a device share the one array, which
 * keeps the last call's contents; each call resets what it reads before
 * reading it.  Calls that overlap on the GPU (other streams, other host
 * threads) race on the array and give wrong results: serialise them. */
pkv_status pkv_paged_attention_decode_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens,
    int S, int H, int D, int bs, int NB, int MB, int max_context_len,
    float scale, pkv_dtype dtype, int partition_tokens, void* stream);

/* ------------------------------------------------------------------ *
 * Cache maintenance kernels
 * ------------------------------------------------------------------ */

/* Slot of each new token (address translation, [P3] 3.1.3 steps 1-3):
 *   slot_mapping[t] = block_tables[seq_idx[t]*MB + pos[t]/bs]*bs + pos[t]%bs
 * pos[t] < 0 gives -1 (no write).  A position past the row (pos/bs >= MB)
 * or a seq_idx outside [0, S) gives -1 and sets PKV_DEVERR_POSITION; a
 * position whose table entry is negative (no block mapped) gives -1 and
 * sets PKV_DEVERR_BLOCK_ID.
 *   slot_mapping  [T] int64 device, written
 *   block_tables  [S][MB] int32 device; seq_idx, pos: [T] int32 device   */
pkv_status pkv_compute_slot_mapping(int64_t* slot_mapping, const int32_t* block_tables,
                                    const int32_t* seq_idx, const int32_t* pos,
                                    int T, int S, int MB, int bs, void* stream);

/* Write new tokens' K and V into their slots (the "write the new KV data
 * into the block" step of [P2] "Copy-on-Write共享解码的显存优化原理"):
 *   k_cache[slot/bs][slot%bs][h][:] = key[t][h][:], same for V,
 * for every t with slot_mapping[t] >= 0 (negative = skip).  Slots must be
 * distinct within a call.
 *   key, value  [T][H][D] dtype device;  slot_mapping [T] int64 device   */
pkv_status pkv_reshape_and_cache(const void* key, const void* value, void* k_cache,
                                 void* v_cache, const int64_t* slot_mapping, int T,
                                 int H, int D, int bs, int NB, pkv_dtype dtype,
                                 void* stream);

/* Copy-on-write block copies ([P2] "Copy-on-Write共享解码的显存优化原理";
 * [P3] 3.1.5 step 3): for each of the P pairs (src, dst) in block_mapping
 * ([P][2] int64 device), copy all bs*H*D elements of K block src to K block
 * dst and likewise for V.  No dst may appear twice or also be a src in the
 * same call (the allocator's copies always target fresh blocks).  P = 0 is
 * a no-op. */
pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping,
                           int P, int H, int D, int bs, int NB, pkv_dtype dtype,
                           void* stream);

/* Host-side check of pkv_copy_blocks' precondition on a copy list the
 * caller holds in host memory (pairs [P][2] int64, (src, dst)): every id in
 * [0, NB), no dst twice, no dst that is also a src.  PKV_OK if it holds,
 * PKV_ERR_INVALID_ARG (naming the first offending pair) if not,
 * PKV_ERR_HOST_MEMORY if the check's scratch cannot be allocated.  Reads
 * only; O(P log P).  pkv_beam_step runs it on its own pairs before the
 * upload. */
pkv_status pkv_check_copy_pairs(const int64_t* pairs, int32_t P, int32_t NB);

/* Swap directions for pkv_swap_blocks. */
#define PKV_SWAP_OUT 0 /* GPU cache -> host cache */
#define PKV_SWAP_IN 1  /* host cache -> GPU cache */

/* Block copies between the GPU caches and host caches (CPU swap, [P1]
 * 3.3.3: the KV of a sequence's blocks is copied page by page to CPU-side
 * blocks so the GPU blocks can be freed, and copied back into freshly
 * allocated GPU blocks later).  For each of the P pairs (src, dst) of
 * block_mapping ([P][2] int64, device memory): PKV_SWAP_OUT copies GPU
 * block src of gpu_k / gpu_v to host block dst of host_k / host_v;
 * PKV_SWAP_IN copies host block src to GPU block dst.
 *   gpu_k, gpu_v    [NB_gpu][bs][H][D] dtype, device memory
 *   host_k, host_v  [NB_host][bs][H][D] dtype, page-locked host memory the
 *                   device can address (cudaHostAlloc / cudaMallocHost, or
 *                   cudaHostRegister'ed); anything else is
 *                   PKV_ERR_INVALID_ARG.  One kernel moves every block over
 *                   the CPU-GPU link, no per-block copy call.
 * No destination block may appear twice in one call.  Ids outside their pool
 * are skipped and set PKV_DEVERR_BLOCK_ID. */
pkv_status pkv_swap_blocks(void* gpu_k, void* gpu_v, void* host_k, void* host_v,
                           const int64_t* block_mapping, int P, int H, int D, int bs,
                           int NB_gpu, int NB_host, pkv_dtype dtype, int direction,
                           void* stream);

/* Waits for `stream`, then returns PKV_ERR_CUDA if any asynchronous CUDA
 * error is pending. */
pkv_status pkv_sync_check(void* stream);

/* Reads and clears the device error word (PKV_DEVERR_* bits) of the
 * current device.  Synchronises with the device. */
pkv_status pkv_get_device_errors(int32_t* flags);

/* Self-test of the give-up path of the library's in-kernel waits.  The
 * tensor-core shared-prefix kernel (PKV_PREFIX_KERNEL=tcgen05) hands work
 * between its warps through shared-memory barriers, and each wait there
 * gives up after at most 2^20 polls (about 0.1 s on GB300): the CTA then
 * sets PKV_DEVERR_TIMEOUT, frees its tensor memory and returns, and the
 * context stays usable.  This call launches one warp on `stream` that takes
 * tensor memory, waits `polls` polls on a barrier that nothing completes,
 * sets PKV_DEVERR_TIMEOUT, frees the tensor memory and returns.
 * Asynchronous; read the bit with pkv_get_device_errors.  `polls` outside
 * [1, 2^20]: PKV_ERR_INVALID_ARG, nothing launched. */
pkv_status pkv_selftest_bounded_wait(int64_t polls, void* stream);

/* ------------------------------------------------------------------ *
 * Host block allocator: one global pool of physical blocks with a free
 * list and a reference count per physical block ([P1] 3.3.2 and 3.3.4;
 * [P2] "Copy-on-Write共享解码的显存优化原理"; [P3] 3.1.2, 3.1.5; [P4]
 * "Memory Sharing与写时复制": the count lives with the physical block).
 * The free list is a stack: the block freed last is handed out first; a
 * fresh pool hands out NB-1 first.  Every operation is all-or-nothing.
 * ------------------------------------------------------------------ */
typedef struct pkv_allocator pkv_allocator;

/* A pool of num_blocks free blocks. */
pkv_status pkv_alloc_create(int32_t num_blocks, pkv_allocator** out);

/* A pool whose free list is initial_free[0..n_free) (the last element is
 * handed out first); every block of [0, num_blocks) not listed is held once
 * (refcount 1).  Ids must be distinct and in range. */
pkv_status pkv_alloc_create_with_order(int32_t num_blocks, const int32_t* initial_free,
                                       int32_t n_free, pkv_allocator** out);

void pkv_alloc_destroy(pkv_allocator* a);

/* Take n blocks (refcount 1 each) into out_ids[0..n).  PKV_ERR_OOM takes
 * nothing ([P1] 3.3.2 allocator sketch checks before taking). */
pkv_status pkv_alloc_blocks(pkv_allocator* a, int32_t n, int32_t* out_ids);

/* One more holder for each block (sharing a prefix / forking a sequence,
 * [P1] 3.3.2 share_blocks; [P3] 3.1.5 step 2).  Every id must be held. */
pkv_status pkv_alloc_incref(pkv_allocator* a, const int32_t* ids, int32_t n);

/* One holder fewer for each block; a block whose count reaches 0 returns to
 * the free list ([P2] "引用计数机制还服务于Block的回收").  Releasing a block
 * that is not held is PKV_ERR_INVALID_ARG (nothing changes).
 * *num_freed (may be NULL) receives the number of blocks freed. */
pkv_status pkv_alloc_decref(pkv_allocator* a, const int32_t* ids, int32_t n,
                            int32_t* num_freed);

/* Copy-on-write before a write into block id: at refcount 1 *out_id = id
 * and *needs_copy = 0; otherwise a new block is taken (PKV_ERR_OOM leaves
 * everything unchanged), id loses one holder, *out_id = the new block and
 * *needs_copy = 1: the caller copies id -> *out_id (pkv_copy_blocks) and
 * points its table at *out_id ([P2] "Copy-on-Write共享解码的显存优化原理";
 * [P3] 3.1.5 steps 3-4). */
pkv_status pkv_alloc_cow(pkv_allocator* a, int32_t id, int32_t* out_id, int32_t* needs_copy);

/* Make room for tokens [ctx_before, ctx_before + n_new) of one sequence
 * whose block table row is table[0..*num_blocks) (capacity max_blocks):
 * first every existing block those tokens land in that has refcount > 1 is
 * copied-on-write (in logical order; its (src, dst) pair is appended to
 * pairs[2*k], pairs[2*k+1] and the table entry repointed); then as many
 * new blocks are appended as ceil((ctx_before + n_new)/bs) requires ([P1]
 * 3.3.2: batch allocation at prefill, one more block whenever the token
 * count exceeds num_blocks*bs).  *n_pairs receives the number of pairs;
 * `pairs` needs room for 2*ceil(n_new/bs + 1) int64.  All-or-nothing:
 * PKV_ERR_OOM or PKV_ERR_INVALID_ARG leave table, counts and pool as they
 * were. */
pkv_status pkv_alloc_append(pkv_allocator* a, int32_t* table, int32_t* num_blocks,
                            int32_t max_blocks, int32_t ctx_before, int32_t n_new,
                            int32_t bs, int64_t* pairs, int32_t* n_pairs);

/* Batched append for S sequences whose tables are the rows of tables
 * ([S][MB] int32, row s has num_blocks[s] valid entries): for s = 0, 1, ...
 * in order, the same as pkv_alloc_append(row s, ctx_before[s], n_new[s]).
 * Copy pairs of all sequences go to pairs[2*k], pairs[2*k+1] (room for
 * max_pairs pairs; sequence s is only started if n_new[s]/bs + 2 more pairs
 * fit); *n_pairs receives their number.  On PKV_ERR_OOM (or a full pairs
 * buffer, PKV_ERR_INVALID_ARG) sequences [0, *n_done) have been extended and
 * the rest are untouched; *n_done = S on success. */
pkv_status pkv_alloc_append_batch(pkv_allocator* a, int32_t* tables, int32_t* num_blocks,
                                  int32_t S, int32_t MB, const int32_t* ctx_before,
                                  const int32_t* n_new, int32_t bs, int64_t* pairs,
                                  int32_t max_pairs, int32_t* n_pairs, int32_t* n_done);

/* Fork (beam search, parallel sampling: [P1] 3.3.2 share_blocks; [P4]
 * "Memory Sharing与写时复制"): row s of tables ([S][MB] int32, num_blocks[s]
 * entries) becomes a copy of row parents[s] of the old tables.  A hold is
 * taken on every block of the new rows before the holds of the old rows are
 * released, so a block that survives the fork never reaches refcount 0.
 * All-or-nothing: an invalid parent, an entry that is not a held block or a
 * release that would underflow changes nothing (PKV_ERR_INVALID_ARG). */
pkv_status pkv_alloc_fork(pkv_allocator* a, int32_t* tables, int32_t* num_blocks, int32_t S,
                          int32_t MB, const int32_t* parents);

/* Reference count of block id (0 = free). */
pkv_status pkv_alloc_refcount(const pkv_allocator* a, int32_t id, int32_t* rc);

int32_t pkv_alloc_num_blocks(const pkv_allocator* a);
int32_t pkv_alloc_num_free(const pkv_allocator* a);
/* Blocks held more than once (refcount > 1). */
int32_t pkv_alloc_num_shared(const pkv_allocator* a);

/* ------------------------------------------------------------------ *
 * Beam-search step in one call ([P1] 3.3.2 share_blocks; [P2]
 * "Copy-on-Write共享解码的显存优化原理"; [P4] "Memory Sharing与写时复制":
 * beams share their blocks until a write diverges them).  The call is
 * exactly this sequence of the entry points above:
 *   1. pkv_alloc_fork(a, tables, num_blocks, S, MB, parents);
 *   2. pkv_alloc_append_batch for one new token per sequence, after
 *      ctx_before[s] = context_lens[parents[s]] (the old lengths): the
 *      copy-on-write pairs of shared last blocks, new blocks at block
 *      boundaries; the pairs then pass pkv_check_copy_pairs;
 *   3. context_lens[s] = ctx_before[s] + 1 (host array, in place);
 *   4. the tables, lengths, token positions (ctx_before), sequence index
 *      (0..S-1) and copy pairs are written into `staging` and uploaded to
 *      `dev_inputs` by one cudaMemcpyAsync on `stream`;
 *   5. pkv_copy_blocks for the pairs, then pkv_decode_step for the S new
 *      tokens (key/value/q [S][H][D], device) with max_context_len = MB*bs
 *      and the G prefix groups (device [G][3], as pkv_decode_step takes
 *      them; G = 0: none).  The beams of one request keep their prompt's
 *      full blocks shared for the whole search (only the ends of the
 *      contexts are written), so a group per request -- its beams, the
 *      prompt's full blocks as the prefix -- reads each prompt once.
 *
 *   tables [S][MB], num_blocks [S], context_lens [S]: host int32, in place
 *   parents [S]: host int32, each in [0, S)
 *   staging: pinned host memory, dev_inputs: device memory, both 256-byte
 *           aligned and inputs_bytes >= pkv_beam_inputs_bytes(S, MB) long.
 *           The copy out of `staging` is asynchronous: the caller does not
 *           pass the same staging buffer again before `stream` has passed
 *           this call (two buffers used in turn, with an event, work).
 *           dev_inputs is read by this step's kernels on `stream`, so one
 *           device buffer serves every step on that stream.
 *   slot_mapping [S] int64 (device, written); workspace of at least
 *           pkv_decode_workspace_size(S, H, D, MB*bs, partition_tokens),
 *           or with G > 0 pkv_decode_shared_prefix_workspace_size(S, H, D,
 *           G, MB*bs, partition_tokens)
 *   *n_pairs  receives the number of copy pairs; they are in `staging`
 *           as int64 [n][2].  Layout of staging and dev_inputs, each part
 *           at a multiple of 256 bytes (r(x) rounds x up to one): tables
 *           [S][MB] int32 at 0; context lengths [S] int32 at
 *           o1 = r(4*S*MB); positions [S] at o2 = o1 + r(4*S); sequence
 *           index [S] at o3 = o2 + r(4*S); copy pairs at o3 + r(4*S), room
 *           for 2*S of them
 * Errors: arguments are checked before step 1 (PKV_ERR_INVALID_ARG: a
 * parent out of range, a context that would pass the table, buffers too
 * small or misaligned).  A failure of step 1 changes nothing; a failure of
 * step 2 (PKV_ERR_OOM, or pairs that fail pkv_check_copy_pairs) leaves the
 * fork done and the first sequences extended, as pkv_alloc_append_batch
 * describes, and launches nothing.  A
 * failure in steps 4-5 (PKV_ERR_CUDA, or an argument pkv_copy_blocks or
 * pkv_decode_step rejects) comes after steps 1-3 have updated the host
 * arrays and the allocator. */
size_t pkv_beam_inputs_bytes(int32_t S, int32_t MB);

pkv_status pkv_beam_step(
    pkv_allocator* a, int32_t* tables, int32_t* num_blocks, int32_t* context_lens,
    const int32_t* parents, int32_t S, int32_t MB, void* staging, void* dev_inputs,
    size_t inputs_bytes, void* out, const void* q, const void* key, const void* value,
    void* k_cache, void* v_cache, int64_t* slot_mapping, const int32_t* prefix_groups, int G,
    int H, int D, int bs, int NB, float scale, pkv_dtype dtype, int partition_tokens,
    void* workspace, size_t workspace_bytes, int32_t* n_pairs, void* stream);

/* ------------------------------------------------------------------ *
 * A beam search held on the native side: pkv_beam_step with everything
 * that stays the same from step to step given once, and the alternation
 * of two staging buffers done here ([P1] 3.3.2 share_blocks; [P4]
 * "Memory Sharing与写时复制": the beams of a search fork and diverge
 * step after step over one pool).
 *
 * pkv_beam_search_create keeps the pointers and sizes (all of them as
 * pkv_beam_step takes them; the caller still owns every buffer and keeps it
 * alive until pkv_beam_search_destroy) and creates one CUDA event per
 * staging buffer on the current device.  staging0 and staging1: pinned
 * host memory, 256-byte aligned, inputs_bytes each.
 * Errors: PKV_ERR_INVALID_ARG (null pointer, bad size, misaligned buffer,
 * inputs_bytes < pkv_beam_inputs_bytes(S, MB)) before any CUDA call;
 * PKV_ERR_CUDA if an event cannot be created; PKV_ERR_HOST_MEMORY. */
typedef struct pkv_beam_search pkv_beam_search;

pkv_status pkv_beam_search_create(
    pkv_allocator* a, int32_t* tables, int32_t* num_blocks, int32_t* context_lens, int32_t S,
    int32_t MB, void* staging0, void* staging1, void* dev_inputs, size_t inputs_bytes, void* out,
    void* k_cache, void* v_cache, int64_t* slot_mapping, const int32_t* prefix_groups, int G,
    int H, int D, int bs, int NB, float scale, pkv_dtype dtype, int partition_tokens,
    void* workspace, size_t workspace_bytes, pkv_beam_search** out_search);

/* One step of the search: waits (on the host) until the upload from the
 * staging buffer used two steps ago has finished, runs pkv_beam_step with
 * that buffer, records the buffer's event on `stream` (whatever the
 * outcome), and returns the step's copy pairs: *n_pairs of them at
 * *pairs ([n][2] int64, (src, dst)), inside that staging buffer and valid
 * until the step after next.  parents [S] host int32; q, key, value
 * [S][H][D] device.  Errors are pkv_beam_step's; PKV_ERR_CUDA if the wait
 * or the event record fails. */
pkv_status pkv_beam_search_step(pkv_beam_search* search, const int32_t* parents, const void* q,
                                const void* key, const void* value, void* stream,
                                int32_t* n_pairs, const int64_t** pairs);

/* Destroys the events and the handle (waits for neither; the caller
 * synchronises its stream first). */
void pkv_beam_search_destroy(pkv_beam_search* search);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
