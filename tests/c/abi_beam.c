/*
 * A plain C11 caller of libpagedkv: a beam search through the C ABI only
 * (pkv_beam_search_create / _step / _destroy), 2 requests x 2 beams x 4
 * heads x 64 dims, fp16, block size 16, 6 steps with forks.
 *
 * The check keeps each beam's logical K/V history on the host: a beam that
 * continues from parent p holds p's tokens and then its own new token ("3.3
 * 页面级显存管理" 3.3.2: forked sequences share blocks until a write
 * diverges them).  After every step
 *   - every token of every beam, gathered through the library's tables from
 *     the device caches, equals that history bit for bit (fork, copy on
 *     write and the cache write together);
 *   - attention equals the C oracle's on a contiguous copy of the same
 *     histories within 2e-3 + 1e-2 |ref|;
 *   - the context lengths grew by one from the parent's, and the copy pairs
 *     are ids of the pool with no target twice and no target that is also
 *     a source.
 * At the end the refcounts add up to the table entries.  Exit status 0 when
 * all hold.
 */
#include <cuda_runtime_api.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "pagedkv.h"

/* from the oracle (test infrastructure) */
int oracle_decode(double* out, const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens, int S, int H, int D,
                  int block_size, int MB, double scale, int is_bf16, const int32_t* row_of_block,
                  const int32_t* items, int n_items, int nthreads);

#define R 2         /* requests */
#define B 2         /* beams per request */
#define S (R * B)   /* sequences */
#define H 4
#define D 64
#define BS 16
#define NB 64
#define MB 8
#define STEPS 6
#define ROW (H * D) /* 16-bit values of one token in one cache */

#define CHECK_PKV(x)                                                         \
    do {                                                                     \
        pkv_status st_ = (x);                                                \
        if (st_ != PKV_OK) {                                                 \
            fprintf(stderr, "%s: %d %s\n", #x, (int)st_, pkv_last_error_string()); \
            return 1;                                                        \
        }                                                                    \
    } while (0)
#define CHECK_CUDA(x)                                                        \
    do {                                                                     \
        cudaError_t e_ = (x);                                                \
        if (e_ != cudaSuccess) {                                             \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));         \
            return 1;                                                        \
        }                                                                    \
    } while (0)

static uint64_t rng_state = 0x2545f4914f6cdd1dull;
static uint64_t next_u64(void) { /* splitmix64 */
    uint64_t z = (rng_state += 0x9e3779b97f4a7c15ull);
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}
/* a random fp16 in [-2, 2): sign, exponent 13..15, random mantissa */
static uint16_t rand_half(void) {
    uint64_t r = next_u64();
    return (uint16_t)(((r & 1) << 15) | ((13 + (r >> 1) % 3) << 10) | ((r >> 8) & 0x3ff));
}
static double half_to_double(uint16_t h) {
    int e = (h >> 10) & 31, f = h & 1023;
    double v = e ? ldexp(1024 + f, e - 25) : ldexp(f, -24);
    return (h >> 15) ? -v : v;
}

/* each beam's logical history: [S][MB * BS tokens][ROW] for K and for V */
static uint16_t hist_k[S][MB * BS][ROW], hist_v[S][MB * BS][ROW];
static uint16_t next_k[S][MB * BS][ROW], next_v[S][MB * BS][ROW];
static uint16_t cache_k[NB * BS * ROW], cache_v[NB * BS * ROW];
static uint16_t cont_k[S * MB * BS * ROW], cont_v[S * MB * BS * ROW];

int main(void) {
    const int prompt[R] = {20, 33};
    /* parents per step, each within its own request (beams r*B .. r*B+B-1) */
    const int32_t parents[STEPS][S] = {{0, 0, 2, 3}, {1, 0, 3, 3}, {1, 1, 2, 2},
                                       {0, 1, 3, 2}, {0, 0, 2, 2}, {1, 0, 3, 2}};
    int32_t tables[S * MB], nblocks[S], ctx[S];
    for (int i = 0; i < S * MB; ++i) tables[i] = -1;

    /* a shuffled pool; each request's prompt blocks are taken once and
     * shared by its beams */
    int32_t order[NB];
    for (int i = 0; i < NB; ++i) order[i] = i;
    for (int i = NB - 1; i > 0; --i) {
        int j = (int)(next_u64() % (uint64_t)(i + 1));
        int32_t t = order[i]; order[i] = order[j]; order[j] = t;
    }
    pkv_allocator* alloc = NULL;
    CHECK_PKV(pkv_alloc_create_with_order(NB, order, NB, &alloc));
    for (size_t i = 0; i < sizeof cache_k / 2; ++i) { cache_k[i] = rand_half(); cache_v[i] = rand_half(); }
    for (int r = 0; r < R; ++r) {
        const int n = (prompt[r] + BS - 1) / BS;
        int32_t ids[MB];
        CHECK_PKV(pkv_alloc_blocks(alloc, n, ids));
        for (int b = 0; b < B; ++b) {
            const int s = r * B + b;
            memcpy(&tables[s * MB], ids, n * sizeof(int32_t));
            nblocks[s] = n;
            ctx[s] = prompt[r];
            if (b > 0) CHECK_PKV(pkv_alloc_incref(alloc, ids, n));
        }
        for (int t = 0; t < prompt[r]; ++t) {
            uint16_t* kr = &cache_k[((size_t)ids[t / BS] * BS + t % BS) * ROW];
            uint16_t* vr = &cache_v[((size_t)ids[t / BS] * BS + t % BS) * ROW];
            for (int b = 0; b < B; ++b) {
                memcpy(hist_k[r * B + b][t], kr, ROW * 2);
                memcpy(hist_v[r * B + b][t], vr, ROW * 2);
            }
        }
    }

    /* device buffers and the search */
    const size_t in_bytes = pkv_beam_inputs_bytes(S, MB);
    const size_t ws_bytes = pkv_decode_workspace_size(S, H, D, MB * BS, 0);
    void *dk, *dv, *dq, *dkey, *dval, *dout, *dws, *din, *stg0, *stg1;
    int64_t* dslot;
    CHECK_CUDA(cudaMalloc(&dk, sizeof cache_k));
    CHECK_CUDA(cudaMalloc(&dv, sizeof cache_v));
    CHECK_CUDA(cudaMalloc(&dq, S * ROW * 2));
    CHECK_CUDA(cudaMalloc(&dkey, S * ROW * 2));
    CHECK_CUDA(cudaMalloc(&dval, S * ROW * 2));
    CHECK_CUDA(cudaMalloc(&dout, S * ROW * 2));
    CHECK_CUDA(cudaMalloc(&dws, ws_bytes));
    CHECK_CUDA(cudaMalloc(&din, in_bytes));
    CHECK_CUDA(cudaMalloc((void**)&dslot, S * sizeof(int64_t)));
    CHECK_CUDA(cudaHostAlloc(&stg0, in_bytes, cudaHostAllocDefault));
    CHECK_CUDA(cudaHostAlloc(&stg1, in_bytes, cudaHostAllocDefault));
    CHECK_CUDA(cudaMemcpy(dk, cache_k, sizeof cache_k, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dv, cache_v, sizeof cache_v, cudaMemcpyHostToDevice));
    const float scale = 0.125f;
    pkv_beam_search* search = NULL;
    CHECK_PKV(pkv_beam_search_create(alloc, tables, nblocks, ctx, S, MB, stg0, stg1, din, in_bytes,
                                     dout, dk, dv, dslot, NULL, 0, H, D, BS, NB, scale, PKV_F16, 0,
                                     dws, ws_bytes, &search));

    double worst = 0.0;
    int total_pairs = 0;
    for (int step = 0; step < STEPS; ++step) {
        uint16_t q[S * ROW], key[S * ROW], val[S * ROW];
        for (int i = 0; i < S * ROW; ++i) { q[i] = rand_half(); key[i] = rand_half(); val[i] = rand_half(); }
        CHECK_CUDA(cudaMemcpy(dq, q, sizeof q, cudaMemcpyHostToDevice));
        CHECK_CUDA(cudaMemcpy(dkey, key, sizeof key, cudaMemcpyHostToDevice));
        CHECK_CUDA(cudaMemcpy(dval, val, sizeof val, cudaMemcpyHostToDevice));
        int32_t old_ctx[S];
        memcpy(old_ctx, ctx, sizeof ctx);

        int32_t np = -1;
        const int64_t* pairs = NULL;
        CHECK_PKV(pkv_beam_search_step(search, parents[step], dq, dkey, dval, NULL, &np, &pairs));
        CHECK_PKV(pkv_sync_check(NULL));
        int32_t flags = -1;
        CHECK_PKV(pkv_get_device_errors(&flags));
        if (flags) { fprintf(stderr, "step %d: device error word %#x\n", step, flags); return 1; }

        /* the histories after this step */
        for (int s = 0; s < S; ++s) {
            const int p = parents[step][s], n = old_ctx[p];
            memcpy(next_k[s], hist_k[p], (size_t)n * ROW * 2);
            memcpy(next_v[s], hist_v[p], (size_t)n * ROW * 2);
            memcpy(next_k[s][n], &key[s * ROW], ROW * 2);
            memcpy(next_v[s][n], &val[s * ROW], ROW * 2);
            if (ctx[s] != n + 1) { fprintf(stderr, "step %d: ctx[%d] = %d, want %d\n", step, s, ctx[s], n + 1); return 1; }
        }
        memcpy(hist_k, next_k, sizeof hist_k);
        memcpy(hist_v, next_v, sizeof hist_v);

        /* copy pairs: pool ids, no target twice, no target that is a source */
        if (np < 0 || (np > 0 && !pairs)) { fprintf(stderr, "step %d: bad pair list\n", step); return 1; }
        for (int i = 0; i < np; ++i) {
            const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
            if (src < 0 || src >= NB || dst < 0 || dst >= NB) { fprintf(stderr, "pair out of the pool\n"); return 1; }
            for (int j = 0; j < np; ++j) {
                if (j != i && pairs[2 * j + 1] == dst) { fprintf(stderr, "target twice\n"); return 1; }
                if (pairs[2 * j] == dst) { fprintf(stderr, "target is a source\n"); return 1; }
            }
        }
        total_pairs += np;

        /* every token through the library's tables equals the history */
        CHECK_CUDA(cudaMemcpy(cache_k, dk, sizeof cache_k, cudaMemcpyDeviceToHost));
        CHECK_CUDA(cudaMemcpy(cache_v, dv, sizeof cache_v, cudaMemcpyDeviceToHost));
        for (int s = 0; s < S; ++s) {
            for (int t = 0; t < ctx[s]; ++t) {
                const int32_t blk = tables[s * MB + t / BS];
                if (blk < 0 || blk >= NB) { fprintf(stderr, "step %d: seq %d token %d: block %d\n", step, s, t, blk); return 1; }
                const size_t at = ((size_t)blk * BS + t % BS) * ROW;
                if (memcmp(&cache_k[at], hist_k[s][t], ROW * 2) || memcmp(&cache_v[at], hist_v[s][t], ROW * 2)) {
                    fprintf(stderr, "step %d: seq %d token %d differs from its history\n", step, s, t);
                    return 1;
                }
            }
        }

        /* attention against the oracle on contiguous copies of the histories */
        int32_t ident[S * MB];
        for (int s = 0; s < S; ++s) {
            for (int j = 0; j < MB; ++j) ident[s * MB + j] = s * MB + j;
            memcpy(&cont_k[(size_t)s * MB * BS * ROW], hist_k[s], sizeof hist_k[s]);
            memcpy(&cont_v[(size_t)s * MB * BS * ROW], hist_v[s], sizeof hist_v[s]);
        }
        double ref[S * ROW];
        oracle_decode(ref, q, cont_k, cont_v, ident, ctx, S, H, D, BS, MB, scale, 0, NULL, NULL, 0, 1);
        uint16_t got[S * ROW];
        CHECK_CUDA(cudaMemcpy(got, dout, sizeof got, cudaMemcpyDeviceToHost));
        for (int i = 0; i < S * ROW; ++i) {
            const double e = fabs(half_to_double(got[i]) - ref[i]);
            if (e > 2e-3 + 1e-2 * fabs(ref[i])) { fprintf(stderr, "step %d: attention differs at %d\n", step, i); return 1; }
            if (e > worst) worst = e;
        }
    }

    /* refcounts add up to the table entries */
    long long held = 0, entries = 0;
    for (int id = 0; id < NB; ++id) {
        int32_t rc = -1;
        CHECK_PKV(pkv_alloc_refcount(alloc, id, &rc));
        held += rc;
    }
    for (int s = 0; s < S; ++s) entries += nblocks[s];
    if (held != entries) { fprintf(stderr, "refcounts %lld, table entries %lld\n", held, entries); return 1; }

    CHECK_CUDA(cudaDeviceSynchronize());
    pkv_beam_search_destroy(search);
    pkv_alloc_destroy(alloc);
    cudaFreeHost(stg0);
    cudaFreeHost(stg1);
    printf("c abi beam ok: %d steps, %d copies, max abs err %.2e\n", STEPS, total_pairs, worst);
    return 0;
}
