/*
 * A plain C11 caller of libpagedkv: one decode step on the GPU through the
 * C ABI only (no C++, no Python), checked against the C oracle.
 *
 *   allocator -> slot mapping -> reshape_and_cache -> decode (workspace and
 *   no-allocation entry points), for 3 sequences x 4 heads x 64 dims, fp16,
 *   block size 16, on random non-contiguous blocks.
 *
 * Exit status 0 when the table/slot results are bit-exact and attention is
 * within 2e-3 + 1e-2 |ref| of the fp64 oracle; non-zero otherwise.
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
void oracle_slot_mapping(int64_t* slot, const int32_t* block_tables, int MB, const int32_t* seq_idx,
                         const int32_t* pos, int T, int block_size);
void oracle_reshape_and_cache(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* key,
                              const uint16_t* value, const int64_t* slot, int T, int H, int D,
                              int block_size, const int32_t* row_of_block);

#define S 3
#define H 4
#define D 64
#define BS 16
#define NB 40
#define MB 8

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

static uint64_t rng_state = 0x9e3779b97f4a7c15ull;
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

int main(void) {
    const size_t block_elems = (size_t)BS * H * D, cache_elems = (size_t)NB * block_elems;
    const int ctx_before[S] = {37, 16, 100};
    int32_t tables[S * MB], nblocks[S] = {0, 0, 0}, ctx[S];
    uint16_t *kc = malloc(cache_elems * 2), *vc = malloc(cache_elems * 2);
    uint16_t q[S * H * D], key[S * H * D], val[S * H * D];
    for (size_t i = 0; i < cache_elems; ++i) { kc[i] = rand_half(); vc[i] = rand_half(); }
    for (int i = 0; i < S * H * D; ++i) { q[i] = rand_half(); key[i] = rand_half(); val[i] = rand_half(); }
    for (int i = 0; i < S * MB; ++i) tables[i] = -1;

    /* host: a shuffled pool, then room for the cached tokens + one new token */
    int32_t order[NB];
    for (int i = 0; i < NB; ++i) order[i] = i;
    for (int i = NB - 1; i > 0; --i) {
        int j = (int)(next_u64() % (uint64_t)(i + 1));
        int32_t t = order[i]; order[i] = order[j]; order[j] = t;
    }
    pkv_allocator* alloc = NULL;
    CHECK_PKV(pkv_alloc_create_with_order(NB, order, NB, &alloc));
    int32_t zeros[S] = {0, 0, 0}, lens[S], ones[S] = {1, 1, 1};
    int64_t pairs[64];
    int32_t npairs = 0, ndone = 0;
    for (int s = 0; s < S; ++s) lens[s] = ctx_before[s];
    CHECK_PKV(pkv_alloc_append_batch(alloc, tables, nblocks, S, MB, zeros, lens, BS, pairs, 32, &npairs, &ndone));
    CHECK_PKV(pkv_alloc_append_batch(alloc, tables, nblocks, S, MB, lens, ones, BS, pairs, 32, &npairs, &ndone));
    for (int s = 0; s < S; ++s) ctx[s] = ctx_before[s] + 1;
    int32_t seq_idx[S] = {0, 1, 2}, pos[S];
    for (int s = 0; s < S; ++s) pos[s] = ctx_before[s];

    /* device buffers */
    void *dk, *dv, *dq, *dkey, *dval, *dout, *dout2, *dws, *dk2, *dv2, *dout3;
    int32_t *dbt, *dctx, *dseq, *dpos;
    int64_t *dslot, *dslot2;
    const size_t ws = pkv_decode_workspace_size(S, H, D, MB * BS, 0);
    CHECK_CUDA(cudaMalloc(&dk, cache_elems * 2));
    CHECK_CUDA(cudaMalloc(&dv, cache_elems * 2));
    CHECK_CUDA(cudaMalloc(&dq, sizeof q));
    CHECK_CUDA(cudaMalloc(&dkey, sizeof key));
    CHECK_CUDA(cudaMalloc(&dval, sizeof val));
    CHECK_CUDA(cudaMalloc(&dout, sizeof q));
    CHECK_CUDA(cudaMalloc(&dout2, sizeof q));
    CHECK_CUDA(cudaMalloc(&dws, ws));
    CHECK_CUDA(cudaMalloc((void**)&dbt, sizeof tables));
    CHECK_CUDA(cudaMalloc((void**)&dctx, sizeof ctx));
    CHECK_CUDA(cudaMalloc((void**)&dseq, sizeof seq_idx));
    CHECK_CUDA(cudaMalloc((void**)&dpos, sizeof pos));
    CHECK_CUDA(cudaMalloc((void**)&dslot, S * sizeof(int64_t)));
    /* a second copy of the caches for the fused step */
    CHECK_CUDA(cudaMalloc(&dk2, cache_elems * 2));
    CHECK_CUDA(cudaMalloc(&dv2, cache_elems * 2));
    CHECK_CUDA(cudaMalloc(&dout3, sizeof q));
    CHECK_CUDA(cudaMalloc((void**)&dslot2, S * sizeof(int64_t)));
    CHECK_CUDA(cudaMemcpy(dk2, kc, cache_elems * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dv2, vc, cache_elems * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dk, kc, cache_elems * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dv, vc, cache_elems * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dq, q, sizeof q, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dkey, key, sizeof key, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dval, val, sizeof val, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dbt, tables, sizeof tables, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dctx, ctx, sizeof ctx, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dseq, seq_idx, sizeof seq_idx, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dpos, pos, sizeof pos, cudaMemcpyHostToDevice));

    /* device: the step */
    const float scale = 0.125f;
    CHECK_PKV(pkv_compute_slot_mapping(dslot, dbt, dseq, dpos, S, S, MB, BS, NULL));
    CHECK_PKV(pkv_reshape_and_cache(dkey, dval, dk, dv, dslot, S, H, D, BS, NB, PKV_F16, NULL));
    CHECK_PKV(pkv_paged_attention_decode(dout, dq, dk, dv, dbt, dctx, S, H, D, BS, NB, MB, 0, scale,
                                         PKV_F16, 0, dws, ws, NULL));
    CHECK_PKV(pkv_paged_attention_decode_noalloc(dout2, dq, dk, dv, dbt, dctx, S, H, D, BS, NB, MB, 0,
                                                 scale, PKV_F16, 0, NULL));
    /* the same step in one call, on the second copy of the caches */
    CHECK_PKV(pkv_decode_step(dout3, dq, dkey, dval, dk2, dv2, dbt, dctx, dseq, dpos, dslot2, NULL, 0,
                              S, S, H, D, BS, NB, MB, 0, scale, PKV_F16, 0, dws, ws, NULL));
    CHECK_PKV(pkv_sync_check(NULL));
    int32_t flags = -1;
    CHECK_PKV(pkv_get_device_errors(&flags));
    if (flags) { fprintf(stderr, "device error word %#x\n", flags); return 1; }

    /* oracle */
    int64_t slot_gpu[S], slot_ref[S];
    CHECK_CUDA(cudaMemcpy(slot_gpu, dslot, sizeof slot_gpu, cudaMemcpyDeviceToHost));
    oracle_slot_mapping(slot_ref, tables, MB, seq_idx, pos, S, BS);
    if (memcmp(slot_gpu, slot_ref, sizeof slot_gpu)) { fprintf(stderr, "slot mapping differs\n"); return 1; }
    oracle_reshape_and_cache(kc, vc, key, val, slot_ref, S, H, D, BS, NULL);
    uint16_t* kg = malloc(cache_elems * 2);
    CHECK_CUDA(cudaMemcpy(kg, dk, cache_elems * 2, cudaMemcpyDeviceToHost));
    if (memcmp(kg, kc, cache_elems * 2)) { fprintf(stderr, "K cache differs\n"); return 1; }
    double ref[S * H * D];
    oracle_decode(ref, q, kc, vc, tables, ctx, S, H, D, BS, MB, scale, 0, NULL, NULL, 0, 1);
    uint16_t got[S * H * D], got2[S * H * D], got3[S * H * D];
    CHECK_CUDA(cudaMemcpy(got, dout, sizeof got, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(got2, dout2, sizeof got2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(got3, dout3, sizeof got3, cudaMemcpyDeviceToHost));
    /* the fused step gives the separate calls' slots, caches and output bit for bit */
    int64_t slot_fused[S];
    CHECK_CUDA(cudaMemcpy(slot_fused, dslot2, sizeof slot_fused, cudaMemcpyDeviceToHost));
    if (memcmp(slot_fused, slot_gpu, sizeof slot_fused)) { fprintf(stderr, "fused slots differ\n"); return 1; }
    uint16_t* kg2 = malloc(cache_elems * 2);
    CHECK_CUDA(cudaMemcpy(kg2, dk2, cache_elems * 2, cudaMemcpyDeviceToHost));
    if (memcmp(kg2, kg, cache_elems * 2)) { fprintf(stderr, "fused K cache differs\n"); return 1; }
    if (memcmp(got3, got, sizeof got)) { fprintf(stderr, "fused output differs\n"); return 1; }
    free(kg2);
    double worst = 0.0;
    for (int i = 0; i < S * H * D; ++i) {
        double e1 = fabs(half_to_double(got[i]) - ref[i]), e2 = fabs(half_to_double(got2[i]) - ref[i]);
        double bound = 2e-3 + 1e-2 * fabs(ref[i]);
        if (e1 > bound || e2 > bound) { fprintf(stderr, "attention differs at %d\n", i); return 1; }
        if (e1 > worst) worst = e1;
    }
    pkv_alloc_destroy(alloc);
    printf("c abi step ok: %d seqs, max abs err %.2e\n", S, worst);
    return 0;
}
