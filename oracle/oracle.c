/*
 * Oracle for the paged decode-attention path -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of what the path computes,
 * in double precision.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header or constant with
 * the CUDA library.
 *
 * Sources (web pages on PagedAttention; section names as printed there):
 *  [P1] "3.3 页面级显存管理"                 (page-level GPU memory management)
 *  [P2] "vLLM三大核心技术分页内存与共享解码"   (vLLM core techniques)
 *  [P3] "3.1 PagedAttention的核心原理"       (PagedAttention core principles)
 *  [P4] notes on "vLLM: Easy, Fast, and Cheap LLM Serving with PagedAttention"
 *
 * Cache layout: k_cache and v_cache are separate arrays of fixed-size
 * blocks ([P3] 3.1.2, "页面结构设计": a page holds the Key and the Value
 * vectors of `page_size` tokens), each [num_blocks][block_size][H][D]; the
 * element of token offset `o` in physical block `p`, head `h`, dim `d` is at
 * p*block_size*kv_dim + o*kv_dim + h*D + d with kv_dim = H*D ([P3] 3.1.3,
 * "逻辑地址到物理地址的转换", step 4).
 *
 * `row_of_block` (may be NULL = identity) lets a caller store only the
 * blocks it uses: physical block p lives in row row_of_block[p] of the
 * arrays passed in.  It changes where the oracle reads, never what it
 * computes.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* IEEE 754 binary16 -> double, from the format's definition: 1 sign bit,
 * 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 -> double: a bfloat16 is the upper half of a binary32. */
double oracle_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

static double to_double(uint16_t v, int is_bf16) {
    return is_bf16 ? oracle_bf16_to_double(v) : oracle_f16_to_double(v);
}

static int64_t row_of(const int32_t* row_of_block, int64_t phys) {
    return row_of_block ? (int64_t)row_of_block[phys] : phys;
}

/* Address translation ([P3] 3.1.3 steps 1-3, [P4] "疑问" 1):
 *   logical = pos / block_size, offset = pos % block_size,
 *   physical = block_table[seq][logical]; the slot is the token's row in the
 * cache viewed as [num_blocks*block_size][kv_dim]: physical*block_size + offset.
 * A negative position yields slot -1 (nothing to write). */
void oracle_slot_mapping(int64_t* slot, const int32_t* block_tables, int MB,
                         const int32_t* seq_idx, const int32_t* pos, int T, int block_size) {
    for (int t = 0; t < T; ++t) {
        if (pos[t] < 0) { slot[t] = -1; continue; }
        int64_t logical = pos[t] / block_size;
        int64_t offset = pos[t] % block_size;
        int64_t physical = block_tables[(int64_t)seq_idx[t] * MB + logical];
        /* no block mapped at that logical block: no slot to write */
        slot[t] = physical < 0 ? -1 : physical * block_size + offset;
    }
}

/* Write each new token's K and V (H*D values) into its slot; slot < 0 means
 * "no write".  Tokens are written in order. */
void oracle_reshape_and_cache(uint16_t* k_cache, uint16_t* v_cache,
                              const uint16_t* key, const uint16_t* value,
                              const int64_t* slot, int T, int H, int D, int block_size,
                              const int32_t* row_of_block) {
    int64_t kv_dim = (int64_t)H * D;
    for (int t = 0; t < T; ++t) {
        if (slot[t] < 0) continue;
        int64_t phys = slot[t] / block_size, off = slot[t] % block_size;
        int64_t dst = (row_of(row_of_block, phys) * block_size + off) * kv_dim;
        memcpy(k_cache + dst, key + (int64_t)t * kv_dim, (size_t)kv_dim * 2);
        memcpy(v_cache + dst, value + (int64_t)t * kv_dim, (size_t)kv_dim * 2);
    }
}

/* Copy-on-write block copies ([P2] "Copy-on-Write共享解码的显存优化原理";
 * [P3] 3.1.5 step 3): for each (src, dst) pair, in order, the whole K block
 * and the whole V block of src are copied to dst. */
void oracle_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, const int64_t* pairs, int P,
                        int H, int D, int block_size, const int32_t* row_of_block) {
    int64_t block_elems = (int64_t)block_size * H * D;
    for (int i = 0; i < P; ++i) {
        int64_t src = row_of(row_of_block, pairs[2 * i]);
        int64_t dst = row_of(row_of_block, pairs[2 * i + 1]);
        memcpy(k_cache + dst * block_elems, k_cache + src * block_elems, (size_t)block_elems * 2);
        memcpy(v_cache + dst * block_elems, v_cache + src * block_elems, (size_t)block_elems * 2);
    }
}

/* Swap copies between two block pools ([P1] 3.3.3, CPU swap: a sequence's
 * blocks are copied page by page to CPU-side blocks, and back later): for
 * each (src, dst) pair, in order, K block src of the source pool is copied to
 * K block dst of the destination pool, and V likewise. */
void oracle_swap_blocks(uint16_t* dst_k, uint16_t* dst_v, const uint16_t* src_k,
                        const uint16_t* src_v, const int64_t* pairs, int P, int H, int D,
                        int block_size) {
    int64_t block_elems = (int64_t)block_size * H * D;
    for (int i = 0; i < P; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        memcpy(dst_k + dst * block_elems, src_k + src * block_elems, (size_t)block_elems * 2);
        memcpy(dst_v + dst * block_elems, src_v + src * block_elems, (size_t)block_elems * 2);
    }
}

/* ---- single-query decode attention, by definition ---------------------- */

typedef struct {
    double* out;
    const uint16_t *q, *k_cache, *v_cache;
    const int32_t *block_tables, *context_lens, *row_of_block, *items;
    int n_items, S, H, D, block_size, MB, is_bf16, nthreads;
    double scale;
} decode_args;

/* o[s,h,:] = sum_j softmax_j(scale * q.K_j) V_j over the sequence's
 * context_lens[s] tokens, each K_j / V_j found through the block table.
 * The softmax subtracts the maximum logit before exponentiating (the same
 * function, kept finite).  An empty context gives o = 0. */
static void decode_one(const decode_args* a, int s, int h) {
    int n = a->context_lens[s];
    int D = a->D;
    int64_t kv_dim = (int64_t)a->H * D;
    double* o = a->out + ((int64_t)s * a->H + h) * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (n <= 0) return;
    const uint16_t* qv = a->q + ((int64_t)s * a->H + h) * D;
    double* qd = (double*)malloc(sizeof(double) * D);
    double* z = (double*)malloc(sizeof(double) * n);
    for (int d = 0; d < D; ++d) qd[d] = to_double(qv[d], a->is_bf16);
    for (int j = 0; j < n; ++j) {
        int64_t logical = j / a->block_size, offset = j % a->block_size;
        int64_t phys = a->block_tables[(int64_t)s * a->MB + logical];
        const uint16_t* kj = a->k_cache
            + (row_of(a->row_of_block, phys) * a->block_size + offset) * kv_dim + (int64_t)h * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[d] * to_double(kj[d], a->is_bf16);
        z[j] = a->scale * dot;
    }
    double m = z[0];
    for (int j = 1; j < n; ++j) if (z[j] > m) m = z[j];
    double denom = 0.0;
    for (int j = 0; j < n; ++j) {
        double w = exp(z[j] - m);
        int64_t logical = j / a->block_size, offset = j % a->block_size;
        int64_t phys = a->block_tables[(int64_t)s * a->MB + logical];
        const uint16_t* vj = a->v_cache
            + (row_of(a->row_of_block, phys) * a->block_size + offset) * kv_dim + (int64_t)h * D;
        for (int d = 0; d < D; ++d) o[d] += w * to_double(vj[d], a->is_bf16);
        denom += w;
    }
    for (int d = 0; d < D; ++d) o[d] /= denom;
    free(z);
    free(qd);
}

typedef struct { const decode_args* a; int tid; } worker_arg;

static void* decode_worker(void* p) {
    const worker_arg* w = (const worker_arg*)p;
    const decode_args* a = w->a;
    int total = a->items ? a->n_items : a->S * a->H;
    for (int i = w->tid; i < total; i += a->nthreads) {
        int s, h;
        if (a->items) { s = a->items[2 * i]; h = a->items[2 * i + 1]; }
        else { s = i / a->H; h = i % a->H; }
        decode_one(a, s, h);
    }
    return NULL;
}

/* out: [S][H][D] doubles.  items: optional list of n_items (seq, head)
 * pairs to compute (NULL = all); the others are left untouched.
 * nthreads >= 1 splits the (seq, head) items across threads; each item is
 * computed by one thread in the same order, so the result does not depend
 * on nthreads.  Returns 0 on success. */
int oracle_decode(double* out, const uint16_t* q, const uint16_t* k_cache,
                  const uint16_t* v_cache, const int32_t* block_tables,
                  const int32_t* context_lens, int S, int H, int D, int block_size, int MB,
                  double scale, int is_bf16, const int32_t* row_of_block,
                  const int32_t* items, int n_items, int nthreads) {
    decode_args a = {out, q, k_cache, v_cache, block_tables, context_lens, row_of_block,
                     items, n_items, S, H, D, block_size, MB, is_bf16,
                     nthreads < 1 ? 1 : nthreads, scale};
    if (a.nthreads == 1) {
        worker_arg w = {&a, 0};
        decode_worker(&w);
        return 0;
    }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * a.nthreads);
    worker_arg* wa = (worker_arg*)malloc(sizeof(worker_arg) * a.nthreads);
    for (int t = 0; t < a.nthreads; ++t) {
        wa[t].a = &a;
        wa[t].tid = t;
        pthread_create(&th[t], NULL, decode_worker, &wa[t]);
    }
    for (int t = 0; t < a.nthreads; ++t) pthread_join(th[t], NULL);
    free(wa);
    free(th);
    return 0;
}
