// Shared-prefix decode on the 5th-generation tensor cores (head_dim 128).
// Included by decode.cu inside its anonymous namespace: it uses that file's
// Workspace, DecodeParams, PrefixParams and merge_partitions.
//
// Two CTAs of 10 warps per SM take the same work items as prefix_kernel --
// (group, prefix partition, group of 4 heads) -- in a static order (the
// items are all the same size), and for each head run, per 128-token tile,
//
//   S^T = K Q^T    tcgen05.mma kind::f16, M = 128 tokens, N = 16 members,
//                  K = 128 dims; A = the K tile (K-major), B = Q (K-major);
//                  accumulator in TMEM, two buffers so the next tile's
//                  scores overlap this tile's softmax
//   softmax        warps 0-7, one token per TMEM lane (tcgen05.ld); warps
//                  w and w + 4 share the lanes and split the members (0-7,
//                  8-15), so a thread handles 8 scores.  Each
//                  member keeps a reference max, moved only when a tile's
//                  max passes it by more than kTcLazy: the common tile costs
//                  one barrier (did any score pass its reference?) and no
//                  exchange of maxima, and O is rescaled only when a
//                  reference moves.  P = 2^(s - reference), rounded to 16
//                  bits, is transposed across lanes and stored as 16-byte
//                  chunks of the B operand of the next product (two
//                  buffers); its sums are kept per lane until the head ends
//   O^T += V^T P^T tcgen05.mma, M = 128 dims, N = 16 members, K = 128
//                  tokens; A = the V tile read MN-major, B = P (K-major)
//
// Warp 8 loads: K and V tiles of 128 tokens by TMA (cp.async.bulk.tensor,
// boxes of min(bs, 16) rows x 128 bytes, 128-byte swizzle; the lanes look up
// their blocks and issue their boxes together) into a 3-stage ring with a
// full and an empty mbarrier per stage.  Warp 9 issues the MMAs (one
// thread), each product as soon as its operands are ready.  mbarriers hand
// each tile and head between the roles; the next
// head's Q is written as soon as the current head's last S^T has completed.
// Each member's (reference, sum, output) partial goes to the decode kernel's
// workspace slots and the same tickets merge it.
//
// Every wait is bounded: on a timeout the roles stop, the kernel sets
// PKV_DEVERR_TIMEOUT, waits (bounded) for its loads in flight, frees its
// TMEM and returns.

#include "tc_wait.cuh"

constexpr int kTcD = 128;                       // head_dim of this path
constexpr int kTcTile = 128;                    // tokens per K or V tile
constexpr int kTcCtasPerSm = 2;                 // CTAs resident per SM
constexpr int kTcStages = 3;                    // tiles in flight per CTA
constexpr int kTcChunkTiles = 1;                // tiles per softmax chunk
constexpr int kTcHalf = kTcTile * 128;          // bytes of one 64-dim half of a tile (16 KB)
constexpr int kTcTileBytes = 2 * kTcHalf;       // 32 KB
constexpr int kTcQOff = kTcStages * kTcTileBytes;       // Q: 16 rows x 256 B (2 halves of 2 KB)
constexpr int kTcPBytes = kTcChunkTiles * 4096;         // P of one chunk
constexpr int kTcPOff = kTcQOff + 4096;                 // P: two chunk buffers, used in turn
constexpr int kTcBarOff = kTcPOff + 2 * kTcPBytes;
constexpr int kTcSmemBytes = kTcBarOff + 2048 + 1024;   // barriers, TMEM slot, reductions; +1 KB alignment
// The softmax keeps a per-member reference max and moves it only when a
// chunk's max passes it by more than this (log2 units): P stays below 2^8,
// and O in TMEM is rescaled (waiting for the previous P.V) only then.
constexpr float kTcLazy = 8.f;
constexpr int kTcSCols = 16 * kTcChunkTiles;    // TMEM columns of one S buffer
constexpr int kTcOCol = 2 * kTcSCols;           // O after the two S buffers
constexpr int kTcTmemCols = kTcOCol + 16 <= 32 ? 32 : kTcOCol + 16 <= 64 ? 64
                          : kTcOCol + 16 <= 128 ? 128 : kTcOCol + 16 <= 256 ? 256 : 512;
constexpr int kTcSmWarps = 8;                  // softmax warps: two per TMEM lane quarter
constexpr int kTcLoadWarp = kTcSmWarps;         // TMA loads
constexpr int kTcMmaWarp = kTcSmWarps + 1;      // MMA issue
constexpr int kTcThreads = 32 * (kTcSmWarps + 2);

static_assert(kTcCtasPerSm * (kTcSmemBytes + 1024) <= 228 * 1024, "prefix_tc shared memory");
static_assert(16 * kTcStages + 72 + 4 <= 256, "prefix_tc barriers overlap the reductions");
static_assert(kTcChunkTiles == 1, "the softmax below handles one tile per chunk");
static_assert(kTcCtasPerSm * kTcTmemCols <= 512, "prefix_tc TMEM");

// ---- PTX helpers (the mbarrier waits and TMEM fences are in tc_wait.cuh) ---
__device__ __forceinline__ void tc_mbar_expect(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// whether phase `parity` of the barrier has completed (never suspends)
__device__ __forceinline__ bool tc_mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void tc_mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_tma_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
// UMMA shared-memory descriptor: 128-byte swizzle, sm_100 family version 1
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// instruction descriptor of kind::f16: fp32 accumulate, A/B f16 or bf16,
// A K-major (0) or MN-major (1), B K-major, N = 16, M = 128
template <class E>
__device__ __forceinline__ uint32_t tc_idesc(uint32_t a_mn_major) {
    constexpr uint32_t fmt = std::is_same<E, pkv::BF16>::value ? 1u : 0u;
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (a_mn_major << 15) | ((16u >> 3) << 17) |
           ((128u >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t ad, uint64_t bd, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(tmem_d), "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate)
        : "memory");
}
// the mbarrier arrives once every tcgen05.mma issued so far has completed
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tc_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_st8(uint32_t taddr, const float (&v)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
        ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
          "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])),
          "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// generic-proxy writes to shared memory visible to the tensor cores
__device__ __forceinline__ void tc_fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// byte offset of (row, element) in a 128-byte-swizzled K-major tile whose
// rows hold 64 16-bit elements (8-row atoms of 1 KB)
__device__ __forceinline__ uint32_t tc_sw128(int row, int el) {
    return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((((el * 2) >> 4) ^ (row & 7)) << 4) +
                      ((el * 2) & 15));
}


// ---- the kernel -----------------------------------------------------------
// Items are the same size, so each CTA takes items b, b + grid, b + 2*grid,
// ... and every role walks that sequence on its own.  Per item, per head,
// per tile (a chunk is one tile):
//   loader warp 8    the head's K tile 0, then K tile c + 1 and V tile c
//                    for each c, into the ring
//   MMA warp 9       wait q_ready; S^T(0); for each c, whichever is ready
//                    first: S^T(c + 1) (K tile landed), commit
//                    s_ready[(c + 1) & 1]; O^T += V^T P^T(c) (p_ready[c & 1]
//                    and the V tile landed), commit pv; after the head:
//                    commit o_ready
//   softmax warps    wait s_ready[c & 1]: reference check (one barrier), P,
//   0-7              sums, arrive p_ready[c & 1]; on the head's last tile
//                    write the next head's Q, arrive q_ready; after the
//                    head: wait o_ready, write the partials; after the item:
//                    tickets and merges
// An item: one (group, prefix partition, head group); its nh heads run one
// after another.
struct TcItem {
    int hg, part, first, n, nh;
    const int32_t* bt_row;
};

__device__ __forceinline__ TcItem tc_item(const PrefixParams& pp, int it) {
    const DecodeParams& a = pp.d;
    TcItem r;
    r.hg = it % a.HG;
    const int packed = a.ws.pitems[it / a.HG];
    const int gi = packed >> 16;
    r.part = packed & 0xffff;
    r.first = pp.groups[3 * gi];
    r.n = pp.groups[3 * gi + 1];
    r.nh = min(kWarps, a.H - r.hg * kWarps);
    r.bt_row = a.block_tables + (int64_t)r.first * a.MB;
    return r;
}

template <class E, int BS>
__global__ void __launch_bounds__(kTcThreads, kTcCtasPerSm)
prefix_tc_kernel(PrefixParams pp, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmv) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    extern __shared__ unsigned char tc_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(tc_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    unsigned char* smem = tc_raw + pad;
    const uint32_t sb = raw + pad;  // 1024-byte aligned: the swizzle atoms line up
    const DecodeParams& a = pp.d;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // barriers: full and empty per stage, then the hand-offs between roles
    const uint32_t bar_full = sb + kTcBarOff;
    const uint32_t bar_empty = bar_full + 8 * kTcStages;
    const uint32_t bar_q = bar_empty + 8 * kTcStages;  // Q written (each softmax thread)
    const uint32_t bar_s0 = bar_q + 8;                 // S buffer 0 ready (commit)
    const uint32_t bar_s1 = bar_s0 + 8;                // S buffer 1 ready (commit)
    // P of chunk k written (and O rescaled), one barrier per P buffer (each
    // softmax thread arrives): the softmax may finish P(k) and P(k + 1) before the MMA
    // warp first looks for P(k), but never P(k + 2), which needs S(k + 2),
    // issued only after P(k) has been taken -- so each barrier is at most
    // one phase ahead of its waiter
    const uint32_t bar_p0 = bar_s1 + 8;
    const uint32_t bar_pv = bar_p0 + 8;                // a chunk's P.V done (commit)
    const uint32_t bar_o = bar_pv + 8;                 // O complete (commit)
    const uint32_t bar_end = bar_o + 8;                // final commit
    const uint32_t bar_p1 = bar_end + 8;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kTcBarOff + 16 * kTcStages + 72);
    float* red = reinterpret_cast<float*>(smem + kTcBarOff + 256);  // [8 warps][8] maxima
    float* reds = red + 64;                                           // [8 warps][8] sums
    float* mrun = reds + 64;  // per member: the reference max of P (log2 units)
    float* lrun = mrun + 16;  // per member: running sum of P
    float* corr = lrun + 16;
    float* mnew = corr + 16;
    // [0] abort, [1] last-partition bits, [2] tiles consumed, [4] tiles issued
    volatile int* sh = reinterpret_cast<volatile int*>(mnew + 16);
    int* s_np = const_cast<int*>(sh) + 32;  // [16] partition counts of the unit's members

    const int PT = *a.ws.pt;
    const int nt = (PT + kTcTile - 1) / kTcTile;
    const int total = *a.ws.n_pitems * a.HG;  // items
    constexpr int R = BS < 16 ? BS : 16;  // rows per TMA box (one block holds them)

    // zero the ring and P once: rows a tile does not load stay finite
    for (int i = tid; i < kTcBarOff / 16; i += kTcThreads)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            tc_mbar_init(bar_full + 8 * s, 1);
            tc_mbar_init(bar_empty + 8 * s, 1);
        }
        tc_mbar_init(bar_q, 32 * kTcSmWarps);
        tc_mbar_init(bar_s0, 1);
        tc_mbar_init(bar_s1, 1);
        tc_mbar_init(bar_p0, 32 * kTcSmWarps);
        tc_mbar_init(bar_p1, 32 * kTcSmWarps);
        tc_mbar_init(bar_pv, 1);
        tc_mbar_init(bar_o, 1);
        tc_mbar_init(bar_end, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        sh[0] = 0;
        sh[2] = 0;
        sh[4] = 0;
        sh[5] = 0;
    }
    tc_fence_async_smem();
    __syncthreads();
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(sb + kTcBarOff + 16 * kTcStages + 72), "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    auto fail = [&]() { sh[0] = 1; };

    if (warp == kTcLoadWarp) {
        // ---------------- loader: lanes look up blocks and issue boxes together
        constexpr int kRowBoxes = kTcTile / R;  // boxes per 64-dim half
        long long g = 0;
        bool stop = false;  // the same in every lane (decided by lane 0)
        const int nch = (nt + kTcChunkTiles - 1) / kTcChunkTiles;
        // the tiles of one chunk (kind 0: K, 1: V) of head h, each into the
        // next stage of the ring
        auto emit = [&](const TcItem& item, int h, int kind, int ch) {
            const CUtensorMap* map = kind == 0 ? &tmk : &tmv;
            const int t1 = min((ch + 1) * kTcChunkTiles, nt);
            for (int t = ch * kTcChunkTiles; t < t1 && !stop; ++t) {
                const int stage = (int)(g % kTcStages);
                int ok = 1;
                if (lane == 0) {
                    if (g >= kTcStages)
                        ok = tc_mbar_wait(bar_empty + 8 * stage,
                                          (uint32_t)(((g / kTcStages) - 1) & 1), sh) ? 1 : 0;
                    if (sh[0]) ok = 0;
                }
                ok = __shfl_sync(kFull, ok, 0);
                if (!ok) {
                    if (lane == 0) fail();
                    stop = true;
                    break;
                }
                // lane l: box (half l / kRowBoxes, rows R*(l % kRowBoxes) ..)
                const int half = lane / kRowBoxes, rb = lane % kRowBoxes;
                int row = -1;
                if (half < 2 && rb * R < PT - t * kTcTile) {
                    const int tok = item.part * PT + t * kTcTile + rb * R;
                    const int p = __ldg(item.bt_row + tok / BS);
                    if ((unsigned)p < (unsigned)a.NB) row = p * BS + tok % BS;
                    else pkv::report(a.err, PKV_DEVERR_BLOCK_ID);
                }
                const unsigned boxes = __popc(__ballot_sync(kFull, row >= 0));
                const uint32_t full = bar_full + 8 * stage;
                if (lane == 0) tc_mbar_expect(full, boxes * (uint32_t)(R * 128));
                __syncwarp();
                if (row >= 0)
                    tc_tma_3d(sb + (uint32_t)stage * kTcTileBytes + half * kTcHalf + rb * R * 128,
                              map, half * 64, h, row, full);
                ++g;
            }
        };
        // per head: K of chunk 0, then for each chunk c: K of chunk c+1, V of
        // chunk c -- the order in which the MMA warp takes them
        for (int it = blockIdx.x; it < total && !stop; it += gridDim.x) {
            const TcItem item = tc_item(pp, it);
            for (int j = 0; j < item.nh && !stop; ++j) {
                const int h = item.hg * kWarps + j;
                emit(item, h, 0, 0);
                for (int c = 0; c < nch && !stop; ++c) {
                    if (c + 1 < nch) emit(item, h, 0, c + 1);
                    emit(item, h, 1, c);
                }
            }
        }
        if (lane == 0) sh[4] = (int)g;  // tiles issued
    }
    else if (warp == kTcMmaWarp) {
        // ---------------- MMAs: one thread issues, the tensor cores run async
        if (lane == 0) {
            const uint32_t idesc_k = tc_idesc<E>(0u), idesc_v = tc_idesc<E>(1u);
            const int nch = (nt + kTcChunkTiles - 1) / kTcChunkTiles;
            long long g = 0;
            uint32_t heads = 0, chunks = 0;  // chunks: global index of the head's chunk 0
            bool ok = true;
            // the heads of the CTA's items, in order
            int nheads = 0;
            for (int it = blockIdx.x; it < total; it += gridDim.x) nheads += tc_item(pp, it).nh;
            // one tile: S^T of chunk k from the K tile at load index gk
            auto s_issue = [&](long long gk, uint32_t k) {
                const int stage = (int)(gk % kTcStages);
                const uint32_t tile = sb + (uint32_t)stage * kTcTileBytes;
                const uint32_t cols = tmem + (k & 1u) * kTcSCols;
#pragma unroll
                for (int kk = 0; kk < kTcD / 16; ++kk) {
                    const uint64_t ad = tc_desc(tile + (kk >> 2) * kTcHalf + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = tc_desc(sb + kTcQOff + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024);
                    tc_mma(cols, ad, bd, idesc_k, kk > 0 ? 1u : 0u);
                }
                tc_commit(bar_empty + 8 * stage);
                tc_commit((k & 1u) ? bar_s1 : bar_s0);
            };
            // O^T += V^T P^T of chunk c (global chunk k) from the V tile at gv
            auto pv_issue = [&](long long gv, int c, uint32_t k) {
                const int stage = (int)(gv % kTcStages);
                const uint32_t tile = sb + (uint32_t)stage * kTcTileBytes;
                const uint32_t pbuf = sb + kTcPOff + (k & 1u) * kTcPBytes;
#pragma unroll
                for (int kk = 0; kk < kTcTile / 16; ++kk) {
                    const uint64_t ad = tc_desc(tile + kk * 2048, kTcHalf, 1024);
                    const uint64_t bd = tc_desc(pbuf + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024);
                    tc_mma(tmem + kTcOCol, ad, bd, idesc_v, (c > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar_empty + 8 * stage);
                tc_commit(bar_pv);
            };
            auto full_ok = [&](long long gi) {
                return tc_mbar_test(bar_full + 8 * (int)(gi % kTcStages), (uint32_t)((gi / kTcStages) & 1));
            };
            for (int u = 0; ok && u < nheads; ++u, ++heads) {
                ok = tc_mbar_wait(bar_q, heads & 1u, sh);  // this head's Q
                if (ok) tc_fence_after();
                // the head's first scores
                ok = ok && tc_mbar_wait(bar_full + 8 * (int)(g % kTcStages),
                                        (uint32_t)((g / kTcStages) & 1), sh);
                if (ok) {
                    tc_fence_after();
                    s_issue(g, chunks);
                    ++g;
                }
                for (int c = 0; ok && c < nch; ++c) {
                    // the next chunk's scores (once its K tile has landed) and
                    // this chunk's P.V (once P is written and its V tile has
                    // landed), whichever can go first: neither waits behind
                    // the other's data
                    const bool next = c + 1 < nch;
                    const long long gk = g, gv = next ? g + 1 : g;  // the loader's order
                    const uint32_t pbar = ((chunks + c) & 1u) ? bar_p1 : bar_p0;
                    const uint32_t ppar = ((chunks + c) >> 1) & 1u;
                    bool s_done = !next, pv_done = false;
                    for (long long polls = 0; !(s_done && pv_done); ++polls) {
                        if (polls >= kTcWaitLimit || ((polls & 255) == 255 && sh[0])) {
                            ok = false;
                            break;
                        }
                        if (!s_done && full_ok(gk)) {
                            tc_fence_after();
                            s_issue(gk, chunks + c + 1);
                            s_done = true;
                        }
                        if (!pv_done && tc_mbar_test(pbar, ppar) && full_ok(gv)) {
                            tc_fence_after();
                            pv_issue(gv, c, chunks + c);
                            pv_done = true;
                        }
                    }
                    g += next ? 2 : 1;
                }
                chunks += nch;
                if (!ok) break;
                // the next head's first P.V waits for its first P, which
                // the softmax hands over only after reading this O out
                tc_commit(bar_o);
            }
            if (!ok) fail();
            tc_commit(bar_end);  // every MMA issued so far
            tc_mbar_wait(bar_end, 0u, sh + 5);
            sh[2] = (int)g;  // tiles consumed
        }
    }
    else {
        // ---------------- softmax and epilogue: warps 0 .. kTcSmWarps - 1.
        // Warp w may reach TMEM lanes 32 (w % 4) .. + 31 only, so warps w and
        // w + 4 read the same lanes -- the tokens 32 (w % 4) + lane of a
        // tile, then the dims of O -- and split the members: warps 0-3 take
        // members 0-7 (columns 0-7 of S and O), warps 4-7 members 8-15.
        constexpr int kSm = 32 * kTcSmWarps;  // threads of this role
        const int quarter = warp & 3, mb = 8 * (warp >> 2);
        const int row = 32 * quarter + lane;  // a token of a tile, then a dim of O
        const uint32_t tlane = tmem + ((uint32_t)(32 * quarter) << 16);
        auto csync = [] { asm volatile("bar.sync 1, %0;" ::"n"(kSm) : "memory"); };
        // barriers over these warps that also AND a flag / count the set flags
        auto csync_and = [](bool v) -> bool {
            uint32_t r;
            asm volatile(
                "{.reg .pred p, q;\n\t"
                "setp.ne.u32 p, %1, 0;\n\t"
                "bar.red.and.pred q, 1, %2, p;\n\t"
                "selp.u32 %0, 1, 0, q;}"
                : "=r"(r)
                : "r"(v ? 1u : 0u), "n"(kSm)
                : "memory");
            return r != 0;
        };
        auto csync_count = [](bool v) -> uint32_t {
            uint32_t r;
            asm volatile(
                "{.reg .pred p;\n\t"
                "setp.ne.u32 p, %1, 0;\n\t"
                "bar.red.popc.u32 %0, 1, %2, p;}"
                : "=r"(r)
                : "r"(v ? 1u : 0u), "n"(kSm)
                : "memory");
            return r;
        };
        // The 8 members' values of one token per lane are transposed in three
        // exchange rounds (lane bits 0, 1, 2): afterwards a lane holds member
        // mb + mt for the eight tokens (lane & 24) + 0..7 of its quarter.
        const int mt = ((lane & 1) << 2) | (((lane >> 1) & 1) << 1) | ((lane >> 2) & 1);
        // this thread's 16 bytes of the members' queries of head h (rows >= n
        // zero): member tid >> 4, dims (tid & 15) * 8 ..
        const int qm = tid >> 4, qd = (tid & 15) * 8;
        auto load_q = [&](const TcItem& item, int h, uint4& v) {
            v = make_uint4(0u, 0u, 0u, 0u);
            if (qm < item.n)
                v = __ldg(reinterpret_cast<const uint4*>(
                    static_cast<const uint16_t*>(a.q) + ((int64_t)(item.first + qm) * a.H + h) * kTcD + qd));
        };
        // ... into Q, the B operand of S^T = K Q^T, then handed to the MMA warp
        auto write_q = [&](const uint4& v) {
            const int c = (qd & 63) >> 3;
            unsigned char* qb = smem + kTcQOff + (qd >> 6) * 2048 + (qm >> 3) * 1024 + (qm & 7) * 128;
            *reinterpret_cast<uint4*>(qb + ((c ^ (qm & 7)) << 4)) = v;
            tc_fence_async_smem();
            tc_mbar_arrive(bar_q);
        };
        // mref[k] without a dynamic register index
        auto pick = [](const float (&v)[8], int k) {
            float x = v[0];
#pragma unroll
            for (int i = 1; i < 8; ++i) x = (i == k) ? v[i] : x;
            return x;
        };
        uint32_t heads = 0, chunks = 0;
        bool ok = true;
        // the CTA's heads in order; the next head's Q is written as soon as
        // the last S^T of the current one has completed
        int it = blockIdx.x, j = 0;
        TcItem item;
        if (it < total) {
            item = tc_item(pp, it);
            uint4 v;
            load_q(item, item.hg * kWarps, v);
            write_q(v);
            if (tid < 16) s_np[tid] = tid < item.n ? a.ws.nparts[item.first + tid] : 0;
        }
        while (ok && it < total) {
            const int h = item.hg * kWarps + j;
            int it2 = it, j2 = j + 1;
            if (j2 >= item.nh) {
                it2 += gridDim.x;
                j2 = 0;
            }
            const bool more = it2 < total;
            const TcItem item2 = (j2 == 0 && more) ? tc_item(pp, it2) : item;
            // the next unit's queries are fetched now and written into Q
            // once this unit's last S^T has completed
            uint4 nq;
            load_q(item2, item2.hg * kWarps + j2, nq);
            // per member mb + k: the reference max of P (the same in every
            // thread), and this lane's share of the running sum of P for
            // member mb + mt (relative to the reference)
            float mref[8], lacc = 0.f;
#pragma unroll
            for (int m = 0; m < 8; ++m) mref[m] = -INFINITY;
            // whether this thread's token of tile c0 is inside the partition
            // with its block id in range, read one tile ahead
            auto token_ok = [&](int c0) -> bool {
                const int rel = c0 * kTcTile + row;
                return rel < PT && (unsigned)__ldg(item.bt_row + (item.part * PT + rel) / BS) < (unsigned)a.NB;
            };
            bool valid_next = nt > 0 && token_ok(0);
            for (int c0 = 0; c0 < nt; ++c0, ++chunks) {
                const uint32_t kb = chunks & 1u;  // this chunk's S and P buffers
                const bool valid = valid_next;
                if (c0 + 1 < nt) valid_next = token_ok(c0 + 1);
                const bool got = tc_mbar_wait(kb ? bar_s1 : bar_s0, (chunks >> 1) & 1u, sh);
                tc_fence_after();
                // every S^T of this head has completed: Q is free
                if (c0 == nt - 1 && got && more) write_q(nq);
                float sc[8];
                {
                    float r[8];
                    tc_ld8(tlane + kb * kTcSCols + mb, r);
#pragma unroll
                    for (int m = 0; m < 8; ++m) sc[m] = valid ? r[m] * a.qscale : -INFINITY;
                }
                // fast path: every score within kTcLazy of its member's
                // reference -- one barrier, no exchange of maxima
                bool over = !got;
#pragma unroll
                for (int m = 0; m < 8; ++m) over = over || sc[m] > mref[m] + kTcLazy;
                if (csync_count(over) != 0) {
                    ok = csync_and(got);
                    if (!ok) break;
                    // the chunk's max per member: a reduce-scatter over the
                    // lanes, then over the four warps that share the members
                    {
                        float r4[4], r2[2];
                        const bool u1 = lane & 1, u2 = lane & 2, u4 = lane & 4;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            r4[q] = fmaxf(u1 ? sc[4 + q] : sc[q],
                                          __shfl_xor_sync(kFull, u1 ? sc[q] : sc[4 + q], 1));
#pragma unroll
                        for (int q = 0; q < 2; ++q)
                            r2[q] = fmaxf(u2 ? r4[2 + q] : r4[q],
                                          __shfl_xor_sync(kFull, u2 ? r4[q] : r4[2 + q], 2));
                        float r1 = fmaxf(u4 ? r2[1] : r2[0], __shfl_xor_sync(kFull, u4 ? r2[0] : r2[1], 4));
                        r1 = fmaxf(r1, __shfl_xor_sync(kFull, r1, 8));
                        r1 = fmaxf(r1, __shfl_xor_sync(kFull, r1, 16));
                        if (lane < 8) red[warp * 8 + mt] = r1;
                    }
                    csync();
                    // a member moves its reference to the chunk's max when
                    // that passes the reference by more than kTcLazy (lane k
                    // of warps 0 and 4: member mb + k)
                    if (quarter == 0 && lane < 8) {
                        const int w0 = warp;  // 0 or 4: the four warps w0 .. w0 + 3
                        const float cm = fmaxf(fmaxf(red[w0 * 8 + lane], red[(w0 + 1) * 8 + lane]),
                                               fmaxf(red[(w0 + 2) * 8 + lane], red[(w0 + 3) * 8 + lane]));
                        const float mo = pick(mref, lane);
                        const bool move = cm > mo + kTcLazy;
                        mnew[mb + lane] = move ? cm : mo;
                        corr[mb + lane] = move ? exp2f(mo - cm) : 1.f;
                    }
                    csync();
#pragma unroll
                    for (int m = 0; m < 8; ++m) mref[m] = mnew[mb + m];
                    lacc *= corr[mb + mt];
                    // what O holds so far is rescaled once the previous
                    // chunk's P.V has landed in it
                    if (c0 > 0) {
                        ok = csync_and(tc_mbar_wait(bar_pv, (chunks - 1) & 1u, sh));
                        if (!ok) break;
                        tc_fence_after();
                        float o[8];
                        tc_ld8(tlane + kTcOCol + mb, o);
#pragma unroll
                        for (int m = 0; m < 8; ++m) o[m] *= corr[mb + m];
                        tc_st8(tlane + kTcOCol + mb, o);
                    }
                }
                // P = 2^(s - reference), 16 bits, into this chunk's P buffer
                // (B operand, K-major, 128-byte swizzle): the values are
                // transposed across lanes so that each lane writes one
                // 16-byte chunk of 8 tokens of member mb + mt and sums them
                {
                    float p[8];
#pragma unroll
                    for (int m = 0; m < 8; ++m) p[m] = valid ? exp2f(sc[m] - mref[m]) : 0.f;
                    float a4[4][2], a2[2][4], a1[8];
                    const bool u1 = lane & 1, u2 = lane & 2, u4 = lane & 4;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float keep = u1 ? p[4 + q] : p[q];
                        const float recv = __shfl_xor_sync(kFull, u1 ? p[q] : p[4 + q], 1);
                        a4[q][0] = u1 ? recv : keep;
                        a4[q][1] = u1 ? keep : recv;
                    }
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            const float keep = u2 ? a4[2 + q][t] : a4[q][t];
                            const float recv = __shfl_xor_sync(kFull, u2 ? a4[q][t] : a4[2 + q][t], 2);
                            a2[q][t] = u2 ? recv : keep;
                            a2[q][2 + t] = u2 ? keep : recv;
                        }
                    }
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const float keep = u4 ? a2[1][t] : a2[0][t];
                        const float recv = __shfl_xor_sync(kFull, u4 ? a2[0][t] : a2[1][t], 4);
                        a1[t] = u4 ? recv : keep;
                        a1[4 + t] = u4 ? keep : recv;
                    }
                    const int tb = 32 * quarter + (lane & 24);  // the first of the lane's 8 tokens
                    unsigned char* pt = smem + kTcPOff + kb * kTcPBytes + (tb >> 6) * 2048;
                    const int ch = (tb & 63) >> 3;               // its 16-byte chunk of a 128-byte row
                    const int m = mb + mt;
                    uint4 v;
                    v.x = E::from_float2(a1[0], a1[1]);
                    v.y = E::from_float2(a1[2], a1[3]);
                    v.z = E::from_float2(a1[4], a1[5]);
                    v.w = E::from_float2(a1[6], a1[7]);
                    *reinterpret_cast<uint4*>(pt + (m >> 3) * 1024 + (m & 7) * 128 + ((ch ^ (m & 7)) << 4)) = v;
                    lacc += ((a1[0] + a1[1]) + (a1[2] + a1[3])) + ((a1[4] + a1[5]) + (a1[6] + a1[7]));
                }
                // each thread hands its part of P to the MMA warp
                tc_fence_async_smem();
                tc_fence_before();
                tc_mbar_arrive(kb ? bar_p1 : bar_p0);
            }
            if (!ok) break;
            // the head's sums per member: over the lanes that share the
            // member (lane bits 3, 4), then over the four warps
            lacc += __shfl_xor_sync(kFull, lacc, 8);
            lacc += __shfl_xor_sync(kFull, lacc, 16);
            if (lane < 8) reds[warp * 8 + mt] = lacc;
            ok = csync_and(tc_mbar_wait(bar_o, heads & 1u, sh));
            if (!ok) break;
            tc_fence_after();
            if (quarter == 0 && lane < 8) {
                const int w0 = warp;
                lrun[mb + lane] = (reds[w0 * 8 + lane] + reds[(w0 + 1) * 8 + lane]) +
                                  (reds[(w0 + 2) * 8 + lane] + reds[(w0 + 3) * 8 + lane]);
                mrun[mb + lane] = pick(mref, lane);
            }
            csync();
            {
                float o[8];
                tc_ld8(tlane + kTcOCol + mb, o);
                const int d = row;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int m = mb + k;
                    if (m < item.n) {
                        const int s = item.first + m;
                        const int np = s_np[m];
                        if (np == 1) {
                            const float l = lrun[m];
                            const float inv = l > 0.f ? 1.f / l : 0.f;
                            static_cast<uint16_t*>(a.out)[((int64_t)s * a.H + h) * kTcD + d] =
                                (uint16_t)(E::from_float2(o[k] * inv, 0.f) & 0xffffu);
                        } else {
                            const int64_t idx = ((int64_t)s * a.H + h) * a.max_parts + item.part;
                            a.ws.acc[idx * kTcD + d] = o[k];
                            if (d == 0) {
                                a.ws.m[idx] = mrun[m];
                                a.ws.l[idx] = lrun[m];
                            }
                        }
                    }
                }
            }
            if (!ok) break;
            ++heads;
            if (j2 == 0) {
                // the item is done: tickets of the members that have more
                // than one partition
                __threadfence();
                csync();
                if (tid < 16) {
                    unsigned bit = 0;
                    if (tid < item.n) {
                        const int s = item.first + tid;
                        const int np = s_np[tid];
                        if (np > 1) {
                            const unsigned done = atomicAdd(&a.ws.tickets[s * a.HG + item.hg], 1u);
                            bit = (done == (unsigned)(np - 1)) ? (1u << tid) : 0u;
                        }
                    }
#pragma unroll
                    for (int o = 8; o >= 1; o >>= 1) bit |= __shfl_xor_sync(0xffffu, bit, o);
                    if (tid == 0) sh[1] = (int)bit;
                }
                csync();
                unsigned last = (unsigned)sh[1];
                if (last && warp < kWarps) {
                    __threadfence();
                    const int hm = item.hg * kWarps + warp;
                    while (last) {
                        const int m = __ffs(last) - 1;
                        last &= last - 1;
                        if (hm < a.H) merge_partitions<E, kTcD>(a, item.first + m, hm, s_np[m], lane);
                    }
                }
                csync();  // sh[1] and s_np read by all before the next item writes them
                if (more && tid < 16) s_np[tid] = tid < item2.n ? a.ws.nparts[item2.first + tid] : 0;
            }
            it = it2;
            j = j2;
            item = item2;
        }
        if (!ok) fail();
    }

    // every role is done: loads still in flight (only after a timeout) land,
    // then TMEM is freed
    __syncthreads();
    if (warp == kTcLoadWarp && lane == 0) {
        for (long long k = sh[2]; k < sh[4]; ++k)
            tc_mbar_wait(bar_full + 8 * (int)(k % kTcStages), (uint32_t)((k / kTcStages) & 1), sh + 5);
        if (sh[0]) pkv::report(a.err, PKV_DEVERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kTcMmaWarp) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols)
                     : "memory");
    }
}
