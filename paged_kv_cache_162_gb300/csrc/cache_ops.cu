// Cache maintenance kernels: slot mapping, the KV write of new tokens
// (reshape_and_cache), the copy-on-write block copy (copy_blocks) and the
// GPU <-> host block copy of CPU swap (swap_blocks).
//
// Each kernel is launched with programmatic dependent launch: it waits for
// the kernel before it to finish (griddepcontrol.wait) before reading
// anything, so only launch latency is overlapped, never data.
//
// All three move 16-byte vectors.  In the [NB][bs][H][D] layout a token's K
// (or V) for all heads is one contiguous row of H*D elements and a block is
// one contiguous run of bs*H*D elements, so both copies are plain streams of
// 16-byte loads and stores.
#include "pagedkv.h"
#include "pkv_device.cuh"

namespace {

// Address translation of "3.1 PagedAttention的核心原理" 3.1.3 steps 1-3:
// logical block = pos / bs, offset = pos % bs, physical = table[logical];
// the slot is the token's row physical*bs + offset (pkv::slot_of).
__global__ void slot_mapping_kernel(int64_t* __restrict__ slot, const int32_t* __restrict__ bt,
                                    const int32_t* __restrict__ seq_idx,
                                    const int32_t* __restrict__ pos, int T, int S, int MB, int bs,
                                    int* err) {
    // inputs may come from the kernel before this one; the next kernel may
    // become resident once every CTA is past this point
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    slot[t] = pkv::slot_of(bt, seq_idx[t], pos[t], S, MB, bs, err);
}

// One CTA per new token: copy its H*D-element K row and V row into the
// slot's row of each cache.
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const uint4* __restrict__ key, const uint4* __restrict__ value, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, const int64_t* __restrict__ slot_mapping, int vec_per_row,
    int64_t num_slots, int* err) {
    // inputs may come from the kernel before this one; the next kernel may
    // become resident once every CTA is past this point
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int t = blockIdx.x;
    const int64_t slot = slot_mapping[t];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (threadIdx.x == 0) pkv::report(err, PKV_DEVERR_SLOT);
        return;
    }
    pkv::write_token_rows(key, value, k_cache, v_cache, t, slot, vec_per_row);
}

// Grid (P, splits): CTA (p, y) copies the y-th 1/splits of pair p's K block
// and V block from the source pool to the destination pool (the same pool
// for copy-on-write, the GPU and the host pool for swaps).
__global__ void __launch_bounds__(256) copy_blocks_kernel(
    uint4* __restrict__ dst_k, uint4* __restrict__ dst_v, const uint4* __restrict__ src_k,
    const uint4* __restrict__ src_v, const int64_t* __restrict__ mapping, int64_t vec_per_block,
    int NB_src, int NB_dst, int* err) {
    // inputs may come from the kernel before this one; the next kernel may
    // become resident once every CTA is past this point
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int p = blockIdx.x;
    const int64_t src = mapping[2 * p], dst = mapping[2 * p + 1];
    if (src < 0 || src >= NB_src || dst < 0 || dst >= NB_dst) {
        if (threadIdx.x == 0 && blockIdx.y == 0) pkv::report(err, PKV_DEVERR_BLOCK_ID);
        return;
    }
    const int64_t per = (vec_per_block + gridDim.y - 1) / gridDim.y;
    const int64_t lo = blockIdx.y * per;
    const int64_t hi = lo + per < vec_per_block ? lo + per : vec_per_block;
    const uint4* ks = src_k + src * vec_per_block;
    const uint4* vs = src_v + src * vec_per_block;
    uint4* kd = dst_k + dst * vec_per_block;
    uint4* vd = dst_v + dst * vec_per_block;
    for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) {
        uint4 a = ks[i];
        uint4 b = vs[i];
        kd[i] = a;
        vd[i] = b;
    }
}

int copy_splits(int64_t vec_per_block) {
    // ~16 KB of K and 16 KB of V per CTA
    int64_t splits = (vec_per_block + 1023) / 1024;
    return (int)(splits < 1 ? 1 : (splits > 64 ? 64 : splits));
}

// Device address of a page-locked host buffer (nullptr if the device cannot
// address it).
void* device_view_of_host(void* p) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (attr.type != cudaMemoryTypeHost) return nullptr;
    return attr.devicePointer;
}

bool supported(int D, int bs) {
    return (D == 64 || D == 128) && (bs == 8 || bs == 16 || bs == 32 || bs == 64);
}

template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*fn)(KArgs...), dim3 grid, int threads, cudaStream_t st,
                       Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, static_cast<KArgs>(args)...);
}

}  // namespace

extern "C" {

pkv_status pkv_compute_slot_mapping(int64_t* slot_mapping, const int32_t* block_tables,
                                    const int32_t* seq_idx, const int32_t* pos, int T, int S,
                                    int MB, int bs, void* stream) {
    PKV_TRACE("pkv_compute_slot_mapping");
    pkv::clear_error();
    if (T < 0 || S < 0 || MB < 0 || bs <= 0)
        return pkv::fail(PKV_ERR_INVALID_ARG, "compute_slot_mapping: bad size");
    if (T == 0) return PKV_OK;
    if (!slot_mapping || !seq_idx || !pos || (S > 0 && MB > 0 && !block_tables))
        return pkv::fail(PKV_ERR_INVALID_ARG, "compute_slot_mapping: null pointer");
    const int threads = 256;
    cudaError_t e = launch_pdl(slot_mapping_kernel, dim3((T + threads - 1) / threads), threads,
                               pkv::as_stream(stream), slot_mapping, block_tables, seq_idx, pos, T,
                               S, MB, bs, pkv::device_error_word());
    return e == cudaSuccess ? PKV_OK : pkv::cuda_fail(e, "compute_slot_mapping launch");
}

pkv_status pkv_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                                 const int64_t* slot_mapping, int T, int H, int D, int bs, int NB,
                                 pkv_dtype dtype, void* stream) {
    PKV_TRACE("pkv_reshape_and_cache");
    pkv::clear_error();
    if (T < 0 || H <= 0 || NB < 0 || (dtype != PKV_F16 && dtype != PKV_BF16))
        return pkv::fail(PKV_ERR_INVALID_ARG, "reshape_and_cache: bad size or dtype");
    if (!supported(D, bs)) return pkv::fail(PKV_ERR_UNSUPPORTED, "reshape_and_cache: unsupported head_dim/block_size");
    if (T == 0) return PKV_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping)
        return pkv::fail(PKV_ERR_INVALID_ARG, "reshape_and_cache: null pointer");
    if (!pkv::aligned16(key) || !pkv::aligned16(value) || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
        return pkv::fail(PKV_ERR_INVALID_ARG, "reshape_and_cache: pointers must be 16-byte aligned");
    const int vec_per_row = H * D / 8;
    const int threads = vec_per_row >= 256 ? 256 : ((vec_per_row + 31) / 32) * 32;
    cudaError_t e = launch_pdl(reshape_and_cache_kernel, dim3(T), threads, pkv::as_stream(stream),
                               static_cast<const uint4*>(key), static_cast<const uint4*>(value),
                               static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                               slot_mapping, vec_per_row, (int64_t)NB * bs,
                               pkv::device_error_word());
    return e == cudaSuccess ? PKV_OK : pkv::cuda_fail(e, "reshape_and_cache launch");
}

pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping, int P,
                           int H, int D, int bs, int NB, pkv_dtype dtype, void* stream) {
    PKV_TRACE("pkv_copy_blocks");
    pkv::clear_error();
    if (P < 0 || H <= 0 || NB < 0 || (dtype != PKV_F16 && dtype != PKV_BF16))
        return pkv::fail(PKV_ERR_INVALID_ARG, "copy_blocks: bad size or dtype");
    if (!supported(D, bs)) return pkv::fail(PKV_ERR_UNSUPPORTED, "copy_blocks: unsupported head_dim/block_size");
    if (P == 0) return PKV_OK;
    if (!k_cache || !v_cache || !block_mapping)
        return pkv::fail(PKV_ERR_INVALID_ARG, "copy_blocks: null pointer");
    if (!pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
        return pkv::fail(PKV_ERR_INVALID_ARG, "copy_blocks: pointers must be 16-byte aligned");
    if (P > 65535 * 64) return pkv::fail(PKV_ERR_INVALID_ARG, "copy_blocks: too many pairs");
    const int64_t vec_per_block = (int64_t)bs * H * D / 8;
    dim3 grid(P, copy_splits(vec_per_block));
    cudaError_t e = launch_pdl(copy_blocks_kernel, grid, 256, pkv::as_stream(stream),
                               static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                               static_cast<const uint4*>(k_cache), static_cast<const uint4*>(v_cache),
                               block_mapping, vec_per_block, NB, NB, pkv::device_error_word());
    return e == cudaSuccess ? PKV_OK : pkv::cuda_fail(e, "copy_blocks launch");
}

pkv_status pkv_swap_blocks(void* gpu_k, void* gpu_v, void* host_k, void* host_v,
                           const int64_t* block_mapping, int P, int H, int D, int bs, int NB_gpu,
                           int NB_host, pkv_dtype dtype, int direction, void* stream) {
    PKV_TRACE("pkv_swap_blocks");
    pkv::clear_error();
    if (P < 0 || H <= 0 || NB_gpu < 0 || NB_host < 0 || (dtype != PKV_F16 && dtype != PKV_BF16) ||
        (direction != PKV_SWAP_OUT && direction != PKV_SWAP_IN))
        return pkv::fail(PKV_ERR_INVALID_ARG, "swap_blocks: bad size, dtype or direction");
    if (!supported(D, bs)) return pkv::fail(PKV_ERR_UNSUPPORTED, "swap_blocks: unsupported head_dim/block_size");
    if (P == 0) return PKV_OK;
    if (P > 65535 * 64) return pkv::fail(PKV_ERR_INVALID_ARG, "swap_blocks: too many pairs");
    if (!gpu_k || !gpu_v || !host_k || !host_v || !block_mapping)
        return pkv::fail(PKV_ERR_INVALID_ARG, "swap_blocks: null pointer");
    if (!pkv::aligned16(gpu_k) || !pkv::aligned16(gpu_v) || !pkv::aligned16(host_k) || !pkv::aligned16(host_v))
        return pkv::fail(PKV_ERR_INVALID_ARG, "swap_blocks: pointers must be 16-byte aligned");
    void* dk = device_view_of_host(host_k);
    void* dv = device_view_of_host(host_v);
    if (!dk || !dv)
        return pkv::fail(PKV_ERR_INVALID_ARG, "swap_blocks: host caches must be page-locked host memory the device can address");
    const int64_t vec_per_block = (int64_t)bs * H * D / 8;
    dim3 grid(P, copy_splits(vec_per_block));
    uint4 *gk = static_cast<uint4*>(gpu_k), *gv = static_cast<uint4*>(gpu_v);
    uint4 *hk = static_cast<uint4*>(dk), *hv = static_cast<uint4*>(dv);
    const bool out = direction == PKV_SWAP_OUT;
    cudaError_t e = launch_pdl(copy_blocks_kernel, grid, 256, pkv::as_stream(stream),
                               out ? hk : gk, out ? hv : gv, out ? gk : hk, out ? gv : hv,
                               block_mapping, vec_per_block, out ? NB_gpu : NB_host,
                               out ? NB_host : NB_gpu, pkv::device_error_word());
    return e == cudaSuccess ? PKV_OK : pkv::cuda_fail(e, "swap_blocks launch");
}

}  // extern "C"
