// Device-side helpers shared by the library's CUDA translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pkv_internal.h"

namespace pkv {

// Address of the device error word (PKV_DEVERR_* bits) of the current
// device; nullptr if the CUDA runtime could not provide it.
int* device_error_word();

// cudaStream_t from the ABI's void*.
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline pkv_status cuda_fail(cudaError_t e, const char* where) {
    set_error(std::string(where) + ": " + cudaGetErrorString(e));
    return PKV_ERR_CUDA;
}

// Number of SMs of the current device (cached per device).
int sm_count();

// ---------------------------------------------------------------------------
// 16-bit element traits.  8 elements travel as one uint4 (16 bytes).
// ---------------------------------------------------------------------------
struct F16 {
    static __device__ __forceinline__ float2 to_float2(uint32_t u) {
        __half2 h = *reinterpret_cast<const __half2*>(&u);
        return __half22float2(h);
    }
    static __device__ __forceinline__ uint32_t from_float2(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
};

struct BF16 {
    // A bfloat16 is the upper half of a binary32: the widening is exact.
    static __device__ __forceinline__ float2 to_float2(uint32_t u) {
        return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
    }
    static __device__ __forceinline__ uint32_t from_float2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
};

template <typename E>
__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
    float2 a = E::to_float2(v.x), b = E::to_float2(v.y), c = E::to_float2(v.z), d = E::to_float2(v.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

template <typename E>
__device__ __forceinline__ uint4 pack8(const float* f) {
    uint4 v;
    v.x = E::from_float2(f[0], f[1]);
    v.y = E::from_float2(f[2], f[3]);
    v.z = E::from_float2(f[4], f[5]);
    v.w = E::from_float2(f[6], f[7]);
    return v;
}

// 16-byte streaming load of data read exactly once (read-only path, no L1
// allocation).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void report(int* err, int bits) {
    if (err) atomicOr(err, bits);
}

// Slot of the token at position p of sequence s: logical block p / bs,
// offset p % bs, physical block from the sequence's table row.  -1 means
// "no write": p < 0; a position past the row or a sequence outside [0, S)
// (PKV_DEVERR_POSITION); a logical block the table has not mapped
// (PKV_DEVERR_BLOCK_ID).
__device__ __forceinline__ int64_t slot_of(const int32_t* __restrict__ bt, int s, int p, int S,
                                           int MB, int bs, int* err) {
    if (p < 0) return -1;
    const int logical = p / bs;
    if (logical >= MB || s < 0 || s >= S) {
        report(err, PKV_DEVERR_POSITION);
        return -1;
    }
    const int64_t phys = bt[(int64_t)s * MB + logical];
    if (phys < 0) {
        report(err, PKV_DEVERR_BLOCK_ID);
        return -1;
    }
    return phys * bs + (p - logical * bs);
}

// One CTA copies new token t's K and V rows (vec_per_row 16-byte vectors
// each) into row `slot` of the caches, two vectors of each in flight per
// thread.  slot must be in range.
__device__ __forceinline__ void write_token_rows(const uint4* __restrict__ key,
                                                 const uint4* __restrict__ value,
                                                 uint4* __restrict__ k_cache,
                                                 uint4* __restrict__ v_cache, int t, int64_t slot,
                                                 int vec_per_row) {
    const uint4* ks = key + (int64_t)t * vec_per_row;
    const uint4* vs = value + (int64_t)t * vec_per_row;
    uint4* kd = k_cache + slot * vec_per_row;
    uint4* vd = v_cache + slot * vec_per_row;
    const int step = blockDim.x;
    int i = threadIdx.x;
    for (; i + step < vec_per_row; i += 2 * step) {
        const uint4 a0 = ks[i], a1 = ks[i + step], b0 = vs[i], b1 = vs[i + step];
        kd[i] = a0; kd[i + step] = a1; vd[i] = b0; vd[i + step] = b1;
    }
    if (i < vec_per_row) {
        const uint4 a = ks[i], b = vs[i];
        kd[i] = a;
        vd[i] = b;
    }
}

}  // namespace pkv
