// Library runtime: last-error text, version, stream check, the device
// error word that kernels set instead of touching an out-of-range address
// or waiting without end, and a self-test of the bounded in-kernel waits.
#include <mutex>
#include <string>

#include "pagedkv.h"
#include "pkv_device.cuh"
#include "tc_wait.cuh"

namespace {

thread_local std::string t_last_error;

// One word per device that loads the library; kernels atomicOr
// PKV_DEVERR_* bits into it.
__device__ int g_pkv_device_errors;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_err_addr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

// The steps a tensor-core prefix CTA takes when one of its waits runs out:
// one warp takes TMEM, waits on an mbarrier that nothing completes for
// `polls` rounds, reports PKV_DEVERR_TIMEOUT, frees the TMEM and returns.
__global__ void __launch_bounds__(32, 1) wait_selftest_kernel(int* err, long long polls) {
    __shared__ __align__(8) unsigned long long bar;
    __shared__ uint32_t tslot;
    __shared__ int abort_flag;
    const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar);
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        tc_mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        abort_flag = 0;
    }
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;"
                 ::"r"((uint32_t)__cvta_generic_to_shared(&tslot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
    __syncwarp();
    tc_fence_after();
    const uint32_t tmem = tslot;
    int ok = 1;
    if (lane == 0) ok = tc_mbar_wait(b, 0u, &abort_flag, polls) ? 1 : 0;  // nothing arrives
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok && lane == 0) pkv::report(err, PKV_DEVERR_TIMEOUT);
    tc_fence_before();
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;" ::"r"(tmem) : "memory");
}

}  // namespace

namespace pkv {

void set_error(const std::string& msg) { t_last_error = msg; }
void clear_error() { t_last_error.clear(); }

int* device_error_word() {
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pkv_device_errors) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_err_addr[dev] = static_cast<int*>(p);
    }
    return g_err_addr[dev];
}

int sm_count() {
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 1;
        }
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

}  // namespace pkv

extern "C" {

const char* pkv_last_error_string(void) { return t_last_error.c_str(); }

const char* pkv_version(void) { return "pagedkv 0.1 (sm_103a)"; }

pkv_status pkv_sync_check(void* stream) {
    PKV_TRACE("pkv_sync_check");
    pkv::clear_error();
    cudaError_t e = cudaStreamSynchronize(pkv::as_stream(stream));
    if (e != cudaSuccess) return pkv::cuda_fail(e, "sync_check");
    e = cudaGetLastError();
    if (e != cudaSuccess) return pkv::cuda_fail(e, "sync_check");
    return PKV_OK;
}

pkv_status pkv_get_device_errors(int32_t* flags) {
    PKV_TRACE("pkv_get_device_errors");
    pkv::clear_error();
    if (!flags) return pkv::fail(PKV_ERR_INVALID_ARG, "get_device_errors: null");
    int* w = pkv::device_error_word();
    if (!w) return pkv::fail(PKV_ERR_CUDA, "get_device_errors: no device error word");
    int v = 0;
    cudaError_t e = cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return pkv::cuda_fail(e, "get_device_errors");
    e = cudaMemset(w, 0, sizeof v);
    if (e != cudaSuccess) return pkv::cuda_fail(e, "get_device_errors");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return pkv::cuda_fail(e, "get_device_errors");
    *flags = v;
    return PKV_OK;
}

pkv_status pkv_selftest_bounded_wait(int64_t polls, void* stream) {
    PKV_TRACE("pkv_selftest_bounded_wait");
    pkv::clear_error();
    if (polls < 1 || polls > kTcWaitLimit)
        return pkv::fail(PKV_ERR_INVALID_ARG, "selftest_bounded_wait: polls must be in [1, 2^20]");
    int* err = pkv::device_error_word();
    if (!err) return pkv::fail(PKV_ERR_CUDA, "selftest_bounded_wait: no device error word");
    wait_selftest_kernel<<<1, 32, 0, pkv::as_stream(stream)>>>(err, (long long)polls);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return pkv::cuda_fail(e, "selftest_bounded_wait launch");
    return PKV_OK;
}

}  // extern "C"
