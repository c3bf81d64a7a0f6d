// Library runtime: last-error text, version, stream check, and the device
// error word that kernels set instead of touching an out-of-range address.
#include <mutex>
#include <string>

#include "pagedkv.h"
#include "pkv_device.cuh"

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
    pkv::clear_error();
    cudaError_t e = cudaStreamSynchronize(pkv::as_stream(stream));
    if (e != cudaSuccess) return pkv::cuda_fail(e, "sync_check");
    e = cudaGetLastError();
    if (e != cudaSuccess) return pkv::cuda_fail(e, "sync_check");
    return PKV_OK;
}

pkv_status pkv_get_device_errors(int32_t* flags) {
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

}  // extern "C"
