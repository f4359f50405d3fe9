// Status reporting, the device error word and cached device facts.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "pkv_internal.h"

namespace {

thread_local char g_last_error[512] = "";

// One error word per device: every kernel of the library ORs its
// PKV_DEVERR_* bits here instead of faulting.
__device__ int32_t g_device_error;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

}  // namespace

namespace pkv {

pkv_status fail(pkv_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

pkv_status cuda_fail(cudaError_t e, const char* what) {
    return fail(PKV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

void clear_last_error() { g_last_error[0] = 0; }

int32_t* device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<int32_t*>(p);
    }
    return g_err_ptr[dev];
}

int sm_count(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

}  // namespace pkv

extern "C" {

const char* pkv_last_error(void) { return g_last_error; }

const char* pkv_version(void) { return "pagedkv 0.1 (sm_103a)"; }

pkv_status pkv_get_device_error(int32_t* bits, int clear, cudaStream_t stream) {
    if (!bits) return pkv::fail(PKV_ERR_INVALID, "pkv_get_device_error: bits is NULL");
    int32_t* word = pkv::device_error_word();
    if (!word) return pkv::fail(PKV_ERR_CUDA, "pkv_get_device_error: no device error word");
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return pkv::cuda_fail(e, "pkv_get_device_error: stream sync");
    int32_t v = 0;
    e = cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return pkv::cuda_fail(e, "pkv_get_device_error: read");
    if (clear && v) {
        const int32_t zero = 0;
        e = cudaMemcpy(word, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return pkv::cuda_fail(e, "pkv_get_device_error: clear");
    }
    *bits = v;
    if (v) return pkv::fail(PKV_ERR_DEVICE, "device error bits 0x%x", (unsigned)v);
    return PKV_OK;
}

}  // extern "C"
