// Error reporting, the device error word and device queries.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace w4 {

// One word per device (each device that loads the module has its own copy of
// this variable); kernels OR W4_DEVERR_* codes into it instead of trapping.
__device__ int g_device_error_word;

static thread_local char t_msg[512] = "no error";

w4_status set_error(w4_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_msg, sizeof t_msg, fmt, ap);
    va_end(ap);
    return st;
}

w4_status cuda_check(cudaError_t e, const char* what) {
    return set_error(W4_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

static constexpr int kMaxDevices = 64;

int* device_error_word() {
    static int* addr[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<int*>(p);
    }
    return addr[dev];
}

int sm_count() {
    static int cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace w4

extern "C" const char* w4_last_error(void) { return w4::t_msg; }

extern "C" int w4_sm_count(void) { return w4::sm_count(); }

extern "C" w4_status w4_device_error(int32_t* flags, int clear) {
    W4_REQUIRE(flags != nullptr, W4_ERR_NULL, "w4_device_error: flags is NULL");
    int* word = w4::device_error_word();
    W4_REQUIRE(word != nullptr, W4_ERR_CUDA, "w4_device_error: no device error word");
    int v = 0;
    W4_CUDA(cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost));
    if (clear) W4_CUDA(cudaMemset(word, 0, sizeof v));
    *flags = v;
    return W4_OK;
}
