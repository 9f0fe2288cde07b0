// Shared host/device helpers for the W4A16 library (sm_103a only).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/w4a16.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "this library targets Blackwell (sm_103a); build with -gencode arch=compute_103a,code=sm_103a"
#endif

namespace w4 {

// ---------------------------------------------------------------- host side
w4_status set_error(w4_status st, const char* fmt, ...);
w4_status cuda_check(cudaError_t e, const char* what);
int* device_error_word();   // device address of this device's error word
int sm_count();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define W4_CUDA(call)                                                   \
    do {                                                                \
        cudaError_t e_ = (call);                                        \
        if (e_ != cudaSuccess) return ::w4::cuda_check(e_, #call);      \
    } while (0)

#define W4_REQUIRE(cond, code, ...)                                     \
    do {                                                                \
        if (!(cond)) return ::w4::set_error((code), __VA_ARGS__);       \
    } while (0)

// -------------------------------------------------------------- device side
__device__ __forceinline__ void record_device_error(int* word, int code) {
    if (word) atomicOr(word, code);
}

__device__ __forceinline__ uint4 ldg_stream_u4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and wait for the previous kernel's results before consuming them.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace w4
