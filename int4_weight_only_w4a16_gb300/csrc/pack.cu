// pack_int4_g128: symmetric group-wise INT4 quantisation (group 128) + packing.
//
// Scheme from "How to build your own LLM runtime from scratch (Towards Data
// Science)", section "What it actually builds" (INT4, symmetric, group-wise,
// group 128), read as: s = fp16(max|w|/7), q = clamp(rint(w/s), -8, 7).
// The packed nibble layout is this library's own (see include/w4a16.h).
//
// One warp per (row, group): each lane holds 4 consecutive weights (one
// 16-byte load), the group max comes from a warp max-reduction, and lane pairs
// merge their nibbles into one 32-bit word.  IEEE division and rintf keep the
// codes bit-identical to an fp32 reference (the library is built without
// fast-math).
#include "common.cuh"

namespace w4 {

__global__ void __launch_bounds__(256)
pack_int4_g128_kernel(const float* __restrict__ w, int64_t n, int64_t k, uint32_t* __restrict__ packed,
                      __half* __restrict__ scales, int32_t* flags, int* errword) {
    const int lane = threadIdx.x & 31;
    const int64_t groups_per_row = k / 128;
    const int64_t gid = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (gid >= n * groups_per_row) return;
    const int64_t row = gid / groups_per_row;
    const int64_t grp = gid % groups_per_row;
    const float4 v = reinterpret_cast<const float4*>(w + row * k + grp * 128)[lane];
    const float e[4] = {v.x, v.y, v.z, v.w};

    bool finite = true;
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        finite = finite && isfinite(e[i]);
        amax = fmaxf(amax, fabsf(e[i]));
    }
    finite = __all_sync(0xffffffffu, finite);
    amax = warp_max(amax);

    const float s32 = __fdiv_rn(amax, 7.0f);
    const __half s16 = __float2half_rn(s32);
    const float sf = __half2float(s16);
    int bad = 0;
    if (!finite) bad = W4_DEVERR_NONFINITE;
    else if (isinf(sf)) bad = W4_DEVERR_SCALE_OVF;

    // codes of this lane's 4 elements: element index within the 8-wide word is
    // (lane & 1) * 4 + i; its slot is 4*(e%2) + e/2
    uint32_t part = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int q = 0;
        if (!bad && sf != 0.f) {
            float r = rintf(__fdiv_rn(e[i], sf));
            r = fminf(fmaxf(r, -8.f), 7.f);
            q = (int)r;
        }
        const int el = (lane & 1) * 4 + i;
        const int slot = 4 * (el & 1) + (el >> 1);
        part |= (uint32_t)(q + 8) << (4 * slot);
    }
    const uint32_t word = part | __shfl_xor_sync(0xffffffffu, part, 1);
    if ((lane & 1) == 0) packed[row * (k / 8) + grp * 16 + (lane >> 1)] = word;
    if (lane == 0) {
        scales[row * groups_per_row + grp] = bad ? __float2half_rn(0.f) : s16;
        if (bad) {
            record_device_error(errword, bad);
            if (flags) atomicOr(flags, bad);
        }
    }
}

}  // namespace w4

extern "C" w4_status w4_pack_int4_g128(const float* w, int64_t n, int64_t k, uint32_t* packed, void* scales,
                                       int32_t* flags, void* stream) {
    W4_REQUIRE(w && packed && scales, W4_ERR_NULL, "pack_int4_g128: null pointer");
    W4_REQUIRE(n >= 1 && k >= 128 && k % 128 == 0, W4_ERR_SHAPE,
               "pack_int4_g128: need n >= 1 and k a positive multiple of 128 (n=%lld k=%lld)",
               (long long)n, (long long)k);
    W4_REQUIRE(w4::aligned16(w) && w4::aligned16(packed), W4_ERR_ALIGN, "pack_int4_g128: w/packed not 16-B aligned");
    W4_REQUIRE((reinterpret_cast<uintptr_t>(scales) & 1) == 0, W4_ERR_ALIGN, "pack_int4_g128: scales misaligned");
    const int64_t groups = n * (k / 128);
    const int warps_per_block = 8;
    const int64_t blocks = (groups + warps_per_block - 1) / warps_per_block;
    W4_REQUIRE(blocks <= 0x7fffffffLL, W4_ERR_SHAPE, "pack_int4_g128: matrix too large");
    w4::pack_int4_g128_kernel<<<(unsigned)blocks, warps_per_block * 32, 0, (cudaStream_t)stream>>>(
        w, n, k, packed, static_cast<__half*>(scales), flags, w4::device_error_word());
    W4_CUDA(cudaGetLastError());
    return W4_OK;
}
