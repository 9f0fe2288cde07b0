// The W4A16 GEMV's shared pieces: parameters, the exact INT4 chunk dot and
// the greedy argmax key (kernels in gemv_tma.cuh at batch 1 and gemv_mma.cuh
// at batches of 2 to 16).
//
// Source of the operation: "How to build your own LLM runtime from scratch
// (Towards Data Science)", section "What it actually builds" (fused GEMVs for
// Q/K/V/O and gate/up/down over INT4 group-128 weights) and "How To Build
// Your Own LLM Runtime From Scratch | daily.dev", third question (fp16
// activations against unpacked INT4 weights beat an INT8-activation path).
//
// Inner products, with exact dequantisation and fp32 accumulation of the
// scaled group partials:
//   V_SUBNORMAL (the batch-1 default): a nibble masked into the low bits of an
//     fp16 is the subnormal u*2^-24, exactly; one mixed-precision
//     fma.rn.f32.f16 per weight accumulates u*x in fp32 with exact products,
//     and the offset is removed per 32-weight chunk:
//     sum(q x) = 2^24*sum(u x 2^-24) - 8*sum(x).
//     Cost per 8 weights: 1 shift + 4 and + 8 FMA.
//   V_MMA_ALL selects the mma.sync kernel (gemv_mma.cuh, the default for
//     batches of 2 to 11) at every batch.
//   V_TC05 selects the tcgen05 kernel (gemv_tc05.cuh, the default for
//     batches of 12 to 16) at every batch.
//   V_INT8 is the W4A8 re-check: activations quantised to INT8 per 128-group
//     while staging, INT4 codes against them by dp4a.
#pragma once

#include "common.cuh"

namespace w4 {

enum GemvVariant { V_SUBNORMAL = 0, V_MMA_ALL = 1, V_INT8 = 2, V_TC05 = 3 };
enum GemvXMode { X_F16 = 0, X_RMSNORM = 1 };
enum GemvEpi { E_STORE_F16 = 0, E_RESID_F32 = 1, E_SWIGLU = 2, E_ARGMAX = 3, E_QKV_ROPE = 4 };

struct GemvParams {
    const __half* x;          // X_F16: [M][K]
    const float* xres;        // X_RMSNORM: fp32 [K]
    const __half* gamma;      // X_RMSNORM: fp16 [K]
    float eps;
    const uint32_t* w0;       // packed [N][K/8]
    const __half* s0;         // scales [N][K/128]
    const uint32_t* w1;       // E_SWIGLU: up matrix (w0 = gate)
    const __half* s1;
    int M;
    int N;
    int K;
    const __half* bias;       // [N] or null   (E_STORE_F16)
    const __half* resid16;    // [M][N] or null (E_STORE_F16)
    __half* y16;              // E_STORE_F16 / E_SWIGLU output
    float* y32;               // E_RESID_F32: residual stream (+=); E_ARGMAX: logits or null
    float* part;              // split-K partials [S][M][N]
    unsigned* counters;       // split-K tickets [row_blocks] ; E_ARGMAX: [1]
    unsigned long long* amax_key;  // E_ARGMAX
    int32_t* token_out;       // E_ARGMAX
    int32_t* pos;             // E_ARGMAX: incremented once by the last CTA (nullable)
    int split;                // S = gridDim.y
    int kc;                   // chunks (32 weights) per split piece
    int* errword;             // device error word (bounded waits)
    // E_QKV_ROPE: the rows are q | k | v of one token; within every q and k
    // head the rows are interleaved (row 2i = dim i, row 2i+1 = dim i+64) so a
    // two-row group holds one rotate-half RoPE pair.  The epilogue adds the
    // bias, rounds to fp16, rotates q and k at position *pos_in, writes q to
    // qout and k, v into the paged pools, and publishes ctx = pos + 1.
    const float2* rope;       // [max_context][64] (cos, sin)
    const int32_t* pos_in;
    const int32_t* pt;        // page table [max_pages]
    __half* qout;             // [hq * 128]
    __half* k_pool;           // [num_pages][hkv][16][128]
    __half* v_pool;
    int32_t* ctx;
    int hq, hkv, max_pages, num_pages, max_context;
    // optional L2 warm-up of the next kernel's weights (two regions), shared
    // out over the CTAs; 16-byte aligned
    const void* pf0;
    size_t pf0_bytes;
    const void* pf1;
    size_t pf1_bytes;
};

__device__ __forceinline__ float fma_f16_lo(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{ .reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %3; }"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fma_f16_hi(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{ .reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, ah, bh, %3; }"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
    return d;
}

// sum_k q_k x_k over one 32-weight chunk (four packed words), returned in fp32.
// xq[j] holds the 8 activations of word j; negx8 = -8 * sum of the 32 activations.
// V_INT8: xq[0..1] hold the chunk's INT8 activations, per word the bytes
// (x0, x4, x1, x5) and (x2, x6, x3, x7) -- the element order of the word's low
// and high nibbles -- and xq[2] holds (fp32 group scale bits, -8 * sum q_x);
// the result is s_x * sum q_w q_x.
template <int VAR>
__device__ __forceinline__ float chunk_dot(const uint4& w, const uint4* xq, float negx8) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    if constexpr (VAR == V_INT8) {
        int acc = (int)xq[2].y;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t lo = ws[j] & 0x0F0F0F0Fu, hi = (ws[j] >> 4) & 0x0F0F0F0Fu;
            const uint4& pc = xq[j >> 1];
            acc = __dp4a((int)lo, (int)((j & 1) ? pc.z : pc.x), acc);
            acc = __dp4a((int)hi, (int)((j & 1) ? pc.w : pc.y), acc);
        }
        (void)negx8;
        return __uint_as_float(xq[2].x) * (float)acc;
    } else {
        float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t v = ws[j], v8 = ws[j] >> 8;
            const uint4 xv = xq[j];
            const uint32_t p01 = v & 0x000F000Fu, p23 = v & 0x00F000F0u;
            const uint32_t p45 = v8 & 0x000F000Fu, p67 = v8 & 0x00F000F0u;
            a0 = fma_f16_lo(p01, xv.x, a0);
            a1 = fma_f16_hi(p01, xv.x, a1);
            b0 = fma_f16_lo(p23, xv.y, b0);
            b1 = fma_f16_hi(p23, xv.y, b1);
            a0 = fma_f16_lo(p45, xv.z, a0);
            a1 = fma_f16_hi(p45, xv.z, a1);
            b0 = fma_f16_lo(p67, xv.w, b0);
            b1 = fma_f16_hi(p67, xv.w, b1);
        }
        // a*: sum u x 2^-24 ; b*: sum 16 u x 2^-24  (exact power-of-two rescaling)
        const float t = fmaf(b0 + b1, 0.0625f, a0 + a1);
        return fmaf(t, 16777216.f, negx8);
    }
}

// Ordered 64-bit key of (logit, row) for the greedy argmax: a larger logit
// wins, and equal logits go to the lower row (the low word is ~row).  -0 and
// +0 compare equal, so -0 is keyed as +0; a NaN logit never wins -- it ranks
// below every number, -inf included (the caller flags it).
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    uint32_t u = v == 0.f ? 0u : __float_as_uint(v);
    u = (v != v) ? 0u : ((u & 0x80000000u) ? ~u : (u | 0x80000000u));
    return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

}  // namespace w4
