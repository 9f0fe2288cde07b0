// W4A16 GEMV kernel template (CUDA cores; dequantisation fused into the dot).
//
// Source of the operation: "How to build your own LLM runtime from scratch
// (Towards Data Science)", section "What it actually builds" (fused GEMVs for
// Q/K/V/O and gate/up/down over INT4 group-128 weights) and "How To Build
// Your Own LLM Runtime From Scratch | daily.dev", third question (fp16
// activations against unpacked INT4 weights beat an INT8-activation path).
//
// Design for sm_103a (HBM-bound at batch 1, so no tensor cores here):
//  * A CTA of 256 threads owns 16*R consecutive output rows; each half-warp
//    streams R rows together (R = 2, or 1 for short matrices; in the fused
//    SwiGLU mode one gate row and the matching up row).  Lane l of a
//    half-warp reads 16-byte chunks l, l+16, l+32, ... of its rows (32 weights
//    each), so a half-warp reads 256 contiguous bytes of a row per step and
//    every load is a full, coalesced 16-byte vector.  Each activation chunk a
//    lane reads from shared memory serves all R rows.
//  * Each lane keeps a ring of 4 chunk loads in flight: the first 4 are issued
//    before the kernel waits on the previous kernel (weights do not depend on
//    it, so with programmatic dependent launch they overlap its tail and the
//    activation staging), and every consumed slot is refilled at once with
//    the chunk 4 steps ahead.
//  * The activation slice is staged once per CTA in shared memory in a
//    chunk-transposed order (piece i of chunk c at [i][c]) so the per-lane
//    16-byte reads are bank-conflict free.
//  * Split-K (grid.y) keeps >= ~3 CTAs per SM for short matrices; partial
//    sums go to a workspace and the last CTA of each row block (atomic
//    ticket, no waiting) reduces them in a fixed order -> deterministic.
//  * Inner product variants (all exact dequantisation; fp32 accumulation of
//    the scaled group partials):
//      V_SUBNORMAL: a nibble masked into the low bits of an fp16 is the
//        subnormal u*2^-24, exactly; one mixed-precision fma.rn.f32.f16 per
//        weight accumulates u*x in fp32 with exact products, and the offset
//        is removed per 32-weight chunk: sum(q x) = 2^24*sum(u x 2^-24) - 8*sum(x).
//        Cost per 8 weights: 1 shift + 4 and + 8 FMA.
//      V_HALF_CHUNK: nibble -> fp16 (1024+u) with one or, then one HFMA2 makes
//        q exactly; HFMA2 accumulates 16 products per lane in fp16 before the
//        fp32 fold.  Cost per 8 weights: 1 shift + 4 lop3 + 8 HFMA2.
//      V_HALF_WORD: as V_HALF_CHUNK but folds into fp32 after every word
//        (4 fp16 products per lane).
#pragma once

#include "common.cuh"

namespace w4 {

// V_TENSOR selects the TMA-fed tensor-core kernel (gemv_tc.cuh) and
// V_MMA_ALL the register-pipelined one (gemv_mma.cuh) at every batch size,
// not a CUDA-core dot
// V_INT8 is the W4A8 measurement variant: activations quantised to INT8 per
// 128-group while staging, INT4 codes against them by dp4a
enum GemvVariant { V_SUBNORMAL = 0, V_HALF_CHUNK = 1, V_HALF_WORD = 2, V_TENSOR = 3, V_MMA_ALL = 4, V_INT8 = 5 };
enum GemvXMode { X_F16 = 0, X_RMSNORM = 1 };
enum GemvEpi { E_STORE_F16 = 0, E_RESID_F32 = 1, E_SWIGLU = 2, E_ARGMAX = 3, E_QKV_ROPE = 4 };

constexpr int kGemvThreads = 256;
constexpr int kGemvRows = 16;      // rows per CTA (one per half-warp)
constexpr int kGemvUnroll = 4;     // chunks in flight per lane per row

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
    } else if constexpr (VAR == V_SUBNORMAL) {
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
    } else {
        const __half2 k1032 = __half2half2(__ushort_as_half(0x6408));   // 1032
        const __half2 k1_16 = __half2half2(__ushort_as_half(0x2c00));   // 1/16
        const __half2 km72 = __half2half2(__ushort_as_half(0xd480));    // -72
        __half2 h = __half2half2(__ushort_as_half(0));
        float dot = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t v = ws[j], v8 = ws[j] >> 8;
            const uint4 xv = xq[j];
            const __half2 q01 = __hsub2(u32_as_h2((v & 0x000F000Fu) | 0x64006400u), k1032);
            const __half2 q23 = __hfma2(u32_as_h2((v & 0x00F000F0u) | 0x64006400u), k1_16, km72);
            const __half2 q45 = __hsub2(u32_as_h2((v8 & 0x000F000Fu) | 0x64006400u), k1032);
            const __half2 q67 = __hfma2(u32_as_h2((v8 & 0x00F000F0u) | 0x64006400u), k1_16, km72);
            h = __hfma2(q01, u32_as_h2(xv.x), h);
            h = __hfma2(q23, u32_as_h2(xv.y), h);
            h = __hfma2(q45, u32_as_h2(xv.z), h);
            h = __hfma2(q67, u32_as_h2(xv.w), h);
            if constexpr (VAR == V_HALF_WORD) {
                const float2 f = __half22float2(h);
                dot += f.x + f.y;
                h = __half2half2(__ushort_as_half(0));
            }
        }
        if constexpr (VAR == V_HALF_CHUNK) {
            const float2 f = __half22float2(h);
            dot = f.x + f.y;
        }
        return dot;
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

// Dynamic shared memory bytes for a CTA: staged activations + chunk sums.
__host__ __device__ inline size_t gemv_smem_bytes(int mt, int kc) {
    return (size_t)mt * kc * (64 + 4) + 64 * sizeof(float);
}

// Two resident CTAs per SM when a lane streams two rows (2 x 64 B in flight
// per lane), three otherwise.
template <int MT, int R, int VAR, int XMODE, int EPI>
__global__ void __launch_bounds__(kGemvThreads, (R * (EPI == E_SWIGLU ? 2 : 1) >= 2) ? 2 : 3)
gemv_w4a16_kernel(const GemvParams p) {
    constexpr int NM = (EPI == E_SWIGLU) ? 2 : 1;   // matrices streamed together
    constexpr int NR = NM * R;                       // rows a lane loads per chunk
    constexpr int U = kGemvUnroll;                   // ring of in-flight chunk loads
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int kc = p.kc;
    uint4* xs = reinterpret_cast<uint4*>(smem_raw);                    // [MT][4][kc]
    float* xneg8 = reinterpret_cast<float*>(xs + (size_t)MT * 4 * kc); // [MT][kc]
    float* red = xneg8 + (size_t)MT * kc;                              // [64]

    const int tid = threadIdx.x;
    const int hw = tid >> 4;          // half-warp: R consecutive rows
    const int l16 = tid & 15;
    const int chunks = p.K >> 5;
    const int cb = blockIdx.y * kc;
    const int ce = min(chunks, cb + kc);
    const int nloc = ce - cb;
    const int gpr = p.K >> 7;         // scale groups per row
    const int row0 = (blockIdx.x * kGemvRows + hw) * R;

    // rows this lane streams (clamped so that every load stays in bounds)
    const uint32_t* wrow[NR];
    const __half* srow[NR];
#pragma unroll
    for (int i = 0; i < NR; ++i) {
        const int r = min(row0 + (i % R), p.N - 1);
        const uint32_t* wb = (NM == 2 && i >= R) ? p.w1 : p.w0;
        const __half* sb = (NM == 2 && i >= R) ? p.s1 : p.s0;
        wrow[i] = wb + (size_t)r * (p.K >> 3);
        srow[i] = sb + (size_t)r * gpr;
    }
    // this lane's chunks: cb + l16 + 16 j, j < J
    const int J = (nloc - l16 + 15) >> 4;

    // ---- weights do not depend on the previous kernel: start the ring now
    uint4 wv[U][NR];
    float sc[U][NR];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (u < J) {
            const int c = cb + l16 + 16 * u;
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                wv[u][i] = ldg_stream_u4(wrow[i] + (size_t)c * 4);
                sc[u][i] = __half2float(srow[i][c >> 2]);
            }
        }
    }
    pdl_trigger();
    // the activations come from the previous kernel in the stream
    pdl_wait();

    // ---- stage the activation slice [cb, ce) chunks into shared memory
    float inv_rms = 1.f;
    if constexpr (XMODE == X_RMSNORM) {
        float ss = 0.f;
        const float4* xr4 = reinterpret_cast<const float4*>(p.xres);
        for (int i = tid; i < (p.K >> 2); i += kGemvThreads) {
            const float4 v = xr4[i];
            ss = fmaf(v.x, v.x, ss);
            ss = fmaf(v.y, v.y, ss);
            ss = fmaf(v.z, v.z, ss);
            ss = fmaf(v.w, v.w, ss);
        }
        ss = warp_sum(ss);
        if ((tid & 31) == 0) red[tid >> 5] = ss;
        __syncthreads();
        if (tid < 32) {
            float t = tid < (kGemvThreads / 32) ? red[tid] : 0.f;
            t = warp_sum(t);
            if (tid == 0) red[32] = 1.0f / sqrtf(t / (float)p.K + p.eps);
        }
        __syncthreads();
        inv_rms = red[32];
    }
    for (int idx = tid; idx < MT * nloc; idx += kGemvThreads) {
        const int m = idx / nloc;
        const int c = idx - m * nloc;
        uint4 pieces[4];
        float csum = 0.f;
        if (m < p.M) {
            const int k0 = (cb + c) * 32;
            if constexpr (XMODE == X_RMSNORM) {
                const float4* xr = reinterpret_cast<const float4*>(p.xres + k0);
                const uint4* gm = reinterpret_cast<const uint4*>(p.gamma + k0);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 a = xr[2 * i], b = xr[2 * i + 1];
                    const uint4 g = gm[i];
                    const float2 g0 = __half22float2(u32_as_h2(g.x)), g1 = __half22float2(u32_as_h2(g.y));
                    const float2 g2 = __half22float2(u32_as_h2(g.z)), g3 = __half22float2(u32_as_h2(g.w));
                    const __half2 h0 = __floats2half2_rn(a.x * inv_rms * g0.x, a.y * inv_rms * g0.y);
                    const __half2 h1 = __floats2half2_rn(a.z * inv_rms * g1.x, a.w * inv_rms * g1.y);
                    const __half2 h2 = __floats2half2_rn(b.x * inv_rms * g2.x, b.y * inv_rms * g2.y);
                    const __half2 h3 = __floats2half2_rn(b.z * inv_rms * g3.x, b.w * inv_rms * g3.y);
                    pieces[i] = make_uint4(h2_as_u32(h0), h2_as_u32(h1), h2_as_u32(h2), h2_as_u32(h3));
                }
            } else {
                const uint4* xg = reinterpret_cast<const uint4*>(p.x + (size_t)m * p.K + k0);
#pragma unroll
                for (int i = 0; i < 4; ++i) pieces[i] = xg[i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t u[4] = {pieces[i].x, pieces[i].y, pieces[i].z, pieces[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 f = __half22float2(u32_as_h2(u[j]));
                    csum += f.x + f.y;
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) pieces[i] = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) xs[((size_t)m * 4 + i) * kc + c] = pieces[i];
        xneg8[(size_t)m * kc + c] = -8.f * csum;
    }
    __syncthreads();

    // ---- main loop: consume slot u, then refill it with the chunk U ahead
    float acc[MT][NR];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int i = 0; i < NR; ++i) acc[m][i] = 0.f;

    for (int j0 = 0; j0 < J; j0 += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = j0 + u;
            if (j < J) {
                const int cl = l16 + 16 * j;   // chunk index within the staged slice
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    uint4 xq[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) xq[q] = xs[((size_t)m * 4 + q) * kc + cl];
                    const float n8 = xneg8[(size_t)m * kc + cl];
#pragma unroll
                    for (int i = 0; i < NR; ++i)
                        acc[m][i] = fmaf(sc[u][i], chunk_dot<VAR>(wv[u][i], xq, n8), acc[m][i]);
                }
                if (j + U < J) {
                    const int c = cb + cl + 16 * U;
#pragma unroll
                    for (int i = 0; i < NR; ++i) {
                        wv[u][i] = ldg_stream_u4(wrow[i] + (size_t)c * 4);
                        sc[u][i] = __half2float(srow[i][c >> 2]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int i = 0; i < NR; ++i)
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) acc[m][i] += __shfl_xor_sync(0xffffffffu, acc[m][i], o);

    // ---- split-K: publish partials, last CTA of the row block reduces
    __shared__ int s_last;
    if (p.split > 1) {
        if (l16 == 0) {
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const int row = row0 + i;
                if (row < p.N)
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        if (m < p.M) p.part[((size_t)blockIdx.y * p.M + m) * p.N + row] = acc[m][i];
            }
            __threadfence();
        }
        __syncthreads();
        if (tid == 0) {
            const unsigned t = atomicAdd(&p.counters[blockIdx.x], 1u);
            s_last = (t == (unsigned)p.split - 1);
        }
        __syncthreads();
        if (!s_last) return;  // uniform for the CTA
        __threadfence();
        if (l16 == 0) {
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const int row = row0 + i;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float s = 0.f;
                    if (m < p.M && row < p.N)
                        for (int sp = 0; sp < p.split; ++sp)
                            s += __ldcg(&p.part[((size_t)sp * p.M + m) * p.N + row]);
                    acc[m][i] = s;
                }
            }
        }
        if (tid == 0) p.counters[blockIdx.x] = 0u;
    }

    // ---- epilogue (lane 0 of each half-warp holds the R row sums)
    if constexpr (EPI == E_ARGMAX) {
        __shared__ unsigned long long s_key[kGemvRows];
        unsigned long long k = 0ull;
        if (l16 == 0) {
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const int row = row0 + i;
                if (row < p.N) {
                    if (p.y32) p.y32[row] = acc[0][i];
                    if (acc[0][i] != acc[0][i]) record_device_error(p.errword, W4_DEVERR_NAN_LOGIT);
                    const unsigned long long kk = argmax_key(acc[0][i], row);
                    k = kk > k ? kk : k;
                }
            }
            s_key[hw] = k;
        }
        __syncthreads();
        if (tid == 0) {
            for (int i = 0; i < kGemvRows; ++i) k = s_key[i] > k ? s_key[i] : k;
            atomicMax(p.amax_key, k);
            __threadfence();
            const unsigned t = atomicAdd(p.counters, 1u);
            if (t == gridDim.x * gridDim.y - 1) {
                __threadfence();
                const unsigned long long kk = atomicExch(p.amax_key, 0ull);
                p.token_out[0] = (int32_t)(0xFFFFFFFFu - (uint32_t)(kk & 0xFFFFFFFFull));
                p.counters[0] = 0u;
                if (p.pos) p.pos[0] += 1;
            }
        }
    } else {
        if (l16 != 0) return;
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int row = row0 + i;
            if (row >= p.N) break;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m >= p.M) break;
                if constexpr (EPI == E_STORE_F16) {
                    float v = acc[m][i];
                    if (p.bias) v += __half2float(p.bias[row]);
                    if (p.resid16) v += __half2float(p.resid16[(size_t)m * p.N + row]);
                    p.y16[(size_t)m * p.N + row] = __float2half_rn(v);
                } else if constexpr (EPI == E_RESID_F32) {
                    p.y32[(size_t)m * p.N + row] += acc[m][i];
                } else if constexpr (EPI == E_SWIGLU) {
                    const float g = acc[m][i], u = acc[m][R + i];
                    p.y16[(size_t)m * p.N + row] = __float2half_rn(g / (1.f + expf(-g)) * u);
                }
            }
        }
    }
}

// ---------------------------------------------------------------- host plan
struct GemvPlan {
    int split;
    int kc;
    int rows;   // rows per half-warp (R)
    dim3 grid;
    size_t smem;
};

// Split-K so that short matrices still give each SM a few CTAs; bounded by
// the shared memory one CTA may stage (96 KiB of activations).
inline GemvPlan gemv_plan(int mt, int n, int k, bool allow_split, int split_override = 0, int rows = 0) {
    GemvPlan pl;
    const int chunks = k / 32;
    const int sms = sm_count();
    // two rows per half-warp halves the shared-memory activation reads per
    // weight byte; fall back to one when that leaves fewer than ~1.5 CTAs per SM
    int R = rows > 0 ? rows : 2;
    if (rows <= 0 && mt > 1) R = 1;
    if (rows <= 0 && (n + 16 * R - 1) / (16 * R) < (3 * sms) / 2) R = 1;
    const int row_blocks = (n + kGemvRows * R - 1) / (kGemvRows * R);
    int s = 1;
    if (allow_split && row_blocks < sms) {
        s = (2 * sms + row_blocks - 1) / row_blocks;
        const int max_s = chunks / 32 > 0 ? chunks / 32 : 1;   // >= 2 chunks per lane
        s = s > max_s ? max_s : s;
    }
    const size_t budget = 96 * 1024;
    while (gemv_smem_bytes(mt, (chunks + s - 1) / s) > budget && s < chunks) ++s;
    if (allow_split && split_override > 0) s = split_override < chunks ? split_override : chunks;
    pl.split = s;
    pl.kc = (chunks + s - 1) / s;
    pl.split = (chunks + pl.kc - 1) / pl.kc;   // drop empty pieces
    pl.rows = R;
    pl.grid = dim3(row_blocks, pl.split, 1);
    pl.smem = gemv_smem_bytes(mt, pl.kc);
    return pl;
}

// Launch one instantiation; sets the dynamic shared memory limit once.
template <int MT, int R, int VAR, int XMODE, int EPI>
inline cudaError_t gemv_launch_r(const GemvParams& p, const GemvPlan& pl, cudaStream_t st, bool pdl) {
    auto kern = gemv_w4a16_kernel<MT, R, VAR, XMODE, EPI>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 100 * 1024);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = pl.grid;
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int MT, int VAR, int XMODE, int EPI>
inline cudaError_t gemv_launch(const GemvParams& p, const GemvPlan& pl, cudaStream_t st, bool pdl) {
    if constexpr (MT == 1 && EPI != E_SWIGLU) {
        if (pl.rows == 2) return gemv_launch_r<MT, 2, VAR, XMODE, EPI>(p, pl, st, pdl);
    }
    return gemv_launch_r<MT, 1, VAR, XMODE, EPI>(p, pl, st, pdl);
}

}  // namespace w4
