// W4A16 GEMM for the prompt pass on the 5th-generation tensor cores.
//
//   Y[t][r] = sum_k X[t][k] * (q[r][k] * s[r][k / 128])      t < n tokens, r < N rows
//
// "How to build your own LLM runtime from scratch (Towards Data Science)",
// section "What it actually builds": the INT4 weights are expanded to fp16 and
// multiplied against fp16 activations with fp32 accumulation; with n prompt
// rows this is a dense contraction, so it runs on tcgen05.mma.
//
// One CTA owns two 128-row weight sub-tiles (rows r0 and r0 + 128 of one
// matrix, or the same 128 rows of gate and up) and bn <= 256 tokens, over a
// range of K (split-K when the tile count alone would leave SMs idle):
//   warp 0      TMA producer: the activation tile [bn][64] (128-byte swizzle)
//               and the packed weight tiles [128][8 words] per stage;
//   warp 1      allocates TMEM (2 * bn fp32 columns) and, from one thread,
//               issues tcgen05.mma (M = 128, N = bn, K = 16) per sub-tile;
//   warps 2..9  expand the packed words to fp16 q * s straight into the
//               canonical K-major 128-byte-swizzled operand layout (warps 2..5
//               sub-tile 0, warps 6..9 sub-tile 1: two expanding warps per
//               scheduler), then run the epilogue from TMEM (tcgen05.ld; each
//               warp reads the lane quarter it is allowed to, the two warps
//               of a quarter taking alternate 16-column chunks): store,
//               residual add, or
//               SiLU(gate) * up to fp16.  With split K every CTA stores its
//               partial tile, and a second kernel adds the partials in split
//               order (deterministic) and applies the same epilogue.
// Every mbarrier wait is bounded in wall time; on expiry the CTA records
// W4_DEVERR_TIMEOUT, drains what it issued (bounded) and frees its TMEM.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"

namespace w4 {

constexpr int kGmThreads = 320;
constexpr int kGmMaxStages = 4;
constexpr int kGmSubBytes = 128 * 128;      // one 128-row x 64-K fp16 operand tile
constexpr int kGmWpBytes = 128 * 32;        // its packed source: 128 rows x 8 words
constexpr size_t kGmSmemBudget = 220 * 1024;

enum { G_STORE = 0, G_RESID = 1, G_SWIGLU = 2 };

struct GemmArgs {
    int n, N, K;               // tokens, rows of each weight matrix, columns
    int bn;                    // tokens per tile: multiple of 16 in [16, 256]
    int tok_tiles, row_tiles;  // tiles = row_tiles * tok_tiles
    int splits, kb_per_split;  // K ranges of kb_per_split 64-column blocks
    int stages;
    int a_tmem;                // 1: the expanded weights go to TMEM (tcgen05.st), not shared memory
    int tile_rows;             // weight rows per CTA for one matrix: 256 (two sub-tiles) or 128
    const __half* s0;          // scales fp16 [N][K/128] of matrix 0
    const __half* s1;          // of matrix 1 (SwiGLU: up)
    float* y;                  // G_STORE / G_RESID: fp32 [n][ldy], columns [0, N)
    int ldy;
    __half* act;               // G_SWIGLU: fp16 [n][N]
    float* part;               // split-K partials fp32 [splits][n][nout]
    int* errword;
};

// TMEM-operand variant: accumulators in columns [0, 2 bn), bn <= 192; the two
// A stages (two sub-tiles of 128 rows x 64 fp16 = 32 columns each) from 384.
constexpr int kGmAtBnMax = 192;
constexpr uint32_t kGmAtCol = 384;
constexpr int kGmAtStages = 2;

__host__ __device__ inline uint32_t gemm_b_bytes(int bn) { return (uint32_t)((bn * 128 + 1023) / 1024 * 1024); }
__host__ __device__ inline uint32_t gemm_stage_bytes(int bn, int a_tmem) {
    return gemm_b_bytes(bn) + (a_tmem ? 0 : 2 * kGmSubBytes) + 2 * kGmWpBytes;
}
__host__ __device__ inline uint32_t gemm_tmem_cols(int bn, int a_tmem) {
    if (a_tmem) return 512;
    uint32_t c = 32;
    while (c < (uint32_t)(2 * bn)) c <<= 1;
    return c;
}

#ifdef W4_DEFINE_GEMM_TC05_KERNEL
constexpr uint64_t kGmWaitNs = 1000000000ull;

__device__ __forceinline__ void gm_tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart (stride byte offset), base 1024-aligned.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Same MMA with A read from tensor memory (128 lanes = rows, 8 columns per 16 K).
__device__ __forceinline__ void tc_mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 consecutive 32-bit TMEM columns of this warp's 32 lanes (one lane per thread),
// waited for before returning.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
          "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
          "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// One packed word (elements e in slot 4 * (e % 2) + e / 2, nibble q + 8) to
// four fp16 pairs q * s: (u | 0x6400) is the fp16 value 1024 + u, minus 1032
// gives q exactly, and one fp16 multiply rounds q * s once.
__device__ __forceinline__ uint4 expand_word(uint32_t w, __half2 s2) {
    const __half2 off = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
    uint32_t o[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t u = ((w >> (4 * p)) & 0x000F000Fu) | 0x64006400u;
        o[p] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(u), off), s2));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float gm_silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// AND of `pred` over the `threads` threads meeting at named barrier `id`.
__device__ __forceinline__ bool bar_and(unsigned id, unsigned threads, bool pred) {
    uint32_t r;
    asm volatile(
        "{ .reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q; }"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

template <int EPI>
__device__ __forceinline__ void gemm_epilogue_one(const GemmArgs& a, int tok, int row0, int row1, int r, int nsub,
                                                  float v0, float v1) {
    if constexpr (EPI == G_SWIGLU) {
        a.act[(size_t)tok * a.N + row0 + r] = __float2half_rn(gm_silu_mul(v0, v1));
    } else if constexpr (EPI == G_RESID) {
        float* y = a.y + (size_t)tok * a.ldy;
        y[row0 + r] += v0;
        if (nsub == 2) y[row1 + r] += v1;
    } else {
        float* y = a.y + (size_t)tok * a.ldy;
        y[row0 + r] = v0;
        if (nsub == 2) y[row1 + r] = v1;
    }
}

template <int EPI, bool AT>
__global__ void __launch_bounds__(kGmThreads, 1)
w4_gemm_tc05_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap tmx,
                    const __grid_constant__ CUtensorMap tmw0, const __grid_constant__ CUtensorMap tmw1) {
    extern __shared__ unsigned char gm_raw[];
    __shared__ uint64_t full[kGmMaxStages], adone[kGmMaxStages], empty[kGmMaxStages], accf;
    __shared__ uint64_t afull[kGmAtStages], aempty[kGmAtStages];   // TMEM operand stages
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tiles = a.row_tiles * a.tok_tiles;
    const int split = blockIdx.x / tiles, tile = blockIdx.x - split * tiles;
    const int rt = tile / a.tok_tiles, tt = tile - rt * a.tok_tiles;
    const int tok0 = tt * a.bn;
    const int kb0 = split * a.kb_per_split;
    const int kb1 = min(a.K / 64, kb0 + a.kb_per_split);
    const int nkb = kb1 - kb0;
    constexpr bool kSwiglu = EPI == G_SWIGLU;
    const int row0 = kSwiglu ? rt * 128 : rt * a.tile_rows;
    const int row1 = kSwiglu ? rt * 128 : row0 + 128;
    const int nsub = (kSwiglu || (a.tile_rows == 256 && row1 < a.N)) ? 2 : 1;
    const int stages = a.stages;
    const uint32_t bbytes = gemm_b_bytes(a.bn);
    constexpr bool at = AT;
    const uint32_t sbytes = gemm_stage_bytes(a.bn, a.a_tmem);
    const uint32_t ncols = gemm_tmem_cols(a.bn, a.a_tmem);
    const uint32_t wpoff = bbytes + (at ? 0u : 2u * kGmSubBytes);   // packed tiles inside a stage
    const uint32_t base = (smem_u32(gm_raw) + 1023u) & ~1023u;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&adone[s], 256);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < kGmAtStages; ++s) {
            mbar_init(&afull[s], 256);
            mbar_init(&aempty[s], 1);
        }
        mbar_init(&accf, 1);
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmx)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmw0)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmw1)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int* abort_flag = &s_abort;
    auto give_up = [&]() {
        record_device_error(a.errword, W4_DEVERR_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            const uint32_t tx = (uint32_t)a.bn * 128 + (uint32_t)nsub * kGmWpBytes;
            int issued = 0;
            for (int i = 0; i < nkb && !*abort_flag; ++i) {
                const int s = i % stages;
                const unsigned ph = (unsigned)(i / stages) & 1u;
                if (!mbar_wait_bounded(&empty[s], ph ^ 1u, kGmWaitNs)) {
                    give_up();
                    break;
                }
                mbar_arrive_expect_tx(&full[s], tx);
                const uint32_t st = base + s * sbytes;
                const int kb = kb0 + i;
                gm_tma_2d(st, &tmx, kb * 64, tok0, &full[s]);
                gm_tma_2d(st + wpoff, &tmw0, kb * 8, row0, &full[s]);
                if (nsub == 2) gm_tma_2d(st + wpoff + kGmWpBytes, kSwiglu ? &tmw1 : &tmw0, kb * 8, row1, &full[s]);
                issued = i + 1;
            }
            // never leave with copies in flight: wait (bounded) for the last stages armed
            for (int i = max(0, issued - stages); i < issued; ++i)
                mbar_wait_bounded(&full[i % stages], (unsigned)(i / stages) & 1u, kGmWaitNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (one thread)
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | ((uint32_t)(a.bn >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
            for (int i = 0; i < nkb && !*abort_flag; ++i) {
                const int s = i % stages;
                const unsigned ph = (unsigned)(i / stages) & 1u;
                const int as = i % kGmAtStages;
                const unsigned aph = (unsigned)(i / kGmAtStages) & 1u;
                if (!mbar_wait_bounded(&full[s], ph, kGmWaitNs) ||
                    !(AT ? mbar_wait_bounded(&afull[as], aph, kGmWaitNs) : mbar_wait_bounded(&adone[s], ph, kGmWaitNs))) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t st = base + s * sbytes;
#pragma unroll
                for (int sub = 0; sub < 2; ++sub) {
                    if (sub < nsub) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            if constexpr (AT)
                                tc_mma_f16_ta(tmem + (uint32_t)(sub * a.bn),
                                              tmem + kGmAtCol + (uint32_t)((as * 2 + sub) * 32 + k * 8),
                                              sw128_desc(st + k * 32), idesc, (uint32_t)(i | k));
                            else
                                tc_mma_f16(tmem + (uint32_t)(sub * a.bn),
                                           sw128_desc(st + bbytes + sub * kGmSubBytes + k * 32), sw128_desc(st + k * 32),
                                           idesc, (uint32_t)(i | k));
                        }
                    }
                }
                tc_commit(&empty[s]);
                if constexpr (AT) tc_commit(&aempty[as]);
            }
            tc_commit(&accf);   // completes when every MMA issued above has
        }
        __syncwarp();
    } else {
        // ---------------- expansion of the packed weights into the A operand
        const int d2 = tid - 64;
        const int sub = d2 >> 7;                 // sub-tile this warp expands
        // row this thread expands: with the TMEM operand it must be the TMEM lane the warp may write
        const int d = AT ? (warp & 3) * 32 + lane : (d2 & 127);
        const bool work = sub < nsub;
        const int groups = a.K / 128;
        const __half* sr = work ? (sub == 0 ? a.s0 + (size_t)(row0 + d) * groups
                                            : (kSwiglu ? a.s1 : a.s0) + (size_t)(row1 + d) * groups)
                                : a.s0;
        __half nxt = sr[kb0 >> 1];
        __half cur = nxt;
        for (int i = 0; i < nkb && !(AT ? __any_sync(0xffffffffu, *abort_flag) : *abort_flag); ++i) {
            const int s = i % stages;
            const unsigned ph = (unsigned)(i / stages) & 1u;
            const int kb = kb0 + i;
            if (i == 0 || (kb & 1) == 0) {   // a new scale group: take the prefetched scale, fetch the next
                cur = nxt;
                const int g = (kb >> 1) + 1;
                if (g < groups) nxt = sr[g];
            }
            // with the TMEM operand, verdicts are warp-uniform: tcgen05.st needs the whole warp
            const bool got = mbar_wait_bounded(&full[s], ph, kGmWaitNs);
            if (!(AT ? __all_sync(0xffffffffu, got) : got)) {
                give_up();
                break;
            }
            const int as = i % kGmAtStages;
            if constexpr (AT) {   // the TMEM stage is free once the MMAs of K-block i - 2 completed
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&aempty[as], ((unsigned)(i / kGmAtStages) & 1u) ^ 1u,
                                                               kGmWaitNs))) {
                    give_up();
                    break;
                }
                tc_fence_after();
            }
            if constexpr (AT) {
              if (work) {
                const uint32_t st = base + s * sbytes;
                const __half2 s2 = __half2half2(cur);
                const uint32_t wp = st + wpoff + sub * kGmWpBytes + d * 32;
                // rows are 32 bytes apart: lanes 4..7 of each 8-lane phase take the other
                // 16-byte half first, so every phase covers all 32 banks once
                const uint32_t hsel = ((uint32_t)d >> 2) & 1u;
                const uint4 wa = lds128(wp + hsel * 16), wb = lds128(wp + (hsel ^ 1u) * 16);
                const uint4 w0 = hsel ? wb : wa, w1 = hsel ? wa : wb;
                const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                uint32_t cols[32];   // column c holds K elements 2c, 2c + 1 of this row
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = expand_word(words[c], s2);
                    cols[4 * c + 0] = v.x;
                    cols[4 * c + 1] = v.y;
                    cols[4 * c + 2] = v.z;
                    cols[4 * c + 3] = v.w;
                }
                tmem_st32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + kGmAtCol + (uint32_t)((as * 2 + sub) * 32), cols);
                tc_fence_before();
              }
            } else if (work) {
                const uint32_t st = base + s * sbytes;
                const __half2 s2 = __half2half2(cur);
                const uint32_t wp = st + wpoff + sub * kGmWpBytes + d * 32;
                // rows are 32 bytes apart: lanes 4..7 of each 8-lane phase take the other
                // 16-byte half first, so every phase covers all 32 banks once
                const uint32_t hsel = ((uint32_t)d >> 2) & 1u;
                const uint4 wa = lds128(wp + hsel * 16), wb = lds128(wp + (hsel ^ 1u) * 16);
                const uint4 w0 = hsel ? wb : wa, w1 = hsel ? wa : wb;
                const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                const uint32_t arow = st + bbytes + sub * kGmSubBytes + (d >> 3) * 1024 + (d & 7) * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = expand_word(words[c], s2);
                    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(arow + ((c ^ (d & 7)) << 4)),
                                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                                 : "memory");
                }
                fence_proxy_async();   // generic-proxy stores -> visible to the tensor core's async proxy
            }
            mbar_arrive(AT ? &afull[as] : &adone[s]);
        }

        // ---------------- epilogue: accumulators from TMEM
        const int q = warp & 3;              // lane quarter this warp may read
        const int r = q * 32 + lane;         // row within the sub-tiles
        const int half = sub;                // 16-column chunks half, half + 2, ...
        // one verdict for all eight warps
        const bool ok = bar_and(1, 256, mbar_wait_bounded(&accf, 0, kGmWaitNs) && !*abort_flag);
        if (!ok) give_up();
        tc_fence_after();
        const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
        if (ok) {
            if (a.splits == 1) {
                for (int c = half * 16; c < a.bn; c += 32) {
                    float v0[16], v1[16];
                    tmem_ld16(tl + c, v0);
                    if (nsub == 2) tmem_ld16(tl + a.bn + c, v1);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int tok = tok0 + c + j;
                        if (tok < a.n) gemm_epilogue_one<EPI>(a, tok, row0, row1, r, nsub, v0[j], nsub == 2 ? v1[j] : 0.f);
                    }
                }
            } else {   // this split's partial sums: gate | up (or the two row blocks) at their output columns
                const int nout = kSwiglu ? 2 * a.N : a.N;
                const int col1 = kSwiglu ? a.N + row0 : row1;
                float* mine = a.part + (size_t)split * a.n * nout;
                for (int c = half * 16; c < a.bn; c += 32) {
                    float v0[16], v1[16];
                    tmem_ld16(tl + c, v0);
                    if (nsub == 2) tmem_ld16(tl + a.bn + c, v1);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int tok = tok0 + c + j;
                        if (tok < a.n) {
                            __stcg(mine + (size_t)tok * nout + row0 + r, v0[j]);
                            if (nsub == 2) __stcg(mine + (size_t)tok * nout + col1 + r, v1[j]);
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
    }
}
// Split-K merge: out = epilogue(sum over splits in order of part[s][t][c]);
// four outputs per thread (columns are multiples of 128).
template <int EPI>
__global__ void __launch_bounds__(256) w4_gemm_reduce_kernel(const GemmArgs a) {
    const int nq = a.N / 4;   // output columns / 4
    const long long total = (long long)a.n * nq;
    const int nout = EPI == G_SWIGLU ? 2 * a.N : a.N;
    const size_t stride = (size_t)a.n * nout;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(i / nq), c = (int)(i - (long long)t * nq) * 4;
        const float* p = a.part + (size_t)t * nout + c;
        float4 g = __ldcg(reinterpret_cast<const float4*>(p));
        float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
        if (EPI == G_SWIGLU) u = __ldcg(reinterpret_cast<const float4*>(p + a.N));
        for (int sp = 1; sp < a.splits; ++sp) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(p + sp * stride));
            g.x += v.x; g.y += v.y; g.z += v.z; g.w += v.w;
            if (EPI == G_SWIGLU) {
                const float4 w = __ldcg(reinterpret_cast<const float4*>(p + sp * stride + a.N));
                u.x += w.x; u.y += w.y; u.z += w.z; u.w += w.w;
            }
        }
        if constexpr (EPI == G_SWIGLU) {
            __half* o = a.act + (size_t)t * a.N + c;
            reinterpret_cast<__half2*>(o)[0] = __floats2half2_rn(gm_silu_mul(g.x, u.x), gm_silu_mul(g.y, u.y));
            reinterpret_cast<__half2*>(o)[1] = __floats2half2_rn(gm_silu_mul(g.z, u.z), gm_silu_mul(g.w, u.w));
        } else {
            float4* y = reinterpret_cast<float4*>(a.y + (size_t)t * a.ldy + c);
            if constexpr (EPI == G_RESID) {
                const float4 o = *y;
                g.x += o.x; g.y += o.y; g.z += o.z; g.w += o.w;
            }
            *y = g;
        }
    }
}
#endif  // W4_DEFINE_GEMM_TC05_KERNEL

// ---------------------------------------------------------------- host side
struct GemmPlan {
    GemmArgs a;
    dim3 grid;
    size_t smem;
};

// Tiles of 256 weight rows (or 128 gate + 128 up rows) by bn tokens; split K
// so that about one CTA per SM is busy when the tiles alone are too few,
// keeping at least eight 64-column blocks per split.
inline GemmPlan gemm_plan(int epi, int n, int N, int K, int sms, int a_tmem = 1, int tile_rows = 0) {
    GemmPlan p = {};
    GemmArgs& a = p.a;
    a.n = n;
    a.N = N;
    a.K = K;
    a.a_tmem = a_tmem;
    const int bn_max = a_tmem ? kGmAtBnMax : 256;
    a.bn = n >= bn_max ? bn_max : (n + 15) / 16 * 16;
    a.tok_tiles = (n + a.bn - 1) / a.bn;
    const int kbs = K / 64;
    auto splits_for = [&](int tiles) {
        const int sp = tiles >= sms ? 1 : sms / tiles;
        return std::max(1, std::min(sp, kbs / 8));
    };
    if (epi == G_SWIGLU) {
        a.tile_rows = 128;   // 128 gate rows + the same 128 up rows
    } else if (tile_rows == 128 || tile_rows == 256) {
        a.tile_rows = tile_rows;
    } else {   // automatic: two sub-tiles share the activation tile -- measured faster than 128-row
               // tiles on every 7B shape, even where it needs more K splits (n = 512: QKV, O, down)
        a.tile_rows = 256;
    }
    a.row_tiles = (N + a.tile_rows - 1) / a.tile_rows;
    const int tiles = a.tok_tiles * a.row_tiles;
    const int splits = splits_for(tiles);
    a.kb_per_split = (kbs + splits - 1) / splits;
    a.splits = (kbs + a.kb_per_split - 1) / a.kb_per_split;
    const uint32_t sb = gemm_stage_bytes(a.bn, a_tmem);
    a.stages = (int)std::min<size_t>(kGmMaxStages, (kGmSmemBudget - 1024) / sb);
    p.grid = dim3((unsigned)(tiles * a.splits));
    // at least 116 KB, so that one CTA holds an SM (and all of its TMEM) at a time
    p.smem = std::max<size_t>((size_t)a.stages * sb + 1024, 116 * 1024);
    return p;
}

inline size_t gemm_part_bytes(int epi, const GemmPlan& p) {
    const size_t nout = epi == G_SWIGLU ? 2 * (size_t)p.a.N : (size_t)p.a.N;
    return p.a.splits > 1 ? (size_t)p.a.splits * p.a.n * nout * sizeof(float) : 0;
}

// Activations fp16 [n][k] as a 2-D tensor: boxes of 64 columns x box_rows rows,
// 128-byte swizzle, rows past n read as zeros (attention.cu).
w4_status make_act_tensor_map(CUtensorMap* map, const void* x, int n, int k, int box_rows);

// Operand placement of the expanded weights for new plans (w4_gemm_tune): 1 TMEM, 0 shared memory;
// weight rows per tile (w4_gemm_tune_tile_rows): 0 automatic, 128 or 256.
int gemm_a_tmem();
int gemm_tile_rows();

// The GEMM kernel, and with split K the merge kernel after it (two launches);
// reduce = false leaves the split partials [splits][n][N] in a.part for the
// caller to add (G_STORE and G_RESID only).
cudaError_t gemm_tc05_launch(int epi, const GemmPlan& p, const CUtensorMap& tmx, const CUtensorMap& tmw0,
                             const CUtensorMap& tmw1, cudaStream_t st, bool reduce = true);

}  // namespace w4
