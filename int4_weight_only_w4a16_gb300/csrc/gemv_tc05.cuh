// Batched W4A16 GEMV (1 <= M <= 16 activation rows) on the 5th-generation
// tensor cores.
//
//   y[m][r] = sum_g s[r][g] * ( sum_{k in group g} x[m][k] * q[r][k] )  (+ bias[r]) (+ residual[m][r])
//
// Same operation as gemv.cuh ("How to build your own LLM runtime from scratch
// (Towards Data Science)", "What it actually builds": GEMVs over INT4
// group-128 weights with fp16 activations and the dequantization fused into
// the product).  With several activation rows this is a dense contraction;
// tcgen05.mma (M = 128 weight rows, N = 16 activation rows, K = 16) runs it,
// and N = 16 covers every batch of 1 to 16 (missing rows are zeros).
//
// Exact in the weights, as the other GEMVs: the tensor cores multiply the
// INT4 codes themselves (q in [-8, 7] is an exact fp16 value, expanded as
// (u | 0x6400) - 1032), every product is exact in fp32, each scale group has
// its own accumulator, and the group's fp16 scale multiplies the group's fp32
// sums in the epilogue: nothing is rounded before fp32.
//
// A CTA owns 128 weight rows over a range of whole groups (split K when the
// row tiles alone would leave SMs idle).  A ring stage holds four groups: the
// packed words of the 128 rows ([4][128][64 B], 64-byte swizzle; 256
// contiguous bytes of each row) and the activations ([8][16 rows][64] fp16
// slices, 128-byte swizzle; rows past M read as zeros), each one TMA copy of
// a 3-D view:
//   warp 0      TMA producer, kTgStages stages ahead;
//   warps 1, 2  TMEM allocation (warp 1), then one thread each issuing the
//               MMAs of the even (warp 1) or odd (warp 2) groups: eight per
//               group (A from TMEM, B the group's activations), one commit per
//               group (its operand slot and accumulator) and one per stage;
//   warps 4..7, 12..15  expansion of the even and the odd groups, one weight
//               row per thread (= TMEM lane): a group's 16 words become 64
//               columns of fp16 code pairs, written with tcgen05.st (no
//               shared-memory round trip);
//   warps 8..11 epilogue, the same rows: per group 16 accumulator columns
//               (tcgen05.ld) times the scale into 16 running sums; at the end
//               the outputs, or the split's partial sums, of which the last
//               CTA of the tile adds every split in split order (deterministic).
// Every mbarrier wait is bounded; on expiry the CTA records
// W4_DEVERR_TIMEOUT, every role stops, and TMEM is freed after the MMAs
// issued have drained.
#pragma once

#include "gemv.cuh"
#include "tc05.cuh"

namespace w4 {

constexpr int kTgThreads = 512;
constexpr int kTgStages = 4;              // ring stages
constexpr int kTgGroupsPerStage = 4;
constexpr int kTgASlots = 4;              // expanded groups in TMEM (64 columns each)
constexpr int kTgDSlots = 4;              // group accumulators in TMEM (16 columns each)
constexpr int kTgGBars = 8;               // per-group completion barriers (a ring)
constexpr int kTgWBytes = 128 * 64;       // one group of 128 rows: 16 packed words a row
constexpr int kTgXBytes = 2 * 16 * 128;   // one group's activations: 16 rows x 128 fp16
constexpr int kTgStageBytes = kTgGroupsPerStage * (kTgWBytes + kTgXBytes);   // 48 KB
constexpr uint32_t kTgTmemCols = 512;
constexpr uint64_t kTgWaitNs = 1000000000ull;

struct TgArgs {
    int M, N, K;
    int tiles;            // 128-row tiles
    int splits, gps;      // K in `splits` ranges of gps groups
    const __half* s;      // scales [N][K/128]
    const __half* bias;   // [N] or null
    const __half* resid;  // [M][N] or null
    __half* y;            // [M][N]
    float* part;          // split partials [splits][M][N]
    unsigned* counters;   // [tiles] split tickets, zero between calls
    int* errword;
};

constexpr size_t kTgSmem = 1024 + (size_t)kTgStages * kTgStageBytes;   // 193 KB: one CTA per SM

#ifdef W4_DEFINE_GEMV_TC05_KERNEL
__global__ void __launch_bounds__(kTgThreads, 1)
gemv_tc05_kernel(const TgArgs a, const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx) {
    extern __shared__ unsigned char tg_raw[];
    __shared__ uint64_t sfull[kTgStages], sdone[kTgStages], gdone[kTgGBars];
    __shared__ uint64_t adone[kTgASlots], dempty[kTgDSlots];
    __shared__ uint64_t drain[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort, s_last;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x % a.tiles, split = blockIdx.x / a.tiles;
    const int row0 = tile * 128;
    const int G = a.K >> 7;
    const int g0 = split * a.gps;
    const int ng = min(G, g0 + a.gps) - g0;
    const int nst = (ng + kTgGroupsPerStage - 1) / kTgGroupsPerStage;
    const uint32_t ring = (smem_u32(tg_raw) + 1023u) & ~1023u;   // [kTgStages][weights | activations]

    if (tid == 0) {
        for (int i = 0; i < kTgStages; ++i) {
            mbar_init(&sfull[i], 1);      // the producer's arrival + the stage's bytes
            mbar_init(&sdone[i], 2);      // one commit per MMA issuer, after its last group of the stage
        }
        for (int i = 0; i < kTgGBars; ++i) mbar_init(&gdone[i], 1);       // the group's MMAs (commit)
        for (int i = 0; i < kTgASlots; ++i) mbar_init(&adone[i], 128);    // every expansion thread
        for (int i = 0; i < kTgDSlots; ++i) mbar_init(&dempty[i], 4);     // one arrival per epilogue warp
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmw)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmx)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(kTgTmemCols)
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
        // ---------------- TMA producer.  Stage t % kTgStages is refilled once both MMA
        // issuers have committed stage t - kTgStages (so its words were expanded, too).
        if (lane == 0) {
            pdl_wait();   // the activations may come from the previous kernel
            int issued = 0;
            for (int t = 0; t < nst && !*abort_flag; ++t) {
                const int ps = t % kTgStages;
                if (t >= kTgStages &&
                    !mbar_wait_bounded(&sdone[ps], ((unsigned)(t / kTgStages) & 1u) ^ 1u, kTgWaitNs)) {
                    give_up();
                    break;
                }
                const uint32_t st = ring + (uint32_t)ps * kTgStageBytes;
                const int g = g0 + t * kTgGroupsPerStage;
                mbar_arrive_expect_tx(&sfull[ps], kTgStageBytes);
                gm_tma_3d(st, &tmw, 0, row0, g, &sfull[ps]);
                gm_tma_3d(st + kTgGroupsPerStage * kTgWBytes, &tmx, 0, 0, 2 * g, &sfull[ps]);
                issued = t + 1;
            }
            // never leave with copies in flight
            for (int t = max(0, issued - kTgStages); t < issued; ++t)
                mbar_wait_bounded(&sfull[t % kTgStages], (unsigned)(t / kTgStages) & 1u, kTgWaitNs);
        }
    } else if (warp == 1 || warp == 2) {
        // ---------------- MMA issuers: warp 1 the even groups, warp 2 the odd ones (one
        // issuing thread keeps the tensor pipe about half busy at N = 16)
        const int e = warp - 1;
        if (lane == 0) {
            // kind::f16: fp32 accumulator, fp16 A and B, both K-major, N = 16, M = 128
            const uint32_t idesc = (1u << 4) | ((uint32_t)(16 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
            for (int i = e; i < ng && !*abort_flag; i += 2) {
                const int s = i % kTgASlots;
                if (!mbar_wait_bounded(&adone[s], (unsigned)(i / kTgASlots) & 1u, kTgWaitNs)) {
                    give_up();
                    break;
                }
                // the epilogue has taken group i - kTgDSlots out of this accumulator
                if (i >= kTgDSlots &&
                    !mbar_wait_bounded(&dempty[s], ((unsigned)(i / kTgDSlots) & 1u) ^ 1u, kTgWaitNs)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const int t = i / kTgGroupsPerStage, j = i % kTgGroupsPerStage;
                const uint32_t ta = tmem + (uint32_t)(s * 64), td = tmem + 256u + (uint32_t)(s * 16);
                const uint32_t xb = ring + (uint32_t)(t % kTgStages) * kTgStageBytes + kTgGroupsPerStage * kTgWBytes +
                                    (uint32_t)j * kTgXBytes;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    tc_mma_f16_ta(td, ta + 8u * k, sw128_desc(xb + (k >> 2) * 2048u + (k & 3) * 32u), idesc,
                                  (uint32_t)k);
                tc_commit(&gdone[i % kTgGBars]);
                // this issuer's last group of the stage
                if (j >= 2 || i + 2 >= ng) tc_commit(&sdone[t % kTgStages]);
            }
            tc_commit(&drain[e]);   // completes once every MMA this thread issued has
            mbar_wait_bounded(&drain[e], 0, kTgWaitNs);
        }
        __syncwarp();
    } else if ((warp >= 4 && warp < 8) || warp >= 12) {
        // ---------------- expansion: row er of the tile, TMEM lane er; warps 4..7 take the
        // even groups (operand slots 0, 2), warps 12..15 the odd ones (slots 1, 3)
        const int er = (warp & 3) * 32 + lane;
        const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t sw = (uint32_t)(er >> 1) & 3u;   // the 64-byte swizzle of this row's 16-byte chunks
        for (int i = warp >= 12 ? 1 : 0; i < ng; i += 2) {
            const int t = i / kTgGroupsPerStage, j = i % kTgGroupsPerStage, s = i % kTgASlots;
            const int ps = t % kTgStages;
            // tcgen05.st needs the whole warp: one verdict per warp
            bool ok = mbar_wait_bounded(&sfull[ps], (unsigned)(t / kTgStages) & 1u, kTgWaitNs);
            if (!__all_sync(0xffffffffu, ok && !*abort_flag)) {
                if (!ok) give_up();
                break;
            }
            const uint32_t rp = ring + (uint32_t)ps * kTgStageBytes + (uint32_t)j * kTgWBytes + (uint32_t)er * 64u;
            uint32_t col[64];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 q = lds128(rp + (((uint32_t)c ^ sw) << 4));
                const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {   // word 4c + w: K values 8(4c+w) .. +7 as four fp16 pairs
                    const uint4 v = expand_codes(wd[w]);
                    col[16 * c + 4 * w + 0] = v.x;
                    col[16 * c + 4 * w + 1] = v.y;
                    col[16 * c + 4 * w + 2] = v.z;
                    col[16 * c + 4 * w + 3] = v.w;
                }
            }
            // the operand slot is free once the MMAs of group i - kTgASlots have completed
            if (i >= kTgASlots) {
                const int jj = i - kTgASlots;
                ok = mbar_wait_bounded(&gdone[jj % kTgGBars], (unsigned)(jj / kTgGBars) & 1u, kTgWaitNs);
                if (!__all_sync(0xffffffffu, ok)) {
                    give_up();
                    break;
                }
            }
            tc_fence_after();
            const uint32_t ta = tmem + lanes + (uint32_t)(s * 64);
            const uint32_t(&c0)[32] = *reinterpret_cast<const uint32_t(*)[32]>(&col[0]);
            const uint32_t(&c1)[32] = *reinterpret_cast<const uint32_t(*)[32]>(&col[32]);
            tmem_st32(ta, c0);
            tmem_st32(ta + 32u, c1);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&adone[s]);
        }
    } else if (warp >= 8) {
        // ---------------- epilogue (warps 8..11): row r of the tile, TMEM lane r
        const int q = warp & 3, r = q * 32 + lane, row = row0 + r;
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        const __half* srow = a.s + (size_t)min(row, a.N - 1) * G + g0;
        float acc[16];
#pragma unroll
        for (int n = 0; n < 16; ++n) acc[n] = 0.f;
        float sc_next = __half2float(srow[0]);
        bool ok = true;
        for (int i = 0; i < ng; ++i) {
            const int d = i % kTgDSlots;
            const float sc = sc_next;
            if (i + 1 < ng) sc_next = __half2float(srow[i + 1]);
            // tcgen05.ld needs the whole warp: one verdict per warp
            if (!__all_sync(0xffffffffu,
                            mbar_wait_bounded(&gdone[i % kTgGBars], (unsigned)(i / kTgGBars) & 1u, kTgWaitNs))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t v[16];
            tmem_ld16(tmem + lanes + 256u + (uint32_t)(d * 16), v);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&dempty[d]);
#pragma unroll
            for (int n = 0; n < 16; ++n) acc[n] = fmaf(sc, __uint_as_float(v[n]), acc[n]);
        }
        if (!ok) give_up();
        ok = bar_and(1, 128, ok && !*abort_flag);   // one verdict for the four epilogue warps
        if (ok) {
            const bool in = row < a.N;
            if (a.splits > 1) {
#pragma unroll
                for (int n = 0; n < 16; ++n)
                    if (n < a.M && in) __stcg(a.part + ((size_t)split * a.M + n) * a.N + row, acc[n]);
                __threadfence();
                named_sync(1, 128);
                if (tid == 256) {
                    const unsigned tk = atomicAdd(&a.counters[tile], 1u);
                    const int last = tk == (unsigned)a.splits - 1;
                    if (last) {
                        __threadfence();
                        a.counters[tile] = 0u;   // ready for the next call
                    }
                    s_last = last;
                }
                named_sync(1, 128);
                if (s_last) {
                    // every split's partials of this row, in split order; a split's loads all
                    // issue before any is added
#pragma unroll
                    for (int n = 0; n < 16; ++n) acc[n] = 0.f;
                    for (int sp = 0; sp < a.splits; ++sp) {
                        float v[16];
#pragma unroll
                        for (int n = 0; n < 16; ++n)
                            v[n] = (n < a.M && in) ? __ldcg(a.part + ((size_t)sp * a.M + n) * a.N + row) : 0.f;
#pragma unroll
                        for (int n = 0; n < 16; ++n) acc[n] += v[n];
                    }
                }
            }
            if (a.splits == 1 || s_last) {
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    if (n < a.M && in) {
                        float v = acc[n];
                        if (a.bias) v += __half2float(a.bias[row]);
                        if (a.resid) v += __half2float(a.resid[(size_t)n * a.N + row]);
                        a.y[(size_t)n * a.N + row] = __float2half_rn(v);
                    }
                }
            }
        }
    }
    // every role meets every other at the end, then TMEM goes back
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTgTmemCols) : "memory");
    }
}
#endif  // W4_DEFINE_GEMV_TC05_KERNEL

// ---------------------------------------------------------------- host side
struct TgPlan {
    TgArgs a;
    dim3 grid;
    size_t smem;
};

// 128-row tiles; K split (in whole groups) so that tiles x splits is near the
// SM count when the tiles alone are too few.
inline TgPlan tg_plan(int m, int n, int k) {
    TgPlan p = {};
    TgArgs& a = p.a;
    a.M = m;
    a.N = n;
    a.K = k;
    a.tiles = (n + 127) / 128;
    const int G = k / 128;
    int splits = (2 * sm_count() + a.tiles) / (2 * a.tiles);   // rounded SMs per tile
    splits = std::max(1, std::min(splits, G));
    a.gps = (G + splits - 1) / splits;
    a.splits = (G + a.gps - 1) / a.gps;
    p.grid = dim3((unsigned)(a.tiles * a.splits));
    p.smem = kTgSmem;
    return p;
}

// split partials, then the tile tickets (zero before the first call)
inline size_t tg_ws_bytes(const TgPlan& p) {
    if (p.a.splits == 1) return 0;
    return ((size_t)p.a.splits * p.a.M * p.a.N * sizeof(float) + 255) / 256 * 256 + (size_t)p.a.tiles * sizeof(unsigned);
}

cudaError_t tg_launch(const TgPlan& p, const CUtensorMap& tmw, const CUtensorMap& tmx, cudaStream_t st);

}  // namespace w4
