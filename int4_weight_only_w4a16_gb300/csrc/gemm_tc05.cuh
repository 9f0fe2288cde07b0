// W4A16 GEMM for the prompt pass on the 5th-generation tensor cores.
//
//   Y[t][r] = sum_g s[r][g] * ( sum_{k in group g} X[t][k] * q[r][k] )     t < n tokens, r < N rows
//
// "How to build your own LLM runtime from scratch (Towards Data Science)",
// section "What it actually builds": INT4 group-128 weights against fp16
// activations with fp32 accumulation; with n prompt rows this is a dense
// contraction, so it runs on tcgen05.mma.
//
// The product is exact in the weights: the tensor cores multiply the INT4
// codes themselves (q in [-8, 7] is an exact fp16 value), each 128-column
// scale group accumulates into its own TMEM accumulator, and the group's
// fp16 scale is applied in fp32 by the epilogue warps, which keep the running
// sums in registers.  Every product is exact and only fp32 sums round, as in
// the decode GEMVs; no weight is rounded to fp16 as q * s.
//
// One CTA owns 128 weight rows (128 rows of one matrix, or 64 gate rows and
// the same 64 up rows, interleaved so that A row 2j is gate row j and A row
// 2j + 1 up row j) and bn in {64, 128, 256} tokens, over a range of whole
// scale groups of K (split K when the tiles alone would leave SMs idle, or
// stream-K, where one CTA per SM takes an equal run of (tile, group) units and
// may finish one tile and start the next; or, when the tiles outnumber the
// SMs, persistent: one CTA per SM walks an equal run of whole tiles):
//   warp 0      TMA producer: the activation tile [bn][64] (128-byte swizzle)
//               and the packed weight tile [128][8 words] per stage;
//   warp 1      allocates TMEM (two group accumulators of bn fp32 columns)
//               and, from one thread, issues tcgen05.mma (M = 128, N = bn,
//               K = 16): eight per scale group into accumulator g % 2, then
//               commits the group to the epilogue;
//   warps 4..7  expand the packed words to fp16 codes straight into the
//               canonical K-major 128-byte-swizzled operand layout;
//   warps 8..15 add each group's accumulator, times its scale, into their
//               running sums (tcgen05.ld; each warp reads the lane quarter it
//               may read, warps 8..11 taking the first half of the columns and
//               12..15 the second); at the end of each tile they store, add
//               into the residual, or write SiLU(gate) * up in fp16 (the
//               lanes 2j, 2j + 1 holding gate and up row j swap halves of the
//               columns by one shuffle).  With split K or
//               stream-K every piece of a tile stores its partial sums, and the
//               next kernel adds the pieces in slot order (deterministic).
// The roles sit in separate warpgroups so that setmaxnreg can give the
// running sums (128 fp32 registers per thread) the registers the producer and
// expansion warps do not need.
// Every mbarrier wait is bounded in wall time; on expiry the CTA records
// W4_DEVERR_TIMEOUT, drains what it issued (bounded) and frees its TMEM.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc05.cuh"

namespace w4 {

constexpr int kGmThreads = 512;          // four warpgroups
constexpr int kGmLaunchRegs = 128;       // registers per thread at launch (64 K / 512)
constexpr int kGmLowRegs = 80;           // producer/MMA and expansion warpgroups after setmaxnreg
constexpr int kGmHighRegs = 176;         // epilogue warpgroups: 2 x (176 - 128) = 2 x (128 - 80)
constexpr int kGmMaxStages = 4;
constexpr int kGmABytes = 128 * 128;        // one 128-row x 64-K fp16 operand tile
constexpr int kGmWpBytes = 128 * 32;        // its packed source: 128 rows x 8 words
constexpr int kGmPStages = 4;               // packed tiles in flight (their own ring, ahead of the stages)
constexpr size_t kGmSmemBudget = 220 * 1024;

enum { G_STORE = 0, G_RESID = 1, G_SWIGLU = 2 };

struct GemmArgs {
    int n, N, K;               // tokens, rows of each weight matrix, columns
    int bn;                    // tokens per tile: 64, 128 or 256
    int tok_tiles, row_tiles;  // tiles = row_tiles * tok_tiles
    int splits, kb_per_split;  // K ranges of kb_per_split 64-column blocks (even: whole scale groups)
    int stream, ctas;          // 1: stream-K, ctas CTAs share the (tile, scale group) units equally;
                               // 2: persistent, ctas CTAs take equal runs of whole tiles
    int stages;
    const uint32_t* w0;        // packed words [N][K/8] of matrix 0 (L2 prefetch; the tiles come by TMA)
    const uint32_t* w1;        // of matrix 1 (SwiGLU: up)
    const __half* s0;          // scales fp16 [N][K/128] of matrix 0
    const __half* s1;          // of matrix 1 (SwiGLU: up)
    float* y;                  // G_STORE / G_RESID: fp32 [n][ldy], columns [0, N)
    int ldy;
    __half* act;               // G_SWIGLU: fp16 [n][N]
    float* part;               // split-K partials fp32 [splits][n][nout]
    int* errword;
};

// Work units are (tile, scale group) pairs in tile-major order, gt = K / 128
// groups per tile.  Split K gives CTA (split, tile) the groups of one K range of
// one tile.  Stream-K gives CTA c the units [c U / ctas, (c + 1) U / ctas) of
// all U = tiles * gt: a CTA may finish one tile and start the next, and each
// tile is covered by consecutive CTAs, piece q of tile t belonging to CTA
// gm_cta_of(t * gt) + q.  Either way a piece's partial sums go to slot q (the
// split) of [splits][n][N], and with stream-K the CTA holding piece 0 of a
// tile zero-fills the slots its tile leaves unused, so the next kernel adds a
// fixed number of slots in slot order (deterministic).
__host__ __device__ inline int gm_cta_of(long long u, long long units, int ctas) {
    return (int)(((u + 1) * ctas + units - 1) / units) - 1;   // the CTA whose range holds unit u
}

__host__ __device__ inline uint32_t gemm_b_bytes(int bn) { return (uint32_t)((bn * 128 + 1023) / 1024 * 1024); }
// a stage: the activation tile and the expanded weight tile of one K-block (the
// packed words travel in a ring of their own, kGmPStages deep, after the stages)
__host__ __device__ inline uint32_t gemm_stage_bytes(int bn) { return gemm_b_bytes(bn) + kGmABytes; }
constexpr uint32_t kGmPRingBytes = (uint32_t)kGmPStages * kGmWpBytes;
__host__ __device__ inline uint32_t gemm_tmem_cols(int bn) { return (uint32_t)(2 * bn); }   // 128, 256 or 512

#ifdef W4_DEFINE_GEMM_TC05_KERNEL
constexpr uint64_t kGmWaitNs = 1000000000ull;

__device__ __forceinline__ float gm_silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// Epilogue warps: running sums of 128 fp32 columns per thread at most (bn / 2
// columns of one TMEM lane).
constexpr int kGmAccCols = 128;

// Warp roles, one warpgroup each so that setmaxnreg (warpgroup-wide) can move
// registers to the running sums:
//   warpgroup 0: warp 0 TMA producer, warp 1 TMEM allocation and MMA issue
//                (warps 2, 3 idle);
//   warpgroup 1: expansion of the packed codes, one A row per thread;
//   warpgroups 2, 3: the scaled group sums (warp w reads TMEM lane quarter
//                w % 4; warpgroup 2 the first half of the columns, 3 the second).
// The register pool balances exactly: 8 warps give up 128 - 80 registers per
// thread and 8 warps take 176 - 128.
template <int EPI>
__global__ void __launch_bounds__(kGmThreads, 1)
w4_gemm_tc05_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap tmx,
                    const __grid_constant__ CUtensorMap tmw0, const __grid_constant__ CUtensorMap tmw1) {
    extern __shared__ unsigned char gm_raw[];
    __shared__ uint64_t bfull[kGmMaxStages], adone[kGmMaxStages], empty[kGmMaxStages];
    __shared__ uint64_t pfull[kGmPStages], pempty[kGmPStages];
    __shared__ uint64_t gfull[2], gempty[2], drain;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wg = warp >> 2;
    const int cta = (int)blockIdx.x;
    const int tiles = a.row_tiles * a.tok_tiles;
    const int gt = a.K >> 7;             // scale groups per tile
    const long long units = (long long)tiles * gt;
    int u0, u1;                          // this CTA's units [u0, u1)
    if (a.stream == 2) {                 // whole tiles: every piece is a tile
        u0 = (int)((long long)cta * tiles / a.ctas) * gt;
        u1 = (int)((long long)(cta + 1) * tiles / a.ctas) * gt;
    } else if (a.stream) {
        u0 = (int)(cta * units / a.ctas);
        u1 = (int)((cta + 1) * units / a.ctas);
    } else {
        const int split = cta / tiles, tile = cta - split * tiles;
        u0 = tile * gt + split * (a.kb_per_split >> 1);
        u1 = min(tile * gt + gt, u0 + (a.kb_per_split >> 1));
    }
    const int ng = u1 - u0;              // scale groups, two 64-column K-blocks each
    const int nkb = 2 * ng;
    constexpr bool kSwiglu = EPI == G_SWIGLU;
    // first row of a tile in each matrix, and its first token
    auto row0_of = [&](int tile) { return (tile / a.tok_tiles) * (kSwiglu ? 64 : 128); };
    auto tok0_of = [&](int tile) { return (tile % a.tok_tiles) * a.bn; };
    const int stages = a.stages;
    const uint32_t bbytes = gemm_b_bytes(a.bn);
    const uint32_t sbytes = gemm_stage_bytes(a.bn);
    const uint32_t ncols = gemm_tmem_cols(a.bn);
    const uint32_t base = (smem_u32(gm_raw) + 1023u) & ~1023u;
    const uint32_t pbase = base + (uint32_t)stages * sbytes;   // the packed-tile ring

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&bfull[s], 1);
            mbar_init(&adone[s], 128);   // every expansion thread
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < kGmPStages; ++s) {
            mbar_init(&pfull[s], 1);
            mbar_init(&pempty[s], 128);  // every expansion thread, once it holds its words
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&gfull[b], 1);
            mbar_init(&gempty[b], 8);    // one arrive per epilogue warp
        }
        mbar_init(&drain, 1);
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

    if (wg < 2) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kGmLowRegs));
    if (warp == 0) {
        // ---------------- TMA producer of the activation tiles: stage s is refilled
        // once the MMAs of the K-block that last used it have completed
        if (lane == 0) {
            const uint32_t tx = (uint32_t)a.bn * 128;
            int issued = 0;
            for (int i = 0; i < nkb && !*abort_flag; ++i) {
                const int s = i % stages;
                const unsigned ph = (unsigned)(i / stages) & 1u;
                if (!mbar_wait_bounded(&empty[s], ph ^ 1u, kGmWaitNs)) {
                    give_up();
                    break;
                }
                const int u = u0 + (i >> 1), tile = u / gt;
                const int kb = 2 * (u - tile * gt) + (i & 1);
                mbar_arrive_expect_tx(&bfull[s], tx);
                gm_tma_2d(base + s * sbytes, &tmx, kb * 64, tok0_of(tile), &bfull[s]);
                issued = i + 1;
            }
            // never leave with copies in flight: wait (bounded) for the last stages armed
            for (int i = max(0, issued - stages); i < issued; ++i)
                mbar_wait_bounded(&bfull[i % stages], (unsigned)(i / stages) & 1u, kGmWaitNs);
        }
    } else if (warp == 2) {
        // ---------------- TMA producer of the packed weight tiles, in their own ring:
        // a slot is refilled as soon as every expansion thread holds its words, so the
        // expansion of a K-block never waits on HBM or L2 latency
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nkb && !*abort_flag; ++i) {
                const int sp = i % kGmPStages;
                const unsigned ph = (unsigned)(i / kGmPStages) & 1u;
                if (!mbar_wait_bounded(&pempty[sp], ph ^ 1u, kGmWaitNs)) {
                    give_up();
                    break;
                }
                mbar_arrive_expect_tx(&pfull[sp], kGmWpBytes);
                const uint32_t dst = pbase + sp * kGmWpBytes;
                const int u = u0 + (i >> 1), tile = u / gt;
                const int kb = 2 * (u - tile * gt) + (i & 1), row0 = row0_of(tile);
                if (kSwiglu) {   // 64 gate rows, then the same 64 up rows
                    gm_tma_2d(dst, &tmw0, kb * 8, row0, &pfull[sp]);
                    gm_tma_2d(dst + kGmWpBytes / 2, &tmw1, kb * 8, row0, &pfull[sp]);
                } else {
                    gm_tma_2d(dst, &tmw0, kb * 8, row0, &pfull[sp]);
                }
                issued = i + 1;
            }
            for (int i = max(0, issued - kGmPStages); i < issued; ++i)
                mbar_wait_bounded(&pfull[i % kGmPStages], (unsigned)(i / kGmPStages) & 1u, kGmWaitNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (one thread): scale group g into accumulator g % 2
        // One wait per scale group: every expansion thread waited for each K-block's
        // activation copy before arriving on its adone, and arrived on adone of the
        // first block before the second, so the second block's adone phase orders both
        // stages' copies and expanded rows before the MMAs (a barrier poll costs this
        // thread a few hundred cycles).
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | ((uint32_t)(a.bn >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
            for (int g = 0; g < ng && !*abort_flag; ++g) {
                const int b = g & 1;
                const int i0 = 2 * g, i1 = i0 + 1;
                const int s0 = i0 % stages, s1 = i1 % stages;
                // the epilogue has taken group g - 2 out of this accumulator
                if (g >= 2 && !mbar_wait_bounded(&gempty[b], ((unsigned)(g >> 1) & 1u) ^ 1u, kGmWaitNs)) {
                    give_up();
                    break;
                }
                if (!mbar_wait_bounded(&adone[s1], (unsigned)(i1 / stages) & 1u, kGmWaitNs)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * a.bn);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t st = base + (h ? s1 : s0) * sbytes;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        tc_mma_f16(d, sw128_desc(st + bbytes + k * 32), sw128_desc(st + k * 32), idesc,
                                   (uint32_t)(h | k));
                }
                tc_commit(&empty[s0]);
                tc_commit(&empty[s1]);
                tc_commit(&gfull[b]);
            }
            tc_commit(&drain);   // completes once every MMA issued above has
            mbar_wait_bounded(&drain, 0, kGmWaitNs);
        }
        __syncwarp();
    } else if (wg == 1) {
        // ---------------- expansion of the packed codes: A row er, all 8 words of a K-block
        const int er = tid - 128;
        // this row's packed words for the CTA's K ranges, into L2 now: the ring's TMA
        // copies then wait on L2, not HBM (one contiguous run per row and tile)
        for (int u = u0; u < u1;) {
            const int tile = u / gt, ue = min(u1, tile * gt + gt), row0 = row0_of(tile);
            const uint32_t* wrow = kSwiglu ? ((er & 1) ? a.w1 : a.w0) + (size_t)(row0 + (er >> 1)) * (a.K / 8)
                                           : a.w0 + (size_t)(row0 + er) * (a.K / 8);
            l2_prefetch_bulk(wrow + (u - tile * gt) * 16, (unsigned)((ue - u) * 64));
            u = ue;
        }
        // SwiGLU: A row 2j is gate row j and A row 2j + 1 up row j (the packed slot
        // holds the 64 gate rows, then the 64 up rows), so that one lane pair of the
        // epilogue holds both sums of an output row.  Slot rows are 32 bytes apart:
        // in every 8-lane phase half the lanes read the other 16-byte half first, so
        // the phase covers all 32 banks once.
        const int srow = kSwiglu ? ((er & 1) ? 64 + (er >> 1) : (er >> 1)) : er;
        const uint32_t hsel = kSwiglu ? ((uint32_t)er & 1u) : (((uint32_t)er >> 2) & 1u);
        for (int i = 0; i < nkb && !*abort_flag; ++i) {
            const int s = i % stages, sp = i % kGmPStages;
            const unsigned ph = (unsigned)(i / stages) & 1u, pph = (unsigned)(i / kGmPStages) & 1u;
            // this row's packed words, then their ring slot back to the producer
            if (!mbar_wait_bounded(&pfull[sp], pph, kGmWaitNs)) {
                give_up();
                break;
            }
            const uint32_t wp = pbase + sp * kGmWpBytes + srow * 32;
            const uint4 wa = lds128(wp + hsel * 16), wb = lds128(wp + (hsel ^ 1u) * 16);
            mbar_arrive(&pempty[sp]);
            const uint4 w0 = hsel ? wb : wa, w1 = hsel ? wa : wb;
            const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            // the stage's weight tile is free once the MMAs of its previous K-block completed
            if (!mbar_wait_bounded(&empty[s], ph ^ 1u, kGmWaitNs)) {
                give_up();
                break;
            }
            const uint32_t arow = base + s * sbytes + bbytes + (er >> 3) * 1024 + (er & 7) * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {   // 16-byte chunk c (8 K values) of the 128-byte row
                const uint4 v = expand_codes(words[c]);
                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(arow + ((c ^ (er & 7)) << 4)), "r"(v.x),
                             "r"(v.y), "r"(v.z), "r"(v.w)
                             : "memory");
            }
            fence_proxy_async();   // generic-proxy stores -> visible to the tensor core's async proxy
            // the K-block is ready for the MMAs once its activation tile has landed too
            if (!mbar_wait_bounded(&bfull[s], ph, kGmWaitNs)) {
                give_up();
                break;
            }
            mbar_arrive(&adone[s]);
        }
    }
        // every role meets every other at the end (bar.sync 0 counts all 512 threads)
        tc_fence_before();
        __syncthreads();
        if (warp == 1) {
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kGmHighRegs));
        // ---------------- scaled group sums: acc += s[r][g] * accumulator (g % 2)
        const int q = warp & 3;                // TMEM lane quarter this warp may read
        const int hc = wg - 2;                 // and its half of the columns
        const int r = q * 32 + lane;           // A row = TMEM lane of this thread
        const int hcols = a.bn >> 1;
        const int nout = kSwiglu ? 2 * a.N : a.N;
        // this row's scale of unit u (its tile's rows, its group)
        auto scale_of = [&](int u) {
            const int tile = u / gt, gi = u - tile * gt;
            if constexpr (kSwiglu)   // lane 2j: gate row j, lane 2j + 1: up row j
                return __half2float(((r & 1) ? a.s1 : a.s0)[(size_t)(row0_of(tile) + (r >> 1)) * gt + gi]);
            else
                return __half2float(a.s0[(size_t)(row0_of(tile) + r) * gt + gi]);
        };
        const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(hc * hcols);
        float acc[kGmAccCols];
#pragma unroll
        for (int j = 0; j < kGmAccCols; ++j) acc[j] = 0.f;
        float sc_next = scale_of(u0);
        bool ok = true;
        for (int g = 0; g < ng; ++g) {
            const int b = g & 1, u = u0 + g;
            const float sc = sc_next;
            if (g + 1 < ng) sc_next = scale_of(u + 1);
            // tcgen05.ld needs the whole warp: one verdict per warp
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&gfull[b], (unsigned)(g >> 1) & 1u, kGmWaitNs))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tb = tl + (uint32_t)(b * a.bn);
#pragma unroll
            for (int c = 0; c < kGmAccCols / 16; c += 2) {
                if (c * 16 < hcols) {   // warp-uniform; hcols is a multiple of 32
                    uint32_t v[16], u[16];
                    tmem_ld16x2(tb + (uint32_t)(c * 16), v, u);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        acc[c * 16 + j] = fmaf(sc, __uint_as_float(v[j]), acc[c * 16 + j]);
                        acc[c * 16 + 16 + j] = fmaf(sc, __uint_as_float(u[j]), acc[c * 16 + 16 + j]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&gempty[b]);
            if (a.splits == 1 && (g + 1 == ng || (u + 1) % gt == 0)) {
                // the end of a whole tile: its results; the MMAs of the next tile go on
                // meanwhile (into the other accumulator, then this one once it is free)
                const int tile = u / gt, row0 = row0_of(tile);
                const int ct0 = tok0_of(tile) + hc * hcols;   // first token of this thread's columns
                const bool wr = __all_sync(0xffffffffu, !*abort_flag);
                if constexpr (kSwiglu) {
                    // lanes 2j and 2j + 1 hold gate and up row j: lane 2j writes the even
                    // columns (tokens), lane 2j + 1 the odd ones
                    const int odd = lane & 1;
                    __half* o = a.act + row0 + (q * 32 + lane) / 2;
#pragma unroll
                    for (int j = 0; j < kGmAccCols; j += 2) {
                        const float mine0 = odd ? acc[j + 1] : acc[j], other0 = odd ? acc[j] : acc[j + 1];
                        const float got = __shfl_xor_sync(0xffffffffu, other0, 1);   // the partner's value
                        // even lane: gate = mine0 (column j), up = got; odd lane: up = mine0 (column j + 1), gate = got
                        const float gv = odd ? got : mine0, uv = odd ? mine0 : got;
                        const int t = ct0 + j + odd;
                        if (wr && j < hcols && t < a.n) o[(size_t)t * a.N] = __float2half_rn(gm_silu_mul(gv, uv));
                    }
                } else {
                    float* y = a.y + row0 + r;
#pragma unroll
                    for (int j = 0; j < kGmAccCols; ++j) {
                        if (wr && j < hcols && ct0 + j < a.n) {
                            float* yy = y + (size_t)(ct0 + j) * a.ldy;
                            if constexpr (EPI == G_RESID) *yy += acc[j];
                            else *yy = acc[j];
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < kGmAccCols; ++j) acc[j] = 0.f;
            }
            if (a.splits > 1 && (g + 1 == ng || (u + 1) % gt == 0)) {
                // the end of a piece: its partial sums (gate | up at their output
                // columns) into its slot; the MMAs of the next piece go on meanwhile
                const int tile = u / gt, row0 = row0_of(tile);
                const int ct0 = tok0_of(tile) + hc * hcols;   // first token of this thread's columns
                const int col = kSwiglu ? ((r & 1) ? a.N + row0 + (r >> 1) : row0 + (r >> 1)) : row0 + r;
                const int first = a.stream ? gm_cta_of((long long)tile * gt, units, a.ctas) : 0;
                const int slot = a.stream ? cta - first : cta / tiles;
                float* mine = a.part + (size_t)slot * a.n * nout + col;
                if (!*abort_flag) {
#pragma unroll
                    for (int j = 0; j < kGmAccCols; ++j)
                        if (j < hcols && ct0 + j < a.n) __stcg(mine + (size_t)(ct0 + j) * nout, acc[j]);
                }
                if (a.stream && slot == 0) {   // the slots no piece of this tile fills
                    const int pieces = gm_cta_of((long long)tile * gt + gt - 1, units, a.ctas) - first + 1;
                    for (int sp = pieces; sp < a.splits; ++sp) {
                        float* z = a.part + (size_t)sp * a.n * nout + col;
#pragma unroll
                        for (int j = 0; j < kGmAccCols; ++j)
                            if (j < hcols && ct0 + j < a.n) __stcg(z + (size_t)(ct0 + j) * nout, 0.f);
                    }
                }
#pragma unroll
                for (int j = 0; j < kGmAccCols; ++j) acc[j] = 0.f;
            }
        }
        if (!ok) give_up();

        tc_fence_before();
        __syncthreads();
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

// Tiles of 128 weight rows (or 64 gate + 64 up rows) by bn tokens; split K
// (in whole scale groups) so that about one CTA per SM is busy when the tiles
// alone are too few, keeping at least eight 64-column blocks per split, or
// stream-K where whole splits fit the SMs badly.
inline GemmPlan gemm_plan(int epi, int n, int N, int K, int sms) {
    GemmPlan p = {};
    GemmArgs& a = p.a;
    a.n = n;
    a.N = N;
    a.K = K;
    a.bn = n > 128 ? 256 : (n > 64 ? 128 : 64);
    a.tok_tiles = (n + a.bn - 1) / a.bn;
    a.row_tiles = N / (epi == G_SWIGLU ? 64 : 128);
    const int kbs = K / 64;
    const int tiles = a.tok_tiles * a.row_tiles;
    const int splits = std::max(1, std::min(tiles >= sms ? 1 : sms / tiles, kbs / 8));
    a.kb_per_split = ((kbs + splits - 1) / splits + 1) / 2 * 2;
    a.splits = (kbs + a.kb_per_split - 1) / a.kb_per_split;
    a.ctas = tiles * a.splits;
    // Stream-K when whole splits would leave more than an eighth of the SMs idle
    // and every CTA gets at least sixteen scale groups (the 7B down projection at
    // 512 tokens: 56 tiles x 2 splits on 152 SMs become 152 runs of 54-55 groups
    // instead of 74).  Each piece costs a partial tile written and read back, so
    // short K stays split (the O projection: 10 groups a CTA, measured slower).
    // Not for SwiGLU, whose tiles outnumber the SMs.
    const long long units = (long long)tiles * (K / 128);
    if (epi != G_SWIGLU && tiles < sms && (long long)a.ctas * 8 < (long long)sms * 7 && units >= 16LL * sms) {
        a.stream = 1;
        a.ctas = sms;
        int pieces = 1;
        for (int t = 0; t < tiles; ++t)
            pieces = std::max(pieces, gm_cta_of((long long)(t + 1) * (K / 128) - 1, units, sms) -
                                          gm_cta_of((long long)t * (K / 128), units, sms) + 1);
        a.splits = pieces;
    }
    // Persistent when the tiles outnumber the SMs (K not split): one CTA per SM
    // walks an equal run of whole tiles, its stage ring and accumulators running on
    // from one tile to the next, so the ring fills once per SM instead of once per
    // tile, and each tile's epilogue overlaps the next tile's MMAs.
    if (a.splits == 1 && tiles > sms) {
        a.stream = 2;
        a.ctas = sms;
    }
    const uint32_t sb = gemm_stage_bytes(a.bn);
    a.stages = (int)std::min<size_t>(kGmMaxStages, (kGmSmemBudget - 1024 - kGmPRingBytes) / sb);
    p.grid = dim3((unsigned)a.ctas);
    // at least 116 KB, so that one CTA holds an SM (and all of its TMEM) at a time
    p.smem = std::max<size_t>((size_t)a.stages * sb + kGmPRingBytes + 1024, 116 * 1024);
    return p;
}

int gemm_ab_mode();
inline size_t gemm_part_bytes(int epi, const GemmPlan& p) {
    const size_t nout = epi == G_SWIGLU ? 2 * (size_t)p.a.N : (size_t)p.a.N;
    return p.a.splits > 1 ? (size_t)p.a.splits * p.a.n * nout * sizeof(float) : 0;
}


// The GEMM kernel, and with split K the merge kernel after it (two launches);
// reduce = false leaves the split partials [splits][n][N] in a.part for the
// caller to add (G_STORE and G_RESID only).
cudaError_t gemm_tc05_launch(int epi, const GemmPlan& p, const CUtensorMap& tmx, const CUtensorMap& tmw0,
                             const CUtensorMap& tmw1, cudaStream_t st, bool reduce = true);

}  // namespace w4
