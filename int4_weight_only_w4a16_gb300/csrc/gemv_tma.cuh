// Batch-1 W4A16 GEMV fed by TMA bulk copies (the decode path's weight stream).
//
// Operation as in gemv.cuh ("How to build your own LLM runtime from scratch
// (Towards Data Science)", "What it actually builds": fused GEMVs over INT4
// group-128 weights; "How To Build Your Own LLM Runtime From Scratch |
// daily.dev", third question: fp16 activations against unpacked INT4).  The
// pages' attention kernels were warp-specialised around Hopper's TMA; this
// kernel applies the same idea to the weight stream.
//
// Why this shape on sm_103a: a read-bandwidth probe on GB300 showed that
// per-thread 16-byte loads only approach HBM peak at full occupancy (64 warps
// per SM), whatever the per-lane prefetch depth, while 1-D bulk copies
// (cp.async.bulk) into a shared-memory ring reach ~7.3 TB/s from one CTA per
// SM.  An exact fp32-accumulating INT4 dot costs ~1.3 issue slots per weight,
// so the consumers must also run without block-wide stalls.  So:
//  * One persistent CTA per SM owns a contiguous, balanced range of output
//    rows: one contiguous run of bytes of the row-major packed matrix.
//  * The last warp (CW, after the CW consumer warps) is the producer: its
//    lane 0 streams the range as stages of whole "row groups" (two rows of one
//    matrix, a gate row and its up row, or one long row, plus their fp16
//    scales) into an ns-deep shared-memory ring with cp.async.bulk, signalling
//    a `full` mbarrier per stage, and refills a slot once every consumer of it
//    has arrived on its `empty` mbarrier.  The first stages are issued before
//    the kernel waits on the previous kernel (programmatic dependent launch):
//    weights do not depend on it.
//  * Warps 0 .. CW-1 (twelve, or eight) are consumers, in units of a half-warp
//    (HPR = 1) or, for long rows, a whole warp (HPR = 2); unit u owns row
//    groups u, u + units, ... of the CTA.  Lanes read 16-byte chunks l,
//    l + 16 (or l + 32), ... of a row (conflict-free); the lanes of a warp
//    read the same activation chunks (broadcast) and each activation chunk
//    serves both rows of a group.  A unit finishes its group with shuffles,
//    writes the epilogue and arrives on the stage's `empty` barrier: no block
//    barrier inside the stream.
//  * Every mbarrier wait is bounded in time; on expiry the waiter records
//    W4_DEVERR_TIMEOUT and carries on without the data, so the CTA always
//    terminates, and the producer does not leave while its copies can land.
#pragma once

#include "gemv.cuh"

namespace w4 {

constexpr int kWsMaxConsumerWarps = 12;
constexpr int kWsMaxHalfWarps = kWsMaxConsumerWarps * 2;
constexpr int kWsMaxStages = 8;
constexpr size_t kWsRingBudget = 176 * 1024;             // weight bytes in the ring
constexpr size_t kTmaSmemMax = 220 * 1024;               // dynamic shared memory the plan may use
constexpr uint64_t kTmaWaitNs = 1000000000ull;
constexpr int kTmaMaxK = 24576;   // inputs the one-round-trip staging holds (8 or 12 pieces per consumer)

struct TmaArgs {
    int cw;           // consumer warps (the block has cw + 1 warps)
    int hpr;          // half-warps per row group: 1, or 2 (a whole warp per long row)
    int rg;           // rows of one matrix per row group (2, or 1 for long rows / gate+up)
    int gs;           // row groups per stage
    int ns;           // stages in the ring
    int wbytes;       // weight bytes of one matrix in a full stage (gs * rg rows)
    int sbytes;       // scale buffer bytes per matrix per stage slot
};

struct TmaPlan {
    TmaArgs a;
    int grid;
    size_t smem;
};

// early: E_RESID_F32's residual value of the row was loaded before the row's
// dot product (into pre), so that its latency hides behind it
template <int EPI>
__device__ __forceinline__ void tma_epilogue(const GemvParams& p, int row, float a0, float a1, bool early, float pre,
                                             unsigned long long& best) {
    if constexpr (EPI == E_STORE_F16) {
        float v = a0;
        if (p.bias) v += __half2float(p.bias[row]);
        if (p.resid16) v += __half2float(p.resid16[row]);
        p.y16[row] = __float2half_rn(v);
    } else if constexpr (EPI == E_RESID_F32) {
        p.y32[row] = (early ? pre : p.y32[row]) + a0;
    } else if constexpr (EPI == E_SWIGLU) {
        p.y16[row] = __float2half_rn(a0 / (1.f + expf(-a0)) * a1);
    } else {
        if (p.y32) p.y32[row] = a0;
        if (a0 != a0) record_device_error(p.errword, W4_DEVERR_NAN_LOGIT);
        const unsigned long long k = argmax_key(a0, row);
        best = k > best ? k : best;
    }
}

// QKV epilogue of one row pair (row even): bias, fp16, RoPE at the token's
// position, q out, k and v into page `page`, slot `slot` of the pools (see
// GemvParams).  b0, b1 (the rows' biases) and cs (the pair's cos, sin at the
// position; q and k rows only) are loaded before the rows' dot products.
__device__ __forceinline__ void qkv_rope_epilogue(const GemvParams& p, int row, float a0, float a1, float b0, float b1,
                                                  float2 cs, int page, int slot) {
    const int qrows = p.hq * 128, krows = p.hkv * 128;
    const __half h0 = __float2half_rn(a0 + b0);
    const __half h1 = __float2half_rn(a1 + b1);
    if (row < qrows + krows) {
        const int r = row < qrows ? row : row - qrows;
        const int head = r >> 7, i = (r & 127) >> 1;
        const float x0 = __half2float(h0), x1 = __half2float(h1);
        const __half o0 = __float2half_rn(x0 * cs.x - x1 * cs.y);
        const __half o1 = __float2half_rn(x1 * cs.x + x0 * cs.y);
        __half* dst = row < qrows ? p.qout + head * 128
                                  : p.k_pool + (((size_t)page * p.hkv + head) * 16 + slot) * 128;
        dst[i] = o0;
        dst[i + 64] = o1;
    } else {
        const int r = row - qrows - krows;
        const int head = r >> 7, d = r & 127;
        __half* dst = p.v_pool + (((size_t)page * p.hkv + head) * 16 + slot) * 128;
        dst[d] = h0;
        dst[d + 1] = h1;
    }
}

// Shared memory: [ns][NM] weights | [ns][NM] scales | x pieces [4][C] | x sums [C] | norm scratch
__host__ __device__ inline size_t tma_smem_bytes(int nm, int k, const TmaArgs& a) {
    const size_t w = (size_t)a.ns * nm * a.wbytes;
    const size_t sc = (size_t)a.ns * nm * a.sbytes;
    const size_t c = (size_t)(k / 32);
    return 128 + w + sc + c * 64 + c * 4 + 64 * sizeof(float);
}

template <int VAR, int XMODE, int EPI, int CW, int HPR>
__global__ void __launch_bounds__((CW + 1) * 32, 1)
gemv_tma_kernel(const GemvParams p, const TmaArgs ta) {
    constexpr int NM = (EPI == E_SWIGLU) ? 2 : 1;   // matrices streamed together
    constexpr int kWsConsumerWarps = CW;
    constexpr int kWsHalfWarps = 2 * CW;
    // a "unit" owns row groups: a half-warp (HPR = 1) or a whole warp (HPR = 2)
    constexpr int NU = kWsHalfWarps / HPR;
    constexpr int UL = 16 * HPR;                     // lanes per unit
    extern __shared__ unsigned char tma_smem_raw[];
    __shared__ __align__(8) uint64_t full[kWsMaxStages];
    __shared__ __align__(8) uint64_t empty[kWsMaxStages];
    __shared__ unsigned long long s_key[kWsMaxHalfWarps];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int C = p.K >> 5;                       // 32-weight chunks per row
    const int rowbytes = p.K >> 1;
    const int gpr = p.K >> 7;
    const int RG = ta.rg;

    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(tma_smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    unsigned char* wst = base;                                               // [ns][NM][wbytes]
    unsigned char* sst = wst + (size_t)ta.ns * NM * ta.wbytes;              // [ns][NM][sbytes]
    uint4* xs = reinterpret_cast<uint4*>(sst + (size_t)ta.ns * NM * ta.sbytes);  // [4][C]
    float* xneg8 = reinterpret_cast<float*>(xs + 4 * C);                    // [C]
    float* nrm = xneg8 + C;                                                  // [64]

    // this CTA's rows: a balanced contiguous share of the N/RG row groups
    const int gtot = (p.N + RG - 1) / RG;
    const int r0 = (int)(((long long)blockIdx.x * gtot) / gridDim.x) * RG;
    const int r1 = min(p.N, (int)(((long long)(blockIdx.x + 1) * gtot) / gridDim.x) * RG);
    const int ngroups = (r1 - r0 + RG - 1) / RG;
    const int nstage = (ngroups + ta.gs - 1) / ta.gs;

    if (warp == kWsConsumerWarps) {
        // ------------------------------------------------------------ producer
        // it sets up the ring itself and starts streaming at once; the consumers
        // meet it at named barrier 2 before their first wait
        if ((tid & 31) == 0) {
            for (int i = 0; i < ta.ns; ++i) {
                mbar_init(&full[i], 1);
                mbar_init(&empty[i], ta.gs);   // one arrival per row group of a full stage
            }
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncwarp();
        asm volatile("bar.arrive 2, %0;" ::"n"((kWsConsumerWarps + 1) * 32) : "memory");
        if ((tid & 31) == 0) {
            const uint64_t policy = l2_evict_first_policy();   // weights are read once per step
            int issued = 0;
            for (int t = 0; t < nstage; ++t) {
                if (t == min(nstage, ta.ns)) {   // ring primed: warm L2 with the next kernel's weights
                    l2_prefetch_share(p.pf0, p.pf0_bytes, blockIdx.x, gridDim.x);
                    l2_prefetch_share(p.pf1, p.pf1_bytes, blockIdx.x, gridDim.x);
                }
                const int slot = t % ta.ns;
                // a slot is reused only after the stage ns earlier (a full stage) was consumed
                if (t >= ta.ns &&
                    !mbar_wait_bounded(&empty[slot], (unsigned)(t / ta.ns - 1) & 1u, kTmaWaitNs)) {
                    record_device_error(p.errword, W4_DEVERR_TIMEOUT);
                    break;
                }
                const int ga = t * ta.gs, gb = min(ngroups, ga + ta.gs);
                const int ra = r0 + ga * RG, rb = min(r1, r0 + gb * RG);
                const unsigned wb = (unsigned)(rb - ra) * (unsigned)rowbytes;
                const long long s_lo = ((long long)ra * gpr * 2) & ~15LL;
                const long long s_hi = (((long long)rb * gpr * 2) + 15) & ~15LL;
                const unsigned sb = (unsigned)(s_hi - s_lo);
                if (t >= ta.ns) fence_proxy_async();
                mbar_arrive_expect_tx(&full[slot], NM * (wb + sb));
#pragma unroll
                for (int i = 0; i < NM; ++i) {
                    const uint32_t* w = i == 0 ? p.w0 : p.w1;
                    const __half* sc = i == 0 ? p.s0 : p.s1;
                    bulk_g2s_hint(wst + ((size_t)slot * NM + i) * ta.wbytes, w + (size_t)ra * (p.K >> 3), wb,
                                  &full[slot], policy);
                    bulk_g2s_hint(sst + ((size_t)slot * NM + i) * ta.sbytes, reinterpret_cast<const char*>(sc) + s_lo,
                                  sb, &full[slot], policy);
                }
                issued = t + 1;
            }
            if (nstage < ta.ns) {   // the whole range fit in the ring: warm L2 now
                l2_prefetch_share(p.pf0, p.pf0_bytes, blockIdx.x, gridDim.x);
                l2_prefetch_share(p.pf1, p.pf1_bytes, blockIdx.x, gridDim.x);
            }
            // do not leave while copies this warp issued may still be landing
            for (int t = max(0, issued - ta.ns); t < issued; ++t)
                mbar_wait_bounded(&full[t % ta.ns], (unsigned)(t / ta.ns) & 1u, kTmaWaitNs);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    constexpr unsigned kConsumers = kWsConsumerWarps * 32;
    const int unit = tid / UL, lu = tid % UL;       // unit index, lane within the unit
    const unsigned umask = HPR == 2 ? 0xFFFFFFFFu : (0xFFFFu << (tid & 16));
    pdl_trigger();
    pdl_wait();  // the activations come from the previous kernel

    int rpos = 0, rpage = 0, rslot = 0;
    bool rope_ok = true;
    if constexpr (EPI == E_QKV_ROPE) {
        rpos = *p.pos_in;
        rope_ok = rpos >= 0 && rpos < p.max_context && rpos < p.max_pages * 16;
        rpage = rope_ok ? p.pt[rpos >> 4] : -1;
        rope_ok = rope_ok && rpage >= 0 && rpage < p.num_pages;
        rslot = rpos & 15;
        if (blockIdx.x == 0 && tid == 0) {
            if (!rope_ok) record_device_error(p.errword, W4_DEVERR_POSITION | W4_DEVERR_PAGE_ID);
            *p.ctx = rope_ok ? rpos + 1 : 0;
        }
    }

    float inv_rms = 1.f;
    // Input staging, one round trip to L2: piece p (8 consecutive inputs) of chunk
    // c = p / 4 goes to xs[(p % 4) * C + c]; the four pieces of a chunk sit in one
    // aligned lane quad, which adds up the chunk's -8 * sum(x) by two shuffles.
    constexpr bool kPieces = VAR != V_INT8;
    static_assert(!(VAR == V_INT8 && XMODE == X_RMSNORM), "the W4A8 variant stages plain fp16 inputs only");
    if constexpr (kPieces && XMODE == X_RMSNORM) {
        constexpr int PPT = CW == 8 ? 4 : 3;   // pieces per thread: 4 * C <= PPT * kConsumers for K <= 8192
        float4 xa[PPT][2];
        uint4 ga[PPT];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < PPT; ++i) {
            const int pc = tid + i * (int)kConsumers;
            if (pc < 4 * C) {
                const float4* xr = reinterpret_cast<const float4*>(p.xres) + 2 * pc;
                xa[i][0] = xr[0];
                xa[i][1] = xr[1];
                ga[i] = reinterpret_cast<const uint4*>(p.gamma)[pc];
            } else {
                xa[i][0] = xa[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                ga[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int i = 0; i < PPT; ++i)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                ss = fmaf(xa[i][h].x, xa[i][h].x, ss);
                ss = fmaf(xa[i][h].y, xa[i][h].y, ss);
                ss = fmaf(xa[i][h].z, xa[i][h].z, ss);
                ss = fmaf(xa[i][h].w, xa[i][h].w, ss);
            }
        ss = warp_sum(ss);
        if ((tid & 31) == 0) nrm[tid >> 5] = ss;
        named_sync(1, kConsumers);
        float t = (tid & 31) < kWsConsumerWarps ? nrm[tid & 31] : 0.f;
        t = warp_sum(t);
        inv_rms = 1.0f / sqrtf(t / (float)p.K + p.eps);
#pragma unroll
        for (int i = 0; i < PPT; ++i) {
            const int pc = tid + i * (int)kConsumers;
            const float2 g0 = __half22float2(u32_as_h2(ga[i].x)), g1 = __half22float2(u32_as_h2(ga[i].y));
            const float2 g2 = __half22float2(u32_as_h2(ga[i].z)), g3 = __half22float2(u32_as_h2(ga[i].w));
            const float4 a = xa[i][0], b = xa[i][1];
            const __half2 h0 = __floats2half2_rn(a.x * inv_rms * g0.x, a.y * inv_rms * g0.y);
            const __half2 h1 = __floats2half2_rn(a.z * inv_rms * g1.x, a.w * inv_rms * g1.y);
            const __half2 h2 = __floats2half2_rn(b.x * inv_rms * g2.x, b.y * inv_rms * g2.y);
            const __half2 h3 = __floats2half2_rn(b.z * inv_rms * g3.x, b.w * inv_rms * g3.y);
            const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
            const float2 f2 = __half22float2(h2), f3 = __half22float2(h3);
            float csum = ((f0.x + f0.y) + (f1.x + f1.y)) + ((f2.x + f2.y) + (f3.x + f3.y));
            csum += __shfl_xor_sync(0xffffffffu, csum, 1);
            csum += __shfl_xor_sync(0xffffffffu, csum, 2);
            if (pc < 4 * C) {
                xs[(pc & 3) * C + (pc >> 2)] = make_uint4(h2_as_u32(h0), h2_as_u32(h1), h2_as_u32(h2), h2_as_u32(h3));
                if ((pc & 3) == 0) xneg8[pc >> 2] = -8.f * csum;
            }
        }
        named_sync(1, kConsumers);
    } else if constexpr (kPieces) {   // X_F16
        constexpr int PPT = CW == 8 ? 12 : 8;   // 4 * C <= PPT * kConsumers for K <= kTmaMaxK
        uint4 xp[PPT];
#pragma unroll
        for (int i = 0; i < PPT; ++i) {
            const int pc = tid + i * (int)kConsumers;
            xp[i] = pc < 4 * C ? reinterpret_cast<const uint4*>(p.x)[pc] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < PPT; ++i) {
            const int pc = tid + i * (int)kConsumers;
            if (i * (int)kConsumers >= 4 * C) break;   // uniform
            const float2 f0 = __half22float2(u32_as_h2(xp[i].x)), f1 = __half22float2(u32_as_h2(xp[i].y));
            const float2 f2 = __half22float2(u32_as_h2(xp[i].z)), f3 = __half22float2(u32_as_h2(xp[i].w));
            float csum = ((f0.x + f0.y) + (f1.x + f1.y)) + ((f2.x + f2.y) + (f3.x + f3.y));
            csum += __shfl_xor_sync(0xffffffffu, csum, 1);
            csum += __shfl_xor_sync(0xffffffffu, csum, 2);
            if (pc < 4 * C) {
                xs[(pc & 3) * C + (pc >> 2)] = xp[i];
                if ((pc & 3) == 0) xneg8[pc >> 2] = -8.f * csum;
            }
        }
        named_sync(1, kConsumers);
    }
    if constexpr (!kPieces)
    for (int c = tid; c < C; c += kConsumers) {
        uint4 pieces[4];
        const int k0 = c * 32;
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
            const uint4* xg = reinterpret_cast<const uint4*>(p.x + k0);
#pragma unroll
            for (int i = 0; i < 4; ++i) pieces[i] = xg[i];
        }
        if constexpr (VAR == V_INT8) {
            // W4A8: quantise the 128-group (chunks 4g..4g+3 sit in one aligned lane
            // quad, all active together) to INT8 with s = max|x| / 127
            float xf[32];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t u[4] = {pieces[i].x, pieces[i].y, pieces[i].z, pieces[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 f = __half22float2(u32_as_h2(u[j]));
                    xf[8 * i + 2 * j] = f.x;
                    xf[8 * i + 2 * j + 1] = f.y;
                }
            }
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(xf[e]));
            const unsigned quad = 0xFu << ((threadIdx.x & 31) & ~3);   // the group's four lanes
            amax = fmaxf(amax, __shfl_xor_sync(quad, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(quad, amax, 2));
            const float sx = amax / 127.f;
            int qv[32], qsum = 0;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                qv[e] = sx > 0.f ? (int)fminf(fmaxf(rintf(xf[e] / sx), -127.f), 127.f) : 0;
                qsum += qv[e];
            }
            auto pack4 = [&](int a, int b, int c2, int d) {
                return (uint32_t)(qv[a] & 0xFF) | ((uint32_t)(qv[b] & 0xFF) << 8) | ((uint32_t)(qv[c2] & 0xFF) << 16) |
                       ((uint32_t)(qv[d] & 0xFF) << 24);
            };
            uint32_t wlo[4], whi[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {   // word j: elements 8j..8j+7 in nibble order
                wlo[j] = pack4(8 * j, 8 * j + 4, 8 * j + 1, 8 * j + 5);
                whi[j] = pack4(8 * j + 2, 8 * j + 6, 8 * j + 3, 8 * j + 7);
            }
            xs[0 * C + c] = make_uint4(wlo[0], whi[0], wlo[1], whi[1]);
            xs[1 * C + c] = make_uint4(wlo[2], whi[2], wlo[3], whi[3]);
            xs[2 * C + c] = make_uint4(__float_as_uint(sx), (uint32_t)(-8 * qsum), 0u, 0u);
            xs[3 * C + c] = make_uint4(0u, 0u, 0u, 0u);
            xneg8[c] = 0.f;
        } else {
            float csum = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t u[4] = {pieces[i].x, pieces[i].y, pieces[i].z, pieces[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 f = __half22float2(u32_as_h2(u[j]));
                    csum += f.x + f.y;
                }
                xs[i * C + c] = pieces[i];
            }
            xneg8[c] = -8.f * csum;
        }
    }
    if constexpr (!kPieces) named_sync(1, kConsumers);
    // the producer has set up the ring before any consumer waits on it
    asm volatile("bar.sync 2, %0;" ::"n"((kWsConsumerWarps + 1) * 32) : "memory");

    unsigned long long best = 0ull;
    const uint32_t xq_stride = (uint32_t)C * 16u;
    const int nj = (C - lu + UL - 1) / UL;   // this lane's chunks of a row: lu, lu+UL, ...
    // stage / slot / parity of this unit's groups, advanced without division:
    // group g sits in stage g / gs; consecutive groups of a unit are st stages apart
    const int st = NU / ta.gs;
    int t = unit / ta.gs, slot = t % ta.ns;
    unsigned parity = (unsigned)(t / ta.ns) & 1u;
    // The epilogue's global operands are loaded before the group's dot product, in
    // flight while the stage lands and the dot runs, where each unit has one group
    // (QKV, O).  With several groups a unit (the down projection's two rows a
    // warp) the residual is read after the dot: measured 1.3 us faster there.
    const bool early = ngroups <= NU;
    for (int g = unit; g < ngroups; g += NU) {
        const int row = r0 + g * RG;                        // first row of the group
        const bool has1 = (NM == 2) || (RG == 2 && row + 1 < r1);
        float e0 = 0.f, e1 = 0.f;
        float2 ecs = make_float2(0.f, 0.f);
        if (lu == 0) {
            if constexpr (EPI == E_RESID_F32) {
                if (early) {
                    e0 = p.y32[row];
                    if (has1) e1 = p.y32[row + 1];
                }
            } else if constexpr (EPI == E_QKV_ROPE) {
                e0 = __half2float(p.bias[row]);
                e1 = __half2float(p.bias[row + 1]);
                if (rope_ok && row < (p.hq + p.hkv) * 128) ecs = p.rope[(size_t)rpos * 64 + ((row & 127) >> 1)];
            }
        }
        const bool ok = mbar_wait_bounded(&full[slot], parity, kTmaWaitNs);
        const int ra = r0 + t * ta.gs * RG;                 // first row of the stage
        float acc0 = 0.f, acc1 = 0.f;
        if (ok) {
            const long long s_lo = ((long long)ra * gpr * 2) & ~15LL;
            const uint32_t soff = (uint32_t)(((long long)row * gpr * 2) - s_lo);
            uint32_t aw0 = smem_u32(wst + (size_t)slot * NM * ta.wbytes + (size_t)(row - ra) * rowbytes) + lu * 16;
            uint32_t aw1 = (NM == 2) ? smem_u32(wst + ((size_t)slot * NM + 1) * ta.wbytes +
                                                (size_t)(row - ra) * rowbytes) + lu * 16
                                     : aw0 + rowbytes;
            uint32_t as0 = smem_u32(sst + (size_t)slot * NM * ta.sbytes) + soff + (lu >> 2) * 2;
            uint32_t as1 = (NM == 2) ? smem_u32(sst + ((size_t)slot * NM + 1) * ta.sbytes) + soff + (lu >> 2) * 2
                                     : as0 + gpr * 2;
            uint32_t ax = smem_u32(xs) + lu * 16;
            uint32_t an = smem_u32(xneg8) + lu * 4;
#pragma unroll 2
            for (int j = 0; j < nj; ++j) {
                uint4 xq[4];
                xq[0] = lds128(ax);
                xq[1] = lds128(ax + xq_stride);
                xq[2] = lds128(ax + 2 * xq_stride);
                xq[3] = lds128(ax + 3 * xq_stride);
                const float n8 = lds_f32(an);
                const uint4 wa = lds128(aw0);
                acc0 = fmaf(lds_f16_as_f32(as0), chunk_dot<VAR>(wa, xq, n8), acc0);
                if (has1) {
                    const uint4 wbv = lds128(aw1);
                    acc1 = fmaf(lds_f16_as_f32(as1), chunk_dot<VAR>(wbv, xq, n8), acc1);
                }
                ax += 16 * UL;
                an += 4 * UL;
                aw0 += 16 * UL;
                aw1 += 16 * UL;
                as0 += UL / 2;
                as1 += UL / 2;
            }
        } else if (lu == 0) {
            record_device_error(p.errword, W4_DEVERR_TIMEOUT);
        }
#pragma unroll
        for (int o = UL / 2; o > 0; o >>= 1) {
            acc0 += __shfl_xor_sync(umask, acc0, o);
            acc1 += __shfl_xor_sync(umask, acc1, o);
        }
        if (lu == 0) {
            mbar_arrive(&empty[slot]);   // this group's bytes are no longer needed
            if (ok) {
                if constexpr (EPI == E_QKV_ROPE) {
                    if (rope_ok) qkv_rope_epilogue(p, row, acc0, acc1, e0, e1, ecs, rpage, rslot);
                } else if constexpr (NM == 2) {
                    tma_epilogue<EPI>(p, row, acc0, acc1, false, 0.f, best);
                } else {
                    tma_epilogue<EPI>(p, row, acc0, 0.f, early, e0, best);
                    if (has1) tma_epilogue<EPI>(p, row + 1, acc1, 0.f, early, e1, best);
                }
            }
        }
        t += st;
        slot += st;
        if (slot >= ta.ns) {   // st divides ns: the slot wraps exactly once per ns stages
            slot -= ta.ns;
            parity ^= 1u;
        }
    }

    if constexpr (EPI == E_ARGMAX) {
        if (lu == 0) s_key[unit] = best;
        named_sync(1, kConsumers);
        if (tid == 0) {
            unsigned long long k = 0ull;
            for (int i = 0; i < NU; ++i) k = s_key[i] > k ? s_key[i] : k;
            atomicMax(p.amax_key, k);
            __threadfence();
            const unsigned tk = atomicAdd(p.counters, 1u);
            if (tk == gridDim.x - 1) {
                __threadfence();
                const unsigned long long kk = atomicExch(p.amax_key, 0ull);
                p.token_out[0] = (int32_t)(0xFFFFFFFFu - (uint32_t)(kk & 0xFFFFFFFFull));
                p.counters[0] = 0u;
                if (p.pos) p.pos[0] += 1;
            }
        }
    }
}

// ---------------------------------------------------------------- host side
// Row groups of two rows when sixteen of them (one per consumer half-warp)
// fit in the ring twice over, else of one row.  A stage holds gs groups, so a
// half-warp's groups lie st = 16/gs stages apart.  The ring depth ns is a
// multiple of st: the stage that last used the slot a half-warp waits on then
// held that half-warp's own previous group, which it has already consumed --
// so no waiter can ever observe an mbarrier phase from two uses back.
// grid = 0 marks a shape whose ring does not fit (callers fall back).
inline TmaPlan tma_plan_cw(int nm, int n, int k, int cw, int hpr) {
    TmaPlan pl = {};
    if (k > kTmaMaxK) return pl;   // beyond what the input staging holds
    const int hws = 2 * cw / hpr;                    // units that own row groups
    const size_t rowbytes = (size_t)k / 2;
    int rg = (nm == 2) ? 1 : 2;
    if (nm == 1 && 2 * rowbytes * 2 * hws > kWsRingBudget) rg = 1;
    const size_t gbytes = (size_t)nm * rg * rowbytes;
    const size_t q = kWsRingBudget / gbytes;       // groups the ring can hold
    // most groups in flight first, then the most (finer) stages
    int gs = 0, ns = 0;
    for (int cand = 8; cand >= 2; cand >>= 1) {
        if (hws % cand) continue;
        const int st = hws / cand;
        int c_ns = (int)(q / cand) / st * st;
        if (c_ns > kWsMaxStages) c_ns = kWsMaxStages / st * st;
        if (c_ns < st || c_ns < 2) continue;
        if (c_ns * cand > ns * gs || (c_ns * cand == ns * gs && c_ns > ns)) {
            gs = cand;
            ns = c_ns;
        }
    }
    if (gs == 0) return pl;
    pl.a.cw = cw;
    pl.a.hpr = hpr;
    pl.a.rg = rg;
    pl.a.gs = gs;
    pl.a.ns = ns;
    pl.a.wbytes = (int)(gs * rg * rowbytes);
    const int gpr = k / 128;
    pl.a.sbytes = ((gs * rg * gpr * 2 + 15) / 16) * 16 + 32;  // 16-byte aligned superset of the rows' scales
    const int sms = sm_count();
    pl.grid = n < sms ? n : sms;
    pl.smem = tma_smem_bytes(nm, k, pl.a);
    if (pl.smem > kTmaSmemMax) pl.grid = 0;
    return pl;
}

// Twelve consumer warps when the ring holds two rounds of their row groups
// (more warps per scheduler hide more latency), else eight.
// Long rows that only fit one row per group, with fewer rows per CTA than
// two per half-warp, are given a whole warp each: twelve warps when the ring
// holds one round of their rows (measured faster on the 18944-long rows of the
// down projection), else eight.
//
// Finally, when every unit owns at most one row group of its CTA (so every ring
// slot is filled once and never reused), the ring shrinks to the CTA's row
// groups (the QKV and O projections): the kernel then leaves shared memory on
// the SM for the stream's next kernel, launched early, to start beside it and
// begin its own loads before this one ends (the paged attention beside QKV).
// The twelve consumer warps stay: with nine, two of these CTAs fit on one SM,
// which then idled other SMs.
inline TmaPlan tma_plan(int nm, int n, int k) {
    TmaPlan pl = tma_plan_cw(nm, n, k, 12, 1);
    if (pl.grid == 0 || pl.a.ns * pl.a.gs < 2 * 2 * 12) {
        const TmaPlan p8 = tma_plan_cw(nm, n, k, 8, 1);
        if (p8.grid > 0) pl = p8;
    }
    if (pl.grid > 0 && nm == 1 && pl.a.rg == 1) {
        const int rows_per_cta = (n + pl.grid - 1) / pl.grid;
        if (rows_per_cta < 2 * 2 * pl.a.cw) {
            // a whole warp per row: twelve warps when the ring holds a round of their rows
            TmaPlan pw = tma_plan_cw(nm, n, k, 12, 2);
            if (pw.grid == 0) pw = tma_plan_cw(nm, n, k, 8, 2);
            if (pw.grid > 0) pl = pw;
        }
    }
    if (pl.grid > 0 && nm == 1 && pl.a.hpr == 1 && pl.a.rg == 2) {
        // at most one row group per whole warp (the O projection): whole-warp units, so
        // that every consumer warp works, each lane on half the chunks (measured slower
        // for QKV's 16 groups, where four warps would take two each)
        const int groups = (n + 1) / 2;
        const int per_cta = (groups + pl.grid - 1) / pl.grid;
        if (per_cta <= pl.a.cw) {
            const TmaPlan pw = tma_plan_cw(nm, n, k, pl.a.cw, 2);
            if (pw.grid > 0 && pw.a.rg == 2) pl = pw;
        }
    }
    if (pl.grid > 0) {
        const int groups = (n + pl.a.rg - 1) / pl.a.rg;
        const int per_cta = (groups + pl.grid - 1) / pl.grid;
        const int units = 2 * pl.a.cw / pl.a.hpr;
        const int need = (per_cta + pl.a.gs - 1) / pl.a.gs;   // stages that hold them all
        if (per_cta <= units && need < pl.a.ns) {
            pl.a.ns = need < 1 ? 1 : need;
            pl.smem = tma_smem_bytes(nm, k, pl.a);
        }
    }
    return pl;
}

template <int VAR, int XMODE, int EPI, int CW, int HPR>
inline cudaError_t tma_launch_cw(const GemvParams& p, const TmaPlan& pl, cudaStream_t st, bool pdl) {
    auto kern = gemv_tma_kernel<VAR, XMODE, EPI, CW, HPR>;
    static size_t attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && attr_set[dev] < pl.smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
        if (e != cudaSuccess) return e;
        // the whole carveout as shared memory, so that the stream's next kernel fits beside it
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        attr_set[dev] = pl.smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.grid, 1, 1);
    cfg.blockDim = dim3((CW + 1) * 32, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p, pl.a);
}

template <int VAR, int XMODE, int EPI>
inline cudaError_t tma_launch(const GemvParams& p, const TmaPlan& pl, cudaStream_t st, bool pdl) {
    if (pl.a.cw == 12 && pl.a.hpr == 1) return tma_launch_cw<VAR, XMODE, EPI, 12, 1>(p, pl, st, pdl);
    if constexpr (EPI != E_SWIGLU && EPI != E_QKV_ROPE) {
        if (pl.a.hpr == 2)
            return pl.a.cw == 12 ? tma_launch_cw<VAR, XMODE, EPI, 12, 2>(p, pl, st, pdl)
                                 : tma_launch_cw<VAR, XMODE, EPI, 8, 2>(p, pl, st, pdl);
    }
    return tma_launch_cw<VAR, XMODE, EPI, 8, 1>(p, pl, st, pdl);
}

}  // namespace w4
