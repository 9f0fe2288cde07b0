// W4A16 GEMV on tensor cores, fed by TMA (1 <= M <= 16 activation rows).
//
// Operation as in gemv.cuh ("How to build your own LLM runtime from scratch
// (Towards Data Science)", "What it actually builds": fused GEMVs over INT4
// group-128 weights, fp16 activations; fp32 accumulation).  The products run
// on mma.sync m16n8k16 with exact unpacking (gemv_mma.cuh explains the
// fragment order and the subnormal nibble trick): the unpack costs one LOP3
// per element pair and the tensor pipe does the multiply-adds, about half the
// issue slots per weight of the CUDA-core dot, so the weight stream rather
// than instruction issue bounds the kernel even at M = 1.
//
// Structure (one persistent CTA per SM, warp-specialised):
//  * Work unit = 64 weight rows x one K piece, served by a group of four
//    consumer warps (16 rows each).  The P pieces split the CTAs: CTA b serves
//    piece floor(b P / G) and a balanced contiguous share of its 64-row
//    blocks, so it stages only that piece of the activations.  A unit is
//    streamed as slices of at most 7 groups (one ring slot each).
//  * Warp CW is the weight producer: per slice, its lane 0 waits for the
//    slot's `empty` barrier (one arrival per warp of the group), arms the
//    `full` barrier with the byte count and the first NM lanes issue one 2-D
//    tensor copy each (a 64-row x slice box of the row-major packed matrix;
//    rows past N arrive as zeros).  A TMA copy instruction costs the issuing
//    warp about the same time whatever its size (measured on GB300: ~2.4 TB/s
//    over all SMs with 7 KiB copies, ~6 TB/s with 28 KiB ones), hence boxes
//    of 64 rows rather than one per warp.
//  * Consumer warps 0..CW-1 stage the activation piece (plain fp16 rows, the
//    RMSNorm of the fp32 residual, or the merge of the attention splits),
//    then, per group, take units g, g+NG, ... of the CTA through the group's
//    ring of Q slots; fp32 accumulators live across a unit's slices.  A unit's fp16
//    group scales (per row, the 16-byte aligned run covering the piece) are
//    fetched one unit ahead with cp.async into a per-warp double buffer.
//  * With P > 1 a unit writes its fp32 partial to the workspace and takes a
//    ticket; the last unit of a row block adds the partials in piece order
//    (deterministic) and runs the epilogue: fp16 store (+bias, +residual),
//    fp32 residual add, SiLU(gate)*up, argmax, or the QKV epilogue (bias,
//    RoPE, paged KV append) of gemv_tma.cuh.
//  * Every mbarrier wait is bounded; on expiry the waiter records
//    W4_DEVERR_TIMEOUT and carries on, and the weight producer waits
//    (bounded) for its last copies before leaving, so no copy outlives the
//    CTA.
#pragma once

#include <cuda.h>

#include <algorithm>

#include "gemv_mma.cuh"
#include "gemv_tma.cuh"

namespace w4 {

constexpr int kTcMaxSlots = 8;                   // ring slots per warp group, at most
constexpr int kTcRB = 4;                         // 16-row blocks (consumer warps) per group
constexpr int kTcMaxSlice = 7;                   // groups per slice, at most
constexpr size_t kTcSmemMax = 224 * 1024;

struct TcArgs {
    int cw;       // consumer warps
    int P;        // K pieces
    int gpp;      // groups per piece (the last piece may be shorter)
    int ssz;      // groups per slice (the tensor-map box is ssz*16 words wide)
    int q;        // ring slots per warp group
    int slot;     // bytes of one ring slot
    int nrb;      // row blocks of 16 rows (the 64-row units are kTcRB of them)
    int m;        // activation rows
};

struct TcPlan {
    TcArgs a;
    int grid;
    size_t smem;
};

// A 2-D tensor map over a packed [n][k/8] uint32 matrix whose box is
// `box_rows` rows by `box_words` words (defined with the other tensor-map
// helpers).
w4_status make_weight_tensor_map(CUtensorMap* map, const uint32_t* packed, int n, int k, int box_words, int box_rows);

// ring slot: weights [NM][64][ssz*64 B]
__host__ __device__ inline int tc_slot_bytes(int nm, int ssz) { return nm * kTcRB * 16 * ssz * 64; }

// bytes per row of a unit's scale buffer: the 16-byte aligned run of the
// packed scale rows that covers gpp groups from any start
__host__ __device__ inline int tc_scale_span(int gpp) { return ((gpp * 2 + 15) / 16 + 1) * 16; }

// the rest of the dynamic shared memory: alignment pad | scale buffers
// [cw][2][nm][16][span] | x [m][gpp*128] halves | group sums [gpp][nt*8] |
// norm scratch [64]
__host__ __device__ inline size_t tc_smem_rest(int xmode, int nm, int m, int gpp, int cw) {
    const int nt = m <= 8 ? 1 : 2;
    size_t b = 128 + (size_t)cw * 2 * nm * 16 * tc_scale_span(gpp);
    b += (size_t)m * gpp * 256 + (size_t)gpp * nt * 8 * 4 + 64 * 4;
    (void)xmode;
    return b;
}

__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

template <int NT, int XMODE, int EPI, int CW>
__global__ void __launch_bounds__((CW + 1) * 32, 1)
gemv_tc_kernel(const GemvParams p, const TcArgs ta, const __grid_constant__ CUtensorMap tm0,
               const __grid_constant__ CUtensorMap tm1) {
    constexpr int NM = (EPI == E_SWIGLU) ? 2 : 1;
    constexpr int NG = CW / kTcRB;                // warp groups
    static_assert(CW % kTcRB == 0, "whole warp groups");
    extern __shared__ unsigned char tc_smem_raw[];
    __shared__ __align__(8) uint64_t full[NG * kTcMaxSlots];
    __shared__ __align__(8) uint64_t empty[NG * kTcMaxSlots];
    __shared__ unsigned long long s_key[CW];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Q = ta.q, ssz = ta.ssz;
    const int gpr = p.K >> 7;
    const int G = gridDim.x, P = ta.P;
    const int piece = (int)(((long long)blockIdx.x * P) / G);
    const int b0 = (int)(((long long)piece * G + P - 1) / P), b1 = (int)(((long long)(piece + 1) * G + P - 1) / P);
    const int nb = b1 - b0, bi = blockIdx.x - b0;
    const int nbb = (ta.nrb + kTcRB - 1) / kTcRB;  // 64-row blocks
    const int bb0 = (int)(((long long)bi * nbb) / nb), bb1 = (int)(((long long)(bi + 1) * nbb) / nb);
    const int my_nbb = bb1 - bb0;
    const int g0 = piece * ta.gpp;
    const int ng = min(ta.gpp, gpr - g0);        // groups of this piece (>= 1)
    const int nsl = (ng + ssz - 1) / ssz;        // slices per unit
    const int k0 = g0 * 128;
    const int units = ng * 16;                   // 16-byte activation units per staged row
    const int wbox = kTcRB * 16 * ssz * 64;      // bytes of one matrix's box

    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(tc_smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    const int span = tc_scale_span(ta.gpp);
    unsigned char* ring = base;                                                   // [NG][Q][slot]
    unsigned char* scb = ring + (size_t)NG * Q * ta.slot;                        // [CW][2][NM][16][span]
    uint4* xs = reinterpret_cast<uint4*>(scb + (size_t)CW * 2 * NM * 16 * span);  // [M][units]
    float* sx = reinterpret_cast<float*>(xs + (size_t)ta.m * ta.gpp * 16);       // [gpp][NT*8]
    float* nrm = sx + ta.gpp * NT * 8;                                            // [64]

    if (tid == 0) {
        for (int i = 0; i < NG * Q; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kTcRB);   // every warp of the group releases the slot
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // stages of group c: r = unit * nsl + slice; units c, c+NG, ... of the CTA
    const int units0 = my_nbb > 0 ? (my_nbb + NG - 1) / NG : 0;   // group 0 has the most
    const int rounds = units0 * nsl;

    if (warp == CW) {
        // ----------------------------------------------------- weight producer
        {
            const uint64_t policy = l2_evict_first_policy();   // weights are read once per step
            int r_stop = rounds, c_stop = 0;                   // first (round, group) not issued
            for (int r = 0; r < rounds; ++r) {
                if (r == min(rounds, Q) && lane == 0) {   // ring primed: warm L2 with the next kernel's weights
                    l2_prefetch_share(p.pf0, p.pf0_bytes, blockIdx.x, G);
                    l2_prefetch_share(p.pf1, p.pf1_bytes, blockIdx.x, G);
                }
                const int u = r / nsl, sl = r - u * nsl;
                bool stop = false;
                for (int c = 0; c < NG; ++c) {
                    const int lbb = c + u * NG;
                    if (lbb >= my_nbb) break;
                    const int s = c * Q + (r % Q);
                    int ok = 1;
                    if (lane == 0 && r >= Q) ok = mbar_wait_bounded(&empty[s], (unsigned)(r / Q - 1) & 1u, kTmaWaitNs);
                    if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
                        if (lane == 0) record_device_error(p.errword, W4_DEVERR_TIMEOUT);
                        r_stop = r;
                        c_stop = c;
                        stop = true;
                        break;
                    }
                    if (lane == 0) {
                        if (r >= Q) fence_proxy_async();
                        mbar_arrive_expect_tx(&full[s], (unsigned)(NM * wbox));
                    }
                    __syncwarp();
                    if (lane < NM) {
                        const int x = (k0 >> 3) + sl * ssz * 16, y = (bb0 + lbb) * kTcRB * 16;
                        tma_load_2d_hint(ring + (size_t)s * ta.slot + lane * wbox, lane == 0 ? &tm0 : &tm1, x, y, &full[s],
                                         policy);
                    }
                }
                if (stop) break;
            }
            if (rounds < Q && lane == 0) {
                l2_prefetch_share(p.pf0, p.pf0_bytes, blockIdx.x, G);
                l2_prefetch_share(p.pf1, p.pf1_bytes, blockIdx.x, G);
            }
            // do not leave while copies may still be landing: per slot, the
            // last round that filled it
            for (int idx = lane; idx < NG * Q; idx += 32) {
                const int c = idx / Q, q = idx - c * Q;
                const int units_c = my_nbb > c ? (my_nbb - c + NG - 1) / NG : 0;
                const int issued = min(units_c * nsl, r_stop + (c < c_stop ? 1 : 0));
                if (issued <= q) continue;
                const int r_last = q + ((issued - 1 - q) / Q) * Q;
                if (!mbar_wait_bounded(&full[idx], (unsigned)(r_last / Q) & 1u, kTmaWaitNs)) {
                    record_device_error(p.errword, W4_DEVERR_TIMEOUT);
                    break;
                }
            }
        }
        return;
    }
    // -------------------------------------------------------------- consumers
    constexpr unsigned kConsumers = CW * 32;
    const int g = lane >> 2, t = lane & 3;
    pdl_trigger();
    pdl_wait();   // the activations come from the previous kernel

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

    // ---- activation piece: [M][units] 16-byte units, swizzled; group sums
    float inv_rms = 1.f;
    if constexpr (XMODE == X_RMSNORM) {
        float ss = 0.f;
        const float4* xr4 = reinterpret_cast<const float4*>(p.xres);
        for (int i = tid; i < (p.K >> 2); i += kConsumers) {
            const float4 v = xr4[i];
            ss = fmaf(v.x, v.x, ss);
            ss = fmaf(v.y, v.y, ss);
            ss = fmaf(v.z, v.z, ss);
            ss = fmaf(v.w, v.w, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) nrm[warp] = ss;
        named_sync(1, kConsumers);
        if (tid < 32) {
            float tt = tid < CW ? nrm[tid] : 0.f;
            tt = warp_sum(tt);
            if (tid == 0) nrm[32] = 1.0f / sqrtf(tt / (float)p.K + p.eps);
        }
        named_sync(1, kConsumers);
        inv_rms = nrm[32];
    }
    const int total = ta.m * units;
    for (int base0 = 0; base0 < total; base0 += kConsumers) {
        const int i = base0 + tid;
        const bool ok = i < total;
        const int m = ok ? i / units : 0, c = ok ? i - m * units : 0;
        const int k = k0 + c * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (ok) {
            if constexpr (XMODE == X_RMSNORM) {
                const float4 a = reinterpret_cast<const float4*>(p.xres + k)[0];
                const float4 b = reinterpret_cast<const float4*>(p.xres + k)[1];
                const uint4 gm = *reinterpret_cast<const uint4*>(p.gamma + k);
                const float2 q0 = __half22float2(u32_as_h2(gm.x)), q1 = __half22float2(u32_as_h2(gm.y));
                const float2 q2 = __half22float2(u32_as_h2(gm.z)), q3 = __half22float2(u32_as_h2(gm.w));
                v.x = h2_as_u32(__floats2half2_rn(a.x * inv_rms * q0.x, a.y * inv_rms * q0.y));
                v.y = h2_as_u32(__floats2half2_rn(a.z * inv_rms * q1.x, a.w * inv_rms * q1.y));
                v.z = h2_as_u32(__floats2half2_rn(b.x * inv_rms * q2.x, b.y * inv_rms * q2.y));
                v.w = h2_as_u32(__floats2half2_rn(b.z * inv_rms * q3.x, b.w * inv_rms * q3.y));
            } else {
                v = *reinterpret_cast<const uint4*>(p.x + (size_t)m * p.K + k);
            }
        }
        const float2 f0 = __half22float2(u32_as_h2(v.x)), f1 = __half22float2(u32_as_h2(v.y));
        const float2 f2 = __half22float2(u32_as_h2(v.z)), f3 = __half22float2(u32_as_h2(v.w));
        float sum = ((f0.x + f0.y) + (f1.x + f1.y)) + ((f2.x + f2.y) + (f3.x + f3.y));
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        if (ok) {
            if ((c & 15) == 0) sx[(c >> 4) * (NT * 8) + m] = sum;
            xs[(size_t)m * units + (c ^ mma_swz(m, (c >> 2) & 3))] = v;
        }
    }
    named_sync(1, kConsumers);

    // ---- this warp's stages
    int xu[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const int m = min(n * 8 + g, ta.m - 1);
        const int swz = mma_swz(m, t);
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) xu[n][wi] = m * units + 4 * t + (wi ^ swz);
    }
    const float* sxl = sx + 2 * t;
    const int grp = warp / kTcRB, sub = warp - grp * kTcRB;   // warp group, 16-row block within the unit
    const int nunits = my_nbb > grp ? (my_nbb - grp + NG - 1) / NG : 0;
    const int nst = nunits * nsl;
    const int srow = ssz * 64;                    // bytes per row of a box
    unsigned long long best = 0ull;
    float acc[NM][NT][4];

    // scales of unit u into buffer u & 1: per row, the aligned 16-byte chunks
    // covering groups g0 .. g0+ng-1 (never past the padded end of the buffer)
    const size_t sc_bytes = (((size_t)p.N * gpr * 2) + 15) & ~(size_t)15;
    const int nch = span / 16;
    unsigned char* wsc = scb + (size_t)warp * 2 * NM * 16 * span;
    auto fetch_scales = [&](int u) {
        const int row0 = ((bb0 + grp + u * NG) * kTcRB + sub) * 16;
        unsigned char* dstb = wsc + (size_t)(u & 1) * NM * 16 * span;
        for (int idx = lane; idx < NM * 16 * nch; idx += 32) {
            const int i = idx / (16 * nch), rem = idx - i * 16 * nch;
            const int rr = rem / nch, ch = rem - rr * nch;
            const int row = min(row0 + rr, p.N - 1);
            const size_t start = (((size_t)row * gpr + g0) * 2) & ~(size_t)15;
            if (start + ch * 16 < sc_bytes)
                cp_async16(smem_u32(dstb + (i * 16 + rr) * span + ch * 16),
                           reinterpret_cast<const unsigned char*>(i == 0 ? p.s0 : p.s1) + start + ch * 16);
        }
        cp_async_commit();
    };
    if (nunits > 0) fetch_scales(0);

    for (int r = 0; r < nst; ++r) {
        const int u = r / nsl, sl = r - u * nsl;
        const int s = grp * Q + (r % Q);
        const int gs0 = sl * ssz, nsz = min(ssz, ng - gs0);   // groups of this slice (piece-relative)
        if (sl == 0) {
#pragma unroll
            for (int i = 0; i < NM; ++i)
#pragma unroll
                for (int n = 0; n < NT; ++n) acc[i][n][0] = acc[i][n][1] = acc[i][n][2] = acc[i][n][3] = 0.f;
            if (u + 1 < nunits) fetch_scales(u + 1);
            else cp_async_commit();
            cp_async_wait<1>();   // this unit's scales (issued a unit ago) have landed
            __syncwarp();
        }
        // this lane's rows g and g+8 in the unit's scale buffer, at group jj
        const int row0u = ((bb0 + grp + u * NG) * kTcRB + sub) * 16;
        const unsigned char* sbu = wsc + (size_t)(u & 1) * NM * 16 * span;
        const uint32_t sra = smem_u32(sbu + g * span) + (uint32_t)((((size_t)min(row0u + g, p.N - 1) * gpr + g0) * 2) & 15);
        const uint32_t srb = smem_u32(sbu + (g + 8) * span) +
                             (uint32_t)((((size_t)min(row0u + g + 8, p.N - 1) * gpr + g0) * 2) & 15);
        const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&full[s], (unsigned)(r / Q) & 1u, kTmaWaitNs));
        if (ok) {
            const uint32_t wb = smem_u32(ring + (size_t)s * ta.slot) + (sub * 16 + g) * srow + 16 * t;
#pragma unroll 2
            for (int j = 0; j < nsz; ++j) {
                const int jj = gs0 + j;                   // group within the piece
                uint4 xb[4][NT];
#pragma unroll
                for (int wi = 0; wi < 4; ++wi)
#pragma unroll
                    for (int n = 0; n < NT; ++n) xb[wi][n] = xs[xu[n][wi] + jj * 16];
#pragma unroll
                for (int i = 0; i < NM; ++i) {
                    const uint32_t wa = wb + i * wbox + j * 64;
                    const uint4 qa = lds128(wa), qb = lds128(wa + 8 * srow);
                    const uint32_t A[4] = {qa.x, qa.y, qa.z, qa.w};
                    const uint32_t B[4] = {qb.x, qb.y, qb.z, qb.w};
                    const float s_a = lds_f16_as_f32(sra + i * 16 * span + jj * 2);
                    const float s_b = lds_f16_as_f32(srb + i * 16 * span + jj * 2);
                    float lo[NT][4], hi[NT][4];
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
                        const uint32_t a8 = A[wi] >> 8, b8 = B[wi] >> 8;
                        const uint32_t fl[4] = {A[wi] & 0x000F000Fu, B[wi] & 0x000F000Fu, a8 & 0x000F000Fu,
                                                b8 & 0x000F000Fu};
                        const uint32_t fh[4] = {A[wi] & 0x00F000F0u, B[wi] & 0x00F000F0u, a8 & 0x00F000F0u,
                                                b8 & 0x00F000F0u};
#pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            if (wi == 0) {
                                mma_16816_f16_z(lo[n], fl, xb[wi][n].x, xb[wi][n].z);
                                mma_16816_f16_z(hi[n], fh, xb[wi][n].y, xb[wi][n].w);
                            } else {
                                mma_16816_f16(lo[n], fl, xb[wi][n].x, xb[wi][n].z);
                                mma_16816_f16(hi[n], fh, xb[wi][n].y, xb[wi][n].w);
                            }
                        }
                    }
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        const float2 sm = *reinterpret_cast<const float2*>(sxl + jj * (NT * 8) + n * 8);
                        const float c0 = -8.f * sm.x, c1 = -8.f * sm.y;
                        acc[i][n][0] = fmaf(s_a, fmaf(16777216.f, lo[n][0], fmaf(1048576.f, hi[n][0], c0)), acc[i][n][0]);
                        acc[i][n][1] = fmaf(s_a, fmaf(16777216.f, lo[n][1], fmaf(1048576.f, hi[n][1], c1)), acc[i][n][1]);
                        acc[i][n][2] = fmaf(s_b, fmaf(16777216.f, lo[n][2], fmaf(1048576.f, hi[n][2], c0)), acc[i][n][2]);
                        acc[i][n][3] = fmaf(s_b, fmaf(16777216.f, lo[n][3], fmaf(1048576.f, hi[n][3], c1)), acc[i][n][3]);
                    }
                }
            }
        } else if (lane == 0) {
            record_device_error(p.errword, W4_DEVERR_TIMEOUT);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);   // the slot's bytes are no longer needed
        if (sl != nsl - 1 || !ok) continue;

        // ---- unit done: split-K partial and ticket, or straight to the epilogue
        const int rb = (bb0 + grp + u * NG) * kTcRB + sub;
        const int row0 = rb * 16;
        if (rb >= ta.nrb) continue;                        // rows past N only
        if (P > 1) {
#pragma unroll
            for (int i = 0; i < NM; ++i)
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int m = n * 8 + 2 * t + (e & 1);
                        const int row = row0 + g + ((e & 2) ? 8 : 0);
                        if (m < ta.m && row < p.N)
                            p.part[(((size_t)piece * NM + i) * ta.m + m) * p.N + row] = acc[i][n][e];
                    }
            __syncwarp();
            unsigned last = 0;
            if (lane == 0) {
                __threadfence();
                last = atomicAdd(&p.counters[rb], 1u) == (unsigned)P - 1;
                if (last) {
                    __threadfence();
                    p.counters[rb] = 0u;
                }
            }
            if (!__shfl_sync(0xFFFFFFFFu, last, 0)) continue;
#pragma unroll
            for (int i = 0; i < NM; ++i)
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int m = n * 8 + 2 * t + (e & 1);
                        const int row = row0 + g + ((e & 2) ? 8 : 0);
                        float v = 0.f;
                        if (m < ta.m && row < p.N)
                            for (int q = 0; q < P; ++q)
                                v += __ldcg(&p.part[(((size_t)q * NM + i) * ta.m + m) * p.N + row]);
                        acc[i][n][e] = v;
                    }
        }

        // ---- epilogue: lane (g, t) holds rows row0+g (e = 0, 1), row0+g+8
        // (e = 2, 3) of activation rows n*8 + 2t + (e & 1)
        if constexpr (EPI == E_QKV_ROPE) {
            // rows 2i and 2i+1 (one RoPE pair) sit in lanes g and g+1
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const float nxt = __shfl_down_sync(0xFFFFFFFFu, acc[0][0][e], 4);
                const int row = row0 + g + ((e & 2) ? 8 : 0);
                if (t == 0 && (g & 1) == 0 && row + 1 < p.N && rope_ok)
                    qkv_rope_epilogue(p, row, acc[0][0][e], nxt, rpos, rpage, rslot);
            }
        } else {
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = n * 8 + 2 * t + (e & 1);
                    const int row = row0 + g + ((e & 2) ? 8 : 0);
                    if (m >= ta.m || row >= p.N) continue;
                    const float v = acc[0][n][e];
                    if constexpr (EPI == E_STORE_F16) {
                        float o = v;
                        if (p.bias) o += __half2float(p.bias[row]);
                        if (p.resid16) o += __half2float(p.resid16[(size_t)m * p.N + row]);
                        p.y16[(size_t)m * p.N + row] = __float2half_rn(o);
                    } else if constexpr (EPI == E_RESID_F32) {
                        p.y32[row] += v;
                    } else if constexpr (EPI == E_SWIGLU) {
                        p.y16[row] = __float2half_rn(v / (1.f + expf(-v)) * acc[NM - 1][n][e]);
                    } else {   // E_ARGMAX
                        if (p.y32) p.y32[row] = v;
                        if (v != v) record_device_error(p.errword, W4_DEVERR_NAN_LOGIT);
                        const unsigned long long kk = argmax_key(v, row);
                        best = kk > best ? kk : best;
                    }
                }
        }
    }

    cp_async_wait<0>();   // no copy outlives the warp

    if constexpr (EPI == E_ARGMAX) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
            best = other > best ? other : best;
        }
        if (lane == 0) s_key[warp] = best;
        named_sync(1, kConsumers);
        if (tid == 0) {
            unsigned long long k = 0ull;
            for (int i = 0; i < CW; ++i) k = s_key[i] > k ? s_key[i] : k;
            if (k) atomicMax(p.amax_key, k);
            __threadfence();
            const unsigned tk = atomicAdd(p.counters + ta.nrb, 1u);
            if (tk == gridDim.x - 1) {
                __threadfence();
                const unsigned long long kk = atomicExch(p.amax_key, 0ull);
                p.token_out[0] = (int32_t)(0xFFFFFFFFu - (uint32_t)(kk & 0xFFFFFFFFull));
                p.counters[ta.nrb] = 0u;
                if (p.pos) p.pos[0] += 1;
            }
        }
    }
}

// ---------------------------------------------------------------- host side
// A plan is scored by a rough time model (microseconds): the busiest SM's
// weight bytes at a per-SM share of HBM bandwidth, its TMA instructions
// (about 0.45 us of the producer each), and the busiest warp's serial work
// (per group of 16 rows, per unit, and the split-K ticket); ties go to fewer
// pieces.  Ring slots per warp group fill the shared-memory budget (at most
// 8, at least 2); twelve consumer warps when that fits, else eight.
inline TcPlan tc_plan(int nm, int xmode, int m, int n, int k) {
    TcPlan best = {};
    const int gpr = k / 128;
    const int nrb = (n + 15) / 16;
    const int nbb = (nrb + kTcRB - 1) / kTcRB;
    const int sms = sm_count();
    double best_cost = 1e30;
    for (int cw : {12, 8}) {
        const int ng = cw / kTcRB;
        for (int P = 1; P <= gpr; ++P) {
            const int gpp = (gpr + P - 1) / P;
            if ((gpr + gpp - 1) / gpp != P) continue;    // P pieces of gpp groups, none empty
            const int nsl = (gpp + kTcMaxSlice - 1) / kTcMaxSlice;
            const int ssz = (gpp + nsl - 1) / nsl;
            TcPlan pl = {};
            pl.a.cw = cw;
            pl.a.P = P;
            pl.a.gpp = gpp;
            pl.a.ssz = ssz;
            pl.a.slot = tc_slot_bytes(nm, ssz);
            pl.a.nrb = nrb;
            pl.a.m = m;
            const size_t rest = tc_smem_rest(xmode, nm, m, gpp, cw);
            if (rest >= kTcSmemMax) continue;
            const size_t qfit = (kTcSmemMax - rest) / ((size_t)ng * pl.a.slot);
            if (qfit < 2) continue;
            pl.a.q = (int)std::min<size_t>(qfit, kTcMaxSlots);
            pl.grid = (int)std::min<long long>(sms, (long long)P * nbb);
            if (pl.grid < P) continue;
            pl.smem = (size_t)pl.a.q * ng * pl.a.slot + rest;
            const int per_piece = pl.grid / P;           // fewest CTAs a piece gets
            const int bb_cta = (nbb + per_piece - 1) / per_piece;
            const int u_grp = (bb_cta + ng - 1) / ng;
            const double t_mem = bb_cta * kTcRB * gpp * nm * 1024.0 / 40e3;   // us at 40 GB/s per SM
            const double t_tma = bb_cta * nsl * 0.45;
            const double t_warp = u_grp * (gpp * nm * 0.15 * (m > 8 ? 1.5 : 1.0) + 0.3 + (P > 1 ? 1.0 : 0.0));
            const double cost = std::max(std::max(t_mem, t_tma), t_warp) + (P > 1 ? 0.5 : 0.0) + 0.001 * P;
            if (cost < best_cost) {
                best_cost = cost;
                best = pl;
            }
        }
        if (best.grid > 0) break;
    }
    return best;
}

inline size_t tc_ws_bytes(const TcPlan& pl, int nm) {
    const size_t part = pl.a.P > 1 ? (size_t)pl.a.P * nm * pl.a.m * pl.a.nrb * 16 * sizeof(float) : 0;
    return ((part + 255) / 256) * 256 + (size_t)(pl.a.nrb + 1) * sizeof(unsigned);
}

template <int NT, int XMODE, int EPI, int CW>
inline cudaError_t tc_launch_cw(const GemvParams& p, const TcPlan& pl, const CUtensorMap& tm0, const CUtensorMap& tm1,
                                cudaStream_t st, bool pdl) {
    auto kern = gemv_tc_kernel<NT, XMODE, EPI, CW>;
    static size_t attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || attr_set[dev] < pl.smem) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = pl.smem;
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
    return cudaLaunchKernelEx(&cfg, kern, p, pl.a, tm0, tm1);
}

template <int XMODE, int EPI>
inline cudaError_t tc_launch(const GemvParams& p, const TcPlan& pl, const CUtensorMap& tm0, const CUtensorMap& tm1,
                             cudaStream_t st, bool pdl) {
    if (pl.a.m > 8) {
        if constexpr (XMODE == X_F16 && EPI == E_STORE_F16) {
            return pl.a.cw == 12 ? tc_launch_cw<2, XMODE, EPI, 12>(p, pl, tm0, tm1, st, pdl)
                                 : tc_launch_cw<2, XMODE, EPI, 8>(p, pl, tm0, tm1, st, pdl);
        }
        return cudaErrorInvalidValue;
    }
    return pl.a.cw == 12 ? tc_launch_cw<1, XMODE, EPI, 12>(p, pl, tm0, tm1, st, pdl)
                         : tc_launch_cw<1, XMODE, EPI, 8>(p, pl, tm0, tm1, st, pdl);
}

}  // namespace w4
