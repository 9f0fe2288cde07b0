// Batched W4A16 GEMV (1 <= M <= 16 activation rows) on tensor cores.
//
// Same operation as gemv.cuh ("How to build your own LLM runtime from
// scratch (Towards Data Science)", "What it actually builds": GEMVs over INT4
// group-128 weights with fp16 activations and the dequantization fused into
// the dot product).  With several activation rows the projection is a real
// dense contraction, so the products run on mma.sync m16n8k16 (fp16 inputs,
// fp32 accumulation) and the CUDA cores only unpack the weights:
//  * A warp owns 16 weight rows over a K range (split-K over grid.y) and all
//    M activation rows (one or two 8-column n-tiles).
//  * Lane (g, t) fetches, per 128-group, the 16 bytes t of rows g and g+8
//    (32 weights each), so a quad of lanes reads one row's 64-byte group
//    segment.  A dot product does not depend on the order of its K terms, so
//    each k-step takes, in lane (g, t), four weights of its own segment from
//    each row, and the activation rows supply the same four K indices.
//  * Unpacking is one AND per element pair: the nibble pair masked in place
//    reads as the fp16 subnormals u * 2^-24 (low nibble of a byte) or
//    u * 2^-20 (high nibble).  Low and high nibbles feed separate MMAs into
//    separate fp32 fragments, so every product is exact, and per group
//        sum q x = 2^24 lo + 2^20 hi - 8 sum x      (q = u - 8),
//    with sum x per activation row and group computed while staging.  The
//    group scale then multiplies the group's fp32 dot product, so no rounding
//    is added before fp32 accumulation.
//  * Weights stream through a per-warp ring of S one-KiB slots in shared
//    memory filled by cp.async (16 bytes per lane and row); every lane reads
//    back only what it copied, so a thread's own cp.async.wait_group is the
//    only synchronisation.  S-1 groups per warp are in flight.
//    Group scales follow in registers, also S-1 groups ahead.
//  * The M activation rows are staged once per CTA by cp.async, the 16-byte
//    units of a row XOR-swizzled so the 128-bit fragment loads are
//    conflict-free; the group sums are then taken from shared memory.
//  * Split-K partials go to the workspace; the last CTA of a row block adds
//    them in a fixed order (deterministic).
#pragma once

#include "gemv.cuh"

namespace w4 {

constexpr int kMmaWarps = 16;                  // warps per CTA
constexpr int kMmaKSplit = 2;                  // warps sharing a 16-row tile, each on its own K part
constexpr int kMmaRows = 16 * kMmaWarps / kMmaKSplit;   // 128 rows per CTA
constexpr int kMmaSlots = 8;                   // ring slots (KiB) per warp, one n-tile (M <= 8)
constexpr int kMmaSlots2 = 4;                  // two n-tiles: leaves room for 16 staged rows
constexpr int kMmaMinBlocks = 1;
constexpr size_t kMmaSmemMax = 200 * 1024;

__device__ __forceinline__ void mma_16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// same with a zero accumulator in
__device__ __forceinline__ void mma_16816_f16_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// staged activation row m: 16-byte unit c (c = 16*group + 4*t + u) sits at
// c ^ swz(m, t); the XOR only permutes the four units of one lane's segment
__host__ __device__ __forceinline__ int mma_swz(int m, int t) { return ((m & 1) << 1) | ((t >> 1) & 1); }

// shared memory: weight rings [W][S][2][32] x 16 B | activations [M][kc*32]
// halves | group sums [kc/4][NT*8] floats
__host__ __device__ inline size_t mma_smem_bytes(int w, int s, int m, int nt, int kc) {
    const size_t ring = (size_t)w * s * 1024;
    const size_t xs = (size_t)m * kc * 32 * 2;
    const size_t sx = (size_t)(kc / 4) * nt * 8 * 4;
    return ring + xs + sx;
}

// NT: 8-column n-tiles (1 for M <= 8, 2 for M <= 16); W warps; S ring slots
// per warp (a power of two); MINB CTAs per SM; KS warps share each 16-row
// tile, warp w taking K part w / (W/KS) of the CTA's range (their partial
// sums meet in shared memory, in a fixed order)
template <int NT, int W = kMmaWarps, int S = kMmaSlots, int MINB = kMmaMinBlocks, int KS = kMmaKSplit>
__global__ void __launch_bounds__(W * 32, MINB)
gemv_mma_kernel(const GemvParams p) {
    static_assert((S & (S - 1)) == 0 && S >= 2, "ring slots: a power of two");
    static_assert(W % KS == 0 && S * 1024 >= 32 * NT * 4 * 4, "K parts; the ring holds a warp's partials");
    constexpr int WR = W / KS;                     // row tiles per CTA
    extern __shared__ __align__(16) unsigned char mma_smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int cb = blockIdx.y * p.kc;
    const int ce = min(p.K >> 5, cb + p.kc);
    const int k0 = cb * 32;
    const int kl = ce * 32 - k0;                   // this CTA's K range, whole groups
    const int ngrp_cta = kl >> 7;
    const int units = kl >> 3;                     // 16-byte units per staged row
    const int rt = warp % WR, kh = warp / WR;      // row tile, K part
    const int gw0 = kh * ngrp_cta / KS;            // this warp's groups: gw0 .. gw0+ngrp-1
    const int ngrp = (kh + 1) * ngrp_cta / KS - gw0;
    uint4* xs = reinterpret_cast<uint4*>(mma_smem_raw + (size_t)W * S * 1024);
    float* sx = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(xs) + (size_t)p.M * units * 16);

    // ---- the weight ring fills first (weights are never written by an
    // earlier kernel, so this may precede the dependency wait); scales ride
    // along in registers, S-1 groups ahead
    const int row0 = blockIdx.x * (16 * WR) + rt * 16;
    const int ra = min(row0 + g, p.N - 1), rb = min(row0 + g + 8, p.N - 1);   // clamped rows stay in bounds
    const uint4* wa = reinterpret_cast<const uint4*>(p.w0 + (size_t)ra * (p.K >> 3) + (k0 >> 3)) + t + 4 * gw0;
    const uint4* wb = reinterpret_cast<const uint4*>(p.w0 + (size_t)rb * (p.K >> 3) + (k0 >> 3)) + t + 4 * gw0;
    const __half* sa = p.s0 + (size_t)ra * (p.K >> 7) + (k0 >> 7) + gw0;
    const __half* sb = p.s0 + (size_t)rb * (p.K >> 7) + (k0 >> 7) + gw0;
    // slot layout: [row g part: 32 lanes x 16 B][row g+8 part: 32 lanes x 16 B]
    const uint32_t ring = smem_u32(mma_smem_raw + (size_t)warp * S * 1024) + lane * 16;
    __half ha[S], hb[S];
#pragma unroll
    for (int s = 0; s < S - 1; ++s) {
        if (s < ngrp) {
            cp_async16(ring + s * 1024, wa + 4 * s);
            cp_async16(ring + s * 1024 + 512, wb + 4 * s);
            ha[s] = sa[s];
            hb[s] = sb[s];
        }
        cp_async_commit();
    }

    pdl_wait();
    // ---- stage the M activation rows: each 16-byte unit straight to its
    // swizzled place
    const uint32_t xs_u32 = smem_u32(xs);
    for (int i = tid; i < p.M * units; i += W * 32) {
        const int m = i / units, c = i - m * units;   // (the CTA stages its whole K range)
        cp_async16(xs_u32 + (uint32_t)(m * units + (c ^ mma_swz(m, (c >> 2) & 3))) * 16,
                   p.x + (size_t)m * p.K + k0 + c * 8);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    // ---- group sums of the activation rows: 16 consecutive units are one
    // group of one row (in swizzled order; the sum does not care).  units is
    // a multiple of 16 and the trip count uniform, so the shuffles are safe.
    for (int base = 0; base < p.M * units; base += W * 32) {
        const int i = base + tid;
        const bool ok = i < p.M * units;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (ok) v = xs[i];
        const float2 f0 = __half22float2(u32_as_h2(v.x)), f1 = __half22float2(u32_as_h2(v.y));
        const float2 f2 = __half22float2(u32_as_h2(v.z)), f3 = __half22float2(u32_as_h2(v.w));
        float sum = ((f0.x + f0.y) + (f1.x + f1.y)) + ((f2.x + f2.y) + (f3.x + f3.y));
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (ok && (i & 15) == 0) {
            const int m = i / units, c = i - m * units;
            sx[(c >> 4) * (NT * 8) + m] = sum;
        }
    }
    __syncthreads();

    // B fragment rows of this lane: activation rows g and 8+g, clamped to
    // M-1 (columns >= M are computed from a copy and never stored); the four
    // units of the lane's segment in swizzled order
    int xu[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const int m = min(n * 8 + g, p.M - 1);
        const int swz = mma_swz(m, t);
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) xu[n][wi] = m * units + 4 * t + (wi ^ swz);
    }
    const float* sxl = sx + 2 * t + gw0 * (NT * 8);
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) xu[n][wi] += gw0 * 16;

    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

    for (int gb = 0; gb < ngrp; gb += S) {
#pragma unroll
        for (int j = 0; j < S; ++j) {
            const int gi = gb + j;
            if (gi >= ngrp) break;   // uniform
            {
                // refill the slot consumed last iteration with group gi + S - 1
                const int gn = gi + S - 1, sn = (j + S - 1) & (S - 1);
                if (gn < ngrp) {
                    cp_async16(ring + sn * 1024, wa + 4 * gn);
                    cp_async16(ring + sn * 1024 + 512, wb + 4 * gn);
                    ha[sn] = sa[gn];
                    hb[sn] = sb[gn];
                }
                cp_async_commit();
            }
            cp_async_wait<S - 1>();   // this thread's copies of group gi have landed
            const uint4 qa = lds128(ring + j * 1024), qb = lds128(ring + j * 1024 + 512);
            const uint32_t A[4] = {qa.x, qa.y, qa.z, qa.w};
            const uint32_t B[4] = {qb.x, qb.y, qb.z, qb.w};
            const float s_a = __half2float(ha[j]), s_b = __half2float(hb[j]);
            float lo[NT][4], hi[NT][4];
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
                uint4 xb[NT];
#pragma unroll
                for (int n = 0; n < NT; ++n) xb[n] = xs[xu[n][wi] + gi * 16];
                const uint32_t a8 = A[wi] >> 8, b8 = B[wi] >> 8;
                // elements 0,1 | 4,5 (x: .x, .z) and 2,3 | 6,7 (x: .y, .w) of word wi
                const uint32_t fl[4] = {A[wi] & 0x000F000Fu, B[wi] & 0x000F000Fu, a8 & 0x000F000Fu, b8 & 0x000F000Fu};
                const uint32_t fh[4] = {A[wi] & 0x00F000F0u, B[wi] & 0x00F000F0u, a8 & 0x00F000F0u, b8 & 0x00F000F0u};
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    if (wi == 0) {
                        mma_16816_f16_z(lo[n], fl, xb[n].x, xb[n].z);
                        mma_16816_f16_z(hi[n], fh, xb[n].y, xb[n].w);
                    } else {
                        mma_16816_f16(lo[n], fl, xb[n].x, xb[n].z);
                        mma_16816_f16(hi[n], fh, xb[n].y, xb[n].w);
                    }
                }
            }
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const float2 sm = *reinterpret_cast<const float2*>(sxl + gi * (NT * 8) + n * 8);
                const float c0 = -8.f * sm.x, c1 = -8.f * sm.y;
                acc[n][0] = fmaf(s_a, fmaf(16777216.f, lo[n][0], fmaf(1048576.f, hi[n][0], c0)), acc[n][0]);
                acc[n][1] = fmaf(s_a, fmaf(16777216.f, lo[n][1], fmaf(1048576.f, hi[n][1], c1)), acc[n][1]);
                acc[n][2] = fmaf(s_b, fmaf(16777216.f, lo[n][2], fmaf(1048576.f, hi[n][2], c0)), acc[n][2]);
                acc[n][3] = fmaf(s_b, fmaf(16777216.f, lo[n][3], fmaf(1048576.f, hi[n][3], c1)), acc[n][3]);
            }
        }
    }
    cp_async_wait<0>();   // no copy outlives the CTA
    pdl_trigger();

    if constexpr (KS > 1) {
        // K parts 1.. leave their partials in their own (now idle) ring; part 0 adds them in order
        __syncwarp();
        float* mine = reinterpret_cast<float*>(mma_smem_raw + (size_t)warp * S * 1024) + lane * NT * 4;
        if (kh > 0) {
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) mine[n * 4 + e] = acc[n][e];
        }
        __syncthreads();
        if (kh == 0) {
#pragma unroll
            for (int q = 1; q < KS; ++q) {
                const float* other =
                    reinterpret_cast<const float*>(mma_smem_raw + (size_t)(warp + q * WR) * S * 1024) + lane * NT * 4;
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[n][e] += other[n * 4 + e];
            }
        }
    }

    // ---- lane holds rows row0+g (e = 0, 1) and row0+g+8 (e = 2, 3) of
    // activation rows n*8 + 2t + (e & 1)
    __shared__ int s_last;
    if (p.split > 1) {
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = n * 8 + 2 * t + (e & 1);
                const int row = row0 + g + ((e & 2) ? 8 : 0);
                if (kh == 0 && m < p.M && row < p.N) p.part[((size_t)blockIdx.y * p.M + m) * p.N + row] = acc[n][e];
            }
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            const unsigned tk = atomicAdd(&p.counters[blockIdx.x], 1u);
            const bool last = tk == (unsigned)p.split - 1;
            if (last) __threadfence();
            s_last = last;
        }
        __syncthreads();
        if (!s_last) return;  // uniform over the CTA
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = n * 8 + 2 * t + (e & 1);
                const int row = row0 + g + ((e & 2) ? 8 : 0);
                float v = 0.f;
                if (kh == 0 && m < p.M && row < p.N)
                    for (int sp = 0; sp < p.split; ++sp) v += __ldcg(&p.part[((size_t)sp * p.M + m) * p.N + row]);
                acc[n][e] = v;
            }
        if (tid == 0) p.counters[blockIdx.x] = 0u;
    }
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int m = n * 8 + 2 * t + (e & 1);
            const int row = row0 + g + ((e & 2) ? 8 : 0);
            if (kh == 0 && m < p.M && row < p.N) {
                float v = acc[n][e];
                if (p.bias) v += __half2float(p.bias[row]);
                if (p.resid16) v += __half2float(p.resid16[(size_t)m * p.N + row]);
                p.y16[(size_t)m * p.N + row] = __float2half_rn(v);
            }
        }
}

struct MmaPlan {
    int split;
    int kc;       // chunks (32 weights) per split piece: whole groups
    dim3 grid;
    size_t smem;
};

// About one CTA per SM: split K into the whole number of pieces that brings
// row blocks x pieces nearest the SM count (measured on GB300: a 148-CTA
// unsplit grid beat a 296-CTA split one for 18944 x 3584), and further while
// the staged rows exceed the shared-memory budget.
inline MmaPlan mma_plan(int m, int n, int k) {
    MmaPlan pl;
    const int nt = m <= 8 ? 1 : 2;
    const int groups = k / 128;
    const int row_blocks = (n + kMmaRows - 1) / kMmaRows;
    int s = (2 * kMmaMinBlocks * sm_count() + row_blocks) / (2 * row_blocks);   // rounded ratio
    s = s < 1 ? 1 : (s > groups ? groups : s);
    const int slots = nt == 1 ? kMmaSlots : kMmaSlots2;
    while (mma_smem_bytes(kMmaWarps, slots, m, nt, ((groups + s - 1) / s) * 4) > kMmaSmemMax && s < groups) ++s;
    const int gpp = (groups + s - 1) / s;
    pl.kc = gpp * 4;
    pl.split = (groups + gpp - 1) / gpp;
    pl.grid = dim3(row_blocks, pl.split, 1);
    pl.smem = mma_smem_bytes(kMmaWarps, slots, m, nt, pl.kc);
    return pl;
}

inline size_t mma_ws_bytes(const MmaPlan& pl, int m, int n) {
    const size_t part = pl.split > 1 ? (size_t)pl.split * m * n * sizeof(float) : 0;
    return ((part + 255) / 256) * 256 + (size_t)pl.grid.x * sizeof(unsigned);
}

template <int NT>
inline cudaError_t mma_launch_nt(const GemvParams& p, const MmaPlan& pl, cudaStream_t st) {
    auto kern = gemv_mma_kernel<NT, kMmaWarps, NT == 1 ? kMmaSlots : kMmaSlots2>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMmaSmemMax);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    kern<<<pl.grid, kMmaWarps * 32, pl.smem, st>>>(p);
    return cudaGetLastError();
}

inline cudaError_t mma_launch(const GemvParams& p, const MmaPlan& pl, cudaStream_t st) {
    return p.M <= 8 ? mma_launch_nt<1>(p, pl, st) : mma_launch_nt<2>(p, pl, st);
}

}  // namespace w4
