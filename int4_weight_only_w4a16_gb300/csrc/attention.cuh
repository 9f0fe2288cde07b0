// Paged GQA decode attention (split over the sequence, merged in one pass).
//
// Operation: "How to build your own LLM runtime from scratch (Towards Data
// Science)", section "What it actually builds" (attention over a paged KV
// cache, 16 tokens per 4 KiB page) and "Two more honest findings" (a block
// barrier inside a warp-id branch corrupted the softmax at page boundaries);
// "How To Build Your Own LLM Runtime From Scratch | daily.dev", second
// question (partial KV tail pages).
//
// Design for sm_103a:
//  * Work unit = (sequence b, KV head g, split s).  A CTA of 4 warps owns
//    4*ppw consecutive pages of the sequence; each warp owns ppw of them and
//    runs its own 2-stage pipeline: every lane copies 16-byte pieces of the
//    4 KiB K and V page tiles with cp.async (in the 128-byte swizzled layout
//    ldmatrix reads without bank conflicts), so 32 lanes issue a page at
//    once instead of one thread issuing tile copies one after another.  No
//    block barrier is ever reached by only some warps: the only
//    __syncthreads() calls sit in code every thread of the CTA executes.
//  * The GQA group (up to 16 query heads sharing head g) is one 16-row MMA
//    tile: S = Q K^T and O += P V run on mma.sync m16n8k16 (fp16 in, fp32
//    accumulate), which makes the 7x16x128 tile products a dense contraction
//    and keeps the kernel HBM-bound.  tcgen05 would need M >= 64 rows for a
//    7-row tile and buys nothing on a bandwidth-bound kernel.
//  * Online softmax in the log2 domain; tokens at or past L in the tail page
//    get score -inf and their V rows are zeroed in shared memory before the
//    PV product, so stale slots (even NaN) never reach the output.
//  * The 4 warps merge in shared memory, each CTA publishes (m, l, O) to the
//    workspace, and the last CTA of (b, g) -- an atomic ticket, no waiting --
//    merges the splits in a fixed order: deterministic output.
#pragma once

#include <cuda.h>

#include <algorithm>

#include "common.cuh"

namespace w4 {

constexpr int kAttnWarps = 4;
constexpr int kAttnMaxCluster = 16;   // splits of one (b, g) merged through distributed shared memory
// Row stride (floats) of the per-warp partial outputs in shared memory: a lane
// quad's 8-byte pairs of rows gid and gid + 4 then fall in different banks.
constexpr int kSoStride = 136;
constexpr int kPageTokens = 16;
constexpr int kHeadDim = 128;
constexpr int kTileBytes = kPageTokens * kHeadDim * 2;      // 4096: one page, one head, K or V
constexpr int kStageBytes = 2 * kTileBytes;                  // K + V
// Cluster merge: what the splits push to the CTA that merges a column slice --
// [split][16 rows][slice columns] fp32 partial outputs (at most 45 * 64 floats,
// for 15 splits of 12 columns) and [split][16 rows] (m, l) pairs.
constexpr int kAttnRecvOFloats = 2880;
constexpr int kAttnRecvBytes = kAttnRecvOFloats * 4 + kAttnMaxCluster * 16 * 2 * 4;
// per-warp page rings of `stages` pages (+ the cluster merge's receive area), plus alignment slack
__host__ __device__ constexpr int attn_smem_bytes(int stages, bool cluster) {
    return kAttnWarps * stages * kStageBytes + (cluster ? kAttnRecvBytes : 0) + 1024;
}

struct AttnParams {
    const __half* q;          // [B][Hq][128]
    __half* out;              // [B][Hq][128]
    const __half* k_pool;     // [num_pages][Hkv][16][128]
    const __half* v_pool;
    const int32_t* pt;        // [B][max_pages]
    const int32_t* lens;      // [B]
    const int32_t* pos_hint;  // decode (B = 1): the new token's position, final before the previous
                              // kernel ends: L = *pos_hint + 1, and every page but the last one may be
                              // loaded before waiting on that kernel (the last gets this step's K/V row)
    float* part_o;            // [B][Hq][max_splits][128]
    float* part_ml;           // [B][Hq][max_splits][2]
    unsigned* counters;       // [B][Hkv]
    int* errword;
    float scale_log2;         // softmax scale * log2(e)
    int B, Hq, Hkv, group;
    int max_pages, num_pages, max_context;
    int ppw;                  // pages per warp
    int max_splits;
    int pt_shared;            // 1: every query reads row 0 of pt (one sequence, many positions)
    const void* pf0;          // optional L2 warm-up of the next kernel's weights
    size_t pf0_bytes;
    const void* pf1;
    size_t pf1_bytes;
};

// Causal attention of a block of prompt rows over one sequence's paged cache:
// prompt row t (position start + t) attends to positions 0 .. start + t.
struct PrefillAttnParams {
    const __half* q;          // [n][Hq][128], RoPE applied
    __half* out;              // [n][Hq][128]
    const int32_t* pt;        // [max_pages] page table of the sequence
    float* part_o;            // split partials [qblocks][Hkv][max_splits][group][16][128]
    float* part_ml;           // [qblocks][Hkv][max_splits][group][16][2]
    unsigned* counters;       // [qblocks][Hkv], zero between launches
    int n, start;
    int Hq, Hkv, group;
    int max_pages, num_pages;
    int ppc, max_splits;      // pages per split, splits per 16-row block
    float scale_log2;         // softmax scale * log2(e)
    int* errword;
};

#ifdef W4_DEFINE_ATTENTION_KERNEL  // the kernels live in attention.cu only
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of (row, column) inside a tile stored as two 64-column boxes of
// [16 rows][128 bytes] with the TMA 128-byte swizzle (16-byte chunk index
// XOR row % 8).  `col` is a multiple of 8 (one 16-byte chunk).
__device__ __forceinline__ uint32_t tile_off(int row, int col) {
    return (uint32_t)((col >> 6) * 2048 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    return h2_as_u32(__floats2half2_rn(lo, hi));
}

constexpr uint64_t kWaitLimit = 1000000000ull;  // 1 s: a page load takes microseconds

// Wait until at most n (0..3) of this thread's cp.async groups are pending.
__device__ __forceinline__ void cp_async_wait_upto(int n) {
    if (n >= 3) asm volatile("cp.async.wait_group 3;" ::: "memory");
    else if (n == 2) asm volatile("cp.async.wait_group 2;" ::: "memory");
    else if (n == 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
    else asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// The CTAs of one cluster (CLUSTER = true) are the splits of one (b, g): every
// CTA reaches both cluster barriers, active or not, and none leaves early.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The same barrier, returning 0 from inside the asm: addresses offset by it
// cannot be computed (and the loads through them cannot be issued) before it.
__device__ __forceinline__ uint32_t cluster_sync_token() {
    uint32_t t;
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;\n\tmov.u32 %0, 0;"
        : "=r"(t)::"memory");
    return t;
}
// Split arrive / wait on the cluster barrier (each thread alternates them).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ void st_cluster_f32(uint32_t cluster_address, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_address), "f"(v) : "memory");
}
// Loads from a peer CTA's shared memory.  Plain (not volatile) so that the
// compiler may issue many of them before the first is used; the cluster barrier
// before them orders them after the peers' writes.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local_addr, uint32_t rank) {
    uint32_t ra;
    asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
    return ra;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t cluster_address) {
    float v;
    asm("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_address));
    return v;
}
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t cluster_address) {
    float4 v;
    asm("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "r"(cluster_address));
    return v;
}

template <bool CLUSTER, int STAGES>
__global__ void __launch_bounds__(kAttnWarps * 32)
paged_attention_kernel(const AttnParams p) {
    extern __shared__ unsigned char att_smem_raw[];
    __shared__ float s_m[kAttnWarps][16], s_l[kAttnWarps][16];
    __shared__ float s_fm[16], s_fl[16];   // this split's merged (m, l) per row
    __shared__ float s_f[kAttnWarps][16];   // per row: each warp's weight exp2(m_w - m)
    static_assert(kAttnWarps * 32 == kHeadDim, "the CTA merge gives each thread one output column");
    __shared__ int s_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    // CLUSTER: the first phase of the cluster barrier only shows that every CTA of the
    // cluster has started (so that its shared memory may be written); it is waited on
    // just before the first remote store, long after every CTA arrived
    if constexpr (CLUSTER) cluster_arrive_relaxed();

    // the next kernel may start streaming its own inputs on SMs this grid leaves free
    pdl_trigger();
    if (tid == 0) {  // this kernel moves little data: warm L2 with the next kernel's weights
        const int ctas = gridDim.x * gridDim.y * gridDim.z;
        const int me = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
        l2_prefetch_share(p.pf0, p.pf0_bytes, me, ctas);
        l2_prefetch_share(p.pf1, p.pf1_bytes, me, ctas);
    }
    const bool early = p.pos_hint != nullptr;
    const int per_cta = kAttnWarps * p.ppw;
    const int cta_p0 = split * per_cta;
    const int32_t* ptb = p.pt + (p.pt_shared ? (size_t)0 : (size_t)b * p.max_pages);
    const int gid = lane >> 2, tig = lane & 3;
    // Q fragments (A operand, 16 rows = GQA group padded with zeros)
    uint32_t qa[8][4];
    auto load_q = [&]() {
        const int r0 = gid, r1 = gid + 8;
        const __half* q0 = p.q + ((size_t)b * p.Hq + (size_t)g * p.group + r0) * kHeadDim;
        const __half* q1 = p.q + ((size_t)b * p.Hq + (size_t)g * p.group + r1) * kHeadDim;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int c = ks * 16 + 2 * tig;
            qa[ks][0] = r0 < p.group ? *reinterpret_cast<const uint32_t*>(q0 + c) : 0u;
            qa[ks][1] = r1 < p.group ? *reinterpret_cast<const uint32_t*>(q1 + c) : 0u;
            qa[ks][2] = r0 < p.group ? *reinterpret_cast<const uint32_t*>(q0 + c + 8) : 0u;
            qa[ks][3] = r1 < p.group ? *reinterpret_cast<const uint32_t*>(q1 + c + 8) : 0u;
        }
    };
    if (!early) pdl_wait();
    // one round trip for the length, this CTA's page ids (read before the length is
    // known: every id of the CTA's range the table holds) and, unless the queries
    // come from the kernel still running, the queries
    const int i0 = cta_p0 + tid;
    const int L = early ? *p.pos_hint + 1 : p.lens[b];
    const int pid0 = (tid < per_cta && i0 < p.max_pages) ? ptb[i0] : 0;
    if (!early) load_q();
    const bool len_ok = L >= 1 && L <= p.max_context && L <= p.max_pages * kPageTokens;
    if (!len_ok) {
        if (tid == 0 && split == 0) record_device_error(p.errword, W4_DEVERR_CONTEXT);
        if constexpr (!CLUSTER) return;   // uniform for the CTA
    }
    const int npages = len_ok ? (L + kPageTokens - 1) / kPageTokens : 0;
    const int nsplit = (npages + per_cta - 1) / per_cta;
    if constexpr (!CLUSTER) {
        if (split >= nsplit) return;  // uniform
    }
    const int cta_p1 = min(npages, cta_p0 + per_cta);

    // validate this CTA's page ids before any copy is issued
    int bad = (tid < per_cta && i0 < cta_p1) ? (pid0 < 0 || pid0 >= p.num_pages) : 0;
    for (int i = i0 + blockDim.x; i < cta_p1; i += blockDim.x) {   // ranges longer than the block
        const int pg = ptb[i];
        bad |= (pg < 0 || pg >= p.num_pages);
    }
    const int anybad = __syncthreads_or(bad);
    if (anybad) {
        if (tid == 0) record_device_error(p.errword, W4_DEVERR_PAGE_ID);
        if constexpr (!CLUSTER) return;  // uniform
    }

    unsigned char* tiles = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(att_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // CLUSTER: this split has pages and none of them is bad (inactive splits still
    // meet the cluster barriers and merge their column slice)
    const bool active = !CLUSTER || (cta_p0 < cta_p1 && !anybad);

    const int wp0 = min(cta_p1, cta_p0 + warp * p.ppw);
    const int wp1 = min(cta_p1, wp0 + p.ppw);
    const int npw = active ? max(0, wp1 - wp0) : 0;
    unsigned char* wtiles = tiles + (size_t)warp * STAGES * kStageBytes;

    // page wp0 + j into stage j % STAGES: lane l copies pieces l, l + 32, ...
    // (row = piece / 16, 16-byte column chunk = piece % 16) of the K and V tiles
    // into the swizzled layout of tile_off, then commits one cp.async group
    auto issue = [&](int j) {
        const int st = j % STAGES;
        const size_t tile = ((size_t)ptb[wp0 + j] * p.Hkv + g) * (kPageTokens * kHeadDim);
        const unsigned char* ks = reinterpret_cast<const unsigned char*>(p.k_pool + tile);
        const unsigned char* vs = reinterpret_cast<const unsigned char*>(p.v_pool + tile);
        const uint32_t kd = smem_u32(wtiles + st * kStageBytes), vd = kd + kTileBytes;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int piece = lane + 32 * i, r = piece >> 4, c = piece & 15;
            const uint32_t off = tile_off(r, c * 8);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(kd + off), "l"(ks + piece * 16) : "memory");
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(vd + off), "l"(vs + piece * 16) : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    // the page holding position L - 1 receives this step's K/V row from the
    // previous kernel: with an early start it is loaded after the wait (it is the
    // last page of the sequence, so its warp issues nothing after it)
    const int last_page = npages - 1;
    int deferred = -1;
    for (int j = 0; j < min(npw, STAGES); ++j) {
        if (early && wp0 + j == last_page) deferred = j;
        else issue(j);
    }
    if (early) {
        pdl_wait();
        if (deferred >= 0) issue(deferred);
        load_q();
    }

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows gid, gid+8

    for (int j = 0; j < npw; ++j) {
        const int st = j % STAGES;
        // this lane's copies of page j have landed (the later pages' may still be in
        // flight: pages j + 1 .. min(npw, j + STAGES) - 1 were issued after it); the
        // warp barrier then makes every lane's pieces visible to all
        cp_async_wait_upto(min(STAGES - 1, npw - 1 - j));
        __syncwarp();
        unsigned char* kt = wtiles + st * kStageBytes;
        unsigned char* vt = kt + kTileBytes;
        const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
        const int valid = min(kPageTokens, L - (wp0 + j) * kPageTokens);

        // ---- S = Q K^T : two 8-token n-tiles, eight 16-dim k-steps (even and odd
        // k-steps in separate accumulators: two independent MMA chains per n-tile)
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
            const int mat = lane >> 3, i = lane & 7;
            const int tok = 8 * (mat >> 1) + i;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t b00, b01, b10, b11;
                ldsm_x4(kbase + tile_off(tok, ks * 16 + 8 * (mat & 1)), b00, b01, b10, b11);
                mma_16816(s[0], qa[ks], b00, b01);
                mma_16816(s[1], qa[ks], b10, b11);
            }
        }
        // ---- mask the tail, online softmax (log2 domain)
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = nt * 8 + 2 * tig + (e & 1);
                const float v = tok < valid ? s[nt][e] * p.scale_log2 : -INFINITY;
                s[nt][e] = v;
                if (e < 2) mx0 = fmaxf(mx0, v);
                else mx1 = fmaxf(mx1, v);
            }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float c0 = exp2f(m0 - mn0), c1 = exp2f(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            s[nt][0] = exp2f(s[nt][0] - mn0);
            s[nt][1] = exp2f(s[nt][1] - mn0);
            s[nt][2] = exp2f(s[nt][2] - mn1);
            s[nt][3] = exp2f(s[nt][3] - mn1);
            ps0 += s[nt][0] + s[nt][1];
            ps1 += s[nt][2] + s[nt][3];
        }
        l0 = l0 * c0 + ps0;
        l1 = l1 * c1 + ps1;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            o[i][0] *= c0;
            o[i][1] *= c0;
            o[i][2] *= c1;
            o[i][3] *= c1;
        }
        // ---- zero V rows past the end of the sequence (tail page only)
        if (valid < kPageTokens) {
            for (int idx = lane; idx < (kPageTokens - valid) * 16; idx += 32) {
                const int r = valid + (idx >> 4), c = idx & 15;
                *reinterpret_cast<uint4*>(vt + (c >> 3) * 2048 + r * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
        }
        // ---- O += P V
        uint32_t pa[4];
        pa[0] = pack_h2(s[0][0], s[0][1]);
        pa[1] = pack_h2(s[0][2], s[0][3]);
        pa[2] = pack_h2(s[1][0], s[1][1]);
        pa[3] = pack_h2(s[1][2], s[1][3]);
        {
            const int mat = lane >> 3, i = lane & 7;
            const int tok = 8 * (mat & 1) + i;
#pragma unroll
            for (int nd = 0; nd < 16; nd += 2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vbase + tile_off(tok, 8 * (nd + (mat >> 1))), b0, b1, b2, b3);
                mma_16816(o[nd], pa, b0, b1);
                mma_16816(o[nd + 1], pa, b2, b3);
            }
        }
        // ---- release the stage and refill it
        __syncwarp();
        if (j + STAGES < npw) issue(j + STAGES);
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    // ---- merge the warps of this CTA (every thread reaches these barriers)
    __syncthreads();
    float* so = reinterpret_cast<float*>(tiles);  // [warps][16][kSoStride]
    if (tig == 0) {
        s_m[warp][gid] = m0;
        s_m[warp][gid + 8] = m1;
        s_l[warp][gid] = l0;
        s_l[warp][gid + 8] = l1;
    }
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
        const int c = nd * 8 + 2 * tig;
        *reinterpret_cast<float2*>(so + ((size_t)warp * 16 + gid) * kSoStride + c) = make_float2(o[nd][0], o[nd][1]);
        *reinterpret_cast<float2*>(so + ((size_t)warp * 16 + gid + 8) * kSoStride + c) = make_float2(o[nd][2], o[nd][3]);
    }
    __syncthreads();
    // per row, once: the merged max, each warp's weight and the merged sum
    if (tid < 16) {
        const int r = tid;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, s_m[w][r]);
        float Ls = 0.f;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) {
            const float f = s_m[w][r] == -INFINITY ? 0.f : exp2f(s_m[w][r] - M);
            s_f[w][r] = f;
            Ls = fmaf(f, s_l[w][r], Ls);
        }
        s_fm[r] = (CLUSTER && !active) ? -INFINITY : M;
        s_fl[r] = (CLUSTER && !active) ? 0.f : Ls;
    }
    __syncthreads();
    // thread = output column: its column of every row of the group, the warps'
    // partials weighted (the rows are independent, so their loads overlap)
    const int col = tid;
    if constexpr (CLUSTER) {
        // Column slice d (four-column groups q0(d) .. q0(d) + q4per) is merged by CTA d
        // of the cluster: every split pushes its rows of each slice, and its (m, l) per
        // row, into that CTA's receive area (distributed shared memory stores, no global
        // round trip); after one cluster barrier each CTA merges from its own shared
        // memory and no CTA reads another's, so none waits for the others to finish.
        const int cs = gridDim.x;                         // splits in the cluster (its size)
        const int q4per = (kHeadDim / 4 + cs - 1) / cs;   // four-column groups per slice
        const int sw = 4 * q4per;                         // columns per slice
        float* recv_o = reinterpret_cast<float*>(tiles + (size_t)kAttnWarps * STAGES * kStageBytes);
        float* recv_ml = recv_o + kAttnRecvOFloats;       // [split][16][2]
        cluster_wait();   // every CTA of the cluster has started
        {
            const int d = col / sw, cc = col - d * sw;
            const uint32_t dst = cluster_addr(smem_u32(recv_o + (size_t)split * 16 * sw + cc), (uint32_t)d);
#pragma unroll 4
            for (int r = 0; r < p.group; ++r) {
                float O = 0.f;
#pragma unroll
                for (int w = 0; w < kAttnWarps; ++w)
                    O = fmaf(s_f[w][r], so[((size_t)w * 16 + r) * kSoStride + col], O);
                st_cluster_f32(dst + 4u * (uint32_t)(r * sw), active ? O : 0.f);
            }
        }
        for (int i = tid; i < 16 * cs; i += blockDim.x) {   // (m, l) of row r to CTA d
            const int r = i & 15, d = i >> 4;
            const uint32_t dst = cluster_addr(smem_u32(recv_ml + ((size_t)split * 16 + r) * 2), (uint32_t)d);
            st_cluster_f32(dst, s_fm[r]);
            st_cluster_f32(dst + 4u, s_fl[r]);
        }
        cluster_sync_all();   // every push into this CTA has landed
        const int q0 = split * q4per, q1 = min(kHeadDim / 4, q0 + q4per);
        const int ncol = max(0, q1 - q0) * 4;
        const int items = nsplit > 0 ? p.group * ncol : 0;   // uniform over the cluster (one sequence)
        for (int it = tid; it < items; it += blockDim.x) {
            const int r = it / ncol, cc = it - r * ncol;
            float M = -INFINITY;
            for (int s2 = 0; s2 < cs; ++s2) M = fmaxf(M, recv_ml[(s2 * 16 + r) * 2]);
            float O = 0.f, Ls = 0.f;
            for (int s2 = 0; s2 < cs; ++s2) {
                const float ms = recv_ml[(s2 * 16 + r) * 2];
                const float f = ms == -INFINITY ? 0.f : exp2f(ms - M);
                O = fmaf(f, recv_o[((size_t)s2 * 16 + r) * sw + cc], O);
                Ls = fmaf(f, recv_ml[(s2 * 16 + r) * 2 + 1], Ls);
            }
            const size_t h = (size_t)b * p.Hq + (size_t)g * p.group + r;
            p.out[h * kHeadDim + 4 * q0 + cc] = __float2half_rn(O / Ls);
        }
        return;
    }
    const bool single = nsplit == 1;
#pragma unroll 4
    for (int r = 0; r < p.group; ++r) {
        float O = 0.f;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) O = fmaf(s_f[w][r], so[((size_t)w * 16 + r) * kSoStride + col], O);
        const size_t h = (size_t)b * p.Hq + (size_t)g * p.group + r;
        if (single) {
            p.out[h * kHeadDim + col] = __float2half_rn(O / s_fl[r]);
        } else {
            p.part_o[(h * p.max_splits + split) * kHeadDim + col] = O;
            if (col == 0) {
                p.part_ml[(h * p.max_splits + split) * 2 + 0] = s_fm[r];
                p.part_ml[(h * p.max_splits + split) * 2 + 1] = s_fl[r];
            }
        }
    }
    if (single) return;  // uniform

    // ---- publish; the last CTA of (b, g) merges every split in order.  The
    // block barrier orders every thread's partial stores before thread 0's
    // fence (cumulative) and ticket; the winner fences again before reading.
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const unsigned t = atomicAdd(&p.counters[b * p.Hkv + g], 1u);
        const bool last = (t == (unsigned)nsplit - 1);
        if (last) __threadfence();
        s_flag = last;
    }
    __syncthreads();
    if (!s_flag) return;  // uniform
    // (m, l) of every split for every row of the group, loaded in parallel,
    // then per-row weights exp2(m_s - M); the tile area is free again here
    float* wml = reinterpret_cast<float*>(tiles);             // [group][nsplit] m, then weight
    float* wl = wml + p.group * nsplit;                       // [group][nsplit] l
    __shared__ float s_L[16];
    for (int base = 0; base < p.group * nsplit; base += 4 * (int)blockDim.x) {   // four loads in flight
        float2 ml[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = base + u * (int)blockDim.x + tid;
            if (idx < p.group * nsplit) {
                const int r = idx / nsplit, s2 = idx - r * nsplit;
                const size_t h = (size_t)b * p.Hq + (size_t)g * p.group + r;
                ml[u] = __ldcg(reinterpret_cast<const float2*>(&p.part_ml[(h * p.max_splits + s2) * 2]));
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = base + u * (int)blockDim.x + tid;
            if (idx < p.group * nsplit) {
                wml[idx] = ml[u].x;
                wl[idx] = ml[u].y;
            }
        }
    }
    __syncthreads();
    if (tid < p.group) {
        float M = -INFINITY;
        for (int s2 = 0; s2 < nsplit; ++s2) M = fmaxf(M, wml[tid * nsplit + s2]);
        float Ls = 0.f;
        for (int s2 = 0; s2 < nsplit; ++s2) {
            const float ms = wml[tid * nsplit + s2];
            const float f = ms == -INFINITY ? 0.f : exp2f(ms - M);
            wml[tid * nsplit + s2] = f;
            Ls += f * wl[tid * nsplit + s2];
        }
        s_L[tid] = Ls;
    }
    __syncthreads();
    // O: four-column items (row r, float4 q4), up to four per thread, with every
    // item's next four splits loaded before any is used
    constexpr int kItems = 16 * 32 / (kAttnWarps * 32);   // group <= 16
    float4 acc[kItems];
#pragma unroll
    for (int it = 0; it < kItems; ++it) acc[it] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < nsplit; s0 += 4) {
        float4 v[kItems][4];
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int item = tid + it * kAttnWarps * 32, r = item >> 5, q4 = item & 31;
            const size_t h = (size_t)b * p.Hq + (size_t)g * p.group + r;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (r < p.group && s0 + u < nsplit)
                    v[it][u] = __ldcg(reinterpret_cast<const float4*>(p.part_o + (h * p.max_splits + s0 + u) * kHeadDim) + q4);
        }
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int item = tid + it * kAttnWarps * 32, r = item >> 5;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (r < p.group && s0 + u < nsplit) {
                    const float f = wml[r * nsplit + s0 + u];
                    acc[it].x = fmaf(f, v[it][u].x, acc[it].x);
                    acc[it].y = fmaf(f, v[it][u].y, acc[it].y);
                    acc[it].z = fmaf(f, v[it][u].z, acc[it].z);
                    acc[it].w = fmaf(f, v[it][u].w, acc[it].w);
                }
        }
    }
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
        const int item = tid + it * kAttnWarps * 32, r = item >> 5, q4 = item & 31;
        if (r < p.group) {
            const size_t h = (size_t)b * p.Hq + (size_t)g * p.group + r;
            const float il = 1.f / s_L[r];
            __half2* dst = reinterpret_cast<__half2*>(p.out + h * kHeadDim + 4 * q4);
            dst[0] = __floats2half2_rn(acc[it].x * il, acc[it].y * il);
            dst[1] = __floats2half2_rn(acc[it].z * il, acc[it].w * il);
        }
    }
    if (tid == 0) p.counters[b * p.Hkv + g] = 0u;
}

// ---------------------------------------------------------------- prompt pass
// A CTA owns KV head g, 16 consecutive prompt rows and one range of at most
// ppc pages of their causal key range; warp w is query head g * group + w, so
// the 16 rows of its MMA tile are 16 tokens of one head.  The K/V page tiles
// are staged once per CTA (TMA, kPaStages-deep ring with full/empty
// mbarriers) and read by every warp of the group.  Keys past a row's own
// position score -inf (causal mask); in the last page, V rows past the
// block's last position are zeroed in the B fragments, so stale slots never
// reach the output.  A block whose range spans several splits leaves
// (m, l, O) per row in the workspace and the last of its CTAs (atomic
// ticket, no waiting) merges them in split order.  Blocks run longest-first.
constexpr int kPaStages = 4;
constexpr int kPaRows = 16;

__global__ void __launch_bounds__(16 * 32)
prefill_attention_kernel(const PrefillAttnParams p, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv) {
    extern __shared__ unsigned char pa_raw[];
    __shared__ uint64_t full[kPaStages], empty[kPaStages];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nwarps = blockDim.x >> 5;
    const int qblocks = gridDim.x / p.max_splits;
    const int qb = qblocks - 1 - (int)blockIdx.x / p.max_splits;   // the longest blocks first
    const int split = (int)blockIdx.x % p.max_splits;
    const int g = blockIdx.y;
    const int t0 = qb * kPaRows;
    const int t_last = min(p.n, t0 + kPaRows) - 1;
    const int pos_last = p.start + t_last;
    const int npages_all = pos_last / kPageTokens + 1;
    const int nsplit = (npages_all + p.ppc - 1) / p.ppc;
    if (split >= nsplit) return;   // uniform: this block's key range is shorter
    const int pg0 = split * p.ppc;
    const int npages = min(npages_all - pg0, p.ppc);   // pages pg0 .. pg0 + npages - 1

    int bad = 0;
    for (int i = tid; i < npages; i += blockDim.x) {
        const int pg = p.pt[pg0 + i];
        bad |= (pg < 0 || pg >= p.num_pages);
    }
    bad |= (npages_all > p.max_pages);
    if (__syncthreads_or(bad)) {
        if (tid == 0) record_device_error(p.errword, W4_DEVERR_PAGE_ID);
        return;  // uniform
    }
    unsigned char* tiles = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(pa_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    if (tid == 0) {
        for (int s = 0; s < kPaStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], nwarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    }
    __syncthreads();

    auto issue = [&](int j) {  // thread 0: page pg0 + j into stage j % kPaStages
        const int st = j % kPaStages;
        const int row = (p.pt[pg0 + j] * p.Hkv + g) * kPageTokens;
        unsigned char* dst = tiles + st * kStageBytes;
        mbar_arrive_expect_tx(&full[st], kStageBytes);
        tma_load_2d(dst, &tmk, 0, row, &full[st]);
        tma_load_2d(dst + 2048, &tmk, 64, row, &full[st]);
        tma_load_2d(dst + kTileBytes, &tmv, 0, row, &full[st]);
        tma_load_2d(dst + kTileBytes + 2048, &tmv, 64, row, &full[st]);
    };
    if (tid == 0)
        for (int j = 0; j < min(npages, kPaStages); ++j) issue(j);

    // Q fragments: rows gid and gid + 8 are prompt rows t0 + gid, t0 + gid + 8 of head h
    const int gid = lane >> 2, tig = lane & 3;
    const int h = g * p.group + warp;
    const int ta = t0 + gid, tb = t0 + gid + 8;
    uint32_t qa[8][4];
    {
        const __half* q0 = p.q + ((size_t)min(ta, p.n - 1) * p.Hq + h) * kHeadDim;
        const __half* q1 = p.q + ((size_t)min(tb, p.n - 1) * p.Hq + h) * kHeadDim;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int c = ks * 16 + 2 * tig;
            qa[ks][0] = *reinterpret_cast<const uint32_t*>(q0 + c);
            qa[ks][1] = *reinterpret_cast<const uint32_t*>(q1 + c);
            qa[ks][2] = *reinterpret_cast<const uint32_t*>(q0 + c + 8);
            qa[ks][3] = *reinterpret_cast<const uint32_t*>(q1 + c + 8);
        }
    }
    const int pa_pos = p.start + ta, pb_pos = p.start + tb;   // key positions each row may see

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool failed = false;
    int issued = min(npages, kPaStages), consumed = 0;

    for (int j = 0; j < npages; ++j) {
        // thread 0 refills the stage every warp has released (the previous page's)
        if (tid == 0 && j >= 1 && j - 1 + kPaStages < npages) {
            const int r = j - 1;
            if (mbar_wait_bounded(&empty[r % kPaStages], (unsigned)(r / kPaStages) & 1u, kWaitLimit)) {
                issue(r + kPaStages);
                issued = r + kPaStages + 1;
            }
        }
        const int st = j % kPaStages;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[st], (unsigned)(j / kPaStages) & 1u,
                                                                  kWaitLimit));
        if (!ok) {
            failed = true;
            break;
        }
        unsigned char* kt = tiles + st * kStageBytes;
        const uint32_t kbase = smem_u32(kt), vbase = smem_u32(kt + kTileBytes);
        const int key0 = (pg0 + j) * kPageTokens;

        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
            const int mat = lane >> 3, i = lane & 7;
            const int tok = 8 * (mat >> 1) + i;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t b00, b01, b10, b11;
                ldsm_x4(kbase + tile_off(tok, ks * 16 + 8 * (mat & 1)), b00, b01, b10, b11);
                mma_16816(s[0], qa[ks], b00, b01);
                mma_16816(s[1], qa[ks], b10, b11);
            }
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
        if (key0 + kPageTokens - 1 <= p.start + t0) {   // every row of the block sees the whole page
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    s[nt][e] *= p.scale_log2;
                    if (e < 2) mx0 = fmaxf(mx0, s[nt][e]);
                    else mx1 = fmaxf(mx1, s[nt][e]);
                }
            }
        } else {   // the causal edge
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int kp = key0 + nt * 8 + 2 * tig + (e & 1);
                    const bool vis = kp <= ((e < 2) ? pa_pos : pb_pos);
                    const float v = vis ? s[nt][e] * p.scale_log2 : -INFINITY;
                    s[nt][e] = v;
                    if (e < 2) mx0 = fmaxf(mx0, v);
                    else mx1 = fmaxf(mx1, v);
                }
            }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        // The reference max m moves only when some row's max grows by more than 2^8 (log2
        // domain); otherwise probabilities exp2(s - m) stay <= 256 and O, l keep their scale.
        // A row that has seen no key yet keeps m = -inf and exactly zero terms.
        if (__any_sync(0xffffffffu, mx0 > m0 + 8.f || mx1 > m1 + 8.f)) {
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float c0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0);
            const float c1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            l0 *= c0;
            l1 *= c1;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                o[i][0] *= c0;
                o[i][1] *= c0;
                o[i][2] *= c1;
                o[i][3] *= c1;
            }
        }
        const float b0 = m0 == -INFINITY ? 0.f : m0, b1 = m1 == -INFINITY ? 0.f : m1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            s[nt][0] = exp2f(s[nt][0] - b0);
            s[nt][1] = exp2f(s[nt][1] - b0);
            s[nt][2] = exp2f(s[nt][2] - b1);
            s[nt][3] = exp2f(s[nt][3] - b1);
            ps0 += s[nt][0] + s[nt][1];
            ps1 += s[nt][2] + s[nt][3];
        }
        l0 += ps0;
        l1 += ps1;
        uint32_t pa[4];
        pa[0] = pack_h2(s[0][0], s[0][1]);
        pa[1] = pack_h2(s[0][2], s[0][3]);
        pa[2] = pack_h2(s[1][0], s[1][1]);
        pa[3] = pack_h2(s[1][2], s[1][3]);
        // in the last page, V rows past the block's last position are not the sequence's
        const int valid = min(kPageTokens, pos_last - key0 + 1);
        {
            const int mat = lane >> 3, i = lane & 7;
            const int tok = 8 * (mat & 1) + i;
            if (valid == kPageTokens) {
#pragma unroll
                for (int nd = 0; nd < 16; nd += 2) {
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_t(vbase + tile_off(tok, 8 * (nd + (mat >> 1))), v0, v1, v2, v3);
                    mma_16816(o[nd], pa, v0, v1);
                    mma_16816(o[nd + 1], pa, v2, v3);
                }
            } else {
                const uint32_t klo = valid > 2 * tig ? 0xFFFFu : 0u, khi = valid > 2 * tig + 1 ? 0xFFFF0000u : 0u;
                const uint32_t klo8 = valid > 2 * tig + 8 ? 0xFFFFu : 0u;
                const uint32_t khi8 = valid > 2 * tig + 9 ? 0xFFFF0000u : 0u;
                const uint32_t mlo = klo | khi, mhi = klo8 | khi8;
#pragma unroll
                for (int nd = 0; nd < 16; nd += 2) {
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_t(vbase + tile_off(tok, 8 * (nd + (mat >> 1))), v0, v1, v2, v3);
                    mma_16816(o[nd], pa, v0 & mlo, v1 & mhi);
                    mma_16816(o[nd + 1], pa, v2 & mlo, v3 & mhi);
                }
            }
        }
        ++consumed;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (failed && tid == 0) {
        record_device_error(p.errword, W4_DEVERR_TIMEOUT);
        // let copies already in flight land before the shared memory is released
        for (int j = consumed; j < issued; ++j)
            mbar_wait_bounded(&full[j % kPaStages], (unsigned)(j / kPaStages) & 1u, kWaitLimit);
    }
    // no CTA leaves while a copy into its shared memory may be in flight; a failure in any warp ends all
    if (__syncthreads_or(failed)) return;
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if (nsplit == 1) {   // the whole key range was here (split 0 always sees key 0, so l > 0)
        const float i0 = 1.f / l0, i1 = 1.f / l1;
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
            const int c = nd * 8 + 2 * tig;
            if (ta < p.n)
                *reinterpret_cast<__half2*>(p.out + ((size_t)ta * p.Hq + h) * kHeadDim + c) =
                    __floats2half2_rn(o[nd][0] * i0, o[nd][1] * i0);
            if (tb < p.n)
                *reinterpret_cast<__half2*>(p.out + ((size_t)tb * p.Hq + h) * kHeadDim + c) =
                    __floats2half2_rn(o[nd][2] * i1, o[nd][3] * i1);
        }
        return;   // uniform
    }
    // ---- publish this split's (m, l, O) rows; the last CTA of the block merges
    const size_t blk = (size_t)qb * p.Hkv + g;
    const size_t slot = (blk * p.max_splits + split) * p.group + warp;   // 16 rows of head h
    float* po = p.part_o + slot * kPaRows * kHeadDim;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
        const int c = nd * 8 + 2 * tig;
        __stcg(reinterpret_cast<float2*>(po + (size_t)gid * kHeadDim + c), make_float2(o[nd][0], o[nd][1]));
        __stcg(reinterpret_cast<float2*>(po + (size_t)(gid + 8) * kHeadDim + c), make_float2(o[nd][2], o[nd][3]));
    }
    if (tig == 0) {
        __stcg(reinterpret_cast<float2*>(p.part_ml + (slot * kPaRows + gid) * 2), make_float2(m0, l0));
        __stcg(reinterpret_cast<float2*>(p.part_ml + (slot * kPaRows + gid + 8) * 2), make_float2(m1, l1));
    }
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned t = atomicAdd(&p.counters[blk], 1u);
        const int last = t == (unsigned)nsplit - 1;
        if (last) {
            __threadfence();
            p.counters[blk] = 0u;
        }
        s_last = last;
    }
    __syncthreads();
    if (!s_last) return;   // uniform
    // merge: warp w takes head h's 16 rows; lane = (row half, 4-column group) -> rows r, columns 4c..4c+3
    for (int r = lane >> 4; r < kPaRows; r += 2) {
        const int t = t0 + r;
        float M = -INFINITY;
        for (int sp = 0; sp < nsplit; ++sp) {
            const size_t sl = (blk * p.max_splits + sp) * p.group + warp;
            M = fmaxf(M, __ldcg(p.part_ml + (sl * kPaRows + r) * 2));
        }
        float L = 0.f;
        float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
        const int c = (lane & 15) * 8;   // eight columns per lane
        for (int sp = 0; sp < nsplit; ++sp) {
            const size_t sl = (blk * p.max_splits + sp) * p.group + warp;
            const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml + (sl * kPaRows + r) * 2));
            const float f = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
            L += f * ml.y;
            const float4* src = reinterpret_cast<const float4*>(p.part_o + (sl * kPaRows + r) * kHeadDim + c);
            const float4 a = __ldcg(src), b = __ldcg(src + 1);
            acc0.x += f * a.x; acc0.y += f * a.y; acc0.z += f * a.z; acc0.w += f * a.w;
            acc1.x += f * b.x; acc1.y += f * b.y; acc1.z += f * b.z; acc1.w += f * b.w;
        }
        if (t < p.n) {
            const float il = 1.f / L;
            __half2* dst = reinterpret_cast<__half2*>(p.out + ((size_t)t * p.Hq + h) * kHeadDim + c);
            dst[0] = __floats2half2_rn(acc0.x * il, acc0.y * il);
            dst[1] = __floats2half2_rn(acc0.z * il, acc0.w * il);
            dst[2] = __floats2half2_rn(acc1.x * il, acc1.y * il);
            dst[3] = __floats2half2_rn(acc1.z * il, acc1.w * il);
        }
    }
}
#endif  // W4_DEFINE_ATTENTION_KERNEL

// ---------------------------------------------------------------- host side
struct AttnPlan {
    int ppw;
    int max_splits;
    int cluster;   // 1: the splits of a (b, g) form one thread-block cluster and merge in shared memory
    int stages;    // pages in flight per warp (2 or 4)
    dim3 grid;
};

// The largest cluster of 4-stage attention CTAs this device co-schedules: 16
// (a non-portable size) where it fits, else 8.  Defined in attention.cu.
int attention_max_cluster();

// Contexts of at most 64 pages keep their splits in one cluster of at most 8
// CTAs (one or two pages per warp); longer ones, while the clusters of every
// (b, g) fit on the GPU at once, in one cluster of up to 16 CTAs with up to
// eight pages per warp in four-page rings.  Either merges through distributed
// shared memory.  The rest spread over more CTAs than a cluster holds and
// merge through the workspace.  sms: the GPU's SMs; cmax: the largest cluster
// it co-schedules; either 0 to ask the device (sm_count(), attention_max_cluster())
// where the plan needs it.
inline AttnPlan attention_plan_for(int B, int hkv, int max_context, int sms, int cmax, int max_splits_cap = 256) {
    auto SMS = [&]() { return sms > 0 ? sms : sm_count(); };
    auto CMAX = [&]() { return cmax > 0 ? cmax : attention_max_cluster(); };
    AttnPlan pl;
    pl.stages = 2;
    const int pages = (max_context + kPageTokens - 1) / kPageTokens;
    if (pages > kAttnWarps * 2 && pages <= 8 * kAttnWarps * 2) {   // two to eight splits
        pl.cluster = 1;
        pl.ppw = pages <= 8 * kAttnWarps ? 1 : 2;
        // 33..64 pages: one page per warp in up to 16 CTAs where such clusters fit
        if (pl.ppw == 2 && CMAX() == kAttnMaxCluster &&
            (long long)B * hkv * ((pages + kAttnWarps - 1) / kAttnWarps) <= SMS())
            pl.ppw = 1;
        const int per_cta = kAttnWarps * pl.ppw;
        pl.max_splits = (pages + per_cta - 1) / per_cta;
        pl.grid = dim3(pl.max_splits, hkv, B);
        return pl;
    }
    if (pages > 8 * kAttnWarps * 2) {
        const int cm = CMAX();
        const int ppw = (pages + cm * kAttnWarps - 1) / (cm * kAttnWarps);
        const int cs = (pages + kAttnWarps * ppw - 1) / (kAttnWarps * ppw);
        if (ppw <= 8 && (long long)B * hkv * cs <= SMS()) {
            pl.cluster = 1;
            pl.ppw = ppw;
            pl.stages = ppw > 2 ? 4 : 2;
            pl.max_splits = cs;
            pl.grid = dim3(cs, hkv, B);
            return pl;
        }
    }
    pl.cluster = 0;
    const long long total = (long long)B * hkv * pages;
    const long long target_warps = (long long)SMS() * 16;
    long long ppw = (total + target_warps - 1) / target_warps;
    const long long min_ppw = (pages + (long long)kAttnWarps * max_splits_cap - 1) /
                              ((long long)kAttnWarps * max_splits_cap);   // <= max_splits_cap splits
    ppw = ppw < min_ppw ? min_ppw : ppw;
    // at least two pages per warp: a split that holds only a page or two per
    // warp costs more in the cross-CTA merge than it saves in parallel loads
    ppw = ppw < 2 ? 2 : ppw;
    pl.ppw = (int)ppw;
    const int per_cta = kAttnWarps * pl.ppw;
    pl.max_splits = (pages + per_cta - 1) / per_cta;
    pl.grid = dim3(pl.max_splits, hkv, B);
    return pl;
}

inline AttnPlan attention_plan(int B, int hkv, int max_context, int max_splits_cap = 256) {
    return attention_plan_for(B, hkv, max_context, 0, 0, max_splits_cap);
}

inline size_t attention_ws_bytes(int B, int hq, int hkv, const AttnPlan& pl) {
    const size_t po = (size_t)B * hq * pl.max_splits * kHeadDim * sizeof(float);
    const size_t pm = (size_t)B * hq * pl.max_splits * 2 * sizeof(float);
    const size_t ct = (size_t)B * hkv * sizeof(unsigned);
    return ((po + 255) / 256) * 256 + ((pm + 255) / 256) * 256 + ct;
}

// Build the 2-D TMA descriptor of one pool: rows of 128 fp16 (256 bytes),
// boxes of 16 rows x 64 columns, 128-byte swizzle.
w4_status make_pool_tensor_map(CUtensorMap* map, const void* pool, int num_pages, int hkv);

cudaError_t attention_launch(const AttnParams& p, const AttnPlan& pl, cudaStream_t st, bool pdl);

// Key-range split of the causal prompt-pass attention for n rows after start:
// at most 8 pages per CTA while the partial slots stay bounded.
struct PrefillAttnPlan {
    int qblocks, ppc, max_splits;
};
inline PrefillAttnPlan prefill_attention_plan(int n, int start) {
    PrefillAttnPlan pl;
    pl.qblocks = (n + 15) / 16;
    const int max_pages = (start + n - 1) / kPageTokens + 1;
    const int cap = std::max(1, std::min(8, 512 / pl.qblocks));
    pl.ppc = std::max(8, (max_pages + cap - 1) / cap);
    pl.max_splits = (max_pages + pl.ppc - 1) / pl.ppc;
    return pl;
}
// Workspace layout: tickets [qblocks][Hkv] first (zeroed per call), then the
// (m, l) and O partials.
inline size_t prefill_attention_ticket_bytes(int n, int hkv) {
    return ((size_t)((n + 15) / 16) * hkv * sizeof(unsigned) + 255) / 256 * 256;
}
// Workspace bytes of the split partials and tickets (a plan for at most n rows
// after at most max_context - n cached positions fits in it).
inline size_t prefill_attention_ws_bytes(int n, int hkv, int group, int max_context) {
    const PrefillAttnPlan pl = prefill_attention_plan(n, std::max(0, max_context - n));
    const size_t slots = (size_t)pl.qblocks * hkv * std::max(pl.max_splits, 8) * group * 16;
    const size_t po = slots * kHeadDim * sizeof(float), pm = slots * 2 * sizeof(float);
    return prefill_attention_ticket_bytes(n, hkv) + (pm + 255) / 256 * 256 + po;
}

// Causal prompt-pass attention: grid (qblocks * max_splits, Hkv), group warps per CTA.
cudaError_t prefill_attention_launch(const PrefillAttnParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                     cudaStream_t st);

}  // namespace w4
