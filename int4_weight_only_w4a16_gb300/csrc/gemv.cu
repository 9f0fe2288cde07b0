// gemv_w4a16: the standalone batch-M W4A16 GEMV entry point.
//
// Batch 1 streams the matrix with the TMA-fed CUDA-core kernel (gemv_tma.cuh)
// when its ring fits the row length; batches of 2 to 11, and batch 1 rows the
// ring cannot hold, run the register-pipelined mma.sync kernel (gemv_mma.cuh);
// batches of 12 to 16 run the tcgen05 kernel (gemv_tc05.cuh).  Measured on
// the layer's projection shapes: the mma.sync kernel's cost doubles with its
// second 8-column n-tile above batch 8, while the tcgen05 kernel's is flat in
// the batch (its N = 16 tile covers every batch), so the two cross near 12.
// w4_gemv_tune can put every batch on the mma.sync kernel, batch 1 on the W4A8
// variant of the streaming kernel, or every batch on the tcgen05 kernel.
#define W4_DEFINE_GEMV_TC05_KERNEL
#include "gemv_mma.cuh"
#include "gemv_tc05.cuh"
#include "gemv_tma.cuh"

namespace w4 {

static int g_variant = V_SUBNORMAL;

static bool use_tma(int m, int64_t n, int64_t k) {
    return m == 1 && g_variant != V_MMA_ALL && g_variant != V_TC05 && tma_plan(1, (int)n, (int)k).grid > 0;
}

constexpr int kTc05MinBatch = 12;   // default: batches of 12..16 on the tcgen05 kernel

static bool use_tc05(int m) { return g_variant == V_TC05 || (g_variant == V_SUBNORMAL && m >= kTc05MinBatch); }

cudaError_t tg_launch(const TgPlan& p, const CUtensorMap& tmw, const CUtensorMap& tmx, cudaStream_t st) {
    static size_t attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && attr_set[dev] < p.smem) {
        const cudaError_t e =
            cudaFuncSetAttribute(gemv_tc05_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = p.smem;
    }
    gemv_tc05_kernel<<<p.grid, kTgThreads, p.smem, st>>>(p.a, tmw, tmx);
    return cudaGetLastError();
}

}  // namespace w4

extern "C" w4_status w4_gemv_plan(int matrices, int64_t n, int64_t k, int32_t* out) {
    W4_REQUIRE(out, W4_ERR_NULL, "gemv_plan: null out");
    W4_REQUIRE((matrices == 1 || matrices == 2) && n >= 1 && k >= 128 && k % 128 == 0 && n <= 0x7fffffff &&
                   k <= 0x7fffffff,
               W4_ERR_SHAPE, "gemv_plan: need matrices 1 or 2, n >= 1, k a positive multiple of 128");
    const w4::TmaPlan p = w4::tma_plan(matrices, (int)n, (int)k);
    const int32_t v[9] = {p.grid, p.a.cw, p.a.hpr, p.a.rg, p.a.gs, p.a.ns, p.a.wbytes, p.a.sbytes, (int32_t)p.smem};
    for (int i = 0; i < 9; ++i) out[i] = p.grid > 0 || i == 0 ? v[i] : 0;
    return W4_OK;
}

extern "C" size_t w4_gemv_workspace_size(int m, int64_t n, int64_t k) {
    if (m < 1 || m > 16 || n < 1 || k < 128 || k % 128 || n > 0x7fffffff || k > 0x7fffffff) return 0;
    if (w4::use_tma(m, n, k)) return 256;
    if (w4::use_tc05(m)) return std::max<size_t>(256, w4::tg_ws_bytes(w4::tg_plan(m, (int)n, (int)k)));
    return w4::mma_ws_bytes(w4::mma_plan(m, (int)n, (int)k), m, (int)n);
}

extern "C" w4_status w4_gemv_tune(int variant) {
    W4_REQUIRE(variant == w4::V_SUBNORMAL || variant == w4::V_MMA_ALL || variant == w4::V_INT8 ||
                   variant == w4::V_TC05,
               W4_ERR_RANGE,
               "gemv_tune: variant must be 0 (default), 1 (mma.sync kernel at every batch), 2 (W4A8 at batch 1) or "
               "3 (tcgen05 kernel at every batch)");
    w4::g_variant = variant;
    return W4_OK;
}

extern "C" w4_status w4_gemv_w4a16(const void* x, int m, int64_t n, int64_t k, const uint32_t* packed,
                                   const void* scales, const void* bias, const void* residual, void* y,
                                   void* workspace, size_t workspace_bytes, void* stream) {
    W4_REQUIRE(x && packed && scales && y, W4_ERR_NULL, "gemv_w4a16: null pointer");
    W4_REQUIRE(m >= 1 && m <= 16, W4_ERR_SHAPE, "gemv_w4a16: m must be in [1, 16] (m=%d)", m);
    W4_REQUIRE(n >= 1 && n <= 0x7fffffff && k >= 128 && k % 128 == 0 && k <= 0x7fffffff, W4_ERR_SHAPE,
               "gemv_w4a16: need n >= 1 and k a positive multiple of 128 (n=%lld k=%lld)", (long long)n,
               (long long)k);
    W4_REQUIRE(w4::aligned16(x) && w4::aligned16(packed) && w4::aligned16(y), W4_ERR_ALIGN,
               "gemv_w4a16: x, packed and y must be 16-byte aligned");
    W4_REQUIRE(x != y, W4_ERR_RANGE, "gemv_w4a16: y must not alias x");
    W4_REQUIRE(w4::aligned16(workspace), W4_ERR_ALIGN, "gemv_w4a16: workspace must be 16-byte aligned");
    cudaStream_t st = (cudaStream_t)stream;
    w4::GemvParams p = {};
    p.x = static_cast<const __half*>(x);
    p.w0 = packed;
    p.s0 = static_cast<const __half*>(scales);
    p.M = m;
    p.N = (int)n;
    p.K = (int)k;
    p.bias = static_cast<const __half*>(bias);
    p.resid16 = static_cast<const __half*>(residual);
    p.y16 = static_cast<__half*>(y);
    p.errword = w4::device_error_word();
    if (w4::use_tma(m, n, k)) {
        W4_REQUIRE(workspace != nullptr && workspace_bytes >= 256, W4_ERR_CAPACITY,
                   "gemv_w4a16: workspace of 256 bytes needed");
        W4_REQUIRE(w4::aligned16(scales), W4_ERR_ALIGN, "gemv_w4a16: scales must be 16-byte aligned");
        const w4::TmaPlan tp = w4::tma_plan(1, (int)n, (int)k);
        const cudaError_t e =
            w4::g_variant == w4::V_INT8
                ? w4::tma_launch<w4::V_INT8, w4::X_F16, w4::E_STORE_F16>(p, tp, st, false)
                : w4::tma_launch<w4::V_SUBNORMAL, w4::X_F16, w4::E_STORE_F16>(p, tp, st, false);
        if (e != cudaSuccess) return w4::cuda_check(e, "gemv_w4a16 launch");
        return W4_OK;
    }
    if (w4::use_tc05(m)) {
        w4::TgPlan tp = w4::tg_plan(m, (int)n, (int)k);
        const size_t need = w4::tg_ws_bytes(tp);
        W4_REQUIRE(workspace != nullptr && workspace_bytes >= need, W4_ERR_CAPACITY,
                   "gemv_w4a16: workspace of %zu bytes needed", need);
        tp.a.s = p.s0;
        tp.a.bias = p.bias;
        tp.a.resid = p.resid16;
        tp.a.y = p.y16;
        tp.a.errword = p.errword;
        if (tp.a.splits > 1) {
            const size_t part_bytes = (size_t)tp.a.splits * m * n * sizeof(float);
            tp.a.part = static_cast<float*>(workspace);
            tp.a.counters = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + (part_bytes + 255) / 256 * 256);
        }
        CUtensorMap tmw, tmx;
        w4_status s = w4::make_weight_group_map(&tmw, packed, (int)n, (int)k, 128, w4::kTgGroupsPerStage);
        if (s == W4_OK) s = w4::make_act_slice_map(&tmx, x, m, (int)k, 16, 2 * w4::kTgGroupsPerStage);
        if (s != W4_OK) return s;
        const cudaError_t e = w4::tg_launch(tp, tmw, tmx, st);
        if (e != cudaSuccess) return w4::cuda_check(e, "gemv_w4a16 launch");
        return W4_OK;
    }
    const w4::MmaPlan mp = w4::mma_plan(m, (int)n, (int)k);
    const size_t need = w4::mma_ws_bytes(mp, m, (int)n);
    W4_REQUIRE(workspace != nullptr && workspace_bytes >= need, W4_ERR_CAPACITY,
               "gemv_w4a16: workspace of %zu bytes needed", need);
    const size_t part_bytes = mp.split > 1 ? (size_t)mp.split * m * n * sizeof(float) : 0;
    p.part = static_cast<float*>(workspace);
    p.counters = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + ((part_bytes + 255) / 256) * 256);
    p.split = mp.split;
    p.kc = mp.kc;
    const cudaError_t e = w4::mma_launch(p, mp, st);
    if (e != cudaSuccess) return w4::cuda_check(e, "gemv_w4a16 launch");
    return W4_OK;
}
