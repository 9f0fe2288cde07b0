// gemv_w4a16: the standalone batch-M W4A16 GEMV entry point.
#include "gemv_tc.cuh"

namespace w4 {

static int g_variant = V_SUBNORMAL;
static int g_split_override = 0;
static int g_rows_override = 0;

template <int VAR>
static cudaError_t launch_store(int mt, const GemvParams& p, const GemvPlan& pl, cudaStream_t st) {
    switch (mt) {
        case 1: return gemv_launch<1, VAR, X_F16, E_STORE_F16>(p, pl, st, false);
        case 2: return gemv_launch<2, VAR, X_F16, E_STORE_F16>(p, pl, st, false);
        case 4: return gemv_launch<4, VAR, X_F16, E_STORE_F16>(p, pl, st, false);
        case 8: return gemv_launch<8, VAR, X_F16, E_STORE_F16>(p, pl, st, false);
        default: return gemv_launch<16, VAR, X_F16, E_STORE_F16>(p, pl, st, false);
    }
}

static int tile_m(int m) { return m <= 1 ? 1 : m <= 2 ? 2 : m <= 4 ? 4 : m <= 8 ? 8 : 16; }

static size_t workspace_for(const GemvPlan& pl, int m, int64_t n) {
    const size_t part = pl.split > 1 ? (size_t)pl.split * m * n * sizeof(float) : 0;
    const size_t ctr = (size_t)pl.grid.x * sizeof(unsigned);
    return ((part + 255) / 256) * 256 + ctr;
}

// The TMA-fed tensor-core kernel (variant 3, opt-in) serves every batch
// size; without it and without a split / row override, batch 1 runs the
// CUDA-core TMA kernel and batches of 2-16 the register-pipelined
// tensor-core kernel, which measured faster on GB300.
static bool use_tc(int m, int64_t n, int64_t k) {
    return g_variant == V_TENSOR && g_split_override == 0 && g_rows_override == 0 &&
           tc_plan(1, X_F16, m, (int)n, (int)k).grid > 0;
}

// Batch 1 streams the matrix with the TMA-fed kernel unless a row-block
// tuning override asks for the blocked kernel.
static bool use_tma(int m, int64_t n, int64_t k) {
    return m == 1 && g_variant != V_MMA_ALL && g_split_override == 0 && g_rows_override == 0 &&
           tma_plan(1, (int)n, (int)k).grid > 0;
}

// Batches of 2..16 run on the tensor cores unless a tuning override asks for
// the blocked kernel.
static bool use_mma(int m) {
    return (m >= 2 || g_variant == V_MMA_ALL) && g_split_override == 0 && g_rows_override == 0;
}

}  // namespace w4

extern "C" size_t w4_gemv_workspace_size(int m, int64_t n, int64_t k) {
    if (m < 1 || m > 16 || n < 1 || k < 128 || k % 128 || n > 0x7fffffff || k > 0x7fffffff) return 0;
    if (w4::use_tc(m, n, k)) return w4::tc_ws_bytes(w4::tc_plan(1, w4::X_F16, m, (int)n, (int)k), 1);
    if (w4::use_tma(m, n, k)) return 256;
    if (w4::use_mma(m)) return w4::mma_ws_bytes(w4::mma_plan(m, (int)n, (int)k), m, (int)n);
    const w4::GemvPlan pl = w4::gemv_plan(w4::tile_m(m), (int)n, (int)k, true, w4::g_split_override, w4::g_rows_override);
    return w4::workspace_for(pl, m, n);
}

extern "C" w4_status w4_gemv_tune(int variant, int split_override, int rows_override) {
    W4_REQUIRE(variant >= 0 && variant <= 5, W4_ERR_RANGE, "gemv_tune: variant must be 0..5");
    W4_REQUIRE(split_override >= 0, W4_ERR_RANGE, "gemv_tune: split_override must be >= 0");
    W4_REQUIRE(rows_override >= 0 && rows_override <= 2, W4_ERR_RANGE, "gemv_tune: rows_override must be 0..2");
    w4::g_variant = variant;
    w4::g_split_override = split_override;
    w4::g_rows_override = rows_override;
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
    const int mt = w4::tile_m(m);
    W4_REQUIRE(w4::aligned16(workspace), W4_ERR_ALIGN, "gemv_w4a16: workspace must be 16-byte aligned");
    cudaStream_t st = (cudaStream_t)stream;
    if (w4::use_tc(m, n, k)) {
        W4_REQUIRE(w4::aligned16(scales), W4_ERR_ALIGN, "gemv_w4a16: scales must be 16-byte aligned");
        const w4::TcPlan tp = w4::tc_plan(1, w4::X_F16, m, (int)n, (int)k);
        const size_t need = w4::tc_ws_bytes(tp, 1);
        W4_REQUIRE(workspace != nullptr && workspace_bytes >= need, W4_ERR_CAPACITY,
                   "gemv_w4a16: workspace of %zu bytes needed", need);
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
        const size_t part_bytes = tp.a.P > 1 ? (size_t)tp.a.P * m * tp.a.nrb * 16 * sizeof(float) : 0;
        p.part = static_cast<float*>(workspace);
        p.counters = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + ((part_bytes + 255) / 256) * 256);
        p.errword = w4::device_error_word();
        CUtensorMap tm;
        const w4_status ms = w4::make_weight_tensor_map(&tm, packed, (int)n, (int)k, tp.a.ssz * 16, w4::kTcRB * 16);
        if (ms != W4_OK) return ms;
        const cudaError_t e = w4::tc_launch<w4::X_F16, w4::E_STORE_F16>(p, tp, tm, tm, st, false);
        if (e != cudaSuccess) return w4::cuda_check(e, "gemv_w4a16 launch");
        return W4_OK;
    }
    if (w4::use_tma(m, n, k)) {
        W4_REQUIRE(workspace != nullptr && workspace_bytes >= 256, W4_ERR_CAPACITY,
                   "gemv_w4a16: workspace of 256 bytes needed");
        W4_REQUIRE(w4::aligned16(scales), W4_ERR_ALIGN, "gemv_w4a16: scales must be 16-byte aligned");
        const w4::TmaPlan tp = w4::tma_plan(1, (int)n, (int)k);
        w4::GemvParams p = {};
        p.x = static_cast<const __half*>(x);
        p.w0 = packed;
        p.s0 = static_cast<const __half*>(scales);
        p.M = 1;
        p.N = (int)n;
        p.K = (int)k;
        p.bias = static_cast<const __half*>(bias);
        p.resid16 = static_cast<const __half*>(residual);
        p.y16 = static_cast<__half*>(y);
        p.errword = w4::device_error_word();
        cudaError_t e;
        switch (w4::g_variant) {
            case w4::V_HALF_CHUNK: e = w4::tma_launch<w4::V_HALF_CHUNK, w4::X_F16, w4::E_STORE_F16>(p, tp, st, false); break;
            case w4::V_HALF_WORD: e = w4::tma_launch<w4::V_HALF_WORD, w4::X_F16, w4::E_STORE_F16>(p, tp, st, false); break;
            case w4::V_INT8: e = w4::tma_launch<w4::V_INT8, w4::X_F16, w4::E_STORE_F16>(p, tp, st, false); break;
            default: e = w4::tma_launch<w4::V_SUBNORMAL, w4::X_F16, w4::E_STORE_F16>(p, tp, st, false); break;
        }
        if (e != cudaSuccess) return w4::cuda_check(e, "gemv_w4a16 launch");
        return W4_OK;
    }
    if (w4::use_mma(m)) {
        const w4::MmaPlan mp = w4::mma_plan(m, (int)n, (int)k);
        const size_t need = w4::mma_ws_bytes(mp, m, (int)n);
        W4_REQUIRE(workspace != nullptr && workspace_bytes >= need, W4_ERR_CAPACITY,
                   "gemv_w4a16: workspace of %zu bytes needed", need);
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
        const size_t part_bytes = mp.split > 1 ? (size_t)mp.split * m * n * sizeof(float) : 0;
        p.part = static_cast<float*>(workspace);
        p.counters = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + ((part_bytes + 255) / 256) * 256);
        p.split = mp.split;
        p.kc = mp.kc;
        const cudaError_t e = w4::mma_launch(p, mp, st);
        if (e != cudaSuccess) return w4::cuda_check(e, "gemv_w4a16 launch");
        return W4_OK;
    }
    const w4::GemvPlan pl = w4::gemv_plan(mt, (int)n, (int)k, true, w4::g_split_override, w4::g_rows_override);
    const size_t need = w4::workspace_for(pl, m, n);
    W4_REQUIRE(workspace != nullptr && workspace_bytes >= need, W4_ERR_CAPACITY,
               "gemv_w4a16: workspace of %zu bytes needed", need);

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
    const size_t part_bytes = pl.split > 1 ? (size_t)pl.split * m * n * sizeof(float) : 0;
    p.part = static_cast<float*>(workspace);
    p.counters = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + ((part_bytes + 255) / 256) * 256);
    p.split = pl.split;
    p.kc = pl.kc;
    cudaError_t e;
    switch (w4::g_variant) {
        case w4::V_HALF_CHUNK: e = w4::launch_store<w4::V_HALF_CHUNK>(mt, p, pl, st); break;
        case w4::V_HALF_WORD: e = w4::launch_store<w4::V_HALF_WORD>(mt, p, pl, st); break;
        default: e = w4::launch_store<w4::V_SUBNORMAL>(mt, p, pl, st); break;
    }
    if (e != cudaSuccess) return w4::cuda_check(e, "gemv_w4a16 launch");
    return W4_OK;
}
