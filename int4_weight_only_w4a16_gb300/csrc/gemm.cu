// gemm_w4a16: the prompt pass's W4A16 GEMM on tcgen05 (kernel in gemm_tc05.cuh).
#include <algorithm>

#define W4_DEFINE_GEMM_TC05_KERNEL
#include "gemm_tc05.cuh"

namespace w4 {

template <int EPI>
static cudaError_t launch_main(const GemmPlan& p, const CUtensorMap& tmx, const CUtensorMap& tmw0,
                               const CUtensorMap& tmw1, cudaStream_t st) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        // setmaxnreg moves registers between the warpgroups inside the launch's
        // allocation; the split only balances at exactly kGmLaunchRegs per thread
        // (otherwise the epilogue's setmaxnreg.inc would wait for registers that never
        // come), so refuse to launch a build that compiled to anything else
        cudaFuncAttributes fa = {};
        cudaError_t e = cudaFuncGetAttributes(&fa, w4_gemm_tc05_kernel<EPI>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != kGmLaunchRegs || fa.maxThreadsPerBlock < kGmThreads) return cudaErrorInvalidKernelImage;
        e = cudaFuncSetAttribute(w4_gemm_tc05_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kGmSmemBudget);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    w4_gemm_tc05_kernel<EPI><<<p.grid, kGmThreads, p.smem, st>>>(p.a, tmx, tmw0, tmw1);
    return cudaGetLastError();
}

template <int EPI>
static cudaError_t launch_epi(const GemmPlan& p, const CUtensorMap& tmx, const CUtensorMap& tmw0,
                              const CUtensorMap& tmw1, cudaStream_t st, bool reduce) {
    cudaError_t e = launch_main<EPI>(p, tmx, tmw0, tmw1, st);
    if (e != cudaSuccess || p.a.splits == 1 || !reduce) return e;
    const long long quads = (long long)p.a.n * (p.a.N / 4);
    const int grid = (int)std::min<long long>((quads + 255) / 256, (long long)sm_count() * 8);
    w4_gemm_reduce_kernel<EPI><<<grid, 256, 0, st>>>(p.a);
    return cudaGetLastError();
}

cudaError_t gemm_tc05_launch(int epi, const GemmPlan& p, const CUtensorMap& tmx, const CUtensorMap& tmw0,
                             const CUtensorMap& tmw1, cudaStream_t st, bool reduce) {
    switch (epi) {
        case G_RESID: return launch_epi<G_RESID>(p, tmx, tmw0, tmw1, st, reduce);
        case G_SWIGLU: return launch_epi<G_SWIGLU>(p, tmx, tmw0, tmw1, st, true);
        default: return launch_epi<G_STORE>(p, tmx, tmw0, tmw1, st, reduce);
    }
}

}  // namespace w4

static size_t gemm_ws_bytes(const w4::GemmPlan& p) { return w4::gemm_part_bytes(w4::G_STORE, p); }

extern "C" w4_status w4_gemm_plan(int epilogue, int n, int N, int K, int sms, int32_t* out) {
    W4_REQUIRE(out, W4_ERR_NULL, "gemm_plan: null out");
    W4_REQUIRE(epilogue >= 0 && epilogue <= 2 && n >= 1 && sms >= 1 && N >= 128 && K >= 128 && N % 128 == 0 &&
                   K % 128 == 0,
               W4_ERR_SHAPE, "gemm_plan: need epilogue 0..2, n >= 1, sms >= 1, N and K positive multiples of 128");
    const w4::GemmPlan p = w4::gemm_plan(epilogue, n, N, K, sms);
    const int32_t v[8] = {p.a.bn, p.a.tok_tiles, p.a.row_tiles, p.a.kb_per_split,
                          p.a.splits, p.a.stream, p.a.ctas, p.a.stages};
    for (int i = 0; i < 8; ++i) out[i] = v[i];
    return W4_OK;
}

extern "C" size_t w4_gemm_workspace_size(int n, int N, int K) {
    if (n < 1 || N < 128 || K < 128) return 0;   // 0 also when K is not split (no scratch)
    return gemm_ws_bytes(w4::gemm_plan(w4::G_STORE, n, N, K, w4::sm_count()));
}

extern "C" w4_status w4_gemm_w4a16(const void* x, int n, int N, int K, const uint32_t* packed, const void* scales,
                                   float* y, void* workspace, size_t workspace_bytes, void* stream) {
    W4_REQUIRE(x && packed && scales && y && workspace, W4_ERR_NULL, "gemm_w4a16: null pointer");
    W4_REQUIRE(n >= 1 && N >= 128 && K >= 128 && N % 128 == 0 && K % 128 == 0, W4_ERR_SHAPE,
               "gemm_w4a16: need n >= 1 and N, K positive multiples of 128 (got n=%d N=%d K=%d)", n, N, K);
    W4_REQUIRE(w4::aligned16(x) && w4::aligned16(packed) && w4::aligned16(workspace) &&
                   (reinterpret_cast<uintptr_t>(scales) & 1) == 0 && (reinterpret_cast<uintptr_t>(y) & 3) == 0,
               W4_ERR_ALIGN, "gemm_w4a16: x, packed and workspace must be 16-byte aligned");
    w4::GemmPlan p = w4::gemm_plan(w4::G_STORE, n, N, K, w4::sm_count());
    const size_t need = gemm_ws_bytes(p);
    W4_REQUIRE(workspace_bytes >= need, W4_ERR_CAPACITY, "gemm_w4a16: workspace of %zu bytes needed", need);
    p.a.w0 = packed;
    p.a.w1 = packed;
    p.a.s0 = static_cast<const __half*>(scales);
    p.a.s1 = p.a.s0;
    p.a.y = y;
    p.a.ldy = N;
    p.a.part = static_cast<float*>(workspace);
    p.a.errword = w4::device_error_word();
    CUtensorMap tmx, tmw;
    w4_status s = w4::make_act_tensor_map(&tmx, x, n, K, p.a.bn);
    if (s == W4_OK) s = w4::make_weight_tensor_map(&tmw, packed, N, K, 8, 128);
    if (s != W4_OK) return s;
    W4_CUDA(w4::gemm_tc05_launch(w4::G_STORE, p, tmx, tmw, tmw, (cudaStream_t)stream));
    return W4_OK;
}
