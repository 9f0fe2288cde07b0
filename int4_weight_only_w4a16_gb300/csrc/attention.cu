// paged_decode_attention and paged_kv_append entry points.
#include <cmath>
#include <mutex>

#define W4_DEFINE_ATTENTION_KERNEL
#include "attention.cuh"

namespace w4 {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

w4_status make_pool_tensor_map(CUtensorMap* map, const void* pool, int num_pages, int hkv) {
    EncodeTiledFn fn = encode_fn();
    W4_REQUIRE(fn != nullptr, W4_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)num_pages * hkv * kPageTokens};
    const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kPageTokens};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(pool), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    W4_REQUIRE(r == CUDA_SUCCESS, W4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return W4_OK;
}

// Packed weights [n][k/8] uint32 as a 2-D tensor (words x rows); a box is
// box_rows rows by box_words words, unswizzled or (swizzle64, 16-word boxes)
// with the 64-byte swizzle; rows past n read as zeros.
w4_status make_weight_tensor_map(CUtensorMap* map, const uint32_t* packed, int n, int k, int box_words, int box_rows,
                                 bool swizzle64) {
    EncodeTiledFn fn = encode_fn();
    W4_REQUIRE(fn != nullptr, W4_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {(cuuint64_t)k / 8, (cuuint64_t)n};
    const cuuint64_t strides[1] = {(cuuint64_t)k / 2};
    const cuuint32_t box[2] = {(cuuint32_t)box_words, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(packed), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    W4_REQUIRE(r == CUDA_SUCCESS, W4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return W4_OK;
}

// Packed weights [n][k/8] uint32 as a 3-D tensor (word of a scale group x row
// x group): a box is 16 words (one group, 64 bytes, 64-byte swizzle) by
// box_rows rows by box_groups consecutive groups, laid out group by group in
// shared memory; rows past n and groups past k/128 read as zeros.
w4_status make_weight_group_map(CUtensorMap* map, const uint32_t* packed, int n, int k, int box_rows, int box_groups) {
    EncodeTiledFn fn = encode_fn();
    W4_REQUIRE(fn != nullptr, W4_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[3] = {16, (cuuint64_t)n, (cuuint64_t)k / 128};
    const cuuint64_t strides[2] = {(cuuint64_t)k / 2, 64};
    const cuuint32_t box[3] = {16, (cuuint32_t)box_rows, (cuuint32_t)box_groups};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(packed), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    W4_REQUIRE(r == CUDA_SUCCESS, W4_ERR_CUDA, "cuTensorMapEncodeTiled (weight groups) failed (%d)", (int)r);
    return W4_OK;
}

// Activations fp16 [n][k] as a 3-D tensor (column of a 64-column slice x row x
// slice): a box is 64 columns (128 bytes, 128-byte swizzle) by box_rows rows by
// box_slices consecutive slices, slice by slice in shared memory; rows past n
// and slices past k/64 read as zeros.
w4_status make_act_slice_map(CUtensorMap* map, const void* x, int n, int k, int box_rows, int box_slices) {
    EncodeTiledFn fn = encode_fn();
    W4_REQUIRE(fn != nullptr, W4_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[3] = {64, (cuuint64_t)n, (cuuint64_t)k / 64};
    const cuuint64_t strides[2] = {(cuuint64_t)k * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_slices};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(x), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    W4_REQUIRE(r == CUDA_SUCCESS, W4_ERR_CUDA, "cuTensorMapEncodeTiled (activation slices) failed (%d)", (int)r);
    return W4_OK;
}

// Activations fp16 [n][k] as a 2-D tensor (columns x rows): boxes of 64
// columns (128 bytes, 128-byte swizzle) by box_rows rows; rows past n read as zeros.
w4_status make_act_tensor_map(CUtensorMap* map, const void* x, int n, int k, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    W4_REQUIRE(fn != nullptr, W4_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)n};
    const cuuint64_t strides[1] = {(cuuint64_t)k * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    W4_REQUIRE(r == CUDA_SUCCESS, W4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return W4_OK;
}

cudaError_t prefill_attention_launch(const PrefillAttnParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                     cudaStream_t st) {
    constexpr int smem = kPaStages * kStageBytes + 1024;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const dim3 grid((unsigned)((p.n + kPaRows - 1) / kPaRows * p.max_splits), (unsigned)p.Hkv);
    prefill_attention_kernel<<<grid, p.group * 32, smem, st>>>(p, tmk, tmv);
    return cudaGetLastError();
}

template <bool CLUSTER, int STAGES>
static cudaError_t attention_set_attributes() {
    auto kern = paged_attention_kernel<CLUSTER, STAGES>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 attn_smem_bytes(STAGES, CLUSTER));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        if (CLUSTER) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    return cudaSuccess;
}

template <bool CLUSTER, int STAGES>
static cudaError_t attention_launch_t(const AttnParams& p, const AttnPlan& pl, cudaStream_t st, bool pdl) {
    cudaError_t e = attention_set_attributes<CLUSTER, STAGES>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = pl.grid;
    cfg.blockDim = dim3(kAttnWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = attn_smem_bytes(STAGES, CLUSTER);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (CLUSTER) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = pl.grid.x;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, paged_attention_kernel<CLUSTER, STAGES>, p);
}

cudaError_t attention_launch(const AttnParams& p, const AttnPlan& pl, cudaStream_t st, bool pdl) {
    if (!pl.cluster) return attention_launch_t<false, 2>(p, pl, st, pdl);
    return pl.stages == 4 ? attention_launch_t<true, 4>(p, pl, st, pdl) : attention_launch_t<true, 2>(p, pl, st, pdl);
}

// 16 when the occupancy calculator places at least one cluster of 16 CTAs of
// the 4-stage kernel (its largest shared-memory footprint), else 8; per device.
int attention_max_cluster() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
    if (cached[dev] != 0) return cached[dev];
    int best = 8;
    if (attention_set_attributes<true, 4>() == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kAttnMaxCluster, 1, 1);
        cfg.blockDim = dim3(kAttnWarps * 32, 1, 1);
        cfg.dynamicSmemBytes = attn_smem_bytes(4, true);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kAttnMaxCluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, paged_attention_kernel<true, 4>, &cfg) == cudaSuccess && n >= 1)
            best = kAttnMaxCluster;
    }
    cudaGetLastError();   // a refused query leaves no error behind
    cached[dev] = best;
    return best;
}

// One thread per 16-byte piece of a K or V row: 2 * b * hkv * 16 threads.
__global__ void kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v, int B, int hkv,
                                 uint4* k_pool, uint4* v_pool, int num_pages, const int32_t* __restrict__ pt,
                                 int max_pages, const int32_t* __restrict__ positions, int* errword) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t per_tensor = (int64_t)B * hkv * 16;
    if (i >= 2 * per_tensor) return;
    const bool is_v = i >= per_tensor;
    const int64_t r = is_v ? i - per_tensor : i;
    const int piece = (int)(r & 15);
    const int h = (int)((r >> 4) % hkv);
    const int b = (int)((r >> 4) / hkv);
    const int pos = positions[b];
    if (pos < 0 || pos >= max_pages * kPageTokens) {
        record_device_error(errword, W4_DEVERR_POSITION);
        return;
    }
    const int page = pt[(int64_t)b * max_pages + pos / kPageTokens];
    if (page < 0 || page >= num_pages) {
        record_device_error(errword, W4_DEVERR_PAGE_ID);
        return;
    }
    const int64_t dst = (((int64_t)page * hkv + h) * kPageTokens + pos % kPageTokens) * 16 + piece;
    (is_v ? v_pool : k_pool)[dst] = (is_v ? v : k)[r];
}

}  // namespace w4

extern "C" w4_status w4_paged_kv_append(const void* k, const void* v, int b, int hkv, int d, void* k_pool,
                                        void* v_pool, int num_pages, const int32_t* page_table, int max_pages,
                                        const int32_t* positions, void* stream) {
    W4_REQUIRE(k && v && k_pool && v_pool && page_table && positions, W4_ERR_NULL, "paged_kv_append: null pointer");
    W4_REQUIRE(d == w4::kHeadDim, W4_ERR_SHAPE, "paged_kv_append: head_dim must be 128 (d=%d)", d);
    W4_REQUIRE(b >= 1 && hkv >= 1 && num_pages >= 1 && max_pages >= 1, W4_ERR_SHAPE, "paged_kv_append: bad sizes");
    W4_REQUIRE((long long)num_pages * hkv * w4::kPageTokens < (1LL << 31), W4_ERR_SHAPE, "paged_kv_append: pool too large");
    W4_REQUIRE(w4::aligned16(k) && w4::aligned16(v) && w4::aligned16(k_pool) && w4::aligned16(v_pool), W4_ERR_ALIGN,
               "paged_kv_append: k, v and pools must be 16-byte aligned");
    const int64_t threads = 2LL * b * hkv * 16;
    const int blk = 256;
    w4::kv_append_kernel<<<(unsigned)((threads + blk - 1) / blk), blk, 0, (cudaStream_t)stream>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), b, hkv, static_cast<uint4*>(k_pool),
        static_cast<uint4*>(v_pool), num_pages, page_table, max_pages, positions, w4::device_error_word());
    W4_CUDA(cudaGetLastError());
    return W4_OK;
}

extern "C" w4_status w4_attention_plan(int b, int hq, int hkv, int max_context, int sms, int max_cluster,
                                       int64_t* out) {
    W4_REQUIRE(out, W4_ERR_NULL, "attention_plan: null out");
    W4_REQUIRE(b >= 1 && hq >= 1 && hkv >= 1 && max_context >= 1 && hq % hkv == 0 && sms >= 0 &&
                   (max_cluster == 0 || max_cluster == 8 || max_cluster == 16),
               W4_ERR_SHAPE, "attention_plan: bad shape, SM count or cluster size");
    const w4::AttnPlan pl = w4::attention_plan_for(b, hkv, max_context, sms, max_cluster);
    const int64_t v[8] = {pl.cluster, pl.ppw, pl.stages, pl.max_splits, (int64_t)pl.grid.x, (int64_t)pl.grid.y,
                          (int64_t)pl.grid.z, (int64_t)w4::attention_ws_bytes(b, hq, hkv, pl)};
    for (int i = 0; i < 8; ++i) out[i] = v[i];
    return W4_OK;
}

extern "C" size_t w4_attention_workspace_size(int b, int hq, int hkv, int max_context) {
    if (b < 1 || hq < 1 || hkv < 1 || max_context < 1) return 0;
    return w4::attention_ws_bytes(b, hq, hkv, w4::attention_plan(b, hkv, max_context));
}

extern "C" w4_status w4_paged_decode_attention(const void* q, int b, int hq, int hkv, int d, float scale,
                                               const void* k_pool, const void* v_pool, int num_pages,
                                               const int32_t* page_table, int max_pages, const int32_t* context_lens,
                                               int max_context, void* out, void* workspace, size_t workspace_bytes,
                                               void* stream) {
    W4_REQUIRE(q && k_pool && v_pool && page_table && context_lens && out, W4_ERR_NULL,
               "paged_decode_attention: null pointer");
    W4_REQUIRE(d == w4::kHeadDim, W4_ERR_SHAPE, "paged_decode_attention: head_dim must be 128 (d=%d)", d);
    W4_REQUIRE(b >= 1 && hkv >= 1 && hq >= hkv && hq % hkv == 0 && hq / hkv <= 16, W4_ERR_SHAPE,
               "paged_decode_attention: need hq %% hkv == 0 and hq/hkv <= 16 (hq=%d hkv=%d)", hq, hkv);
    W4_REQUIRE(num_pages >= 1 && max_pages >= 1 && max_context >= 1, W4_ERR_SHAPE, "paged_decode_attention: bad sizes");
    W4_REQUIRE(max_context <= max_pages * w4::kPageTokens, W4_ERR_RANGE,
               "paged_decode_attention: max_context exceeds the page table (%d > %d)", max_context,
               max_pages * w4::kPageTokens);
    W4_REQUIRE((long long)num_pages * hkv * w4::kPageTokens < (1LL << 31), W4_ERR_SHAPE,
               "paged_decode_attention: pool too large");
    W4_REQUIRE(std::isfinite(scale), W4_ERR_RANGE, "paged_decode_attention: scale must be finite");
    W4_REQUIRE(w4::aligned16(k_pool) && w4::aligned16(v_pool) && w4::aligned16(q) && w4::aligned16(out), W4_ERR_ALIGN,
               "paged_decode_attention: q, out and pools must be 16-byte aligned");
    const w4::AttnPlan pl = w4::attention_plan(b, hkv, max_context);
    const size_t need = w4::attention_ws_bytes(b, hq, hkv, pl);
    W4_REQUIRE(workspace && workspace_bytes >= need, W4_ERR_CAPACITY,
               "paged_decode_attention: workspace of %zu bytes needed", need);
    W4_REQUIRE(w4::aligned16(workspace), W4_ERR_ALIGN, "paged_decode_attention: workspace must be 16-byte aligned");
    w4::AttnParams p = {};
    p.q = static_cast<const __half*>(q);
    p.out = static_cast<__half*>(out);
    p.k_pool = static_cast<const __half*>(k_pool);
    p.v_pool = static_cast<const __half*>(v_pool);
    p.pt = page_table;
    p.lens = context_lens;
    const size_t po = (size_t)b * hq * pl.max_splits * w4::kHeadDim * sizeof(float);
    const size_t pm = (size_t)b * hq * pl.max_splits * 2 * sizeof(float);
    char* ws = static_cast<char*>(workspace);
    p.part_o = reinterpret_cast<float*>(ws);
    p.part_ml = reinterpret_cast<float*>(ws + ((po + 255) / 256) * 256);
    p.counters = reinterpret_cast<unsigned*>(ws + ((po + 255) / 256) * 256 + ((pm + 255) / 256) * 256);
    p.errword = w4::device_error_word();
    p.scale_log2 = scale * 1.4426950408889634f;
    p.B = b;
    p.Hq = hq;
    p.Hkv = hkv;
    p.group = hq / hkv;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    p.max_context = max_context;
    p.ppw = pl.ppw;
    p.max_splits = pl.max_splits;
    // programmatic dependent launch: the kernel touches no input or output before
    // griddepcontrol.wait, so its launch may overlap the end of the previous kernel
    cudaError_t e = w4::attention_launch(p, pl, (cudaStream_t)stream, true);
    if (e != cudaSuccess) return w4::cuda_check(e, "paged_decode_attention launch");
    return W4_OK;
}

// ----------------------------------------------------------------------------
// paged_decode_attention without caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run
// attention: a process that reserved its whole device-memory budget up front
// and may not grow it, an allocator-less embedded host or plugin, or a caller
// that holds only borrowed pointers.  For them the split-merge scratch lives
// in a fixed array of this module.  It is a file-scope device array: every
// GPU that loads this library holds kNoAllocScratchBytes of it until exit.
//
// In host code the array's name is only a host-side stand-in for the device
// variable, so its device address is looked up once per device with
// cudaGetSymbolAddress (on the first call made while that device is current)
// and cached for the life of the process.  The cached address belongs to the
// device's primary context: after cudaDeviceReset (or anything else that
// destroys that context) it is stale, so this entry point must not be used
// across a device reset.  Every call shares the one array: calls that overlap on the GPU
// (concurrent streams) race on it and must be serialised by the caller.  The
// split tickets inside it must start at zero; each call clears them on its
// stream before the kernel runs.
// ----------------------------------------------------------------------------
namespace w4 {

constexpr size_t kNoAllocScratchBytes = 8u << 20;   // 8 MiB
static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

static w4_status noalloc_scratch(void** out) {
    static void* addr[64] = {};
    static std::mutex mu;
    int dev = 0;
    W4_CUDA(cudaGetDevice(&dev));
    W4_REQUIRE(dev >= 0 && dev < 64, W4_ERR_STATE, "paged_decode_attention_noalloc: device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess) return cuda_check(e, "cudaGetSymbolAddress(attention scratch)");
        addr[dev] = p;
    }
    *out = addr[dev];
    return W4_OK;
}

}  // namespace w4

extern "C" size_t w4_paged_decode_attention_noalloc_max_scratch(void) { return w4::kNoAllocScratchBytes; }

extern "C" w4_status w4_paged_decode_attention_noalloc(const void* q, int b, int hq, int hkv, int d, float scale,
                                                       const void* k_pool, const void* v_pool, int num_pages,
                                                       const int32_t* page_table, int max_pages,
                                                       const int32_t* context_lens, int max_context, void* out,
                                                       void* stream) {
    W4_REQUIRE(q && k_pool && v_pool && page_table && context_lens && out, W4_ERR_NULL,
               "paged_decode_attention_noalloc: null pointer");
    W4_REQUIRE(d == w4::kHeadDim, W4_ERR_SHAPE, "paged_decode_attention_noalloc: head_dim must be 128 (d=%d)", d);
    W4_REQUIRE(b >= 1 && hkv >= 1 && hq >= hkv && hq % hkv == 0 && hq / hkv <= 16, W4_ERR_SHAPE,
               "paged_decode_attention_noalloc: need hq %% hkv == 0 and hq/hkv <= 16 (hq=%d hkv=%d)", hq, hkv);
    W4_REQUIRE(num_pages >= 1 && max_pages >= 1 && max_context >= 1, W4_ERR_SHAPE,
               "paged_decode_attention_noalloc: bad sizes");
    W4_REQUIRE(max_context <= max_pages * w4::kPageTokens, W4_ERR_RANGE,
               "paged_decode_attention_noalloc: max_context exceeds the page table (%d > %d)", max_context,
               max_pages * w4::kPageTokens);
    W4_REQUIRE((long long)num_pages * hkv * w4::kPageTokens < (1LL << 31), W4_ERR_SHAPE,
               "paged_decode_attention_noalloc: pool too large");
    W4_REQUIRE(std::isfinite(scale), W4_ERR_RANGE, "paged_decode_attention_noalloc: scale must be finite");
    W4_REQUIRE(w4::aligned16(k_pool) && w4::aligned16(v_pool) && w4::aligned16(q) && w4::aligned16(out), W4_ERR_ALIGN,
               "paged_decode_attention_noalloc: q, out and pools must be 16-byte aligned");
    const w4::AttnPlan pl = w4::attention_plan(b, hkv, max_context);
    const size_t need = w4::attention_ws_bytes(b, hq, hkv, pl);
    W4_REQUIRE(need <= w4::kNoAllocScratchBytes, W4_ERR_CAPACITY,
               "paged_decode_attention_noalloc: this batch/context needs %zu bytes of scratch, more than the "
               "library's fixed %zu; use w4_paged_decode_attention with a workspace",
               need, w4::kNoAllocScratchBytes);
    void* scratch = nullptr;
    w4_status s = w4::noalloc_scratch(&scratch);
    if (s != W4_OK) return s;
    w4::AttnParams p = {};
    p.q = static_cast<const __half*>(q);
    p.out = static_cast<__half*>(out);
    p.k_pool = static_cast<const __half*>(k_pool);
    p.v_pool = static_cast<const __half*>(v_pool);
    p.pt = page_table;
    p.lens = context_lens;
    const size_t po = (size_t)b * hq * pl.max_splits * w4::kHeadDim * sizeof(float);
    const size_t pm = (size_t)b * hq * pl.max_splits * 2 * sizeof(float);
    char* ws = static_cast<char*>(scratch);
    p.part_o = reinterpret_cast<float*>(ws);
    p.part_ml = reinterpret_cast<float*>(ws + ((po + 255) / 256) * 256);
    p.counters = reinterpret_cast<unsigned*>(ws + ((po + 255) / 256) * 256 + ((pm + 255) / 256) * 256);
    // the split tickets must start at zero; the partials are written before they are read
    W4_CUDA(cudaMemsetAsync(p.counters, 0, (size_t)b * hkv * sizeof(unsigned), (cudaStream_t)stream));
    p.errword = w4::device_error_word();
    p.scale_log2 = scale * 1.4426950408889634f;
    p.B = b;
    p.Hq = hq;
    p.Hkv = hkv;
    p.group = hq / hkv;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    p.max_context = max_context;
    p.ppw = pl.ppw;
    p.max_splits = pl.max_splits;
    // programmatic dependent launch, as in w4_paged_decode_attention
    const cudaError_t e = w4::attention_launch(p, pl, (cudaStream_t)stream, true);
    if (e != cudaSuccess) return w4::cuda_check(e, "paged_decode_attention_noalloc launch");
    return W4_OK;
}
