// decode_step: one greedy token of a Qwen2-style decoder over INT4 weights,
// eager or captured as one CUDA graph.
//
// "How to build your own LLM runtime from scratch (Towards Data Science)",
// opening paragraph (decode-only engine, greedy sampling) and section "The one
// lesson that generalizes" (280+ launches per token made launch overhead
// dominate; the same kernels submitted as one graph were 7x faster).
//
// Launches per step: embedding (1) + per layer [QKV GEMV with fused RMSNorm,
// bias, RoPE and paged KV append; paged attention; O GEMV + residual; gate/up
// GEMV with fused RMSNorm and SiLU(gate)*up; down GEMV + residual] (5) + LM
// head GEMV with fused final RMSNorm and argmax (1) = 5 * layers + 2.
// Position and context length live on the device and are advanced by the
// last kernel, so a captured graph replays unchanged token after token.
#include "model.cuh"

namespace w4 {

__global__ void embed_kernel(const int32_t* __restrict__ token, const __half* __restrict__ embed, int vocab,
                             int hidden, float* __restrict__ x, int* errword) {
    pdl_wait();
    int t = token[0];
    if (t < 0 || t >= vocab) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_device_error(errword, W4_DEVERR_TOKEN);
        t = -1;
    }
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < hidden; i += gridDim.x * blockDim.x)
        x[i] = t < 0 ? 0.f : __half2float(embed[(size_t)t * hidden + i]);
}

// cos/sin of pos * theta^(-2i/128) for every position and i < 64, in double
// precision once at set-up, stored as fp32 pairs.
__global__ void rope_table_kernel(float2* table, int max_context, double theta) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= max_context * 64) return;
    const int pos = idx / 64, i = idx % 64;
    const double inv = pow(theta, -2.0 * i / 128.0);
    double s, c;
    sincos((double)pos * inv, &s, &c);
    table[idx] = make_float2((float)c, (float)s);
}

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// The decode workspace of one cache: laid out from the model's shape and plans
// and the cache's capacity (the RoPE table and the attention split partials).
static ModelLayout build_layout(const w4_model* m, const w4_kv_config& kc, const AttnPlan& p_att) {
    const w4_model_config& c = m->cfg;
    ModelLayout L = {};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    L.x = take((size_t)c.hidden * 4);
    L.qr = take((size_t)c.hidden * 2);
    L.att = take((size_t)c.hidden * 2);
    L.ctx = take(16);
    L.mlp = take((size_t)c.ffn * 2);
    L.lmctr = take(16);
    L.attws = take(attention_ws_bytes(1, c.n_q_heads, c.n_kv_heads, p_att));
    L.key = take(16);
    L.rope = take((size_t)kc.max_context * 64 * sizeof(float2));
    L.total = off;
    return L;
}

static AttnPlan decode_attention_plan(const w4_model_config& c, int max_context) {
    return attention_plan(1, c.n_kv_heads, max_context);
}

static bool same_shape(const w4_model_config& a, const w4_model_config& b) {
    return a.hidden == b.hidden && a.ffn == b.ffn && a.n_layers == b.n_layers && a.n_q_heads == b.n_q_heads &&
           a.n_kv_heads == b.n_kv_heads && a.head_dim == b.head_dim && a.vocab == b.vocab;
}

w4_status check_pair(const w4_model* m, const w4_kv* kv) {
    W4_REQUIRE(m != nullptr && kv != nullptr, W4_ERR_NULL, "decode: null model or cache");
    W4_REQUIRE(same_shape(m->cfg, kv->mcfg), W4_ERR_SHAPE, "decode: the cache was laid out for another model shape");
    int dev = -1;
    W4_CUDA(cudaGetDevice(&dev));
    W4_REQUIRE(dev == m->device && dev == kv->device, W4_ERR_STATE,
               "decode: model on device %d, cache on device %d, current is %d", m->device, kv->device, dev);
    return W4_OK;
}

// Launch kernel `which` (W4_K_*) of layer `li` exactly as the decode step does.
w4_status launch_one(const w4_model* m, const w4_kv* kv, const StepArgs& a, int which, int li) {
    const w4_model_config& c = m->cfg;
    const w4_kv_config& kc = kv->kc;
    const ModelLayout& L = kv->lay;
    char* ws = kv->ws;
    cudaStream_t st = a.st;
    const int kvdim = c.n_kv_heads * c.head_dim;
    const int nqkv = c.hidden + 2 * kvdim;
    int* err = device_error_word();
    float* x = reinterpret_cast<float*>(ws + L.x);
    __half* qr = reinterpret_cast<__half*>(ws + L.qr);
    int32_t* ctx = reinterpret_cast<int32_t*>(ws + L.ctx);
    __half* mlp = reinterpret_cast<__half*>(ws + L.mlp);
    // the first kernel of a step follows ordinary stream order
    const bool pdl = m->pdl && which != W4_K_EMBED;

    cudaLaunchAttribute pattr[1];
    pattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pattr[0].val.programmaticStreamSerializationAllowed = 1;
    auto small_cfg = [&](unsigned grid, unsigned block) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(block);
        cfg.stream = st;
        cfg.attrs = pattr;
        cfg.numAttrs = pdl ? 1 : 0;
        return cfg;
    };
    const w4_layer_weights* lw = (li >= 0 && li < c.n_layers) ? &m->layers[li] : nullptr;
    const w4_kv_layer* lp = (li >= 0 && li < c.n_layers) ? &kv->pools[li] : nullptr;
    GemvParams g = {};
    g.M = 1;
    g.errword = err;
    switch (which) {
        case W4_K_EMBED: {
            cudaLaunchConfig_t cfg = small_cfg((c.hidden + 255) / 256, 256);
            W4_CUDA(cudaLaunchKernelEx(&cfg, embed_kernel, a.token_in, m->embed, c.vocab, c.hidden, x, err));
            return W4_OK;
        }
        case W4_K_QKV:  // RMSNorm(x) -> QKV rows + bias -> RoPE; q out, k/v into the pools, ctx = pos + 1
            g.xres = x;
            g.gamma = static_cast<const __half*>(lw->ln1);
            g.eps = c.rms_eps;
            g.w0 = lw->wqkv.packed;
            g.s0 = static_cast<const __half*>(lw->wqkv.scales);
            g.N = nqkv;
            g.K = c.hidden;
            g.bias = static_cast<const __half*>(lw->bqkv);
            g.rope = reinterpret_cast<const float2*>(ws + L.rope);
            g.pos_in = kv->pos;
            g.pt = kv->pt;
            g.qout = qr;
            g.k_pool = static_cast<__half*>(lp->k_pool);
            g.v_pool = static_cast<__half*>(lp->v_pool);
            g.ctx = ctx;
            g.hq = c.n_q_heads;
            g.hkv = c.n_kv_heads;
            g.max_pages = kc.max_pages;
            g.num_pages = kc.num_pages;
            g.max_context = kc.max_context;
            W4_CUDA((tma_launch<V_SUBNORMAL, X_RMSNORM, E_QKV_ROPE>(g, m->tp[CTR_QKV], st, pdl)));
            return W4_OK;
        case W4_K_ATTENTION: {   // splits merged by the last CTA of each KV head: fp16 output
            AttnParams ap = {};
            ap.q = qr;
            ap.out = reinterpret_cast<__half*>(ws + L.att);
            ap.k_pool = static_cast<const __half*>(lp->k_pool);
            ap.v_pool = static_cast<const __half*>(lp->v_pool);
            ap.pt = kv->pt;
            ap.lens = ctx;
            ap.pos_hint = kv->pos;   // pages before this step's row are loaded while QKV runs
            const AttnPlan& pa = kv->p_att;
            const size_t po = (size_t)c.n_q_heads * pa.max_splits * kHeadDim * sizeof(float);
            const size_t pm = (size_t)c.n_q_heads * pa.max_splits * 2 * sizeof(float);
            char* aw = ws + L.attws;
            ap.part_o = reinterpret_cast<float*>(aw);
            ap.part_ml = reinterpret_cast<float*>(aw + align_up(po, 256));
            ap.counters = reinterpret_cast<unsigned*>(aw + align_up(po, 256) + align_up(pm, 256));
            ap.errword = err;
            ap.scale_log2 = (float)(1.0 / std::sqrt((double)c.head_dim) * 1.4426950408889634);
            ap.B = 1;
            ap.Hq = c.n_q_heads;
            ap.Hkv = c.n_kv_heads;
            ap.group = c.n_q_heads / c.n_kv_heads;
            ap.max_pages = kc.max_pages;
            ap.num_pages = kc.num_pages;
            ap.max_context = kc.max_context;
            ap.ppw = pa.ppw;
            ap.max_splits = pa.max_splits;
            W4_CUDA(attention_launch(ap, pa, st, pdl));
            return W4_OK;
        }
        case W4_K_O: {  // O projection of the attention output + residual into x
            g.x = reinterpret_cast<const __half*>(ws + L.att);
            g.w0 = lw->wo.packed;
            g.s0 = static_cast<const __half*>(lw->wo.scales);
            g.N = c.hidden;
            g.K = c.hidden;
            g.y32 = x;
            W4_CUDA((tma_launch<V_SUBNORMAL, X_F16, E_RESID_F32>(g, m->tp[CTR_O], st, pdl)));
            return W4_OK;
        }
        case W4_K_GATE_UP:  // RMSNorm prologue, SiLU(gate)*up epilogue
            g.xres = x;
            g.gamma = static_cast<const __half*>(lw->ln2);
            g.eps = c.rms_eps;
            g.w0 = lw->wgate.packed;
            g.s0 = static_cast<const __half*>(lw->wgate.scales);
            g.w1 = lw->wup.packed;
            g.s1 = static_cast<const __half*>(lw->wup.scales);
            g.N = c.ffn;
            g.K = c.hidden;
            g.y16 = mlp;
            W4_CUDA((tma_launch<V_SUBNORMAL, X_RMSNORM, E_SWIGLU>(g, m->tp[CTR_GU], st, pdl)));
            return W4_OK;
        case W4_K_DOWN:  // down projection + residual into x
            g.x = mlp;
            g.w0 = lw->wdown.packed;
            g.s0 = static_cast<const __half*>(lw->wdown.scales);
            g.N = c.hidden;
            g.K = c.ffn;
            g.y32 = x;
            if (li + 1 < c.n_layers) {  // the next layer's QKV weights, into L2 while this streams
                const w4_layer_weights& nx = m->layers[li + 1];
                g.pf0 = nx.wqkv.packed;
                g.pf0_bytes = (size_t)nqkv * c.hidden / 2;
                g.pf1 = nx.wqkv.scales;
                g.pf1_bytes = ((size_t)nqkv * (c.hidden / 128) * 2) & ~(size_t)15;
            }
            W4_CUDA((tma_launch<V_SUBNORMAL, X_F16, E_RESID_F32>(g, m->tp[CTR_DOWN], st, pdl)));
            return W4_OK;
        case W4_K_LM_HEAD:  // final RMSNorm -> LM head -> argmax -> token_out, pos += 1
            g.xres = x;
            g.gamma = m->final_norm;
            g.eps = c.rms_eps;
            g.w0 = m->lm.packed;
            g.s0 = static_cast<const __half*>(m->lm.scales);
            g.N = c.vocab;
            g.K = c.hidden;
            g.y32 = a.logits;
            g.counters = reinterpret_cast<unsigned*>(ws + L.lmctr);
            g.amax_key = reinterpret_cast<unsigned long long*>(ws + L.key);
            g.token_out = a.token_out;
            g.pos = kv->pos;
            W4_CUDA((tma_launch<V_SUBNORMAL, X_RMSNORM, E_ARGMAX>(g, m->tp[CTR_LM], st, pdl)));
            return W4_OK;
        default:
            return set_error(W4_ERR_RANGE, "decode: unknown kernel id %d", which);
    }
}

static w4_status launch_step(const w4_model* m, const w4_kv* kv, const StepArgs& a) {
    w4_status s = launch_one(m, kv, a, W4_K_EMBED, -1);
    for (int li = 0; li < m->cfg.n_layers && s == W4_OK; ++li)
        for (int k = W4_K_QKV; k <= W4_K_DOWN && s == W4_OK; ++k) s = launch_one(m, kv, a, k, li);
    if (s == W4_OK) s = launch_one(m, kv, a, W4_K_LM_HEAD, -1);
    return s;
}

}  // namespace w4

extern "C" w4_status w4_model_create(const w4_model_config* cfg, const w4_layer_weights* layers, const void* embed,
                                     const void* final_norm, w4_qmatrix lm_head, w4_model** out) {
    W4_REQUIRE(cfg && layers && embed && final_norm && lm_head.packed && lm_head.scales && out, W4_ERR_NULL,
               "model_create: null pointer");
    const w4_model_config& c = *cfg;
    W4_REQUIRE(c.head_dim == 128, W4_ERR_SHAPE, "model_create: head_dim must be 128");
    W4_REQUIRE(c.n_layers >= 1 && c.n_kv_heads >= 1 && c.n_q_heads % c.n_kv_heads == 0 &&
                   c.n_q_heads / c.n_kv_heads <= 16 && c.n_q_heads <= 64,
               W4_ERR_SHAPE, "model_create: bad head counts");
    W4_REQUIRE(c.hidden == c.n_q_heads * c.head_dim, W4_ERR_SHAPE, "model_create: hidden must be n_q_heads*128");
    W4_REQUIRE(c.hidden % 128 == 0 && c.ffn % 128 == 0 && c.ffn > 0 && c.vocab > 0, W4_ERR_SHAPE,
               "model_create: hidden and ffn must be multiples of 128");
    W4_REQUIRE(c.rms_eps >= 0.f && c.rope_theta > 0.f, W4_ERR_RANGE, "model_create: bad eps/theta");
    for (int i = 0; i < c.n_layers; ++i) {
        const w4_layer_weights& l = layers[i];
        W4_REQUIRE(l.ln1 && l.ln2 && l.wqkv.packed && l.wqkv.scales && l.bqkv && l.wo.packed && l.wo.scales &&
                       l.wgate.packed && l.wgate.scales && l.wup.packed && l.wup.scales && l.wdown.packed &&
                       l.wdown.scales,
                   W4_ERR_NULL, "model_create: layer %d has a null pointer", i);
        W4_REQUIRE(w4::aligned16(l.wqkv.packed) && w4::aligned16(l.wo.packed) && w4::aligned16(l.wgate.packed) &&
                       w4::aligned16(l.wup.packed) && w4::aligned16(l.wdown.packed) && w4::aligned16(l.ln1) &&
                       w4::aligned16(l.ln2),
                   W4_ERR_ALIGN, "model_create: layer %d buffer not 16-byte aligned", i);
    }
    W4_REQUIRE(w4::aligned16(lm_head.packed) && w4::aligned16(final_norm), W4_ERR_ALIGN,
               "model_create: LM head / final norm not 16-byte aligned");
    w4_model* m = new w4_model();
    m->cfg = c;
    m->layers.assign(layers, layers + c.n_layers);
    m->embed = static_cast<const __half*>(embed);
    m->final_norm = static_cast<const __half*>(final_norm);
    m->lm = lm_head;
    m->pdl = true;
    cudaGetDevice(&m->device);
    const int kv = c.n_kv_heads * c.head_dim;
    using namespace w4;
    m->tp[CTR_QKV] = tma_plan(1, c.hidden + 2 * kv, c.hidden);
    m->tp[CTR_O] = tma_plan(1, c.hidden, c.hidden);
    m->tp[CTR_GU] = tma_plan(2, c.ffn, c.hidden);
    m->tp[CTR_DOWN] = tma_plan(1, c.hidden, c.ffn);
    m->tp[CTR_LM] = tma_plan(1, c.vocab, c.hidden);
    for (int i = 0; i < CTR_COUNT; ++i)
        if (m->tp[i].grid == 0 || (i == CTR_QKV && m->tp[i].a.rg != 2)) {
            delete m;
            return set_error(W4_ERR_SHAPE, "model_create: hidden/ffn too large for the streaming GEMV's shared memory");
        }
    *out = m;
    return W4_OK;
}

extern "C" void w4_model_destroy(w4_model* m) { delete m; }

extern "C" w4_status w4_model_set_pdl(w4_model* m, int enable) {
    W4_REQUIRE(m != nullptr, W4_ERR_NULL, "model_set_pdl: null model");
    m->pdl = enable != 0;
    return W4_OK;
}

static w4_status check_kv_config(const w4_kv_config* kc, int n_kv_heads) {
    W4_REQUIRE(kc != nullptr, W4_ERR_NULL, "kv: null config");
    W4_REQUIRE(kc->max_context >= 1 && kc->max_pages >= 1 && kc->num_pages >= 1 &&
                   (long long)kc->max_context <= (long long)kc->max_pages * 16,
               W4_ERR_RANGE, "kv: max_context must be in [1, 16*max_pages]");
    W4_REQUIRE((long long)kc->num_pages * n_kv_heads * 16 < (1LL << 31), W4_ERR_SHAPE, "kv: pool too large");
    return W4_OK;
}

extern "C" size_t w4_kv_workspace_size(const w4_model* m, const w4_kv_config* kc) {
    if (!m || check_kv_config(kc, m->cfg.n_kv_heads) != W4_OK) return 0;
    return w4::build_layout(m, *kc, w4::decode_attention_plan(m->cfg, kc->max_context)).total;
}

extern "C" w4_status w4_kv_create(const w4_model* m, const w4_kv_config* kc, const w4_kv_layer* layers,
                                  const int32_t* page_table, int32_t* pos, void* workspace, size_t workspace_bytes,
                                  void* stream, w4_kv** out) {
    W4_REQUIRE(m && layers && page_table && pos && workspace && out, W4_ERR_NULL, "kv_create: null pointer");
    w4_status s = check_kv_config(kc, m->cfg.n_kv_heads);
    if (s != W4_OK) return s;
    const w4_model_config& c = m->cfg;
    for (int i = 0; i < c.n_layers; ++i) {
        W4_REQUIRE(layers[i].k_pool && layers[i].v_pool, W4_ERR_NULL, "kv_create: layer %d has a null pool", i);
        W4_REQUIRE(w4::aligned16(layers[i].k_pool) && w4::aligned16(layers[i].v_pool), W4_ERR_ALIGN,
                   "kv_create: layer %d pool not 16-byte aligned", i);
    }
    W4_REQUIRE(w4::aligned16(workspace), W4_ERR_ALIGN, "kv_create: workspace must be 16-byte aligned");
    const w4::AttnPlan pa = w4::decode_attention_plan(c, kc->max_context);
    const w4::ModelLayout lay = w4::build_layout(m, *kc, pa);
    W4_REQUIRE(workspace_bytes >= lay.total, W4_ERR_CAPACITY, "kv_create: workspace of %zu bytes needed", lay.total);
    int dev = -1;
    W4_CUDA(cudaGetDevice(&dev));
    W4_REQUIRE(dev == m->device, W4_ERR_STATE, "kv_create: model was created on device %d, current is %d", m->device,
               dev);
    w4_kv* kv = new w4_kv();
    kv->mcfg = c;
    kv->kc = *kc;
    kv->pools.assign(layers, layers + c.n_layers);
    kv->pt = page_table;
    kv->pos = pos;
    kv->ws = static_cast<char*>(workspace);
    kv->ws_bytes = workspace_bytes;
    kv->p_att = pa;
    kv->lay = lay;
    kv->device = dev;
    kv->tmk.resize(c.n_layers);
    kv->tmv.resize(c.n_layers);
    for (int i = 0; i < c.n_layers && s == W4_OK; ++i) {
        s = w4::make_pool_tensor_map(&kv->tmk[i], layers[i].k_pool, kc->num_pages, c.n_kv_heads);
        if (s == W4_OK) s = w4::make_pool_tensor_map(&kv->tmv[i], layers[i].v_pool, kc->num_pages, c.n_kv_heads);
    }
    if (s != W4_OK) {
        delete kv;
        return s;
    }
    // a zero-filled workspace (its split tickets and argmax key start at zero), then the RoPE table
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(workspace, 0, lay.total, st);
    if (e == cudaSuccess) {
        const int n = kc->max_context * 64;
        w4::rope_table_kernel<<<(n + 255) / 256, 256, 0, st>>>(
            reinterpret_cast<float2*>(kv->ws + lay.rope), kc->max_context, (double)c.rope_theta);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        delete kv;
        return w4::cuda_check(e, "kv_create");
    }
    *out = kv;
    return W4_OK;
}

extern "C" void w4_kv_destroy(w4_kv* kv) { delete kv; }

extern "C" int w4_decode_launches_per_step(const w4_model* m) { return m ? 5 * m->cfg.n_layers + 2 : 0; }

extern "C" w4_status w4_decode_step(const w4_model* m, w4_kv* kv, const int32_t* token_in, int32_t* token_out,
                                    float* logits, void* stream) {
    w4_status s = w4::check_pair(m, kv);
    if (s != W4_OK) return s;
    W4_REQUIRE(token_in && token_out, W4_ERR_NULL, "decode_step: null token pointer");
    return w4::launch_step(m, kv, {token_in, token_out, logits, (cudaStream_t)stream});
}

extern "C" w4_status w4_decode_launch_kernel(const w4_model* m, w4_kv* kv, int kernel, int layer,
                                             const int32_t* token_in, int32_t* token_out, float* logits,
                                             void* stream) {
    w4_status s = w4::check_pair(m, kv);
    if (s != W4_OK) return s;
    W4_REQUIRE(token_in && token_out, W4_ERR_NULL, "decode_launch_kernel: null token pointer");
    const bool per_layer = kernel >= W4_K_QKV && kernel <= W4_K_DOWN;
    W4_REQUIRE(!per_layer || (layer >= 0 && layer < m->cfg.n_layers), W4_ERR_RANGE,
               "decode_launch_kernel: layer %d out of range", layer);
    return w4::launch_one(m, kv, {token_in, token_out, logits, (cudaStream_t)stream}, kernel, layer);
}

extern "C" w4_status w4_decode_graph_create(const w4_model* m, w4_kv* kv, const int32_t* token_in,
                                            int32_t* token_out, float* logits, void* stream, w4_graph** out) {
    w4_status s = w4::check_pair(m, kv);
    if (s != W4_OK) return s;
    W4_REQUIRE(token_in && token_out && out, W4_ERR_NULL, "decode_graph_create: null pointer");
    W4_REQUIRE(stream != nullptr, W4_ERR_STATE, "decode_graph_create: capture needs a non-default stream");
    cudaStream_t st = (cudaStream_t)stream;
    W4_CUDA(cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal));
    s = w4::launch_step(m, kv, {token_in, token_out, logits, st});
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(st, &graph);
    if (s != W4_OK) {
        if (graph) cudaGraphDestroy(graph);
        return s;
    }
    if (e != cudaSuccess) return w4::cuda_check(e, "cudaStreamEndCapture");
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    if (e != cudaSuccess) {
        cudaGraphDestroy(graph);
        return w4::cuda_check(e, "cudaGraphInstantiate");
    }
    w4_graph* g = new w4_graph();
    g->graph = graph;
    g->exec = exec;
    g->device = m->device;
    *out = g;
    return W4_OK;
}

extern "C" w4_status w4_decode_graph_launch(w4_graph* g, void* stream) {
    W4_REQUIRE(g != nullptr, W4_ERR_NULL, "decode_graph_launch: null graph");
    W4_CUDA(cudaGraphLaunch(g->exec, (cudaStream_t)stream));
    return W4_OK;
}

extern "C" void w4_decode_graph_destroy(w4_graph* g) {
    if (!g) return;
    cudaGraphExecDestroy(g->exec);
    cudaGraphDestroy(g->graph);
    delete g;
}
