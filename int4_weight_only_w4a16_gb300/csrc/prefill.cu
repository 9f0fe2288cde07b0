// prefill: run a prompt of n tokens through the model in one pass and leave
// the decode stream ready for the token after it.
//
// "How to build your own LLM runtime from scratch (Towards Data Science)",
// section "What the numbers say": time to first token is the prompt pass plus
// the first sampled token.  The pages give no prefill design; this one is the
// plain reading of the same Qwen2 block as the decode step, applied to all
// prompt rows at once:
//
//   x[t] = E[token t]                                       (t = 0 .. n-1)
//   per layer:  h = RMSNorm(x) g1 -> [q k v] = h Wqkv^T + b -> RoPE(q, k) at
//               start + t -> K/V rows appended at start + t -> causal paged
//               attention (query t sees positions 0 .. start + t) -> x += a Wo^T
//               -> h = RMSNorm(x) g2 -> x += (SiLU(h Wg^T) * (h Wu^T)) Wd^T
//   the last row: final RMSNorm -> LM head -> argmax -> token_out, pos
//
// Every matrix product here is a real GEMM (n rows of activations): the
// fused W4A16 tcgen05 kernel of gemm_tc05.cuh (the INT4 codes multiplied
// exactly on the tensor cores, each scale group's sum scaled in fp32), with
// the residual add and SiLU(gate) * up in its epilogue.  Attention is the
// causal prompt-pass kernel of attention.cuh (16 prompt rows of one query head
// per warp, the group's K/V pages staged once per CTA); the rest are kernels
// of this file and the decode step's fused LM head for the last row.
#include "model.cuh"

namespace w4 {

namespace {

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

struct PrefillLayout {
    size_t x, hn, q, att_out, act, y, gpart, apart, total;
};

// The four fused GEMMs of a layer for an n-token prompt: QKV, O, gate/up, down.
struct LayerPlans {
    GemmPlan qkv, o, gu, down;
};

int nqkv_of(const w4_model_config& c) { return c.hidden + 2 * c.n_kv_heads * c.head_dim; }

LayerPlans layer_plans(const w4_model_config& c, int n) {
    const int sms = sm_count();
    return {gemm_plan(G_STORE, n, nqkv_of(c), c.hidden, sms), gemm_plan(G_RESID, n, c.hidden, c.hidden, sms),
            gemm_plan(G_SWIGLU, n, c.ffn, c.hidden, sms), gemm_plan(G_RESID, n, c.hidden, c.ffn, sms)};
}

PrefillLayout prefill_layout(const w4_model_config& c, const w4_kv_config& kc, int n) {
    PrefillLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align256(off + bytes);
        return o;
    };
    const size_t H = c.hidden, F = c.ffn, N3 = nqkv_of(c);
    L.x = take((size_t)n * H * 4);
    L.hn = take((size_t)n * H * 2);
    L.q = take((size_t)n * H * 2);
    L.att_out = take((size_t)n * H * 2);
    L.act = take((size_t)n * F * 2);
    L.y = take((size_t)n * N3 * 4);
    const LayerPlans lp = layer_plans(c, n);   // split-K partials of the largest GEMM of a layer
    L.gpart = take(std::max(std::max(gemm_part_bytes(G_STORE, lp.qkv), gemm_part_bytes(G_RESID, lp.o)),
                            std::max(gemm_part_bytes(G_SWIGLU, lp.gu), gemm_part_bytes(G_RESID, lp.down))));
    L.apart = take(prefill_attention_ws_bytes(n, c.n_kv_heads, c.n_q_heads / c.n_kv_heads, kc.max_context));
    L.total = off;
    return L;
}

__global__ void embed_rows_kernel(const int32_t* __restrict__ tokens, const __half* __restrict__ embed, int vocab,
                                  int hidden, float* __restrict__ x, int* errword) {
    const int t = blockIdx.x;
    int tok = tokens[t];
    if (tok < 0 || tok >= vocab) {
        if (threadIdx.x == 0) record_device_error(errword, W4_DEVERR_TOKEN);
        tok = -1;
    }
    float* xr = x + (size_t)t * hidden;
    const __half* er = embed + (size_t)(tok < 0 ? 0 : tok) * hidden;
    for (int i = threadIdx.x; i < hidden; i += blockDim.x) xr[i] = tok < 0 ? 0.f : __half2float(er[i]);
}

// h[t] = fp16(x[t] / sqrt(mean(x[t]^2) + eps) * gamma); one CTA of 128 threads
// per row, the row held in registers as float4s (hidden <= 128 * 4 * ITEMS).
// With nsplit > 0 the residual first takes the split-K partial sums of the
// GEMM before it: x[t] += sum over s in order of part[s][t] (written back).
template <int ITEMS>
__global__ void __launch_bounds__(128) rmsnorm_rows_kernel(float* __restrict__ x, const __half* __restrict__ gamma,
                                                           float eps, int hidden, __half* __restrict__ out,
                                                           const float* __restrict__ part, int nsplit,
                                                           size_t split_stride) {
    __shared__ float red[4];
    const int t = blockIdx.x, tid = threadIdx.x;
    float4* xr = reinterpret_cast<float4*>(x + (size_t)t * hidden);
    const int n4 = hidden / 4;
    float4 v[ITEMS];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        const int idx = tid + i * 128;
        v[i] = idx < n4 ? xr[idx] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (nsplit > 0) {
        // the split partials in split order, every item's load of a split issued together
        const float4* pr = reinterpret_cast<const float4*>(part + (size_t)t * hidden);
        float4 a[ITEMS];
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) {
            const int idx = tid + i * 128;
            a[i] = idx < n4 ? __ldcg(pr + idx) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int sp = 1; sp < nsplit; ++sp) {
            const float4* ps = reinterpret_cast<const float4*>(part + sp * split_stride + (size_t)t * hidden);
            float4 b[ITEMS];
#pragma unroll
            for (int i = 0; i < ITEMS; ++i) {
                const int idx = tid + i * 128;
                b[i] = idx < n4 ? __ldcg(ps + idx) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i = 0; i < ITEMS; ++i) {
                a[i].x += b[i].x; a[i].y += b[i].y; a[i].z += b[i].z; a[i].w += b[i].w;
            }
        }
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) {
            const int idx = tid + i * 128;
            if (idx < n4) {
                v[i].x += a[i].x; v[i].y += a[i].y; v[i].z += a[i].z; v[i].w += a[i].w;
                xr[idx] = v[i];
            }
        }
    }
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        ss = fmaf(v[i].x, v[i].x, ss);
        ss = fmaf(v[i].y, v[i].y, ss);
        ss = fmaf(v[i].z, v[i].z, ss);
        ss = fmaf(v[i].w, v[i].w, ss);
    }
    ss = warp_sum(ss);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    const float r = 1.0f / sqrtf((red[0] + red[1] + red[2] + red[3]) / (float)hidden + eps);
    const uint2* gr = reinterpret_cast<const uint2*>(gamma);
    uint2* o = reinterpret_cast<uint2*>(out + (size_t)t * hidden);
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        const int idx = tid + i * 128;
        if (idx < n4) {
            const uint2 g = gr[idx];
            const float2 g0 = __half22float2(u32_as_h2(g.x)), g1 = __half22float2(u32_as_h2(g.y));
            o[idx] = make_uint2(h2_as_u32(__floats2half2_rn(v[i].x * r * g0.x, v[i].y * r * g0.y)),
                                h2_as_u32(__floats2half2_rn(v[i].z * r * g1.x, v[i].w * r * g1.y)));
        }
    }
}

// Bias, fp16, RoPE of every q/k row pair at position start + t; q rows out,
// k and v rows into the pools.  One CTA per row t.
// y holds the QKV rows, or with nsplit > 1 the GEMM's split-K partials (added
// here in split order).
__global__ void rope_append_rows_kernel(const float* __restrict__ y, int ldy, int nsplit, size_t split_stride,
                                        const __half* __restrict__ bias,
                                        const float2* __restrict__ rope, const int32_t* __restrict__ pt, int start,
                                        int hq, int hkv, int num_pages, int max_pages, int max_context,
                                        __half* __restrict__ q_out, __half* __restrict__ k_pool,
                                        __half* __restrict__ v_pool, int* errword) {
    const int t = blockIdx.x;
    const int pos = start + t;
    const bool pos_ok = pos >= 0 && pos < max_context && pos < max_pages * 16;
    const int page = pos_ok ? pt[pos >> 4] : -1;
    const bool ok = pos_ok && page >= 0 && page < num_pages;
    const int slot = pos & 15;
    if (threadIdx.x == 0 && !ok) record_device_error(errword, W4_DEVERR_POSITION | W4_DEVERR_PAGE_ID);
    const int qrows = hq * 128, krows = hkv * 128;
    const int pairs = (qrows + 2 * krows) / 2;
    const float* yr = y + (size_t)t * ldy;
    // four pairs per thread at a time: every load of the four is issued before any is used
    constexpr int U = 4;
    for (int base = threadIdx.x; base < pairs; base += U * blockDim.x) {
        float2 a[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int pr = base + u * blockDim.x;
            a[u] = pr < pairs ? *reinterpret_cast<const float2*>(yr + 2 * pr) : make_float2(0.f, 0.f);
        }
        for (int sp = 1; sp < nsplit; ++sp) {   // split partials in split order
            float2 b[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int pr = base + u * blockDim.x;
                b[u] = pr < pairs ? __ldcg(reinterpret_cast<const float2*>(yr + sp * split_stride + 2 * pr))
                                  : make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                a[u].x += b[u].x;
                a[u].y += b[u].y;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int pr = base + u * blockDim.x;
            if (pr >= pairs) break;
            const int row = 2 * pr;
            const __half h0 = __float2half_rn(a[u].x + __half2float(bias[row]));
            const __half h1 = __float2half_rn(a[u].y + __half2float(bias[row + 1]));
            if (row < qrows + krows) {
                const int r = row < qrows ? row : row - qrows;
                const int head = r >> 7, i = (r & 127) >> 1;
                const float x0 = __half2float(h0), x1 = __half2float(h1);
                const float2 cs = rope[(size_t)(ok ? pos : 0) * 64 + i];
                const __half o0 = __float2half_rn(x0 * cs.x - x1 * cs.y);
                const __half o1 = __float2half_rn(x1 * cs.x + x0 * cs.y);
                if (row < qrows) {
                    __half* dst = q_out + (size_t)t * qrows + head * 128;
                    dst[i] = o0;
                    dst[i + 64] = o1;
                } else if (ok) {
                    __half* dst = k_pool + (((size_t)page * hkv + head) * 16 + slot) * 128;
                    dst[i] = o0;
                    dst[i + 64] = o1;
                }
            } else if (ok) {
                const int r = row - qrows - krows;
                const int head = r >> 7, d = r & 127;
                __half* dst = v_pool + (((size_t)page * hkv + head) * 16 + slot) * 128;
                dst[d] = h0;
                dst[d + 1] = h1;
            }
        }
    }
}

// The decode stream's state after the prompt: its residual row is the last
// prompt row and *pos = start + n - 1 (the LM head kernel then adds one).
// With nsplit > 0 the last row first takes the split-K partials of the last
// down projection (part_last: that row of split 0).
__global__ void prefill_tail_kernel(const float* __restrict__ x_last, int hidden, float* __restrict__ x_dec,
                                    int32_t* pos, int pos_value, const float* __restrict__ part_last, int nsplit,
                                    size_t split_stride) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < hidden; i += gridDim.x * blockDim.x) {
        float v = x_last[i];
        if (nsplit > 0) {
            float a = __ldcg(part_last + i);
            for (int sp = 1; sp < nsplit; ++sp) a += __ldcg(part_last + sp * split_stride + i);
            v += a;
        }
        x_dec[i] = v;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) *pos = pos_value;
}

struct Prefill {
    const w4_model* m;
    const w4_kv* kv;
    char* ws;
    PrefillLayout L;
    LayerPlans lp_;
    CUtensorMap tm_hn, tm_att, tm_act;   // the GEMM inputs as TMA tensors
    int n;
    cudaStream_t st;
    int* err;

    // split-K partial sums left in the workspace for the next kernel to add
    // (QKV: the RoPE kernel; O and down: the RMSNorm after them; the last down:
    // the tail), instead of a separate merge launch: [nsplit][n][N] fp32
    int pend_splits = 0;
    size_t pend_stride = 0;

    w4_status fused(int epi, GemmPlan p, const CUtensorMap& tmx, const CUtensorMap& tmw0, const CUtensorMap& tmw1,
                    const w4_qmatrix& m0, const w4_qmatrix* m1, float* y, int ldy, __half* act) {
        const void* s0 = m0.scales;
        const void* s1 = m1 ? m1->scales : nullptr;
        p.a.w0 = m0.packed;
        p.a.w1 = m1 ? m1->packed : m0.packed;
        p.a.s0 = static_cast<const __half*>(s0);
        p.a.s1 = static_cast<const __half*>(s1);
        p.a.y = y;
        p.a.ldy = ldy;
        p.a.act = act;
        p.a.part = reinterpret_cast<float*>(ws + L.gpart);
        p.a.errword = err;
        const bool defer = epi != G_SWIGLU && p.a.splits > 1;
        W4_CUDA(gemm_tc05_launch(epi, p, tmx, tmw0, tmw1, st, !defer));
        pend_splits = defer ? p.a.splits : 0;
        pend_stride = (size_t)n * p.a.N;
        return W4_OK;
    }

    w4_status rmsnorm(const void* gamma, __half* out) {   // adds any pending residual partials first
        float* x = reinterpret_cast<float*>(ws + L.x);
        const __half* g = static_cast<const __half*>(gamma);
        const float* part = reinterpret_cast<const float*>(ws + L.gpart);
        if (m->cfg.hidden <= 128 * 4 * 8)
            rmsnorm_rows_kernel<8><<<n, 128, 0, st>>>(x, g, m->cfg.rms_eps, m->cfg.hidden, out, part, pend_splits,
                                                      pend_stride);
        else   // hidden = n_q_heads * 128 <= 8192
            rmsnorm_rows_kernel<16><<<n, 128, 0, st>>>(x, g, m->cfg.rms_eps, m->cfg.hidden, out, part, pend_splits,
                                                       pend_stride);
        pend_splits = 0;
        W4_CUDA(cudaGetLastError());
        return W4_OK;
    }

    w4_status layer(int li, int start, const float2* rope) {
        const w4_model_config& c = m->cfg;
        const w4_kv_config& kc = kv->kc;
        const w4_layer_weights& lw = m->layers[li];
        const w4_kv_layer& lp = kv->pools[li];
        const int H = c.hidden, N3 = nqkv_of(c);
        float* x = reinterpret_cast<float*>(ws + L.x);
        __half* hn = reinterpret_cast<__half*>(ws + L.hn);
        __half* q = reinterpret_cast<__half*>(ws + L.q);
        __half* ao = reinterpret_cast<__half*>(ws + L.att_out);
        __half* act = reinterpret_cast<__half*>(ws + L.act);
        float* y = reinterpret_cast<float*>(ws + L.y);

        const CUtensorMap* wm = &m->pf_maps[(size_t)li * 5];   // qkv, o, gate, up, down
        w4_status s = rmsnorm(lw.ln1, hn);
        if (s == W4_OK) s = fused(G_STORE, lp_.qkv, tm_hn, wm[0], wm[0], lw.wqkv, nullptr, y, N3, nullptr);
        if (s != W4_OK) return s;
        const bool qkv_split = pend_splits > 0;   // QKV sums still in split partials
        rope_append_rows_kernel<<<n, 256, 0, st>>>(qkv_split ? reinterpret_cast<const float*>(ws + L.gpart) : y, N3,
                                                   qkv_split ? pend_splits : 1, pend_stride,
                                                   static_cast<const __half*>(lw.bqkv), rope, kv->pt, start,
                                                   c.n_q_heads, c.n_kv_heads, kc.num_pages, kc.max_pages,
                                                   kc.max_context, q, static_cast<__half*>(lp.k_pool),
                                                   static_cast<__half*>(lp.v_pool), err);
        pend_splits = 0;
        W4_CUDA(cudaGetLastError());

        PrefillAttnParams ap = {};   // causal: row t sees positions 0 .. start + t
        const PrefillAttnPlan apl = prefill_attention_plan(n, start);
        const size_t slots = (size_t)apl.qblocks * c.n_kv_heads * apl.max_splits * (c.n_q_heads / c.n_kv_heads) * 16;
        ap.q = q;
        ap.out = ao;
        ap.pt = kv->pt;
        const size_t tb = prefill_attention_ticket_bytes(n, c.n_kv_heads);
        ap.counters = reinterpret_cast<unsigned*>(ws + L.apart);
        ap.part_ml = reinterpret_cast<float*>(ws + L.apart + tb);
        ap.part_o = reinterpret_cast<float*>(ws + L.apart + tb + align256(slots * 2 * sizeof(float)));
        ap.ppc = apl.ppc;
        ap.max_splits = apl.max_splits;
        ap.n = n;
        ap.start = start;
        ap.Hq = c.n_q_heads;
        ap.Hkv = c.n_kv_heads;
        ap.group = c.n_q_heads / c.n_kv_heads;
        ap.max_pages = kc.max_pages;
        ap.num_pages = kc.num_pages;
        ap.scale_log2 = (float)(1.0 / std::sqrt((double)c.head_dim) * 1.4426950408889634);
        ap.errword = err;
        W4_CUDA(prefill_attention_launch(ap, kv->tmk[li], kv->tmv[li], st));

        // O + residual; gate/up with SiLU(gate) * up; down + residual
        s = fused(G_RESID, lp_.o, tm_att, wm[1], wm[1], lw.wo, nullptr, x, H, nullptr);
        if (s == W4_OK) s = rmsnorm(lw.ln2, hn);
        if (s == W4_OK) s = fused(G_SWIGLU, lp_.gu, tm_hn, wm[2], wm[3], lw.wgate, &lw.wup, nullptr, 0, act);
        if (s == W4_OK) s = fused(G_RESID, lp_.down, tm_act, wm[4], wm[4], lw.wdown, nullptr, x, H, nullptr);
        return s;
    }
};

}  // namespace

}  // namespace w4

extern "C" size_t w4_prefill_workspace_size(const w4_model* m, const w4_kv* kv, int max_tokens) {
    if (!m || !kv || max_tokens < 1) return 0;
    // The split-K partials grow with splits x n, and the split count drops when a
    // new token tile starts (tiles of 64, 128, then 256 tokens), so the need is not
    // monotonic in n: take the largest layout over the ends of every tile regime up
    // to max_tokens.
    size_t need = w4::prefill_layout(m->cfg, kv->kc, max_tokens).total;
    for (int n = 64; n < max_tokens; n = n < 256 ? 2 * n : n + 256)
        need = std::max(need, w4::prefill_layout(m->cfg, kv->kc, n).total);
    return need;
}

extern "C" w4_status w4_prefill(const w4_model* m, w4_kv* kv, void* prefill_workspace, size_t prefill_workspace_bytes,
                                const int32_t* tokens, int n_tokens, int start_pos, int32_t* token_out, float* logits,
                                void* stream) {
    using namespace w4;
    W4_REQUIRE(m && kv && prefill_workspace && tokens && token_out, W4_ERR_NULL, "prefill: null pointer");
    W4_REQUIRE(aligned16(prefill_workspace), W4_ERR_ALIGN, "prefill: workspace must be 16-byte aligned");
    w4_status s = check_pair(m, kv);
    if (s != W4_OK) return s;
    const w4_model_config& c = m->cfg;
    W4_REQUIRE(n_tokens >= 1, W4_ERR_SHAPE, "prefill: n_tokens must be >= 1");
    W4_REQUIRE(start_pos >= 0 && (long long)start_pos + n_tokens <= kv->kc.max_context, W4_ERR_RANGE,
               "prefill: positions [%d, %lld) outside the context capacity %d", start_pos,
               (long long)start_pos + n_tokens, kv->kc.max_context);
    const PrefillLayout L = prefill_layout(c, kv->kc, n_tokens);
    W4_REQUIRE(prefill_workspace_bytes >= L.total, W4_ERR_CAPACITY, "prefill: workspace of %zu bytes needed for %d tokens",
               L.total, n_tokens);

    cudaStream_t st = (cudaStream_t)stream;
    char* ws = static_cast<char*>(prefill_workspace);
    const int n = n_tokens;
    Prefill pf{m, kv, ws, L, layer_plans(c, n), {}, {}, {}, n, st, device_error_word()};
    {
        std::lock_guard<std::mutex> lock(m->pf_mu);
        if (m->pf_maps.empty()) {   // packed weights as 2-D tensors: boxes of 8 words x 128 rows (64 for gate, up)
            std::vector<CUtensorMap> maps((size_t)c.n_layers * 5);
            const int N3 = nqkv_of(c);
            for (int li = 0; li < c.n_layers; ++li) {
                const w4_layer_weights& l = m->layers[li];
                const struct {
                    const w4_qmatrix* q;
                    int rows, cols, box_rows;
                } mats[5] = {{&l.wqkv, N3, c.hidden, 128}, {&l.wo, c.hidden, c.hidden, 128},
                             {&l.wgate, c.ffn, c.hidden, 64}, {&l.wup, c.ffn, c.hidden, 64},
                             {&l.wdown, c.hidden, c.ffn, 128}};
                for (int j = 0; j < 5; ++j) {
                    s = make_weight_tensor_map(&maps[(size_t)li * 5 + j], mats[j].q->packed, mats[j].rows,
                                               mats[j].cols, 8, mats[j].box_rows);
                    if (s != W4_OK) return s;
                }
            }
            m->pf_maps.swap(maps);
        }
    }
    s = make_act_tensor_map(&pf.tm_hn, ws + L.hn, n, c.hidden, pf.lp_.qkv.a.bn);
    if (s == W4_OK) s = make_act_tensor_map(&pf.tm_att, ws + L.att_out, n, c.hidden, pf.lp_.o.a.bn);
    if (s == W4_OK) s = make_act_tensor_map(&pf.tm_act, ws + L.act, n, c.ffn, pf.lp_.down.a.bn);
    if (s != W4_OK) return s;
    // attention split tickets start at zero (the last CTA of a block resets its own)
    W4_CUDA(cudaMemsetAsync(ws + L.apart, 0, prefill_attention_ticket_bytes(n, c.n_kv_heads), st));
    embed_rows_kernel<<<n, 256, 0, st>>>(tokens, m->embed, c.vocab, c.hidden, reinterpret_cast<float*>(ws + L.x),
                                         pf.err);
    W4_CUDA(cudaGetLastError());
    const float2* rope = reinterpret_cast<const float2*>(kv->ws + kv->lay.rope);
    for (int li = 0; li < c.n_layers; ++li) {
        s = pf.layer(li, start_pos, rope);
        if (s != W4_OK) return s;
    }
    // the last row continues as the decode stream: LM head + argmax of the decode step
    prefill_tail_kernel<<<(c.hidden + 255) / 256, 256, 0, st>>>(
        reinterpret_cast<const float*>(ws + L.x) + (size_t)(n - 1) * c.hidden, c.hidden,
        reinterpret_cast<float*>(kv->ws + kv->lay.x), kv->pos, start_pos + n - 1,
        reinterpret_cast<const float*>(ws + L.gpart) + (size_t)(n - 1) * c.hidden, pf.pend_splits, pf.pend_stride);
    W4_CUDA(cudaGetLastError());
    return launch_one(m, kv, {tokens, token_out, logits, st}, W4_K_LM_HEAD, -1);
}
