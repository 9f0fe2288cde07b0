// The decode model handle shared by the decode step (decode.cu) and the
// prompt prefill (prefill.cu): weights, plans, tensor maps and the layout of
// the decode workspace.
#pragma once

#include <cmath>
#include <mutex>
#include <vector>

#include "attention.cuh"
#include "gemm_tc05.cuh"
#include "gemv_tma.cuh"

namespace w4 {

enum { CTR_QKV = 0, CTR_O, CTR_GU, CTR_DOWN, CTR_LM, CTR_COUNT };

struct ModelLayout {
    size_t x, qr, att, ctx, mlp, lmctr, attws, key, rope, total;
};

}  // namespace w4

// The weights of one model: shared, read-only, by every sequence (w4_kv).
struct w4_model {
    w4_model_config cfg;
    std::vector<w4_layer_weights> layers;
    const __half* embed;
    const __half* final_norm;
    w4_qmatrix lm;
    int device;
    bool pdl;
    w4::TmaPlan tp[w4::CTR_COUNT];   // qkv, o, gate/up, down, LM head
    // prefill: the packed-weight tensor maps of the fused GEMM (qkv, o, gate, up,
    // down per layer), built on first use
    mutable std::mutex pf_mu;
    mutable std::vector<CUtensorMap> pf_maps;
};

// One sequence's paged KV cache and decode state over a model's shape: the
// caller's pools (and their tensor maps), page table, device position and
// decode workspace (activations, attention split partials, RoPE table).
struct w4_kv {
    w4_model_config mcfg;            // the model shape this cache was laid out for
    w4_kv_config kc;
    std::vector<w4_kv_layer> pools;
    std::vector<CUtensorMap> tmk, tmv;
    const int32_t* pt;
    int32_t* pos;
    char* ws;
    size_t ws_bytes;
    w4::AttnPlan p_att;
    w4::ModelLayout lay;
    int device;
};

struct w4_graph {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
    int device;
};

namespace w4 {
// Launch kernel `which` (W4_K_*) of layer `li` of the decode step of sequence
// `kv`; the workspace layout is kv->lay.  Defined in decode.cu.
struct StepArgs {
    const int32_t* token_in;
    int32_t* token_out;
    float* logits;
    cudaStream_t st;
};
w4_status launch_one(const w4_model* m, const w4_kv* kv, const StepArgs& a, int which, int li);
// The model and cache agree on the shape, and the model's device is current.
w4_status check_pair(const w4_model* m, const w4_kv* kv);
}  // namespace w4
