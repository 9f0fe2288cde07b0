/*
 * w4a16.h -- C ABI of the GB300 (sm_103a) W4A16 single-token decode library.
 *
 * What it computes comes from the build-log "How to build your own LLM runtime
 * from scratch (Towards Data Science)" (wiki summary), section "What it
 * actually builds": INT4 weights, symmetric and group-wise with group size
 * 128; a paged KV cache of 16 tokens per 4 KiB page; fused GEMVs for the
 * Q/K/V/O projections and the MLP gate/up/down; CUDA-graph capture of the
 * token loop; greedy sampling only.  "How To Build Your Own LLM Runtime From
 * Scratch | daily.dev", section "Questions this post answers", adds that the
 * softmax must stay correct at partial KV tail pages and that activations
 * are fp16 against unpacked INT4 weights.
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers unless a comment says "host".  fp16 data is
 *     IEEE binary16 passed as void*; every buffer is owned by the caller and
 *     the library keeps no reference after a call returns (the model and graph
 *     handles below hold the caller's pointers until destroyed).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  All work is enqueued on it; no call synchronises unless
 *     stated.
 *   - Arguments are validated on the host before anything is launched; a
 *     failed check returns an error code and launches nothing.  Values that
 *     live on the device (page ids, positions, context lengths) are checked by
 *     the kernels: a bad value makes the kernel skip that access and record a
 *     code in the device error word (w4_device_error); outputs that depend on
 *     it are then unspecified.  No kernel traps.
 *   - w4_last_error() returns a message for the last failing call of the
 *     calling thread.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4_OK = 0,
    W4_ERR_NULL = 1,         /* a required pointer is NULL                        */
    W4_ERR_SHAPE = 2,        /* a size is out of range or inconsistent            */
    W4_ERR_ALIGN = 3,        /* a pointer is not 16-byte aligned                  */
    W4_ERR_RANGE = 4,        /* a host-visible value is out of range              */
    W4_ERR_CAPACITY = 5,     /* workspace or pool too small                       */
    W4_ERR_NONFINITE = 6,    /* pack saw a NaN/Inf weight or an fp16 scale overflow */
    W4_ERR_CUDA = 7,         /* a CUDA runtime call failed                        */
    W4_ERR_DEVICE_CHECK = 8, /* a kernel recorded a device-side check failure     */
    W4_ERR_STATE = 9,        /* handle misuse (e.g. wrong device)                 */
    W4_ERR_IO = 10           /* file I/O failed, or a container is malformed      */
} w4_status;

/* Device error word codes (bit flags, OR-ed by kernels). */
#define W4_DEVERR_PAGE_ID     0x1  /* page id outside [0, num_pages)              */
#define W4_DEVERR_POSITION    0x2  /* position/context outside the page table     */
#define W4_DEVERR_CONTEXT     0x4  /* context length < 1 or above the launch bound */
#define W4_DEVERR_TIMEOUT     0x8  /* a bounded wait on an mbarrier gave up        */
#define W4_DEVERR_NONFINITE   0x10 /* pack: non-finite weight                     */
#define W4_DEVERR_SCALE_OVF   0x20 /* pack: scale above fp16 range                */
#define W4_DEVERR_TOKEN       0x40 /* decode: input token outside [0, vocab)       */
#define W4_DEVERR_NAN_LOGIT   0x80 /* LM head: a logit is NaN (it never wins the argmax) */

const char* w4_last_error(void);

/* Read (and optionally clear) the device error word of the current device.
 * Synchronous (copies 4 bytes).  *flags (host) receives the OR of W4_DEVERR_*. */
w4_status w4_device_error(int32_t* flags, int clear);

/* Number of streaming multiprocessors of the current device (for planning). */
int w4_sm_count(void);

/* ------------------------------------------------------------------------
 * pack_int4_g128 -- symmetric group-wise INT4 quantisation and packing.
 * Source: TDS build-log summary, "What it actually builds" (INT4, symmetric,
 * group-wise, group size 128).  Per row n and 128-group j of W:
 *     s = fp16_rne(max|w| / 7)  (IEEE fp32 division)
 *     q = clamp(rint(w / float(s)), -8, 7)   (fp32 quotient, ties to even)
 *     s == 0  ->  q = 0
 * Layout written (the library's own format):
 *     packed uint32 [n][k/8] row-major; word j of row r holds k = 8j..8j+7;
 *     nibble u = q + 8; element e (0..7) of a word sits in bits
 *     [4*slot, 4*slot+4) with slot = 4*(e%2) + e/2;
 *     scales fp16 [n][k/128] row-major, in a buffer of at least
 *     round_up(n*(k/128)*2, 16) bytes (the GEMV copies scales in whole
 *     16-byte blocks, so the allocation is padded to a 16-byte multiple).
 * w: fp32 [n][k] row-major.  k % 128 == 0, n >= 1.  w, packed 16-B aligned.
 * flags: optional device int32; W4_DEVERR_NONFINITE / W4_DEVERR_SCALE_OVF are
 * OR-ed into it (and into the device error word) for bad groups, whose
 * codes and scale are written as 0.  Stream-ordered; no synchronisation.
 * ------------------------------------------------------------------------ */
w4_status w4_pack_int4_g128(const float* w, int64_t n, int64_t k,
                            uint32_t* packed, void* scales, int32_t* flags, void* stream);

/* ------------------------------------------------------------------------
 * gemv_w4a16 -- y[m][:] = W_deq x[m][:] (+ bias) (+ residual), batch m rows.
 * Source: TDS build-log summary, "What it actually builds" (fused GEMVs for
 * Q/K/V/O and gate/up/down over INT4 group-128 weights); daily.dev FAQ,
 * third question (fp16 activations against unpacked INT4 weights).
 *     y[i][r] = fp16( sum_k x[i][k] * q[r][k] * s[r][k/128]
 *                     + bias[r] + residual[i][r] )
 * Dequantisation is fused into the dot product; products and sums are fp32.
 * x: fp16 [m][k]; packed/scales as written by w4_pack_int4_g128 for an
 * [n][k] matrix (scales in a 16-byte padded, 16-byte aligned buffer); bias
 * fp16 [n] or NULL; residual fp16 [m][n] or NULL; y fp16 [m][n] (must not
 * alias x).  1 <= m <= 16, n >= 1, k % 128 == 0.  x, packed, y 16-B aligned.
 * At m = 1 the weights are streamed by one persistent CTA per SM through a
 * TMA (cp.async.bulk) shared-memory ring into an exact CUDA-core dot; at
 * 2 <= m <= 11, and at m = 1 for rows longer than that ring holds beside
 * the staged input (k > 21632), the products run on the tensor cores (mma.sync, fp32
 * accumulation, exact INT4 unpack) with the weights software-pipelined
 * through a per-warp cp.async ring; at 12 <= m <= 16 on the 5th-generation
 * tensor cores (tcgen05: TMA-fed, exact codes expanded into TMEM, one TMEM
 * accumulator per scale group, scaled in fp32).  w4_gemv_tune selects the
 * alternatives; the workspace size depends on the variant and the batch, so
 * call w4_gemv_workspace_size after w4_gemv_tune.
 * workspace: device scratch of at least
 * w4_gemv_workspace_size(m, n, k) bytes, zero-filled before its first use;
 * every call leaves it zero-filled again where that matters (its counters).
 * Calls sharing one workspace must not run concurrently.
 * ------------------------------------------------------------------------ */
size_t w4_gemv_workspace_size(int m, int64_t n, int64_t k);
w4_status w4_gemv_w4a16(const void* x, int m, int64_t n, int64_t k,
                        const uint32_t* packed, const void* scales,
                        const void* bias, const void* residual, void* y,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Measurement hook: the GEMV variant.  0 = default (at m = 1 the streaming
 * kernel's subnormal-nibble + mixed fp16/fp32 FMA dot, at m = 2..11 the
 * mma.sync kernel, at m = 12..16 the tcgen05 kernel); 1 = the mma.sync kernel
 * at every m; 2 = W4A8 at m = 1: the activations quantised to INT8 per
 * 128-group in the streaming kernel (s = max|x|/127, round half to even) and
 * multiplied with the codes by dp4a -- a different product, a re-check of the
 * pages' negative INT8-activation result, for measurement only; 3 = the
 * tcgen05 kernel at every m.  W4_ERR_RANGE for other values.  Process-wide;
 * not thread-safe. */
w4_status w4_gemv_tune(int variant);

/* gemv_plan -- how the batch-1 streaming kernel lays out one matrix
 * (matrices = 1) or a gate/up pair (2) of n rows by k columns: one CTA per SM
 * (grid = min(n, SMs); without a GPU, 148), cw consumer warps whose units
 * (half-warps, hpr = 1, or whole warps, hpr = 2) own row groups of rg rows,
 * a ring of ns stages of gs row groups.  grid = 0: the rows are too long for
 * the ring beside the staged input, and the tensor-core kernel takes them.
 * Host only.  out[9]: grid, cw, hpr, rg, gs, ns, weight bytes per stage per
 * matrix, scale bytes per stage per matrix, shared-memory bytes.
 * Errors: W4_ERR_NULL (out), W4_ERR_SHAPE (matrices outside 1..2, n < 1, k
 * not a positive multiple of 128, n or k above 2^31 - 1). */
w4_status w4_gemv_plan(int matrices, int64_t n, int64_t k, int32_t* out);

/* ------------------------------------------------------------------------
 * paged_kv_append -- write one new token's K and V rows into the paged cache.
 * Source: TDS build-log summary, "What it actually builds" (paged KV cache,
 * 16 tokens per 4 KiB page); "Build Crude Implementations for Learning",
 * "Paged KV cache" (blocks reached through a table).
 *   pool layout fp16 [num_pages][hkv][16][d]; entry b writes
 *   k[b][h][:] to k_pool[page_table[b*max_pages + p/16]][h][p%16][:], p =
 *   positions[b], and likewise v.  k, v: fp16 [b][hkv][d].
 * d == 128.  page_table int32 [b][max_pages], positions int32 [b] (device).
 * Device checks: p in [0, 16*max_pages), page id in [0, num_pages).
 * ------------------------------------------------------------------------ */
w4_status w4_paged_kv_append(const void* k, const void* v, int b, int hkv, int d,
                             void* k_pool, void* v_pool, int num_pages,
                             const int32_t* page_table, int max_pages,
                             const int32_t* positions, void* stream);

/* ------------------------------------------------------------------------
 * paged_decode_attention -- GQA decode attention over the paged cache.
 * Source: TDS build-log summary, "What it actually builds" (attention over
 * the paged cache) and "Two more honest findings" (softmax corrupted at page
 * boundaries by a misplaced block barrier); daily.dev FAQ, second question
 * (partial KV tail pages).
 *   out[b][h] = sum_{t < L_b} softmax_t(scale * q[b][h] . K_t) V_t
 *   with K_t = k_pool[page_table[b][t/16]][g][t%16], g = h / (hq/hkv).
 * Online softmax over pages; the last page holds L - 16*(pages-1) valid
 * tokens and slots past L are never used (they may hold anything, NaN too).
 * q, out: fp16 [b][hq][d].  d == 128, hq % hkv == 0, hq/hkv <= 16.
 * context_lens int32 [b] (device), each in [1, max_context] and
 * <= 16*max_pages; max_context is the host-side bound the grid is sized for.
 * workspace: >= w4_attention_workspace_size(b, hq, hkv, max_context) bytes,
 * zero-filled before first use and left zero-filled where that matters.
 * k_pool, v_pool 16-B aligned; num_pages*hkv*16 < 2^31.
 * ------------------------------------------------------------------------ */
size_t w4_attention_workspace_size(int b, int hq, int hkv, int max_context);
w4_status w4_paged_decode_attention(const void* q, int b, int hq, int hkv, int d, float scale,
                                    const void* k_pool, const void* v_pool, int num_pages,
                                    const int32_t* page_table, int max_pages,
                                    const int32_t* context_lens, int max_context,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    void* stream);

/* attention_plan -- how w4_paged_decode_attention divides a batch of b
 * sequences over hkv KV heads, for caches of max_context tokens, on a GPU of
 * `sms` SMs co-scheduling clusters of up to `max_cluster` CTAs (8 or 16; 0 for
 * either: ask the device).  Host only when both are given.  A (sequence, KV
 * head) takes `splits` CTAs of four warps, each warp `ppw` pages of 16 tokens
 * (the pages of max_context in order); with cluster = 1 the splits form one
 * thread-block cluster and merge in distributed shared memory, otherwise the
 * last CTA merges them through the workspace.
 * out[8]: cluster, ppw, stages (pages in flight per warp), splits, grid x, y,
 * z, workspace bytes.
 * Errors: W4_ERR_NULL (out), W4_ERR_SHAPE (b, hq, hkv or max_context < 1, hq
 * not a multiple of hkv, sms < 0, max_cluster not 0, 8 or 16). */
w4_status w4_attention_plan(int b, int hq, int hkv, int max_context, int sms, int max_cluster, int64_t* out);

/* ------------------------------------------------------------------------
 * paged_decode_attention_noalloc -- the same attention for callers that
 * cannot allocate device memory where they run it: a process that reserved
 * its whole device-memory budget up front and may not grow it, an
 * allocator-less host or plugin, a caller that only holds borrowed pointers.
 * The pages have no counterpart to this entry point: it exists for this
 * library's callers.
 * Arguments and results are those of w4_paged_decode_attention without the
 * workspace.  The split-merge scratch is a fixed array inside the library
 * (w4_paged_decode_attention_noalloc_max_scratch() bytes, 8 MiB, held on
 * every GPU that loads the library until exit); a batch/context needing more
 * returns W4_ERR_CAPACITY before anything is launched.  Nothing is
 * allocated: the first call on a device looks up the array's device address
 * and keeps it for the life of the process, so the entry point must not be
 * used across a cudaDeviceReset.  Each call clears the array's split tickets on `stream`
 * before launching.  All calls share the one array, so calls that overlap on
 * the GPU race: serialise them.
 * ------------------------------------------------------------------------ */
size_t w4_paged_decode_attention_noalloc_max_scratch(void);
w4_status w4_paged_decode_attention_noalloc(const void* q, int b, int hq, int hkv, int d, float scale,
                                            const void* k_pool, const void* v_pool, int num_pages,
                                            const int32_t* page_table, int max_pages,
                                            const int32_t* context_lens, int max_context,
                                            void* out, void* stream);

/* ------------------------------------------------------------------------
 * decode_step -- one greedy token of a Qwen2-style decoder with INT4 weights.
 * Source: TDS build-log summary, opening paragraph (decode-only engine,
 * greedy sampling) and "The one lesson that generalizes" (capture the step
 * as one CUDA graph: 280+ launches per token otherwise).
 * Per layer: RMSNorm -> fused QKV GEMV + bias -> RoPE + paged KV append ->
 * paged attention -> O GEMV + residual -> RMSNorm -> gate/up GEMV with
 * SiLU(gate)*up -> down GEMV + residual; then final RMSNorm, INT4 LM head,
 * argmax (lowest index on ties; -0 ties with +0; a NaN logit never wins and
 * sets W4_DEVERR_NAN_LOGIT).  The residual stream is fp32.
 * Row order of wqkv: q (hidden rows), k (kv rows), v (kv rows); inside every
 * q and k head of 128 rows, row 2i holds head dimension i and row 2i+1 holds
 * dimension i+64 (the rotate-half RoPE pairs), likewise for bqkv; v rows and
 * all other matrices are in natural order.
 * ------------------------------------------------------------------------ */
typedef struct {
    int hidden;        /* 3584 for the 7B shape; multiple of 128             */
    int ffn;           /* 18944; multiple of 128                             */
    int n_layers;      /* 28                                                 */
    int n_q_heads;     /* 28                                                 */
    int n_kv_heads;    /* 4                                                  */
    int head_dim;      /* must be 128                                        */
    int vocab;         /* 152064                                             */
    float rms_eps;     /* 1e-6                                               */
    float rope_theta;  /* 1e6                                                */
} w4_model_config;

typedef struct {
    const uint32_t* packed;   /* [rows][cols/8], 16-byte aligned             */
    const void* scales;       /* fp16 [rows][cols/128], 16-byte aligned, buffer
                                 padded to a 16-byte multiple                */
} w4_qmatrix;

typedef struct {
    const void* ln1;          /* fp16 [hidden]                               */
    const void* ln2;          /* fp16 [hidden]                               */
    w4_qmatrix wqkv;          /* rows: q (hidden) | k (kv) | v (kv); cols hidden */
    const void* bqkv;         /* fp16 [hidden + 2*kv]                        */
    w4_qmatrix wo;            /* [hidden][hidden]                            */
    w4_qmatrix wgate;         /* [ffn][hidden]                               */
    w4_qmatrix wup;           /* [ffn][hidden]                               */
    w4_qmatrix wdown;         /* [hidden][ffn]                               */
} w4_layer_weights;

typedef struct w4_model w4_model;

/* Create a model handle: the weights only, shared read-only by every sequence
 * (w4_kv) run over them, on any number of streams.  `layers` (host array of
 * n_layers entries) and the struct are copied; the device buffers they point
 * to stay caller-owned and must outlive the handle.  embed fp16
 * [vocab][hidden]; final_norm fp16 [hidden]. */
w4_status w4_model_create(const w4_model_config* cfg, const w4_layer_weights* layers, const void* embed,
                          const void* final_norm, w4_qmatrix lm_head, w4_model** out);
void w4_model_destroy(w4_model* m);
/* Launch the step's kernels with programmatic dependent launch (default on):
 * each kernel may start its prologue while the previous one drains, and waits
 * (griddepcontrol.wait) before reading what that kernel produced. */
w4_status w4_model_set_pdl(w4_model* m, int enable);

/* ------------------------------------------------------------------------
 * kv -- one sequence's paged KV cache and decode state.
 * Source: TDS build-log summary, "What it actually builds" (a paged KV cache
 * of 16-token, 4 KiB pages as its own component of the engine); "Build Crude
 * Implementations for Learning", "Paged KV cache" (a sequence's blocks found
 * through a table).
 * The handle wraps caller-owned device memory: per layer a K and a V pool
 * fp16 [num_pages][n_kv_heads][16][128] (16-byte aligned), the page table
 * int32 [max_pages] (shared by all layers: position p of the sequence lives in
 * page page_table[p / 16], slot p % 16), the position pos (int32 [1]: the
 * position of the next token, i.e. the number of tokens already cached;
 * advanced by every decode step and prompt pass), and a workspace of
 * w4_kv_workspace_size(m, kc) bytes (activations, attention split partials,
 * the RoPE table) that the handle owns until destroyed.  Several caches may
 * share one model; each decodes independently (one stream at a time per
 * cache).  w4_kv_create zero-fills the workspace and writes its RoPE table on
 * `stream`.  max_context <= 16 * max_pages; num_pages * n_kv_heads * 16 < 2^31.
 * Errors: W4_ERR_NULL, _ALIGN, _RANGE (cache sizes), _SHAPE, _CAPACITY
 * (workspace too small), _CUDA.
 * ------------------------------------------------------------------------ */
typedef struct {
    int max_context;   /* capacity in tokens; <= 16 * max_pages              */
    int num_pages;     /* pages in each layer's pool                         */
    int max_pages;     /* entries of the page table                          */
} w4_kv_config;

typedef struct {
    void* k_pool;      /* fp16 [num_pages][n_kv_heads][16][128]              */
    void* v_pool;
} w4_kv_layer;

typedef struct w4_kv w4_kv;

size_t w4_kv_workspace_size(const w4_model* m, const w4_kv_config* kc);
w4_status w4_kv_create(const w4_model* m, const w4_kv_config* kc, const w4_kv_layer* layers,
                       const int32_t* page_table, int32_t* pos, void* workspace, size_t workspace_bytes,
                       void* stream, w4_kv** out);
void w4_kv_destroy(w4_kv* kv);

/* ------------------------------------------------------------------------
 * decode_step -- one greedy token of a Qwen2-style decoder with INT4 weights.
 * Source: TDS build-log summary, opening paragraph (decode-only engine,
 * greedy sampling) and "The one lesson that generalizes" (capture the step
 * as one CUDA graph: 280+ launches per token otherwise).
 * Per layer: RMSNorm -> fused QKV GEMV + bias -> RoPE + paged KV append ->
 * paged attention -> O GEMV + residual -> RMSNorm -> gate/up GEMV with
 * SiLU(gate)*up -> down GEMV + residual; then final RMSNorm, INT4 LM head,
 * argmax (lowest index on ties; -0 ties with +0; a NaN logit never wins and
 * sets W4_DEVERR_NAN_LOGIT).  The residual stream is fp32.
 * Row order of wqkv: q (hidden rows), k (kv rows), v (kv rows); inside every
 * q and k head of 128 rows, row 2i holds head dimension i and row 2i+1 holds
 * dimension i+64 (the rotate-half RoPE pairs), likewise for bqkv; v rows and
 * all other matrices are in natural order.
 * The step reads *token_in (device int32 [1]), writes K/V at position *pos of
 * kv, then the greedy token to *token_out (may alias token_in) and the logits
 * (device fp32 [vocab], or NULL), and increments *pos -- all on the device,
 * so a captured graph replays unchanged token after token.  Eager: 5 launches
 * per layer + 2.  Errors: W4_ERR_NULL, _SHAPE (kv laid out for another model
 * shape), _STATE (wrong device), _CUDA.
 * ------------------------------------------------------------------------ */
w4_status w4_decode_step(const w4_model* m, w4_kv* kv, const int32_t* token_in, int32_t* token_out,
                         float* logits, void* stream);

/* Capture one decode step of (m, kv) into a CUDA graph (same kernels, one
 * launch); stream must not be the legacy default stream. */
typedef struct w4_graph w4_graph;
w4_status w4_decode_graph_create(const w4_model* m, w4_kv* kv, const int32_t* token_in, int32_t* token_out,
                                 float* logits, void* stream, w4_graph** out);
w4_status w4_decode_graph_launch(w4_graph* g, void* stream);
void w4_decode_graph_destroy(w4_graph* g);
/* Kernel launches one decode step makes (for reporting). */
int w4_decode_launches_per_step(const w4_model* m);

/* Profiling hook: launch only kernel `kernel` (W4_K_*) of layer `layer`
 * exactly as w4_decode_step would (same grid, same buffers), so one kernel
 * can be timed in isolation.  `layer` is ignored for the embedding and LM
 * head kernels.  The cache's workspace must hold the state the kernel expects. */
enum {
    W4_K_EMBED = 0, W4_K_QKV = 1 /* + RoPE + paged KV append */, W4_K_ATTENTION = 2,
    W4_K_O = 3, W4_K_GATE_UP = 4, W4_K_DOWN = 5, W4_K_LM_HEAD = 6
};
w4_status w4_decode_launch_kernel(const w4_model* m, w4_kv* kv, int kernel, int layer, const int32_t* token_in,
                                  int32_t* token_out, float* logits, void* stream);

/* ------------------------------------------------------------------------
 * gemm_w4a16 -- y[t][r] = sum_k x[t][k] * q[r][k] * s[r][k/128] for n rows of
 * activations at once (the prompt pass's matrix products).
 * Source: TDS build-log summary, "What it actually builds" (INT4 group-128
 * weights against fp16 activations, fp32 accumulation); with many activation
 * rows the product is a dense GEMM rather than a GEMV.
 * Runs on the 5th-generation tensor cores: TMA stages the activation tile
 * (128-byte swizzle) and the packed weight tile, eight warps expand the INT4
 * codes to fp16 (exact: q in [-8, 7]) in the MMA's shared-memory layout, one
 * thread issues tcgen05.mma (M = 128 weight rows, N = 64, 128 or 256 rows of
 * x, K = 16) into one TMEM accumulator per 128-column scale group (two, used
 * in turn), and the same eight warps add each group's sums times its fp16
 * scale into fp32 running sums.  Every product is exact and only fp32 sums
 * round, as in w4_gemv_w4a16.  K is split across CTAs (in whole scale groups)
 * when the tiles alone leave SMs idle, or, for long K, shared out stream-K
 * (one CTA per SM, each an equal run of (tile, scale group) units, a tile's
 * pieces in consecutive CTAs); a second kernel adds the partial sums in a
 * fixed order (deterministic).
 * x: fp16 [n][K], 16-byte aligned.  packed/scales: as w4_gemv_w4a16 (scales
 * need only 2-byte alignment here).  y: fp32 [n][N].  N and K positive
 * multiples of 128, n >= 1.  workspace: device, 16-byte aligned, at least
 * w4_gemm_workspace_size(n, N, K) bytes (the partial sums of the split-K or
 * stream-K pieces; 0 when K is not divided).
 * Errors: W4_ERR_NULL, _SHAPE, _ALIGN, _CAPACITY, _CUDA.
 * ------------------------------------------------------------------------ */
size_t w4_gemm_workspace_size(int n, int N, int K);
w4_status w4_gemm_w4a16(const void* x, int n, int N, int K, const uint32_t* packed, const void* scales,
                        float* y, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * gemm_plan -- how the GEMM above, and each projection of the prompt pass,
 * divides its work among CTAs on a GPU of `sms` SMs.  Host only: no device
 * call, so it answers for any SM count.
 * The work is 128-row (SwiGLU: 64 gate + 64 up rows) by bn-token tiles, each
 * of K/128 scale groups.  Mode 0, split K: CTA c = split * tiles + tile takes
 * kb_per_split / 2 groups of one tile (splits == 1: the whole tile).  Mode 1,
 * stream-K: CTA c takes the (tile, group) units [c U / ctas, (c + 1) U /
 * ctas) of all U, a tile's pieces in consecutive CTAs, piece q in slot q.
 * Mode 2, persistent: CTA c takes the whole tiles [c T / ctas, (c + 1) T /
 * ctas).  Partial sums, when splits > 1, fill [splits][n][N (SwiGLU: 2N)].
 * epilogue: 0 store, 1 residual add, 2 SwiGLU (N = rows of gate and of up).
 * out[8]: bn, token tiles, row tiles, K-blocks (64 columns) per split,
 * splits (partial slots), mode, CTAs, stages of the operand ring.
 * Errors: W4_ERR_NULL (out), W4_ERR_SHAPE (epilogue outside 0..2, n < 1,
 * sms < 1, N or K not positive multiples of 128).
 * ------------------------------------------------------------------------ */
w4_status w4_gemm_plan(int epilogue, int n, int N, int K, int sms, int32_t* out);

/* ------------------------------------------------------------------------
 * prefill -- run a prompt through the model in one pass (time to first token).
 * Source: TDS build-log summary, "What the numbers say" (time to first token
 * of the engine against llama.cpp).  The pages give no prefill design; this
 * is the decode step's block applied to n prompt rows at once, with causal
 * attention: prompt row t sits at position start_pos + t and attends to
 * positions 0 .. start_pos + t of the paged cache (rows 0 .. start_pos - 1
 * must already be there).  Every projection is a W4A16 GEMM over the n
 * rows (w4_gemm_w4a16's kernel: exact INT4 codes on the tensor cores, each
 * scale group's sum scaled in fp32); RMSNorm, bias + RoPE + paged KV append
 * and the embedding are this library's kernels; attention is a causal paged
 * kernel (16 prompt rows of one query head per warp on mma.sync, the GQA
 * group's K/V pages staged once per CTA by TMA); the last row goes through
 * the decode step's fused final RMSNorm + LM head + argmax.
 *
 * kv: the sequence's cache -- its RoPE table is read from the cache's
 * workspace, the last row's residual is left there, and its position advances.
 * prefill_workspace: device, 16-byte aligned, at least
 * w4_prefill_workspace_size(m, kv, n_tokens) bytes (a buffer sized for n
 * serves every prompt of at most n tokens); caller-owned scratch, no state
 * kept.  tokens: device int32 [n_tokens].  On return (stream order) K/V rows
 * start_pos .. start_pos + n_tokens - 1 of every layer are in the pools,
 * *token_out holds the greedy next token, the cache's position is
 * start_pos + n_tokens and logits (device fp32 [vocab], or NULL) the last
 * row's logits -- exactly the state w4_decode_step continues from.  Errors:
 * W4_ERR_NULL, _ALIGN, _SHAPE (n_tokens < 1, or kv laid out for another model
 * shape), _RANGE (positions past max_context), _CAPACITY (workspace too
 * small), _STATE (wrong device), _CUDA (a CUDA call failed); bad tokens or
 * page ids set W4_DEVERR_TOKEN / _PAGE_ID in the error word.
 * ------------------------------------------------------------------------ */
size_t w4_prefill_workspace_size(const w4_model* m, const w4_kv* kv, int max_tokens);
w4_status w4_prefill(const w4_model* m, w4_kv* kv, void* prefill_workspace, size_t prefill_workspace_bytes,
                     const int32_t* tokens, int n_tokens, int start_pos, int32_t* token_out, float* logits,
                     void* stream);

/* ------------------------------------------------------------------------
 * Model container -- this library's own on-disk format for a packed model.
 * Source: "How to build your own LLM runtime from scratch (Towards Data
 * Science)", "What it actually builds": the engine keeps its packed INT4
 * weights in its own binary file, opened by memory mapping and recognised by
 * a magic-byte header.  The pages give no layout, so this one is the
 * library's.
 *
 * File (little-endian):
 *   [0, 4096)          header: magic "W4A16MC\0", u32 version = 1,
 *                      u32 n_tensors, u64 file_bytes, the model config
 *                      (i32 hidden, ffn, n_layers, n_q_heads, n_kv_heads,
 *                      head_dim, vocab; f32 rms_eps, rope_theta), u32 CRC-32
 *                      of the header bytes before it;
 *   [4096, data0)      directory: n_tensors entries of 112 bytes: name[64]
 *                      (NUL-terminated), u32 dtype (W4_DT_*), u32 ndim (1 or
 *                      2), u64 dims[2], u64 offset, u64 bytes, u32 CRC-32 of
 *                      the blob, u32 zero;
 *   blobs              each at a 4096-byte aligned offset, row-major, tightly
 *                      packed (scales are NOT padded in the file).
 * CRC-32 is the IEEE 802.3 polynomial (reflected 0xEDB88320, init and final
 * xor 0xFFFFFFFF).  A container holds whatever tensors the writer passes; the
 * Python side stores a decoder's packed weights under the names "embed",
 * "final_norm", "lm_head.packed", "lm_head.scales" and "layers.<i>.<field>".
 * ------------------------------------------------------------------------ */
enum { W4_DT_U32 = 1, W4_DT_F16 = 2, W4_DT_F32 = 3, W4_DT_I32 = 4 };

typedef struct {
    const char* name;     /* at most 63 bytes */
    int dtype;            /* W4_DT_* */
    int ndim;             /* 1 or 2 */
    int64_t dims[2];      /* dims[1] ignored when ndim == 1 */
    const void* data;     /* host memory (write); the read-only mapping (read) */
    size_t bytes;         /* must equal prod(dims) * element size */
} w4_tensor_desc;

typedef struct w4_container w4_container;

/* Write a container from host buffers (blocking; the file is created or
 * truncated).  cfg is stored in the header.  W4_ERR_SHAPE for bad
 * descriptors or duplicate names, W4_ERR_IO when the file cannot be
 * written. */
w4_status w4_container_write(const char* path, const w4_model_config* cfg, const w4_tensor_desc* tensors,
                             int n_tensors);
/* Map a container read-only and validate its header and directory (bounds,
 * alignment, sizes, header CRC); verify != 0 also checks every blob's CRC.
 * W4_ERR_IO for any mismatch.  The handle owns the mapping and two pinned
 * staging buffers; close it with w4_container_close. */
w4_status w4_container_open(const char* path, int verify, w4_container** out);
void w4_container_close(w4_container* c);
/* The stored model config. */
w4_status w4_container_config(const w4_container* c, w4_model_config* cfg);
int w4_container_count(const w4_container* c);
/* Descriptor of tensor `index`, or of the tensor called `name`
 * (W4_ERR_RANGE if absent); data points into the mapping, valid until close. */
w4_status w4_container_tensor(const w4_container* c, int index, w4_tensor_desc* out);
w4_status w4_container_find(const w4_container* c, const char* name, int* index);
/* Copy tensor `index` into device memory dst (dst_bytes >= its bytes),
 * staged through pinned buffers in 8 MiB chunks with cudaMemcpyAsync on
 * `stream`.  Returns once every chunk is queued; the copy is complete when
 * the stream reaches that point.  Not thread-safe per handle. */
w4_status w4_container_upload(w4_container* c, int index, void* dst, size_t dst_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* W4A16_H */
