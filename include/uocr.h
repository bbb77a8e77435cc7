/*
 * uocr.h — C ABI of the GB300 quantized MoE decode step.
 *
 * One decode step of a DeepSeek-V2-style OCR text decoder whose weights are
 * block-quantized (Q8_0, Q4_0, per-group int8-asymmetric) and dequantized
 * inside the matmul kernels, with fp16 activations, a KV cache made of a fixed
 * prefix followed by a ring of generated tokens, optional attention sinks,
 * batched rows that share one weight read, and a greedy argmax over the LM
 * head.
 *
 * Sources (page title, section):
 *  - "Unlimited-OCR on Apple Silicon with C and Metal":
 *      "Il decoder e il Mixture of Experts" (layer stack, 64 routed experts,
 *      top-6, 2 shared, grouping tokens by expert, KV append, 128-token ring,
 *      argmax over the language head);
 *      "Quantizzazione: Q8 prima, Q4 dove conviene" (Q8_0 / Q4_0 profiles,
 *      fused dequantisation, attention kept Q8, norms and activations fp16);
 *      "Memoria: il vincolo principale" (per-category working set checked
 *      against a budget before running, refused with a detailed error);
 *      "Dall'ABI C all'API Python" (a deliberately small C ABI, one lock per
 *      engine, one instance per execution lane).
 *  - "Falcon-OCR INT8 OpenVINO IR" model card: intro (the sink as one more
 *      key with value zero; the KV cache is an input written in place, never
 *      rebuilt); "How it is meant to be run" (dynamic batch: rows share one
 *      weight read; lengths are explicit, never inferred from shapes).
 *
 * Each declaration below names the passage that defines what it computes or
 * enforces ("Source:").  Page titles are abbreviated as
 *   [Metal]  "Unlimited-OCR on Apple Silicon with C and Metal"
 *   [Falcon] "Falcon-OCR INT8 OpenVINO IR" model card
 *
 * Conventions
 *  - Every call returns a uocr_status; uocr_last_error() gives the text of
 *    the last failure on that context.  Calls on one context are serialised
 *    by a per-context mutex; use one context per execution lane.
 *  - The library owns all device memory it allocates (one arena sized at
 *    uocr_create).  Pointers documented as "device" must point to device
 *    memory of the context's GPU; "host" pointers are ordinary memory.
 *  - Device work is enqueued on an internal stream ordered after the caller's
 *    stream (uocr_config.stream, 0 = legacy default stream) and the caller's
 *    stream is made to wait for it, so the calls are asynchronous with respect
 *    to the host unless stated otherwise.
 *  - Kernels never trap.  Invalid device-side inputs (a token id outside
 *    [0, vocab), a negative position) set bits of a device status word that
 *    uocr_sync() reports as UOCR_E_TOKEN / UOCR_E_POSITION; the offending
 *    row uses id 0 / position 0 for that step.
 */
#ifndef UOCR_H
#define UOCR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define UOCR_API __attribute__((visibility("default")))
#else
#define UOCR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  UOCR_OK = 0,
  UOCR_E_INVALID_ARG = 1, /* a NULL pointer, a size or a config value out of range */
  UOCR_E_OOM = 2,         /* device allocation failed */
  UOCR_E_BUDGET = 3,      /* the working set exceeds uocr_config.mem_budget */
  UOCR_E_FORMAT = 4,      /* weight tensor with wrong kind/format/shape/byte size */
  UOCR_E_STATE = 5,       /* call not valid in the context's current state */
  UOCR_E_CUDA = 6,        /* a CUDA runtime error (text in uocr_last_error) */
  UOCR_E_POSITION = 7,    /* a device-side position was invalid */
  UOCR_E_TOKEN = 8,       /* a device-side token id was outside [0, vocab) */
  UOCR_E_TIMEOUT = 9      /* a kernel's bounded wait for its asynchronous copies ran out;
                             the kernel returned without the data, the context stays usable */
} uocr_status;

/* Canonical weight formats.  Source: [Metal] "Quantizzazione: Q8 prima, Q4
 * dove conviene" (Q8_0 / Q4_0 block formats dequantised inside the kernels);
 * [Falcon] "How it is meant to be run" (INT8_ASYM weights, u8 codes); the block
 * size 32 and the value formulas are the decode-step statement's definitions.
 * Blocks hold 32 consecutive values of one row;
 * blocks run along the row (K), rows follow each other.  fp16 little endian.
 *   UOCR_F16     plain fp16 [rows][cols]
 *   UOCR_Q8_0    {fp16 d; int8 q[32]}           34 B   value = d*q
 *   UOCR_Q4_0    {fp16 d; uint8 qs[16]}         18 B   value = d*(q-8), q of
 *                element j<16 = low nibble of qs[j], j>=16 = high nibble of qs[j-16]
 *   UOCR_I8ASYM  {fp16 s; fp16 z; uint8 q[32]}  36 B   value = s*(q-z)      */
typedef enum {
  UOCR_F16 = 0,
  UOCR_Q8_0 = 1,
  UOCR_Q4_0 = 2,
  UOCR_I8ASYM = 3,
  UOCR_Q8_0_G64 = 4, /* {fp16 d; int8 q[64]}   66 B   value = d*q                      */
  UOCR_Q4_0_G64 = 5  /* {fp16 d; uint8 qs[32]} 34 B   value = d*(q-8), q of element
                        j<32 = low nibble of qs[j], j>=32 = high nibble of qs[j-32]
                        ([Metal] "Quantizzazione": groups of 64 values)          */
} uocr_format;

/* Weight tensor kinds.  Source: [Metal] "Il decoder e il Mixture of Experts"
 * (attention, one dense MLP layer, MoE layers with a router, 64 routed and 2
 * shared SwiGLU experts, embedding and language head).  Shapes use H = hidden, S = n_heads*head_dim,
 * I = dense_inter, Ie = expert_inter, E = n_experts, V = vocab.
 * Matrices are [out_features][in_features] (y = W x).                       */
typedef enum {
  UOCR_T_EMBED = 0,         /* [V][H]   F16 only                     layer 0 */
  UOCR_T_FINAL_NORM = 1,    /* [1][H]   F16                          layer 0 */
  UOCR_T_LM_HEAD = 2,       /* [V][H]   F16 only                     layer 0 */
  UOCR_T_ATTN_NORM = 3,     /* [1][H]   F16                                  */
  UOCR_T_WQ = 4,            /* [S][H]   fmt_attn                             */
  UOCR_T_WK = 5,            /* [S][H]   fmt_attn                             */
  UOCR_T_WV = 6,            /* [S][H]   fmt_attn                             */
  UOCR_T_WO = 7,            /* [H][S]   fmt_attn                             */
  UOCR_T_MLP_NORM = 8,      /* [1][H]   F16                                  */
  UOCR_T_GATE = 9,          /* [I][H]   fmt_dense      dense layers only     */
  UOCR_T_UP = 10,           /* [I][H]   fmt_dense                            */
  UOCR_T_DOWN = 11,         /* [H][I]   fmt_dense                            */
  UOCR_T_ROUTER = 12,       /* [E][H]   F16 only       MoE layers only       */
  UOCR_T_SHARED_GATE = 13,  /* [Ie][H]  fmt_shared     expert = shared index */
  UOCR_T_SHARED_UP = 14,    /* [Ie][H]  fmt_shared                           */
  UOCR_T_SHARED_DOWN = 15,  /* [H][Ie]  fmt_shared                           */
  UOCR_T_EXPERT_GATE = 16,  /* [Ie][H]  fmt_routed     expert = routed index */
  UOCR_T_EXPERT_UP = 17,    /* [Ie][H]  fmt_routed                           */
  UOCR_T_EXPERT_DOWN = 18,  /* [H][Ie]  fmt_routed                           */
  UOCR_T_PROJ = 19,         /* [H][proj_in]  fmt_proj   projector (proj_in > 0) layer 0 */
  UOCR_T_PROJ_BIAS = 20     /* [1][H]   F16             projector bias          layer 0 */
} uocr_tensor_kind;

/* Source: [Metal] "Il decoder e il Mixture of Experts" (model constants, the
 * 128-token ring for generated tokens); [Falcon] intro (the sink, the cache
 * as an input); "Dall'ABI C all'API Python" (one engine per execution lane). */
typedef struct {
  /* model */
  int32_t hidden;          /* H, multiple of 64                                  */
  int32_t n_heads;
  int32_t head_dim;        /* D, multiple of 16, <= 256                          */
  int32_t n_layers;
  int32_t n_dense_layers;  /* layers [0, n_dense_layers) use the dense MLP       */
  int32_t dense_inter;     /* multiple of 64 (0 if no dense layer)               */
  int32_t n_experts;       /* routed experts E (0 = every layer dense), <= 256   */
  int32_t top_k;           /* 1..8                                               */
  int32_t n_shared;        /* shared experts (weight 1 each), 0..4               */
  int32_t expert_inter;    /* multiple of 64                                     */
  int32_t vocab;           /* 0 = no embedding / LM head                         */
  int32_t fmt_attn, fmt_dense, fmt_shared, fmt_routed; /* uocr_format           */
  /* cache */
  int32_t prefix_len;      /* P: slots [0, P) hold positions [0, P)              */
  int32_t ring_len;        /* R: positions p >= P live in slot P + (p-P) mod R   */
  int32_t max_rows;        /* rows of one step, 1..64                            */
  int32_t use_sink;        /* 1: per-layer, per-head sink logit (uocr_set_sinks) */
  float rms_eps;           /* RMSNorm epsilon                                    */
  float rope_theta;        /* rotary base                                        */
  /* runtime */
  uint64_t mem_budget;     /* bytes; 0 = no limit                                */
  void* stream;            /* cudaStream_t the calls are ordered with (0 = legacy) */
  int32_t device;          /* CUDA device ordinal                                */
  int32_t use_graphs;      /* 1: capture each step shape in a CUDA graph         */
  /* cache format (after the runtime fields so that older callers' layout holds)  */
  int32_t kv_int8;         /* 1: INT8 KV cache, one fp32 scale per (row, K|V,
                              head, slot): value = scale * code, the key / value
                              vector of a head quantised when written
                              (s = max|x| / 127, code = round(x / s)) -- [Falcon]
                              "How it is meant to be run" (an INT8 KV cache)   */
  /* projector of visual features into the hidden space ([Metal] "Il modello":
     2048 -> 1280; "Quantizzazione": the Q8 profile covers the projector)       */
  int32_t proj_in;         /* input width, multiple of 64 (0 = no projector)     */
  int32_t fmt_proj;        /* uocr_format of UOCR_T_PROJ                         */
  /* dynamic int8 activations ([Falcon] "How it is meant to be run": the linear
     layers' inputs quantised dynamically in groups of 32).  1: the inputs of
     the dense projections (Q/K/V, O, dense gate/up and down) are quantised
     per group of 32 (s = max|x| / 127, code = round(x / s), fp32 decisions)
     and multiplied on the int8 tensor cores; fmt_attn and fmt_dense must then
     be quantised formats and hidden, n_heads*head_dim and dense_inter at most
     8192 (else uocr_create returns UOCR_E_INVALID_ARG).  Router, experts, LM
     head and projector unchanged.  0 or 1. */
  int32_t act_int8;
} uocr_config;

typedef struct {
  int32_t kind;     /* uocr_tensor_kind                                   */
  int32_t layer;    /* 0..n_layers-1 (0 for global tensors)               */
  int32_t expert;   /* routed or shared expert index, else 0              */
  int32_t format;   /* uocr_format                                        */
  int32_t rows;     /* out features                                       */
  int32_t cols;     /* in features                                        */
  const void* data; /* host pointer to the canonical bytes                */
  uint64_t bytes;   /* byte size of data                                  */
} uocr_tensor;

/* Bytes per category.  Source: [Metal] "Memoria: il vincolo principale"
 * (every buffer belongs to a category; the working set is estimated per
 * category before running). */
typedef struct {
  uint64_t weights;      /* packed weights, norms, router, embedding, LM head  */
  uint64_t kv_cache;     /* [layer][row][K|V][head][P+R][D] fp16               */
  uint64_t activations;  /* residual stream, q, attention partials, MLP/expert scratch */
  uint64_t routing;      /* router logits, top-k, counts, offsets, permutation */
  uint64_t logits;       /* [max_rows][vocab] fp32 readback buffer             */
  uint64_t total;        /* the arena allocated at uocr_create                 */
} uocr_mem_report;

typedef struct uocr_ctx uocr_ctx;

/* Source: [Metal] "Memoria: il vincolo principale" (estimate, compare with the
 * budget, refuse with a detailed error) and "Dall'ABI C all'API Python" (engine
 * open).
 * Validate cfg, size the arena per category, compare it with cfg->mem_budget
 * (UOCR_E_BUDGET with a per-category message when it does not fit), allocate
 * it, zero the KV cache.  Launches no compute kernel.  *out receives the
 * context (NULL on failure).  cfg is copied.                                 */
UOCR_API uocr_status uocr_create(const uocr_config* cfg, uocr_ctx** out);

/* Source: [Metal] "Dall'ABI C all'API Python" (engine close).
 * Release everything; NULL-safe; the context must not be used afterwards.   */
UOCR_API void uocr_destroy(uocr_ctx* ctx);

/* Source: [Metal] "Quantizzazione" (no fp16 copy of the weights: the packed
 * quantised blocks are what the kernels read).
 * Copy and pack weight tensors (host pointers, caller keeps ownership and may
 * free them on return).  Tensors may come in any order and over several
 * calls; a group (Q/K/V of a layer, gate/up of an MLP or expert, the shared
 * experts of a layer) is packed once all its members have arrived.  Wrong
 * kind, index, format, shape or byte size -> UOCR_E_FORMAT (nothing of that
 * tensor is kept).  Synchronous.                                             */
UOCR_API uocr_status uocr_load_weights(uocr_ctx* ctx, const uocr_tensor* t, size_t n);

/* Source: [Falcon] intro (the KV cache is an input the caller owns; lengths
 * are explicit).
 * Write n cached prefix positions [start, start+n) of one row and layer.
 * k, v: host fp16 [n_heads][n][head_dim].  Requires start+n <= prefix_len.
 * Synchronous.                                                               */
UOCR_API uocr_status uocr_kv_write_prefix(uocr_ctx* ctx, int32_t row, int32_t layer,
                                 const uint16_t* k, const uint16_t* v,
                                 int32_t start, int32_t n);

/* Source: [Falcon] intro (the cache is caller-visible state).
 * Read back cache slots [slot0, slot0+n) of one row and layer into host fp16
 * [n_heads][n][head_dim] buffers.  Synchronous.                               */
UOCR_API uocr_status uocr_kv_read(uocr_ctx* ctx, int32_t row, int32_t layer, int32_t slot0,
                         int32_t n, uint16_t* k, uint16_t* v);

/* Write cache slots [slot0, slot0+n) of one row and layer (prefix or ring)
 * from host fp16 [n_heads][n][head_dim] buffers: the cache is caller-visible
 * state the step reads and writes in place (Falcon-OCR INT8 OpenVINO IR model
 * card, intro).  Requires slot0+n <= prefix_len+ring_len.  Synchronous.       */
UOCR_API uocr_status uocr_kv_write(uocr_ctx* ctx, int32_t row, int32_t layer, int32_t slot0,
                          int32_t n, const uint16_t* k, const uint16_t* v);

/* Source: [Falcon] "How it is meant to be run" (an INT8 KV cache).
 * The INT8 cache's entries of slots [slot0, slot0+n) of one row and layer,
 * exactly: codes host int8 [n_heads][n][head_dim] and scales host fp32
 * [n_heads][n] for keys and for values (value = scale * code).  Read copies
 * them out; write copies them in as they are (no quantisation).  Synchronous.
 * UOCR_E_STATE when the context's cache is fp16 (kv_int8 = 0).  With an INT8
 * cache, uocr_kv_write_prefix / uocr_kv_write quantise the given fp16 vectors
 * (one scale per head vector) and uocr_kv_read returns scale * code rounded to
 * fp16.                                                                      */
UOCR_API uocr_status uocr_kv_read_i8(uocr_ctx* ctx, int32_t row, int32_t layer, int32_t slot0, int32_t n,
                                     int8_t* k_codes, float* k_scales, int8_t* v_codes, float* v_scales);
UOCR_API uocr_status uocr_kv_write_i8(uocr_ctx* ctx, int32_t row, int32_t layer, int32_t slot0, int32_t n,
                                      const int8_t* k_codes, const float* k_scales, const int8_t* v_codes,
                                      const float* v_scales);

/* Source: [Falcon] intro (the sink is one more key whose logit is the sink and
 * whose value is zero; equivalent to rescaling by sigmoid(lse - sink)).
 * Per-layer, per-head sink logits, host fp32 [n_layers][n_heads]; they enter
 * the softmax unscaled as one more key with value zero.  Synchronous.        */
UOCR_API uocr_status uocr_set_sinks(uocr_ctx* ctx, const float* sinks);

/* Source: [Metal] "Il decoder e il Mixture of Experts" (the decode loop:
 * append to the KV cache, generated tokens in a 128-token ring, argmax over the
 * language head; route, group tokens by expert, recompose) and
 * "Quantizzazione" (dequantisation inside GEMV/SwiGLU/combine/argmax, fp16
 * activations); [Falcon] "How it is meant to be run" (the rows of a step share
 * one read of the weights).
 * One decode step for rows 0..rows-1 (row i uses KV row i).
 *   token_ids  device int32 [rows]  (embedding lookup; requires vocab > 0)
 *   positions  device int32 [rows]  absolute positions; slot(p) is written
 *              with the new key/value, then attention reads every slot whose
 *              position q has q <= p and (q < P or q > p - R)
 *   next_ids   device int32 [rows]  greedy argmax (lowest index on ties)
 *   logits     device fp32 [rows][vocab] or NULL
 * Asynchronous (see conventions).                                            */
UOCR_API uocr_status uocr_decode_step(uocr_ctx* ctx, int32_t rows, const int32_t* token_ids,
                             const int32_t* positions, int32_t* next_ids, float* logits);

/* Source: as uocr_decode_step; [Metal] "Il modello: una pipeline
 * vision-language completa" (visual tokens enter the decoder as embeddings).
 * The same step fed with hidden vectors instead of token ids.
 *   x         device fp16 [rows][hidden]
 *   y         device fp32 [rows][hidden] or NULL: residual stream after the
 *             last layer (before the final norm)
 *   y_f16     device fp16 [rows][hidden] or NULL: the same, rounded to fp16
 *             (the activation precision of [Metal] "Quantizzazione")
 *   next_ids  device int32 [rows] or NULL (requires vocab > 0 when given)
 *   logits    device fp32 [rows][vocab] or NULL                              */
UOCR_API uocr_status uocr_decode_step_embeds(uocr_ctx* ctx, int32_t rows, const uint16_t* x,
                                    const int32_t* positions, float* y, uint16_t* y_f16,
                                    int32_t* next_ids, float* logits);

/* Source: [Metal] "Il modello: una pipeline vision-language completa" (the
 * encoders' features pass through a projector from 2048 to 1280 dimensions,
 * then take the image placeholder's span of the prompt) and "Quantizzazione"
 * (the projector is quantised in the Q8 profile, biases stay fp16).
 * out = fp16(W_proj feats + b_proj) for n feature vectors: one launch of the
 * fused dequant GEMM (every weight read serves 16 features per token group,
 * on the tensor cores).  Needs proj_in > 0 and UOCR_T_PROJ / UOCR_T_PROJ_BIAS
 * loaded (the decoder's weights are not needed).
 *   feats  device fp16 [n][proj_in]
 *   out    device fp16 [n][hidden] (e.g. the x of uocr_prefill)
 * Asynchronous (see conventions); not captured in a graph.                  */
UOCR_API uocr_status uocr_project(uocr_ctx* ctx, int32_t n, const uint16_t* feats, uint16_t* out);

/* Source: [Metal] intro and "Il modello" (prefill of the prompt, with the
 * visual tokens in the placeholder span, before token-by-token decoding);
 * [Falcon] file table (a separate prompt pass over the whole prompt).
 * Prefill of one row: n consecutive positions [start_pos, start_pos + n) of
 * cache row `row`, all layers, in chunks of up to 64 tokens.  Each chunk runs
 * the decode-step kernels once over its tokens (every weight read serves all
 * of them, on the tensor cores), writes their keys and values, and attends
 * causally (position p sees the slots of positions <= p).  The result is the
 * one n decode steps of this row would give.
 *   token_ids  device int32 [n] or NULL   exactly one of token_ids, x
 *   x          device fp16 [n][hidden] or NULL
 *   next_id    device int32 [1] or NULL: greedy argmax after the last token
 *   logits     device fp32 [vocab] or NULL: logits of the last token
 * Requires 0 <= start_pos and start_pos + n <= prefix_len + ring_len (no ring
 * wrap inside one call).  Invalid ids / positions are reported by uocr_sync as
 * for a step.  Asynchronous (see conventions); not captured in a graph.      */
UOCR_API uocr_status uocr_prefill(uocr_ctx* ctx, int32_t row, const int32_t* token_ids, const uint16_t* x,
                                  int32_t n, int32_t start_pos, int32_t* next_id, float* logits);

/* Source: as uocr_decode_step; [Metal] "Dall'ABI C all'API Python" (token
 * results returned to the host).
 * uocr_decode_step with HOST buffers: copies token_ids/positions to the
 * device, runs the step, copies next_ids back, and returns when they are on
 * the host.                                                                  */
UOCR_API uocr_status uocr_decode_step_host(uocr_ctx* ctx, int32_t rows, const int32_t* token_ids,
                                  const int32_t* positions, int32_t* next_ids);

/* Source: as uocr_decode_step ([Metal]: the decode loop generates token by
 * token, greedy argmax).
 * n_steps greedy steps chained on the device: step s uses positions+s and
 * the ids produced by step s-1 (token_ids for s = 0).  out_ids: device int32
 * [n_steps][rows].  Asynchronous.                                            */
UOCR_API uocr_status uocr_generate(uocr_ctx* ctx, int32_t rows, const int32_t* token_ids,
                          const int32_t* positions, int32_t n_steps, int32_t* out_ids);

/* Source: [Metal] "Il decoder e il Mixture of Experts" (the ring bounds the
 * memory of generated tokens).
 * Zero the ring slots (and the prefix when keep_prefix == 0) of one row
 * (row = -1: all rows).  Attention never reads a slot not written for the
 * current sequence, so this is hygiene, not a correctness requirement.      */
UOCR_API uocr_status uocr_kv_reset(uocr_ctx* ctx, int32_t row, int32_t keep_prefix);

/* Source: [Metal] "Dall'ABI C all'API Python" (errors reported through the
 * ABI, never by aborting).
 * Wait for the context's work; report a device-side status raised since the
 * last uocr_sync (UOCR_E_TIMEOUT, UOCR_E_TOKEN, UOCR_E_POSITION, in that order
 * of precedence) and clear it.                                               */
UOCR_API uocr_status uocr_sync(uocr_ctx* ctx);

/* Source: [Metal] "Memoria" (refusals carry a detailed message).
 * Text of the last failure on ctx ("" if none); valid until the next call.
 * uocr_last_error(NULL) gives the text of the last failed uocr_create on the
 * calling thread.                                                            */
UOCR_API const char* uocr_last_error(uocr_ctx* ctx);

/* Source: [Metal] "Dall'ABI C all'API Python" (memory report) and "Memoria".
 * The bytes of each category of the context's arena (host output).         */
UOCR_API uocr_status uocr_memory_report(uocr_ctx* ctx, uocr_mem_report* out);

/* Source: as uocr_decode_step (the intermediate values it defines: residual
 * after attention and after each layer; the router's choice, weights and
 * grouping of [Metal] "Il decoder e il Mixture of Experts").
 * Debug taps of the last completed step or prefill chunk (synchronous, host
 * outputs; rows up to 64, the tokens of the last pass).
 *   uocr_debug_hidden: fp32 [rows][hidden] residual stream at tap `layer`:
 *     2*l   = after attention of layer l, 2*l+1 = output of layer l,
 *     -1    = input of layer 0.
 *   uocr_debug_router: MoE layer l: idx int32 [rows][k], w fp32 [rows][k],
 *     count int32 [E], offset int32 [E+1], perm int32 [rows*k]; any output
 *     may be NULL.                                                           */
UOCR_API uocr_status uocr_debug_hidden(uocr_ctx* ctx, int32_t tap, int32_t rows, float* out);
UOCR_API uocr_status uocr_debug_router(uocr_ctx* ctx, int32_t layer, int32_t rows, int32_t* idx,
                              float* w, int32_t* count, int32_t* offset, int32_t* perm);
/* Source: as uocr_debug_router.
 * The fp32 router logits [rows][E] of MoE layer `layer` from the last step
 * (the values the top-k was taken on).  Host output buffer; E_INVALID_ARG for
 * a dense layer or bad rows. */
UOCR_API uocr_status uocr_debug_router_logits(uocr_ctx* ctx, int32_t layer, int32_t rows, float* logits);

/* Source: [Metal] "Dall'ABI C all'API Python" (profiling through the ABI).
 * Per-kernel-class device time (ms per step).  One whole step runs first with
 * the given rows, input kind and inputs; then, for each kernel class, that
 * class's launches of one step (every layer, with the step's real arguments
 * and programmatic dependent launch between them) are captured alone in a
 * CUDA graph and replayed 5 times, timed with CUDA events on the library
 * stream.  names[i] points into static storage.  n_inout: in = capacity, out
 * = number of classes.  The step mutates the KV cache like a real step (the
 * replays rewrite the current slot with the same values).                  */
UOCR_API uocr_status uocr_profile(uocr_ctx* ctx, int32_t rows, int32_t input_kind,
                         const int32_t* token_ids, const uint16_t* x, const int32_t* positions,
                         const char** names, float* ms, int32_t* n_inout);

/* Final RMSNorm + LM head + greedy argmax on final hidden states the caller
 * provides, without allocating any memory.  (The pages have no counterpart:
 * this entry point exists for callers, not for the method.)
 *
 * Who needs it: code that may not call cudaMalloc/cudaFree while it runs,
 * e.g. a serving loop whose device memory is owned by a fixed pool (cudaMalloc
 * synchronises the device and stalls every other stream), or a host framework
 * that hands the library only the buffers it already owns.  The regular steps
 * keep their scratch in the context arena; this call instead keeps the
 * kernel's scratch (one argmax key per row, a CTA counter and, for more than
 * 16 rows, the rows staged for the tensor-core kernel: 1 KB + 256 KB in all)
 * in a static device array of the library, which every GPU that loads the
 * library holds until the process exits.  It runs the same kernel as the
 * decode step at the same row count, so its logits and ids equal the step's.
 *   hidden    device fp32 [rows][hidden]: residual stream after the last layer
 *   next_ids  device int32 [rows]: argmax id per row (lowest index on ties)
 *   logits    device fp32 [rows][vocab] or NULL
 *   stream    cudaStream_t the work is enqueued on (0 = legacy default stream)
 * rows must be in [1, 64] and, above 16 rows, hidden <= 2048 (the scratch
 * capacity), else UOCR_E_INVALID_ARG and nothing is launched.  Uses the context's loaded LM head and final norm.
 * The first call on a device looks up the scratch address on that device
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * All calls share the one scratch array and each call clears it first, so
 * calls whose work overlaps on the GPU (on different streams, or from
 * different contexts on the same device) race and must be serialised by the
 * caller.  The launch goes to the context's device (cfg.device), whatever
 * device the calling thread has current; the thread's current device is left
 * as it was.  The kernel raises no device-side status of its own (the ids
 * and positions it would check belong to the step that produced `hidden`).
 * Asynchronous with respect to the host.                                    */
UOCR_API uocr_status uocr_lm_head_argmax_noalloc(uocr_ctx* ctx, int32_t rows, const float* hidden,
                                                 int32_t* next_ids, float* logits, void* stream);

/* Source: [Falcon] intro and [Metal] "Dall'ABI C all'API Python" (failures are
 * reported, never fatal); the kernels' TMA waits poll an mbarrier with an
 * iteration limit and report UOCR_E_TIMEOUT through uocr_sync.
 * Runs that bounded wait alone, with a short limit, on a 16-byte bulk copy
 * that is issued (issue_copy = 1: the wait succeeds and no status is raised)
 * or never issued (issue_copy = 0: the wait runs out, and the next uocr_sync
 * returns UOCR_E_TIMEOUT).  Asynchronous; no copy is left in flight.        */
UOCR_API uocr_status uocr_debug_wait_probe(uocr_ctx* ctx, int32_t issue_copy);

#ifdef __cplusplus
}
#endif
#endif /* UOCR_H */
