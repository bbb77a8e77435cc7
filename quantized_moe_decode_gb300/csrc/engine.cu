// Host side of the library: configuration checks, the per-category memory
// plan and its single device arena, weight loading and packing, the launch
// sequence of one decode step (captured once per step shape into a CUDA
// graph), and the C ABI declared in include/uocr.h.
//
// Memory categories and the budget check follow "Unlimited-OCR on Apple
// Silicon with C and Metal", "Memoria: il vincolo principale" (every buffer
// belongs to a category; the working set is estimated per category and
// compared with the configured budget before running; a request that does
// not fit is refused with a detailed error).  The per-context lock follows
// "Dall'ABI C all'API Python" (one lock per engine, one instance per lane).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <cstdlib>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "launch.h"
#include "uocr.h"

using namespace uocr;

namespace {

struct DMat {
  uint8_t* q = nullptr;
  uint8_t* s = nullptr;
  int fmt = 0, cfmt = 0, n_slabs = 0, U = 0, K = 0;  // packed and canonical format
  size_t qbytes = 0, sbytes = 0;  // of one matrix (one expert for expert arrays)
  PMat view(int n_experts_stride = 0) const {
    PMat p;
    p.q = q;
    p.s = s;
    p.n_slabs = n_slabs;
    p.U = U;
    p.K = K;
    p.q_stride = n_experts_stride ? (long long)qbytes : 0;
    p.s_stride = n_experts_stride ? (long long)sbytes : 0;
    return p;
  }
};

size_t packed_q_bytes(int n_rows_packed, int K, int fmt) {
  const size_t slabs = (size_t)(n_rows_packed + 15) / 16;
  return slabs * (K / unit_k(fmt)) * unit_bytes(fmt);
}
size_t packed_s_bytes(int n_rows_packed, int K, int fmt) {
  const size_t slabs = (size_t)(n_rows_packed + 15) / 16;
  return slabs * (K / unit_k(fmt)) * unit_scale_bytes(fmt);
}
// Canonical block formats: values per block and bytes per block.  The group-64
// variants pack into the layout of their 32-value format (a Q8_0 unit of 32
// inputs is half a block and takes the block's scale; a Q4_0 unit of 64
// inputs is one block), so every kernel runs on the packed format kf(fmt).
int fmt_group(int fmt) { return fmt == UOCR_Q8_0_G64 || fmt == UOCR_Q4_0_G64 ? 64 : 32; }
int fmt_block_bytes(int fmt) {
  switch (fmt) {
    case UOCR_Q8_0: return 34;
    case UOCR_Q4_0: return 18;
    case UOCR_I8ASYM: return 36;
    case UOCR_Q8_0_G64: return 66;
    case UOCR_Q4_0_G64: return 34;
  }
  return 0;
}
int kf(int fmt) { return fmt == UOCR_Q8_0_G64 ? Q8_0 : fmt == UOCR_Q4_0_G64 ? Q4_0 : fmt; }
size_t blob_bytes(int fmt, int rows, int cols) {
  if (fmt == F16) return (size_t)rows * cols * 2;
  return (size_t)rows * (cols / fmt_group(fmt)) * fmt_block_bytes(fmt);
}

struct LayerW {
  DMat qkv, o, gateup, down, router, sh_gateup, sh_down, ex_gateup, ex_down;
  __half* attn_norm = nullptr;
  __half* mlp_norm = nullptr;
  float* sink = nullptr;
  bool dense = true;
};

// bump allocator over the arena, with a measuring pass
struct Carver {
  char* base = nullptr;
  size_t off = 0;
  template <class T>
  T* take(size_t count, uint64_t& cat) {
    const size_t bytes = ((count * sizeof(T)) + 255) / 256 * 256;
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += bytes;
    cat += bytes;
    return p;
  }
};

constexpr int kMaxSplits = 8;  // attention splits of a (row, head): one portable thread-block cluster
// Tokens one pass of the kernels can carry (four token groups of 16): the rows
// of a decode step (max_rows <= 64) or one chunk of a prefill.  Activation and
// routing buffers are sized for it; the KV cache is sized by max_rows.
constexpr int kTokCap = 64;
thread_local std::string g_create_err;  // text of the last failed uocr_create on this thread
constexpr int kHistCap = 1024;

enum Group : int { G_SINGLE = 0, G_QKV, G_DENSE_GU, G_SHARED_GU, G_SHARED_DOWN, G_EXPERT_GU };

struct Pending {
  std::vector<void*> dev;  // staged canonical blobs (device), by member index
  int have = 0;
};

}  // namespace

struct uocr_ctx {
  uocr_config cfg{};
  std::mutex mu;
  std::string err;
  int n_sm = 148;
  cudaStream_t st = nullptr;
  cudaStream_t ust = nullptr;
  cudaEvent_t ev_in = nullptr, ev_out = nullptr;
  char* arena = nullptr;
  uocr_mem_report rep{};
  std::vector<LayerW> L;
  __half* emb = nullptr;
  __half* final_norm = nullptr;
  DMat lm;
  uint8_t* lm_tc = nullptr;  // LM head in the tensor-core operand layout (max_rows > 16)
  uint8_t* lm_xc = nullptr;  // the rows staged for it [H/64][64 x 64] fp16
  int lm_mtiles = 0;
  DMat proj;                 // projector [H][proj_in]
  __half* proj_b = nullptr;  // its bias [H]
  double* inv_freq = nullptr;
  float2* rope = nullptr;  // [max_rows][head_dim/2] (cos, sin) of the step's positions
  __half* kv = nullptr;        // fp16 cache [L][MR][2][nh][SL][D]
  int8_t* kv8 = nullptr;       // INT8 cache codes, same shape
  float* kvs = nullptr;        // INT8 cache scales [L][MR][2][nh][SLp]
  float* kv_new = nullptr;     // INT8 cache: the pass's new keys / values in fp32 [kTokCap][2][nh][D]
  size_t kv_layer = 0;         // entries (codes or fp16 values) per layer
  size_t kvs_layer = 0;        // scales per layer
  int SLp = 0;                 // scale slots per (row, K|V, head): SL rounded up to 16
  int S = 0, SL = 0;
  float* hid = nullptr;  // [2L+1][kTokCap][H]
  __half* x_in = nullptr;
  float* q = nullptr;
  __half* attn_out = nullptr;
  __half* act_dense = nullptr;
  __half* xhat = nullptr;
  uint8_t* act8 = nullptr;   // int8 activations: staging blocks of the 16-row token groups (written once per projection)
  uint8_t* act_r = nullptr;  // B-fragment order, padded expert entries x Ie
  uint8_t* act_s = nullptr;  // B-fragment order, rows x n_shared*Ie
  float* part_r = nullptr;
  float* part_s = nullptr;
  float* r_logits = nullptr;
  int *r_idx = nullptr, *r_count = nullptr, *r_offset = nullptr, *r_perm = nullptr, *r_inv = nullptr;
  int4* r_rec = nullptr;  // [L][token groups][E] routing records

  float* r_w = nullptr;
  float* sinks = nullptr;
  float* logits = nullptr;
  unsigned long long* keys = nullptr;
  int *lm_counter = nullptr, *next_ids = nullptr, *ids_buf = nullptr, *pos_buf = nullptr;
  int *hist = nullptr, *hist_ctr = nullptr, *status = nullptr;
  // loading
  std::map<std::vector<int>, bool> loaded;  // (kind, layer, expert) -> present
  bool complete = false;  // every tensor the config needs has been loaded (set once checked; loads only add)
  std::map<std::vector<int>, Pending> pending;
  bool sinks_set = false;
  // graphs
  std::map<uint64_t, cudaGraphExec_t> graphs;
  bool pdl = true;  // programmatic dependent launch between the step's kernels
  int gemv_ctas_per_sm = 2;    // streaming CTAs per SM of a GEMV launch
  int expert_ctas_per_sm = 2;  // CTAs per SM an expert launch is sized for (active experts only)
  int attn_min_splits = 1;     // lower bound of the attention splits per (row, head)
  int attn_slots = 0;          // attention CTAs resident on the whole GPU at once
  // tensor-core expert kernels for steps of more than 16 rows (one CTA per SM)
  bool tc_experts = false;
  TcxPlan tcx_gu{}, tcx_dn{};

  int H() const { return cfg.hidden; }
  int MR() const { return cfg.max_rows; }
  int TC() const { return kTokCap; }
  bool layer_dense(int l) const { return l < cfg.n_dense_layers || cfg.n_experts == 0; }
  bool any_moe() const {
    for (int l = 0; l < cfg.n_layers; ++l)
      if (!layer_dense(l)) return true;
    return false;
  }
  int shared_fmt() const { return kf(cfg.n_shared > 0 ? cfg.fmt_shared : cfg.fmt_routed); }

  uocr_status fail(uocr_status s, const char* fmt, ...) {
    char buf[1024];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    err = buf;
    return s;
  }
  uocr_status cuda(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return UOCR_OK;
    return fail(UOCR_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
  }
};

#define CK(expr, what)                                        \
  do {                                                        \
    uocr_status _s = ctx->cuda((expr), what);                 \
    if (_s != UOCR_OK) return _s;                             \
  } while (0)

// ------------------------------------------------------------------ config
static bool fmt_ok(int f) { return f >= UOCR_F16 && f <= UOCR_Q4_0_G64; }
static bool quant_fmt(int f) { return f != UOCR_F16 && fmt_ok(f); }
static bool expert_pair_ok(int fr, int fs) {
  fr = kf(fr);
  fs = kf(fs);
  return (fr == Q8_0 && fs == Q8_0) || (fr == Q4_0 && fs == Q8_0) || (fr == Q4_0 && fs == Q4_0) ||
         (fr == Q8_0 && fs == Q4_0) || (fr == I8ASYM && fs == I8ASYM);
}

// dynamic shared memory a streaming kernel may plan (the device offers 227 KB
// per block; the kernels' static shared memory is below 13 KB)
constexpr int kSmemLimit = 214 * 1024;

static uocr_status check_config(uocr_ctx* ctx, const uocr_config& c) {
  auto bad = [&](const char* m) { return ctx->fail(UOCR_E_INVALID_ARG, "invalid config: %s", m); };
  if (c.hidden <= 0 || c.hidden % 64) return bad("hidden must be a positive multiple of 64");
  if (c.n_heads <= 0) return bad("n_heads must be positive");
  if (!(c.head_dim == 16 || c.head_dim == 32 || c.head_dim == 64 || c.head_dim == 128 || c.head_dim == 256))
    return bad("head_dim must be 16, 32, 64, 128 or 256");
  if ((c.n_heads * c.head_dim) % 64) return bad("n_heads*head_dim must be a multiple of 64");
  if (c.n_layers <= 0 || c.n_dense_layers < 0 || c.n_dense_layers > c.n_layers) return bad("layer counts");
  if (c.n_experts < 0 || c.n_experts > 256) return bad("n_experts must be in [0, 256]");
  const bool has_dense = c.n_dense_layers > 0 || c.n_experts == 0;
  const bool has_moe = c.n_experts > 0 && c.n_layers > c.n_dense_layers;
  if (has_dense && (c.dense_inter <= 0 || c.dense_inter % 64)) return bad("dense_inter must be a positive multiple of 64");
  if (!fmt_ok(c.fmt_attn) || !fmt_ok(c.fmt_dense) || !fmt_ok(c.fmt_shared) || !fmt_ok(c.fmt_routed))
    return bad("unknown weight format");
  if (has_moe) {
    if (c.top_k < 1 || c.top_k > 8 || c.top_k > c.n_experts) return bad("top_k must be in [1, min(8, n_experts)]");
    if (c.expert_inter <= 0 || c.expert_inter % 64) return bad("expert_inter must be a positive multiple of 64");
    if (c.n_shared < 0 || c.n_shared > 4) return bad("n_shared must be in [0, 4]");
    const int fs = c.n_shared > 0 ? c.fmt_shared : c.fmt_routed;
    if (!quant_fmt(c.fmt_routed) || !expert_pair_ok(c.fmt_routed, fs))
      return bad("unsupported (routed, shared) expert format pair");
    if (plan_stream(2, kf(c.fmt_routed), c.hidden, 16).bytes > kSmemLimit)
      return bad("hidden too large for the expert kernels");
    const int kmax = c.n_shared * c.expert_inter > c.expert_inter ? c.n_shared * c.expert_inter : c.expert_inter;
    if (plan_stream(2, kf(c.fmt_routed), 0, 0, 2 * (kmax / 32) * 512).bytes > kSmemLimit)
      return bad("expert_inter * n_shared too large for the expert kernels");
  }
  if (c.vocab < 0) return bad("vocab must be >= 0");
  {
    const int kmax = c.hidden > c.dense_inter ? (c.hidden > c.n_heads * c.head_dim ? c.hidden : c.n_heads * c.head_dim)
                                              : c.dense_inter;
    if (plan_stream(2, F16, kmax, 16, 16 * (c.head_dim / 2) * 8).bytes > kSmemLimit)
      return bad("a projection input is too long for the shared-memory activation tile");
  }
  if (c.prefix_len < 0 || c.ring_len < 1) return bad("prefix_len >= 0 and ring_len >= 1 required");
  if ((long long)c.prefix_len + c.ring_len > (1 << 24)) return bad("cache too long");
  if (c.max_rows < 1 || c.max_rows > 64) return bad("max_rows must be in [1, 64]");
  if (c.use_sink != 0 && c.use_sink != 1) return bad("use_sink must be 0 or 1");
  if (!(c.rms_eps >= 0.f) || !(c.rope_theta > 0.f)) return bad("rms_eps >= 0 and rope_theta > 0 required");
  if (c.kv_int8 != 0 && c.kv_int8 != 1) return bad("kv_int8 must be 0 or 1");
  if (c.act_int8 != 0 && c.act_int8 != 1) return bad("act_int8 must be 0 or 1");
  if (c.act_int8 && (!quant_fmt(c.fmt_attn) || (has_dense && !quant_fmt(c.fmt_dense))))
    return bad("act_int8 needs quantised fmt_attn and fmt_dense (int8 codes against int8 activations)");
  if (c.act_int8 && (c.hidden > kActMaxChunks * kActChunk || c.n_heads * c.head_dim > kActMaxChunks * kActChunk ||
                     (has_dense && c.dense_inter > kActMaxChunks * kActChunk)))
    return bad("act_int8: projection inputs are limited to 8192");
  if (c.proj_in < 0 || c.proj_in % 64) return bad("proj_in must be 0 or a positive multiple of 64");
  if (c.proj_in > 0) {
    if (!quant_fmt(c.fmt_proj)) return bad("fmt_proj must be a quantised format");
    if (plan_stream(2, kf(c.fmt_proj), c.proj_in).bytes > kSmemLimit) return bad("proj_in too large");
  }
  return UOCR_OK;
}

// ------------------------------------------------------------------ memory plan
static void carve(uocr_ctx* ctx, Carver& cv) {
  const uocr_config& c = ctx->cfg;
  uocr_mem_report& r = ctx->rep;
  r = uocr_mem_report{};
  const int H = c.hidden, S = c.n_heads * c.head_dim, MR = c.max_rows, Lc = c.n_layers, V = c.vocab;
  const int E = c.n_experts, k = c.top_k, Ie = c.expert_inter, Ish = c.n_shared * c.expert_inter;
  const int TC = kTokCap;  // tokens of one pass (decode rows or a prefill chunk)
  auto mat = [&](DMat& m, int rows_packed, int K, int cfmt, int count = 1) {
    const int fmt = kf(cfmt);
    m.cfmt = cfmt;
    m.fmt = fmt;
    m.K = K;
    m.U = K / unit_k(fmt);
    m.n_slabs = (rows_packed + 15) / 16;
    m.qbytes = packed_q_bytes(rows_packed, K, fmt);
    m.sbytes = packed_s_bytes(rows_packed, K, fmt);
    m.q = cv.take<uint8_t>(m.qbytes * count, r.weights);
    m.s = m.sbytes ? cv.take<uint8_t>(m.sbytes * count, r.weights) : nullptr;
  };
  ctx->L.assign(Lc, LayerW{});
  for (int l = 0; l < Lc; ++l) {
    LayerW& w = ctx->L[l];
    w.dense = ctx->layer_dense(l);
    mat(w.qkv, 3 * S, H, c.fmt_attn);
    mat(w.o, H, S, c.fmt_attn);
    w.attn_norm = cv.take<__half>(H, r.weights);
    w.mlp_norm = cv.take<__half>(H, r.weights);
    if (w.dense) {
      mat(w.gateup, 2 * c.dense_inter, H, c.fmt_dense);
      mat(w.down, H, c.dense_inter, c.fmt_dense);
    } else {
      mat(w.router, E, H, F16);
      if (c.n_shared > 0) {
        mat(w.sh_gateup, 2 * Ish, H, c.fmt_shared);
        mat(w.sh_down, H, Ish, c.fmt_shared);
      }
      mat(w.ex_gateup, 2 * Ie, H, c.fmt_routed, E);
      mat(w.ex_down, H, Ie, c.fmt_routed, E);
    }
  }
  if (V > 0) {
    ctx->emb = cv.take<__half>((size_t)V * H, r.weights);
    ctx->final_norm = cv.take<__half>(H, r.weights);
    mat(ctx->lm, V, H, F16);
    if (MR > 16) {  // steps of more than 16 rows run the LM head on the tensor cores (tcgen05)
      ctx->lm_mtiles = (V + 127) / 128;
      ctx->lm_tc = cv.take<uint8_t>((size_t)ctx->lm_mtiles * (H / 64) * 16384, r.weights);
      ctx->lm_xc = cv.take<uint8_t>((size_t)(H / 64) * 64 * 64 * 2, r.activations);
    }
  }
  if (c.proj_in > 0) {
    mat(ctx->proj, H, c.proj_in, c.fmt_proj);
    ctx->proj_b = cv.take<__half>(H, r.weights);
  }
  ctx->inv_freq = cv.take<double>(c.head_dim / 2, r.weights);
  ctx->rope = cv.take<float2>((size_t)TC * (c.head_dim / 2), r.activations);
  ctx->sinks = cv.take<float>((size_t)Lc * c.n_heads, r.weights);
  // KV cache [L][MR][2][nh][SL][D]
  ctx->S = S;
  ctx->SL = c.prefix_len + c.ring_len;
  ctx->kv_layer = (size_t)MR * 2 * c.n_heads * ctx->SL * c.head_dim;
  ctx->SLp = (ctx->SL + 15) / 16 * 16;
  if (c.kv_int8) {
    ctx->kvs_layer = (size_t)MR * 2 * c.n_heads * ctx->SLp;
    ctx->kv8 = cv.take<int8_t>(ctx->kv_layer * Lc, r.kv_cache);
    ctx->kvs = cv.take<float>(ctx->kvs_layer * Lc, r.kv_cache);
    ctx->kv_new = cv.take<float>((size_t)TC * 2 * S, r.activations);
  } else {
    ctx->kv = cv.take<__half>(ctx->kv_layer * Lc, r.kv_cache);
  }
  // activations
  ctx->hid = cv.take<float>((size_t)(2 * Lc + 1) * TC * H, r.activations);
  ctx->x_in = cv.take<__half>((size_t)TC * H, r.activations);
  ctx->q = cv.take<float>((size_t)TC * S, r.activations);
  ctx->attn_out = cv.take<__half>((size_t)TC * S, r.activations);
  if (c.n_dense_layers > 0 || E == 0) ctx->act_dense = cv.take<__half>((size_t)TC * c.dense_inter, r.activations);
  if (c.act_int8) {
    int kmax = c.hidden > c.n_heads * c.head_dim ? c.hidden : c.n_heads * c.head_dim;
    if ((c.n_dense_layers > 0 || E == 0) && c.dense_inter > kmax) kmax = c.dense_inter;
    ctx->act8 = cv.take<uint8_t>((size_t)(TC / 8) * act_i8_bytes(8, kmax) > (size_t)(TC / 16) * act_i8_bytes(16, kmax)
                                     ? (size_t)(TC / 8) * act_i8_bytes(8, kmax)
                                     : (size_t)(TC / 16) * act_i8_bytes(16, kmax),
                                 r.activations);
  }
  if (ctx->any_moe()) {
    ctx->xhat = cv.take<__half>((size_t)TC * H, r.activations);
    const int TG = (TC + 15) / 16;
    ctx->act_r = cv.take<uint8_t>((size_t)E * TG * 16 * Ie * 2, r.activations);  // 16 tokens per (expert, group)
    ctx->act_s = cv.take<uint8_t>((size_t)(TC + 7) / 8 * 8 * (Ish > 0 ? Ish : 32) * 2, r.activations);
    ctx->part_r = cv.take<float>((size_t)TC * k * H, r.activations);
    ctx->part_s = cv.take<float>((size_t)TC * H, r.activations);
    ctx->r_logits = cv.take<float>((size_t)Lc * TC * E, r.routing);
    ctx->r_idx = cv.take<int>((size_t)Lc * TC * k, r.routing);
    ctx->r_w = cv.take<float>((size_t)Lc * TC * k, r.routing);
    ctx->r_count = cv.take<int>((size_t)Lc * E, r.routing);
    ctx->r_offset = cv.take<int>((size_t)Lc * (E + 1), r.routing);
    ctx->r_perm = cv.take<int>((size_t)Lc * TC * k, r.routing);
    ctx->r_inv = cv.take<int>((size_t)Lc * TC * k, r.routing);
    ctx->r_rec = cv.take<int4>((size_t)Lc * TG * E, r.routing);
  }
  if (V > 0) {
    ctx->logits = cv.take<float>((size_t)MR * V, r.logits);
    ctx->keys = cv.take<unsigned long long>(MR, r.logits);
    ctx->lm_counter = cv.take<int>(1, r.logits);
  }
  ctx->next_ids = cv.take<int>(MR, r.activations);
  ctx->ids_buf = cv.take<int>(TC, r.activations);
  ctx->pos_buf = cv.take<int>(TC, r.activations);
  ctx->hist = cv.take<int>((size_t)kHistCap * MR, r.activations);
  ctx->hist_ctr = cv.take<int>(1, r.activations);
  ctx->status = cv.take<int>(1, r.activations);
  r.total = cv.off;
}

// ------------------------------------------------------------------ step
namespace {

// A step that launches the kernels of one class only (`only`), for timing that
// class on its own; `launches` counts them.
struct Prof {
  const char* only = nullptr;
  int launches = 0;
};

// kernel classes of a step, in launch order
const char* const kClasses[] = {"embed",       "qkv",      "kv_quant", "attention",      "o_proj",
                                "mlp_gate_up", "mlp_down", "router",   "expert_gate_up", "expert_down", "expert_combine",
                                "lm_head_argmax"};

struct StepShape {
  int rows;
  bool ids;     // input: token ids (else hidden vectors)
  bool lm;      // run the LM head + argmax
  bool logits;  // store logits
  bool chain;   // feed the argmax into the next step (uocr_generate)
  // prefill chunk: every token belongs to cache row `kv_row`, at positions
  // pos_base + t; the LM head (when lm) runs on the last token only
  bool prefill = false;
  int kv_row = 0;
  int pos_base = -1;
};

}  // namespace

static uocr_status enqueue_step(uocr_ctx* ctx, const StepShape& sh, Prof* prof) {
  const uocr_config& c = ctx->cfg;
  cudaStream_t st = ctx->st;
  const int H = c.hidden, S = ctx->S, TC = ctx->TC(), rows = sh.rows;
  const int kv_row0 = sh.prefill ? sh.kv_row : 0, kv_rstep = sh.prefill ? 0 : 1;
  const int nt = rows <= 8 ? 1 : 2;
  const int tg = (rows + 15) / 16;  // token groups of 16 rows (one n-tile pair)
  // streaming CTAs per launch
  const int G = ctx->gemv_ctas_per_sm * ctx->n_sm;
  const int GE = ctx->expert_ctas_per_sm * ctx->n_sm;
  const bool pdl = ctx->pdl;
  auto gx_for = [&](int slabs) {
    int g = G / tg;
    if (g < 1) g = 1;
    return slabs < g ? slabs : g;
  };
  // with prof->only set, only that class's kernels are launched
  auto want = [&](const char* name) {
    if (!prof || !prof->only) return true;
    if (std::strcmp(prof->only, name) != 0) return false;
    ++prof->launches;
    return true;
  };
  auto hid = [&](int idx) { return ctx->hid + (size_t)idx * TC * H; };

  EmbedArgs ea{};
  ea.ids = sh.ids ? ctx->ids_buf : nullptr;
  ea.x = ctx->x_in;
  ea.emb = ctx->emb;
  ea.pos = ctx->pos_buf;
  ea.pos_base = sh.prefill ? sh.pos_base : -1;
  ea.out = hid(0);
  ea.H = H;
  ea.V = c.vocab;
  ea.inv_freq = ctx->inv_freq;
  ea.rope = ctx->rope;
  ea.half_d = c.head_dim / 2;
  ea.status = ctx->status;
  if (want("embed")) {
    CK(launch_embed(ea, rows, st), "embed launch");
  }

  // int8 activations from 4 rows: each projection's input quantised once per
  // token group by its own small kernel instead of in every streaming CTA (below
  // that, the extra launch costs more than the CTAs' own quantisation)
  const bool a8g = c.act_int8 && rows >= 4;
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerW& w = ctx->L[l];
    __half* kvl = ctx->kv ? ctx->kv + ctx->kv_layer * l : nullptr;
    int8_t* kv8l = ctx->kv8 ? ctx->kv8 + ctx->kv_layer * l : nullptr;
    float* kvsl = ctx->kvs ? ctx->kvs + ctx->kvs_layer * l : nullptr;
    // QKV + RoPE + in-place KV append
    GemvArgs qa{};
    qa.w = w.qkv.view();
    qa.sp = plan_stream(nt, kf(c.fmt_attn), H, nt * 8, nt * 8 * (c.head_dim / 2) * 8);
    qa.ntok = rows;
    qa.xf = hid(2 * l);
    qa.ld_src = H;
    qa.norm_w = w.attn_norm;
    qa.eps = c.rms_eps;
    qa.pos = ctx->pos_buf;
    qa.q_out = ctx->q;
    qa.kv = kvl;
    qa.rope = ctx->rope;
    qa.nh = c.n_heads;
    qa.D = c.head_dim;
    qa.S = S;
    qa.P = c.prefix_len;
    qa.R = c.ring_len;
    qa.SL = ctx->SL;
    qa.kv_row0 = kv_row0;
    qa.kv_rstep = kv_rstep;
    qa.kv_new = kv8l ? ctx->kv_new : nullptr;
    qa.status = ctx->status;
    if (want("qkv")) {
      if (a8g) {
        qa.x8 = ctx->act8;
        CK(launch_act_quant(kf(c.fmt_attn), true, qa, ctx->act8, st, pdl), "qkv int8 staging launch");
      }
      CK(launch_gemv(kf(c.fmt_attn), a8g ? SRC_I8_COPY : c.act_int8 ? SRC_NORM_I8 : SRC_NORM, EPI_QKV, qa, gx_for(w.qkv.n_slabs), tg, st, pdl), "qkv launch");
    }
    if (kv8l) {  // INT8 cache: quantise the new keys / values into their slots
      KvQuantArgs ka{};
      ka.src32 = ctx->kv_new;
      ka.kv8 = kv8l;
      ka.kvs = kvsl;
      ka.pos = ctx->pos_buf;
      ka.nh = c.n_heads;
      ka.D = c.head_dim;
      ka.P = c.prefix_len;
      ka.R = c.ring_len;
      ka.SL = ctx->SL;
      ka.SLp = ctx->SLp;
      ka.kv_row0 = kv_row0;
      ka.kv_rstep = kv_rstep;
      if (want("kv_quant")) {
        CK(launch_kv_quant(ka, rows, st, pdl), "kv quant launch");
      }
    }
    // attention
    AttnArgs aa{};
    aa.q = ctx->q;
    aa.kv = kvl;
    aa.kv8 = kv8l;
    aa.kvs = kvsl;
    aa.SLp = ctx->SLp;
    aa.pos = ctx->pos_buf;
    aa.out = ctx->attn_out;
    aa.sink = c.use_sink ? ctx->sinks + (size_t)l * c.n_heads : nullptr;
    aa.nh = c.n_heads;
    aa.D = c.head_dim;
    aa.P = c.prefix_len;
    aa.R = c.ring_len;
    aa.SL = ctx->SL;
    aa.kv_row0 = kv_row0;
    aa.kv_rstep = kv_rstep;
    aa.early = sh.prefill ? 0 : 1;
    aa.status = ctx->status;
    {
      const int pairs = rows * c.n_heads;
      int ns = (2 * ctx->n_sm + pairs - 1) / pairs;
      // more than one wave of resident CTAs with the last one less than half full:
      // one more split (at most doubling) evens the waves out, where each split
      // keeps at least 512 slots (64 rows x 10 heads over 2176 slots: 640 CTAs on
      // 456 resident -> 1280, 124 -> 108 us per launch; over 478 slots the merge
      // costs more than the fuller last wave gains)
      if (const int slots = ctx->attn_slots; slots > 0 && pairs * ns > slots) {
        const int last = pairs * ns - (pairs * ns - 1) / slots * slots;
        const int ns2 = ns + 1;
        const int last2 = pairs * ns2 - (pairs * ns2 - 1) / slots * slots;
        if (2 * last < slots && ns2 <= 2 * ns && last2 > last && ctx->SL >= 512 * ns2) ns = ns2;
      }
      if (ns < ctx->attn_min_splits) ns = ctx->attn_min_splits;
      const int cap = (ctx->SL + 63) / 64;
      if (ns > cap) ns = cap;
      if (ns > kMaxSplits) ns = kMaxSplits;
      if (ns < 1) ns = 1;
      aa.nsplit = ns;
      aa.chunk = (ctx->SL + ns - 1) / ns;
      if (kv8l) aa.chunk = (aa.chunk + 15) / 16 * 16;  // scale runs start on 16-byte boundaries
    }
    aa.scale = 1.0f / sqrtf((float)c.head_dim);
    if (want("attention")) {
      CK(launch_attn(aa, rows, st, pdl), "attention launch");
    }
    // O projection + residual
    GemvArgs oa{};
    oa.w = w.o.view();
    oa.sp = plan_stream(nt, kf(c.fmt_attn), S);
    oa.ntok = rows;
    oa.xh = ctx->attn_out;
    oa.ld_src = S;
    oa.res_in = hid(2 * l);
    oa.out_f = hid(2 * l + 1);
    oa.ld_out = H;
    oa.status = ctx->status;
    if (want("o_proj")) {
      if (a8g) {
        oa.x8 = ctx->act8;
        CK(launch_act_quant(kf(c.fmt_attn), false, oa, ctx->act8, st, pdl), "o_proj int8 staging launch");
      }
      CK(launch_gemv(kf(c.fmt_attn), a8g ? SRC_I8_COPY : c.act_int8 ? SRC_F16_I8 : SRC_F16, EPI_RESID, oa, gx_for(w.o.n_slabs), tg, st, pdl), "o_proj launch");
    }
    if (w.dense) {
      GemvArgs ga{};
      ga.w = w.gateup.view();
      ga.sp = plan_stream(nt, kf(c.fmt_dense), H);
      ga.ntok = rows;
      ga.xf = hid(2 * l + 1);
      ga.ld_src = H;
      ga.norm_w = w.mlp_norm;
      ga.eps = c.rms_eps;
      ga.out_h = ctx->act_dense;
      ga.ld_out = c.dense_inter;
      ga.status = ctx->status;
      if (want("mlp_gate_up")) {
        if (a8g) {
          ga.x8 = ctx->act8;
          CK(launch_act_quant(kf(c.fmt_dense), true, ga, ctx->act8, st, pdl), "gate/up int8 staging launch");
        }
        CK(launch_gemv(kf(c.fmt_dense), a8g ? SRC_I8_COPY : c.act_int8 ? SRC_NORM_I8 : SRC_NORM, EPI_SWIGLU, ga, gx_for(w.gateup.n_slabs), tg, st, pdl),
           "gate/up launch");
      }
      GemvArgs da{};
      da.w = w.down.view();
      da.sp = plan_stream(nt, kf(c.fmt_dense), c.dense_inter);
      da.ntok = rows;
      da.xh = ctx->act_dense;
      da.ld_src = c.dense_inter;
      da.res_in = hid(2 * l + 1);
      da.out_f = hid(2 * l + 2);
      da.ld_out = H;
      da.status = ctx->status;
      if (want("mlp_down")) {
        if (a8g) {
          da.x8 = ctx->act8;
          CK(launch_act_quant(kf(c.fmt_dense), false, da, ctx->act8, st, pdl), "down int8 staging launch");
        }
        CK(launch_gemv(kf(c.fmt_dense), a8g ? SRC_I8_COPY : c.act_int8 ? SRC_F16_I8 : SRC_F16, EPI_RESID, da, gx_for(w.down.n_slabs), tg, st, pdl), "down launch");
      }
    } else {
      const int E = c.n_experts, k = c.top_k;
      // Routed units: active slots when few experts are expected to receive a
      // token (one token group only), else expert ids (their CTAs stream before
      // the routing is known; the grid is one wave of CTAs that all have work).
      // Expected experts with a token: E (1 - (1 - k/E)^rows).
      const int max_act = E < rows * k ? E : rows * k;
      const double exp_act = E * (1.0 - pow(1.0 - (double)k / E, rows));
      const int by_slot = exp_act < 0.75 * E && tg == 1;
      // more than 16 rows: the expert contraction on the tensor cores (expert-id units)
      const bool tcx = ctx->tc_experts && rows > 16 && !by_slot;
      const int n_units = by_slot ? max_act : E;
      int4* rec = ctx->r_rec + (size_t)l * ((TC + 15) / 16) * E;

      RouterArgs ra{};
      ra.w = w.router.view();
      ra.sp = plan_stream(nt, F16, H);
      ra.ntok = rows;
      ra.H = H;
      ra.E = E;
      ra.k = k;
      ra.h = hid(2 * l + 1);
      ra.norm_w = w.mlp_norm;
      ra.eps = c.rms_eps;
      ra.logits = ctx->r_logits + (size_t)l * TC * E;
      ra.tg = tg;
      ra.by_slot = by_slot;
      ra.n_units = n_units;
      ra.idx = ctx->r_idx + (size_t)l * TC * k;
      ra.wts = ctx->r_w + (size_t)l * TC * k;
      ra.rec = rec;
      ra.status = ctx->status;
      if (want("router")) {
        CK(launch_router(ra, st, pdl), "router launch");
      }

      const int fs = ctx->shared_fmt();
      ExpertArgs xa{};
      xa.ntok = rows;
      xa.E = E;
      xa.k = k;
      xa.H = H;
      xa.Ie = c.expert_inter;
      xa.Ish = c.n_shared * c.expert_inter;
      xa.tg = tg;
      xa.rec = rec;
      xa.idx = ra.idx;
      xa.wts = ra.wts;
      xa.count = ctx->r_count + (size_t)l * E;
      xa.offset = ctx->r_offset + (size_t)l * (E + 1);
      xa.perm = ctx->r_perm + (size_t)l * TC * k;
      xa.inv = ctx->r_inv + (size_t)l * TC * k;
      xa.h = hid(2 * l + 1);
      xa.norm_w = w.mlp_norm;
      xa.eps = c.rms_eps;
      xa.act_r = ctx->act_r;
      xa.act_s = ctx->act_s;
      xa.part_r = ctx->part_r;
      xa.part_s = ctx->part_s;
      xa.out = hid(2 * l + 2);
      xa.status = ctx->status;
      xa.by_slot = by_slot;
      xa.n_units = n_units;
      const double units = by_slot ? exp_act : E;
      // CTAs per routed unit and for the shared experts, in proportion to the
      // bytes each streams (the shared experts once per 16-row pass), about GE
      // in all: one grid row covers every token group
      auto split = [&](const DMat& r, const DMat* sh, int rslabs, int sslabs) {
        const double br = (double)(r.qbytes + r.sbytes);
        // the shared experts are streamed once per pass: 16 rows (GEMV), 32 (tensor cores)
        const int sh_passes = tcx ? (rows + kTcxRowsShared - 1) / kTcxRowsShared : tg;
        const double bs = sh ? (double)(sh->qbytes + sh->sbytes) * sh_passes : 0.0;
        const double tot = units * br + bs;
        const int gt = tcx ? ctx->n_sm : GE;  // the tensor-core kernels run one CTA per SM
        // parts of whole rounds (G_w slabs; a 128-row tile of 8 slabs on the tensor
        // cores); the fewest parts that give the rounds per CTA the byte-proportional
        // target gives
        auto parts = [&](double target, int slabs, int U) {
          const int gw = tcx ? 8 : kWarps / warps_per_slab(U);
          const int nr = (slabs + gw - 1) / gw;
          int t = (int)ceil(target);
          t = t < 1 ? 1 : t > nr ? nr : t;
          const int per = (nr + t - 1) / t;
          return (nr + per - 1) / per;
        };
        if (by_slot) {
          xa.cpe = parts(gt * br / tot, rslabs, r.U);
          xa.cpes = sh ? parts(gt * bs / tot, sslabs, sh->U) : 0;
        } else {
          // expert ids: the routed parts rounded down so that the grid stays one
          // wave; the shared experts take the rest of it
          xa.cpe = parts(floor(gt * br / tot), rslabs, r.U);
          const int left = gt - E * xa.cpe;
          xa.cpes = sh ? parts(left > 1 ? left : 1, sslabs, sh->U) : 0;
        }
        // active-slot units: the routed CTAs fill the rest of the wave and are
        // dealt out over the experts that did receive a token (at least one each)
        const int rest = gt - xa.cpes;
        xa.n_rctas = by_slot ? (rest > n_units ? rest : n_units) : 0;
      };
      const DMat* shg = c.n_shared > 0 ? &w.sh_gateup : nullptr;
      const DMat* shd = c.n_shared > 0 ? &w.sh_down : nullptr;
      // gate/up + SwiGLU (and the routing of every row)
      xa.wr = w.ex_gateup.view(1);
      xa.ws = shg ? shg->view() : PMat{};
      xa.sp = plan_stream(nt, kf(c.fmt_routed), H, 16);
      split(w.ex_gateup, shg, w.ex_gateup.n_slabs, shg ? shg->n_slabs : 0);
      if (want("expert_gate_up")) {
        if (tcx)
          CK(launch_tc_expert(0, kf(c.fmt_routed), fs, xa, ctx->tcx_gu, st, pdl), "tensor-core expert gate/up launch");
        else
          CK(launch_expert_gateup(kf(c.fmt_routed), fs, xa, st, pdl), "expert gate/up launch");
      }
      // down + combine
      xa.wr = w.ex_down.view(1);
      xa.ws = shd ? shd->view() : PMat{};
      {
        const int kmax = xa.Ish > xa.Ie ? xa.Ish : xa.Ie;
        xa.sp = plan_stream(nt, kf(c.fmt_routed), 0, 0, nt * (kmax / 32) * 512);
      }
      split(w.ex_down, shd, H / 16, H / 16);
      if (want("expert_down")) {
        if (tcx)
          CK(launch_tc_expert(1, kf(c.fmt_routed), fs, xa, ctx->tcx_dn, st, pdl), "tensor-core expert down launch");
        else
          CK(launch_expert_down(kf(c.fmt_routed), fs, xa, st, pdl), "expert down launch");
      }
      if (want("expert_combine")) {
        CK(launch_expert_combine(xa, st, pdl), "expert combine launch");
      }
    }
  }

  if (sh.lm && ctx->lm_tc && !sh.prefill && rows > 16) {
    // many rows: one read of every weight tile for all of them, on the tensor cores
    TcLmArgs ta{};
    ta.w = ctx->lm_tc;
    ta.xc = ctx->lm_xc;
    ta.x = hid(2 * c.n_layers);
    ta.ld_x = H;
    ta.norm_w = ctx->final_norm;
    ta.eps = c.rms_eps;
    ta.K = H;
    ta.V = c.vocab;
    ta.n_mtiles = ctx->lm_mtiles;
    ta.ntok = rows;
    ta.npad = tc_lm_npad(rows);
    ta.logits = sh.logits ? ctx->logits : nullptr;
    ta.keys = ctx->keys;
    ta.counter = ctx->lm_counter;
    ta.next_ids = ctx->next_ids;
    ta.status = ctx->status;
    if (sh.chain) {
      ta.feed_ids = ctx->ids_buf;
      ta.feed_pos = ctx->pos_buf;
      ta.hist = ctx->hist;
      ta.hist_ctr = ctx->hist_ctr;
    }
    if (want("lm_head_argmax")) {
      CK(launch_tc_lm(ta, ctx->n_sm, st, pdl), "tensor-core lm head launch");
    }
  } else if (sh.lm) {
    // a prefill chunk needs the next id after its last token only
    const int lm_rows = sh.prefill ? 1 : rows;
    const int lm_nt = lm_rows <= 8 ? 1 : 2, lm_tg = (lm_rows + 15) / 16;
    GemvArgs la{};
    la.w = ctx->lm.view();
    la.sp = plan_stream(lm_nt, F16, H);
    la.ntok = lm_rows;
    la.xf = hid(2 * c.n_layers) + (size_t)(rows - lm_rows) * H;
    la.ld_src = H;
    la.norm_w = ctx->final_norm;
    la.eps = c.rms_eps;
    la.out_f = sh.logits ? ctx->logits : nullptr;
    la.n_valid = c.vocab;
    la.keys = ctx->keys;
    la.counter = ctx->lm_counter;
    la.next_ids = ctx->next_ids;
    la.status = ctx->status;
    if (sh.chain) {
      la.feed_ids = ctx->ids_buf;
      la.feed_pos = ctx->pos_buf;
      la.hist = ctx->hist;
      la.hist_ctr = ctx->hist_ctr;
    }
    if (want("lm_head_argmax")) {
      int lgx = G / lm_tg;
      lgx = lgx < 1 ? 1 : lgx > ctx->lm.n_slabs ? ctx->lm.n_slabs : lgx;
      CK(launch_gemv(F16, SRC_NORM, EPI_LOGITS, la, lgx, lm_tg, st, pdl), "lm head launch");
    }
  }
  return UOCR_OK;
}

static uocr_status run_step(uocr_ctx* ctx, const StepShape& sh) {
  if (!ctx->cfg.use_graphs) return enqueue_step(ctx, sh, nullptr);
  const uint64_t key = (uint64_t)sh.rows | ((uint64_t)sh.ids << 8) | ((uint64_t)sh.lm << 9) |
                       ((uint64_t)sh.logits << 10) | ((uint64_t)sh.chain << 11);
  auto it = ctx->graphs.find(key);
  if (it == ctx->graphs.end()) {
    cudaGraph_t g = nullptr;
    CK(cudaStreamBeginCapture(ctx->st, cudaStreamCaptureModeThreadLocal), "begin capture");
    uocr_status s = enqueue_step(ctx, sh, nullptr);
    cudaError_t e = cudaStreamEndCapture(ctx->st, &g);
    if (s != UOCR_OK) {
      if (g) cudaGraphDestroy(g);
      return s;
    }
    CK(e, "end capture");
    cudaGraphExec_t ge = nullptr;
    e = cudaGraphInstantiate(&ge, g, 0);
    cudaGraphDestroy(g);
    CK(e, "graph instantiate");
    it = ctx->graphs.emplace(key, ge).first;
  }
  CK(cudaGraphLaunch(it->second, ctx->st), "graph launch");
  return UOCR_OK;
}

// ------------------------------------------------------------------ weights
namespace {

struct Expect {
  int fmt;  // -1: any quantised? no: exact format required
  int rows, cols;
  Group group;
  int n_members;  // members of the group
  int member;     // index of this tensor in the group
};

}  // namespace

static bool expect_for(uocr_ctx* ctx, const uocr_tensor& t, Expect& ex, std::string& why) {
  const uocr_config& c = ctx->cfg;
  const int H = c.hidden, S = ctx->S, V = c.vocab, E = c.n_experts;
  const bool proj = t.kind == UOCR_T_PROJ || t.kind == UOCR_T_PROJ_BIAS;
  const bool glob = t.kind == UOCR_T_EMBED || t.kind == UOCR_T_FINAL_NORM || t.kind == UOCR_T_LM_HEAD || proj;
  if (glob) {
    if (proj && c.proj_in <= 0) return why = "the config has no projector (proj_in = 0)", false;
    if (!proj && V <= 0) return why = "the config has no vocabulary", false;
    if (t.layer != 0 || t.expert != 0) return why = "global tensors use layer 0, expert 0", false;
  } else if (t.layer < 0 || t.layer >= c.n_layers) {
    return why = "layer out of range", false;
  }
  const bool dense = glob ? true : ctx->layer_dense(t.layer);
  ex.group = G_SINGLE;
  ex.n_members = 1;
  ex.member = 0;
  auto need_expert0 = [&]() { return t.expert == 0 ? true : (why = "expert must be 0", false); };
  switch (t.kind) {
    case UOCR_T_EMBED: ex = {UOCR_F16, V, H, G_SINGLE, 1, 0}; return true;
    case UOCR_T_FINAL_NORM: ex = {UOCR_F16, 1, H, G_SINGLE, 1, 0}; return true;
    case UOCR_T_LM_HEAD: ex = {UOCR_F16, V, H, G_SINGLE, 1, 0}; return true;
    case UOCR_T_PROJ: ex = {c.fmt_proj, H, c.proj_in, G_SINGLE, 1, 0}; return true;
    case UOCR_T_PROJ_BIAS: ex = {UOCR_F16, 1, H, G_SINGLE, 1, 0}; return true;
    case UOCR_T_ATTN_NORM:
    case UOCR_T_MLP_NORM: ex = {UOCR_F16, 1, H, G_SINGLE, 1, 0}; return need_expert0();
    case UOCR_T_WQ:
    case UOCR_T_WK:
    case UOCR_T_WV:
      ex = {c.fmt_attn, S, H, G_QKV, 3, t.kind - UOCR_T_WQ};
      return need_expert0();
    case UOCR_T_WO: ex = {c.fmt_attn, H, S, G_SINGLE, 1, 0}; return need_expert0();
    case UOCR_T_GATE:
    case UOCR_T_UP:
      if (!dense) return why = "dense MLP tensor on a MoE layer", false;
      ex = {c.fmt_dense, c.dense_inter, H, G_DENSE_GU, 2, t.kind - UOCR_T_GATE};
      return need_expert0();
    case UOCR_T_DOWN:
      if (!dense) return why = "dense MLP tensor on a MoE layer", false;
      ex = {c.fmt_dense, H, c.dense_inter, G_SINGLE, 1, 0};
      return need_expert0();
    case UOCR_T_ROUTER:
      if (dense) return why = "router on a dense layer", false;
      ex = {UOCR_F16, E, H, G_SINGLE, 1, 0};
      return need_expert0();
    case UOCR_T_SHARED_GATE:
    case UOCR_T_SHARED_UP:
    case UOCR_T_SHARED_DOWN:
      if (dense) return why = "expert tensor on a dense layer", false;
      if (t.expert < 0 || t.expert >= c.n_shared) return why = "shared expert index out of range", false;
      if (t.kind == UOCR_T_SHARED_DOWN)
        ex = {c.fmt_shared, H, c.expert_inter, G_SHARED_DOWN, c.n_shared, t.expert};
      else
        ex = {c.fmt_shared, c.expert_inter, H, G_SHARED_GU, 2 * c.n_shared,
              2 * t.expert + (t.kind == UOCR_T_SHARED_UP ? 1 : 0)};
      return true;
    case UOCR_T_EXPERT_GATE:
    case UOCR_T_EXPERT_UP:
    case UOCR_T_EXPERT_DOWN:
      if (dense) return why = "expert tensor on a dense layer", false;
      if (t.expert < 0 || t.expert >= E) return why = "routed expert index out of range", false;
      if (t.kind == UOCR_T_EXPERT_DOWN)
        ex = {c.fmt_routed, H, c.expert_inter, G_SINGLE, 1, 0};
      else
        ex = {c.fmt_routed, c.expert_inter, H, G_EXPERT_GU, 2, t.kind == UOCR_T_EXPERT_UP ? 1 : 0};
      return true;
  }
  why = "unknown tensor kind";
  return false;
}

static uocr_status pack_into(uocr_ctx* ctx, const DMat& dst, size_t expert_off_q, size_t expert_off_s, int map,
                             const std::vector<void*>& srcs, int src_rows, int src_cols, int I) {
  PackArgs pa{};
  pa.q = dst.q + expert_off_q;
  pa.s = dst.s ? dst.s + expert_off_s : nullptr;
  pa.fmt = dst.fmt;
  pa.group = fmt_group(dst.cfmt);
  pa.bb = fmt_block_bytes(dst.cfmt);
  pa.n_slabs = dst.n_slabs;
  pa.U = dst.U * (unit_bytes(dst.fmt) / 512);  // the packer counts 512-byte (sub-)units
  pa.K = dst.K;
  pa.map = map;
  pa.nsrc = (int)srcs.size();
  for (size_t i = 0; i < srcs.size() && i < 8; ++i) pa.src[i] = reinterpret_cast<const uint8_t*>(srcs[i]);
  pa.src_rows = src_rows;
  pa.src_cols = src_cols;
  pa.S = ctx->S;
  pa.D = ctx->cfg.head_dim;
  pa.I = I;
  CK(launch_pack(pa, ctx->st), "pack launch");
  CK(cudaStreamSynchronize(ctx->st), "pack");
  return UOCR_OK;
}

static uocr_status finish_group(uocr_ctx* ctx, int kind, int layer, int expert, Group grp, std::vector<void*>& srcs) {
  const uocr_config& c = ctx->cfg;
  const int H = c.hidden;
  LayerW* w = (kind == UOCR_T_EMBED || kind == UOCR_T_FINAL_NORM || kind == UOCR_T_LM_HEAD || kind == UOCR_T_PROJ)
                  ? nullptr
                  : &ctx->L[layer];
  switch (grp) {
    case G_QKV: return pack_into(ctx, w->qkv, 0, 0, MAP_QKV, srcs, ctx->S, H, 0);
    case G_DENSE_GU: return pack_into(ctx, w->gateup, 0, 0, MAP_SWIGLU, srcs, c.dense_inter, H, c.dense_inter);
    case G_SHARED_GU: return pack_into(ctx, w->sh_gateup, 0, 0, MAP_SWIGLU, srcs, c.expert_inter, H, c.expert_inter);
    case G_SHARED_DOWN: return pack_into(ctx, w->sh_down, 0, 0, MAP_KCAT, srcs, H, c.expert_inter, c.expert_inter);
    case G_EXPERT_GU:
      return pack_into(ctx, w->ex_gateup, w->ex_gateup.qbytes * expert, w->ex_gateup.sbytes * expert, MAP_SWIGLU,
                       srcs, c.expert_inter, H, c.expert_inter);
    case G_SINGLE: break;
  }
  switch (kind) {
    case UOCR_T_WO: return pack_into(ctx, w->o, 0, 0, MAP_IDENT, srcs, H, ctx->S, 0);
    case UOCR_T_DOWN: return pack_into(ctx, w->down, 0, 0, MAP_IDENT, srcs, H, c.dense_inter, 0);
    case UOCR_T_ROUTER: return pack_into(ctx, w->router, 0, 0, MAP_IDENT, srcs, c.n_experts, H, 0);
    case UOCR_T_EXPERT_DOWN:
      return pack_into(ctx, w->ex_down, w->ex_down.qbytes * expert, w->ex_down.sbytes * expert, MAP_IDENT, srcs, H,
                       c.expert_inter, 0);
    case UOCR_T_LM_HEAD: {
      uocr_status s = pack_into(ctx, ctx->lm, 0, 0, MAP_IDENT, srcs, c.vocab, H, 0);
      if (s == UOCR_OK && ctx->lm_tc) {
        CK(launch_pack_canon(srcs[0], ctx->lm_tc, c.vocab, H, ctx->st), "lm head tensor-core pack");
        CK(cudaStreamSynchronize(ctx->st), "lm head tensor-core pack");
      }
      return s;
    }
    case UOCR_T_PROJ: return pack_into(ctx, ctx->proj, 0, 0, MAP_IDENT, srcs, H, c.proj_in, 0);
  }
  return ctx->fail(UOCR_E_FORMAT, "internal: no packer for kind %d", kind);
}

static uocr_status load_one(uocr_ctx* ctx, const uocr_tensor& t) {
  Expect ex{};
  std::string why;
  if (!expect_for(ctx, t, ex, why))
    return ctx->fail(UOCR_E_FORMAT, "tensor kind %d layer %d expert %d: %s", t.kind, t.layer, t.expert, why.c_str());
  if (t.format != ex.fmt)
    return ctx->fail(UOCR_E_FORMAT, "tensor kind %d layer %d expert %d: format %d, expected %d", t.kind, t.layer,
                     t.expert, t.format, ex.fmt);
  if (t.rows != ex.rows || t.cols != ex.cols)
    return ctx->fail(UOCR_E_FORMAT, "tensor kind %d layer %d expert %d: shape [%d][%d], expected [%d][%d]", t.kind,
                     t.layer, t.expert, t.rows, t.cols, ex.rows, ex.cols);
  const size_t want = blob_bytes(t.format, t.rows, t.cols);
  if (t.bytes != want || t.data == nullptr)
    return ctx->fail(UOCR_E_FORMAT, "tensor kind %d layer %d expert %d: %llu bytes, expected %zu", t.kind, t.layer,
                     t.expert, (unsigned long long)t.bytes, want);
  // plain copies
  const uocr_config& c = ctx->cfg;
  if (t.kind == UOCR_T_EMBED || t.kind == UOCR_T_FINAL_NORM || t.kind == UOCR_T_ATTN_NORM ||
      t.kind == UOCR_T_MLP_NORM || t.kind == UOCR_T_PROJ_BIAS) {
    void* dst = t.kind == UOCR_T_EMBED        ? (void*)ctx->emb
                : t.kind == UOCR_T_FINAL_NORM ? (void*)ctx->final_norm
                : t.kind == UOCR_T_PROJ_BIAS  ? (void*)ctx->proj_b
                : t.kind == UOCR_T_ATTN_NORM  ? (void*)ctx->L[t.layer].attn_norm
                                              : (void*)ctx->L[t.layer].mlp_norm;
    CK(cudaMemcpy(dst, t.data, t.bytes, cudaMemcpyHostToDevice), "weight copy");
    ctx->loaded[{t.kind, t.layer, t.expert}] = true;
    return UOCR_OK;
  }
  void* dev = nullptr;
  CK(cudaMalloc(&dev, t.bytes), "staging allocation");
  cudaError_t e = cudaMemcpy(dev, t.data, t.bytes, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(dev);
    return ctx->cuda(e, "staging copy");
  }
  // group key: (group, layer, expert for per-expert groups)
  const int gexp = ex.group == G_EXPERT_GU ? t.expert : 0;
  std::vector<int> gk = {(int)ex.group, t.layer, ex.group == G_SINGLE ? t.kind : gexp,
                         ex.group == G_SINGLE ? t.expert : 0};
  Pending& p = ctx->pending[gk];
  if (p.dev.empty()) p.dev.assign(ex.n_members, nullptr);
  if (p.dev[ex.member]) {
    cudaFree(p.dev[ex.member]);
    --p.have;
  }
  p.dev[ex.member] = dev;
  ++p.have;
  uocr_status s = UOCR_OK;
  if (p.have == ex.n_members) {
    s = finish_group(ctx, t.kind, t.layer, t.expert, ex.group, p.dev);
    for (void* d : p.dev) cudaFree(d);
    ctx->pending.erase(gk);
  }
  (void)c;
  if (s == UOCR_OK) ctx->loaded[{t.kind, t.layer, t.expert}] = true;
  return s;
}

static uocr_status check_complete(uocr_ctx* ctx) {
  if (ctx->complete) return UOCR_OK;  // the walk below costs hundreds of µs of host time per step
  const uocr_config& c = ctx->cfg;
  auto has = [&](int k, int l, int e) { return ctx->loaded.count({k, l, e}) > 0; };
  auto miss = [&](int k, int l, int e) {
    return ctx->fail(UOCR_E_STATE, "weight tensor kind %d layer %d expert %d has not been loaded", k, l, e);
  };
  if (c.vocab > 0)
    for (int k : {UOCR_T_EMBED, UOCR_T_FINAL_NORM, UOCR_T_LM_HEAD})
      if (!has(k, 0, 0)) return miss(k, 0, 0);
  for (int l = 0; l < c.n_layers; ++l) {
    for (int k : {UOCR_T_ATTN_NORM, UOCR_T_WQ, UOCR_T_WK, UOCR_T_WV, UOCR_T_WO, UOCR_T_MLP_NORM})
      if (!has(k, l, 0)) return miss(k, l, 0);
    if (ctx->layer_dense(l)) {
      for (int k : {UOCR_T_GATE, UOCR_T_UP, UOCR_T_DOWN})
        if (!has(k, l, 0)) return miss(k, l, 0);
    } else {
      if (!has(UOCR_T_ROUTER, l, 0)) return miss(UOCR_T_ROUTER, l, 0);
      for (int s = 0; s < c.n_shared; ++s)
        for (int k : {UOCR_T_SHARED_GATE, UOCR_T_SHARED_UP, UOCR_T_SHARED_DOWN})
          if (!has(k, l, s)) return miss(k, l, s);
      for (int e = 0; e < c.n_experts; ++e)
        for (int k : {UOCR_T_EXPERT_GATE, UOCR_T_EXPERT_UP, UOCR_T_EXPERT_DOWN})
          if (!has(k, l, e)) return miss(k, l, e);
    }
  }
  if (c.use_sink && !ctx->sinks_set) return ctx->fail(UOCR_E_STATE, "use_sink = 1 but uocr_set_sinks was not called");
  ctx->complete = true;
  return UOCR_OK;
}

// ------------------------------------------------------------------ scratch-free LM head
// Scratch of uocr_lm_head_argmax_noalloc: one 64-bit argmax key per row (up to
// kNoAllocMaxRows) and the kernel's finished-CTA counter, then room for the
// rows staged in the tensor cores' operand layout (steps of more than 16 rows).
// It lives in this file-scope device array (1 KB + 256 KB), so every GPU that
// loads the library holds it until the process exits and no call ever
// allocates.  Host code must not pass the symbol itself to a kernel: its
// device address is fetched per device with cudaGetSymbolAddress.
constexpr int kNoAllocMaxRows = 64;
// Beyond 16 rows the LM head runs on the tensor cores, which need the rows
// staged in their operand layout: 128 bytes per input for 64 rows, here for
// hidden sizes up to kNoAllocMaxHidden.
constexpr int kNoAllocMaxHidden = 2048;
constexpr size_t kNoAllocKeysBytes = 1024;  // keys [64] + counter, rounded up
constexpr size_t kNoAllocBytes = kNoAllocKeysBytes + (size_t)kNoAllocMaxHidden * 128;
static __device__ __align__(256) unsigned long long g_lm_noalloc_scratch[kNoAllocBytes / 8];
static std::mutex g_noalloc_mu;
static std::map<int, unsigned long long*> g_noalloc_addr;  // device ordinal -> device address

// Looks the scratch address up once per device, with that device current.
static cudaError_t noalloc_scratch(int device, unsigned long long** out) {
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  auto it = g_noalloc_addr.find(device);
  if (it != g_noalloc_addr.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  int prev = 0;
  cudaError_t e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return e;
  if (prev != device && (e = cudaSetDevice(device)) != cudaSuccess) return e;
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_lm_noalloc_scratch);
  if (prev != device) cudaSetDevice(prev);
  if (e != cudaSuccess) return e;
  g_noalloc_addr[device] = reinterpret_cast<unsigned long long*>(p);
  *out = reinterpret_cast<unsigned long long*>(p);
  return cudaSuccess;
}

static uocr_status noalloc_launch(uocr_ctx* ctx, int rows, const float* hidden, int32_t* next_ids, float* logits,
                                  unsigned long long* scratch, cudaStream_t st);

// ------------------------------------------------------------------ C ABI
extern "C" {

uocr_status uocr_create(const uocr_config* cfg, uocr_ctx** out) {
  if (!out) return UOCR_E_INVALID_ARG;
  *out = nullptr;
  if (!cfg) return UOCR_E_INVALID_ARG;
  uocr_ctx* ctx = new uocr_ctx();
  ctx->cfg = *cfg;
  uocr_status s = check_config(ctx, ctx->cfg);
  if (s != UOCR_OK) {
    g_create_err = ctx->err;
    delete ctx;
    return s;
  }
  // measuring pass for the budget check
  Carver m;
  carve(ctx, m);
  if (cfg->mem_budget && ctx->rep.total > cfg->mem_budget) {
    const uocr_mem_report& r = ctx->rep;
    g_create_err = ctx->fail(UOCR_E_BUDGET,
              "working set %llu B exceeds the budget %llu B (weights %llu, kv_cache %llu, activations %llu, "
              "routing %llu, logits %llu)",
              (unsigned long long)r.total, (unsigned long long)cfg->mem_budget, (unsigned long long)r.weights,
              (unsigned long long)r.kv_cache, (unsigned long long)r.activations, (unsigned long long)r.routing,
              (unsigned long long)r.logits) == UOCR_E_BUDGET ? ctx->err : std::string();
    delete ctx;
    return UOCR_E_BUDGET;
  }
  cudaError_t e = cudaSetDevice(cfg->device);
  if (e != cudaSuccess) {
    g_create_err = std::string("cudaSetDevice: ") + cudaGetErrorString(e);
    delete ctx;
    return UOCR_E_CUDA;
  }
  cudaDeviceGetAttribute(&ctx->n_sm, cudaDevAttrMultiProcessorCount, cfg->device);
  e = init_kernel_attributes();
  if (e == cudaSuccess) e = cudaMalloc(&ctx->arena, m.off);
  if (e != cudaSuccess) {
    const bool oom = e == cudaErrorMemoryAllocation;
    g_create_err = std::string("arena allocation / kernel set-up: ") + cudaGetErrorString(e);
    cudaGetLastError();
    delete ctx;
    return oom ? UOCR_E_OOM : UOCR_E_CUDA;
  }
  Carver a;
  a.base = ctx->arena;
  carve(ctx, a);
  e = cudaStreamCreateWithFlags(&ctx->st, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ctx->ev_in, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ctx->ev_out, cudaEventDisableTiming);
  ctx->ust = reinterpret_cast<cudaStream_t>(cfg->stream);
  {
    const char* v = std::getenv("UOCR_NO_PDL");  // A/B switch for measuring the launch overlap
    ctx->pdl = !(v && v[0] == '1');
    // grid sizing knobs for tuning sweeps (CTAs per SM, 1..8)
    auto knob = [](const char* name, int def) {
      const char* e = std::getenv(name);
      const int x = e ? atoi(e) : def;
      return x >= 1 && x <= 8 ? x : def;
    };
    ctx->gemv_ctas_per_sm = knob("UOCR_GEMV_CTAS_PER_SM", ctx->gemv_ctas_per_sm);
    ctx->expert_ctas_per_sm = knob("UOCR_EXPERT_CTAS_PER_SM", ctx->expert_ctas_per_sm);
    ctx->attn_min_splits = knob("UOCR_ATTN_MIN_SPLITS", ctx->attn_min_splits);
    ctx->attn_slots = attn_ctas_per_sm(cfg->head_dim, cfg->kv_int8 != 0) * ctx->n_sm;
    // the tensor-core expert kernels on request (UOCR_TC_EXPERTS=1) where the formats and
    // the shared memory allow them.  Off by default: at the few rows per expert of a
    // decode step they stream the weights at about 0.6 the speed of the fragment-GEMV
    // kernels (dequantising into shared memory costs the SM what the mma.sync products
    // cost it there, and one CTA per SM keeps fewer weight bytes in flight).
    const char* tv = std::getenv("UOCR_TC_EXPERTS");
    const bool want_tc = tv && tv[0] == '1';
    if (want_tc && ctx->any_moe() && tcx_format_ok(kf(cfg->fmt_routed), ctx->shared_fmt())) {
      int optin = 0;
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, cfg->device);
      const int limit = optin - 8 * 1024;  // the kernel's static routing state and slack
      const int H = cfg->hidden, Ie = cfg->expert_inter, Ish = cfg->n_shared * cfg->expert_inter;
      const int bg = kTcxRowsRouted * H * 2 > kTcxRowsShared * H * 2 * (Ish > 0) ? kTcxRowsRouted * H * 2
                                                                                  : kTcxRowsShared * H * 2;
      const int bd = kTcxRowsRouted * Ie * 2 > kTcxRowsShared * Ish * 2 ? kTcxRowsRouted * Ie * 2
                                                                         : kTcxRowsShared * Ish * 2;
      ctx->tcx_gu = tcx_plan(bg, limit);
      ctx->tcx_dn = tcx_plan(bd, limit);
      ctx->tc_experts = ctx->tcx_gu.stages >= 2 && ctx->tcx_dn.stages >= 2;
    }
  }
  // zero everything (KV cache, counters, argmax keys, status)
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->arena, 0, m.off, ctx->st);
  if (e == cudaSuccess) {
    std::vector<double> inv(cfg->head_dim / 2);
    for (int i = 0; i < cfg->head_dim / 2; ++i)
      inv[i] = std::pow((double)cfg->rope_theta, -2.0 * i / cfg->head_dim);
    e = cudaMemcpyAsync(ctx->inv_freq, inv.data(), inv.size() * sizeof(double), cudaMemcpyHostToDevice, ctx->st);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->st);
  if (e != cudaSuccess) {
    g_create_err = std::string("context set-up: ") + cudaGetErrorString(e);
    uocr_destroy(ctx);
    return UOCR_E_CUDA;
  }
  g_create_err.clear();
  *out = ctx;
  return UOCR_OK;
}

void uocr_destroy(uocr_ctx* ctx) {
  if (!ctx) return;
  {
    std::lock_guard<std::mutex> lk(ctx->mu);
    if (ctx->st) cudaStreamSynchronize(ctx->st);
    for (auto& kv : ctx->graphs) cudaGraphExecDestroy(kv.second);
    for (auto& kv : ctx->pending)
      for (void* d : kv.second.dev)
        if (d) cudaFree(d);
    if (ctx->arena) cudaFree(ctx->arena);
    if (ctx->ev_in) cudaEventDestroy(ctx->ev_in);
    if (ctx->ev_out) cudaEventDestroy(ctx->ev_out);
    if (ctx->st) cudaStreamDestroy(ctx->st);
  }
  delete ctx;
}

uocr_status uocr_load_weights(uocr_ctx* ctx, const uocr_tensor* t, size_t n) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (!t && n) return ctx->fail(UOCR_E_INVALID_ARG, "tensor list is NULL");
  for (size_t i = 0; i < n; ++i) {
    uocr_status s = load_one(ctx, t[i]);
    if (s != UOCR_OK) return s;
  }
  return UOCR_OK;
}

}  // extern "C"

// Slots [slot0, slot0 + n) of one (row, layer) from host fp16 [nh][n][D]
// keys and values; the INT8 cache quantises them on the device.
static uocr_status kv_put(uocr_ctx* ctx, int row, int layer, int slot0, int n, const uint16_t* k, const uint16_t* v) {
  const uocr_config& c = ctx->cfg;
  const size_t D = c.head_dim, nh = c.n_heads;
  if (n == 0) return UOCR_OK;
  if (!ctx->kv8) {
    for (int kv = 0; kv < 2; ++kv) {
      const uint16_t* src = kv ? v : k;
      for (size_t h = 0; h < nh; ++h) {
        __half* dst = ctx->kv + ctx->kv_layer * layer + ((((size_t)row * 2 + kv) * nh + h) * ctx->SL + slot0) * D;
        CK(cudaMemcpyAsync(dst, src + h * n * D, (size_t)n * D * 2, cudaMemcpyHostToDevice, ctx->st), "kv copy");
      }
    }
    CK(cudaStreamSynchronize(ctx->st), "kv copy");
    return UOCR_OK;
  }
  const size_t bytes = nh * n * D * 2;
  void* stage = nullptr;
  CK(cudaMalloc(&stage, 2 * bytes), "kv staging allocation");
  uint8_t* st8 = reinterpret_cast<uint8_t*>(stage);
  cudaError_t e = cudaMemcpyAsync(st8, k, bytes, cudaMemcpyHostToDevice, ctx->st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(st8 + bytes, v, bytes, cudaMemcpyHostToDevice, ctx->st);
  if (e == cudaSuccess) {
    KvQuantArgs ka{};
    ka.src16k = reinterpret_cast<const __half*>(st8);
    ka.src16v = reinterpret_cast<const __half*>(st8 + bytes);
    ka.kv8 = ctx->kv8 + ctx->kv_layer * layer;
    ka.kvs = ctx->kvs + ctx->kvs_layer * layer;
    ka.slot0 = slot0;
    ka.nh = c.n_heads;
    ka.D = c.head_dim;
    ka.P = c.prefix_len;
    ka.R = c.ring_len;
    ka.SL = ctx->SL;
    ka.SLp = ctx->SLp;
    ka.kv_row0 = row;
    ka.kv_rstep = 0;
    e = launch_kv_quant(ka, n, ctx->st, false);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->st);
  cudaFree(stage);
  return ctx->cuda(e, "kv quantise");
}

// Slots [slot0, slot0 + n) of one (row, layer) into host fp16 [nh][n][D]
// (the INT8 cache gives scale * code rounded to fp16).
static uocr_status kv_get(uocr_ctx* ctx, int row, int layer, int slot0, int n, uint16_t* k, uint16_t* v) {
  const uocr_config& c = ctx->cfg;
  const size_t D = c.head_dim, nh = c.n_heads;
  CK(cudaStreamSynchronize(ctx->st), "kv read");
  if (n == 0) return UOCR_OK;
  if (!ctx->kv8) {
    for (int kv = 0; kv < 2; ++kv) {
      uint16_t* dst = kv ? v : k;
      for (size_t h = 0; h < nh; ++h) {
        const __half* src = ctx->kv + ctx->kv_layer * layer + ((((size_t)row * 2 + kv) * nh + h) * ctx->SL + slot0) * D;
        CK(cudaMemcpy(dst + h * n * D, src, (size_t)n * D * 2, cudaMemcpyDeviceToHost), "kv read");
      }
    }
    return UOCR_OK;
  }
  const size_t bytes = nh * n * D * 2;
  void* stage = nullptr;
  CK(cudaMalloc(&stage, 2 * bytes), "kv staging allocation");
  __half* sk = reinterpret_cast<__half*>(stage);
  __half* sv = sk + nh * n * D;
  cudaError_t e = launch_kv_dequant(ctx->kv8 + ctx->kv_layer * layer + (size_t)row * 2 * nh * ctx->SL * D,
                                    ctx->kvs + ctx->kvs_layer * layer + (size_t)row * 2 * nh * ctx->SLp, c.n_heads,
                                    c.head_dim, ctx->SL, ctx->SLp, slot0, n, sk, sv, ctx->st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->st);
  if (e == cudaSuccess) e = cudaMemcpy(k, sk, bytes, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(v, sv, bytes, cudaMemcpyDeviceToHost);
  cudaFree(stage);
  return ctx->cuda(e, "kv read");
}

// INT8 cache entries of slots [slot0, slot0 + n) of one (row, layer), exactly:
// codes [nh][n][D] and scales [nh][n] per K and V; `put` writes them, else reads.
static uocr_status kv_i8_io(uocr_ctx* ctx, int row, int layer, int slot0, int n, int8_t* kc, float* ks, int8_t* vc,
                            float* vs, bool put) {
  const uocr_config& c = ctx->cfg;
  const size_t D = c.head_dim, nh = c.n_heads;
  CK(cudaStreamSynchronize(ctx->st), "kv sync");
  for (int kv = 0; kv < 2; ++kv) {
    int8_t* codes = kv ? vc : kc;
    float* scales = kv ? vs : ks;
    for (size_t h = 0; h < nh; ++h) {
      const size_t vec = ((size_t)row * 2 + kv) * nh + h;
      int8_t* dc = ctx->kv8 + ctx->kv_layer * layer + (vec * ctx->SL + slot0) * D;
      float* ds = ctx->kvs + ctx->kvs_layer * layer + vec * ctx->SLp + slot0;
      if (put) {
        CK(cudaMemcpy(dc, codes + h * n * D, (size_t)n * D, cudaMemcpyHostToDevice), "kv write");
        CK(cudaMemcpy(ds, scales + h * n, (size_t)n * 4, cudaMemcpyHostToDevice), "kv write");
      } else {
        CK(cudaMemcpy(codes + h * n * D, dc, (size_t)n * D, cudaMemcpyDeviceToHost), "kv read");
        CK(cudaMemcpy(scales + h * n, ds, (size_t)n * 4, cudaMemcpyDeviceToHost), "kv read");
      }
    }
  }
  return UOCR_OK;
}

extern "C" {

uocr_status uocr_kv_write_prefix(uocr_ctx* ctx, int32_t row, int32_t layer, const uint16_t* k, const uint16_t* v,
                                 int32_t start, int32_t n) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  const uocr_config& c = ctx->cfg;
  if (!k || !v || row < 0 || row >= c.max_rows || layer < 0 || layer >= c.n_layers || start < 0 || n < 0 ||
      start + n > c.prefix_len)
    return ctx->fail(UOCR_E_INVALID_ARG, "kv_write_prefix: bad row/layer/range");
  return kv_put(ctx, row, layer, start, n, k, v);
}

uocr_status uocr_kv_write(uocr_ctx* ctx, int32_t row, int32_t layer, int32_t slot0, int32_t n, const uint16_t* k,
                          const uint16_t* v) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  const uocr_config& c = ctx->cfg;
  if (!k || !v || row < 0 || row >= c.max_rows || layer < 0 || layer >= c.n_layers || slot0 < 0 || n < 0 ||
      slot0 + n > ctx->SL)
    return ctx->fail(UOCR_E_INVALID_ARG, "kv_write: bad row/layer/slot range");
  return kv_put(ctx, row, layer, slot0, n, k, v);
}

uocr_status uocr_kv_read(uocr_ctx* ctx, int32_t row, int32_t layer, int32_t slot0, int32_t n, uint16_t* k,
                         uint16_t* v) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  const uocr_config& c = ctx->cfg;
  if (!k || !v || row < 0 || row >= c.max_rows || layer < 0 || layer >= c.n_layers || slot0 < 0 || n < 0 ||
      slot0 + n > ctx->SL)
    return ctx->fail(UOCR_E_INVALID_ARG, "kv_read: bad row/layer/range");
  return kv_get(ctx, row, layer, slot0, n, k, v);
}

uocr_status uocr_kv_read_i8(uocr_ctx* ctx, int32_t row, int32_t layer, int32_t slot0, int32_t n, int8_t* k_codes,
                            float* k_scales, int8_t* v_codes, float* v_scales) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  const uocr_config& c = ctx->cfg;
  if (!ctx->kv8) return ctx->fail(UOCR_E_STATE, "kv_read_i8: the cache is fp16 (kv_int8 = 0)");
  if (!k_codes || !k_scales || !v_codes || !v_scales || row < 0 || row >= c.max_rows || layer < 0 ||
      layer >= c.n_layers || slot0 < 0 || n < 0 || slot0 + n > ctx->SL)
    return ctx->fail(UOCR_E_INVALID_ARG, "kv_read_i8: bad row/layer/range");
  return kv_i8_io(ctx, row, layer, slot0, n, k_codes, k_scales, v_codes, v_scales, false);
}

uocr_status uocr_kv_write_i8(uocr_ctx* ctx, int32_t row, int32_t layer, int32_t slot0, int32_t n,
                             const int8_t* k_codes, const float* k_scales, const int8_t* v_codes,
                             const float* v_scales) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  const uocr_config& c = ctx->cfg;
  if (!ctx->kv8) return ctx->fail(UOCR_E_STATE, "kv_write_i8: the cache is fp16 (kv_int8 = 0)");
  if (!k_codes || !k_scales || !v_codes || !v_scales || row < 0 || row >= c.max_rows || layer < 0 ||
      layer >= c.n_layers || slot0 < 0 || n < 0 || slot0 + n > ctx->SL)
    return ctx->fail(UOCR_E_INVALID_ARG, "kv_write_i8: bad row/layer/range");
  return kv_i8_io(ctx, row, layer, slot0, n, const_cast<int8_t*>(k_codes), const_cast<float*>(k_scales),
                  const_cast<int8_t*>(v_codes), const_cast<float*>(v_scales), true);
}

uocr_status uocr_set_sinks(uocr_ctx* ctx, const float* sinks) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (!sinks) return ctx->fail(UOCR_E_INVALID_ARG, "sinks is NULL");
  if (!ctx->cfg.use_sink) return ctx->fail(UOCR_E_STATE, "the config has use_sink = 0");
  CK(cudaMemcpy(ctx->sinks, sinks, sizeof(float) * ctx->cfg.n_layers * ctx->cfg.n_heads, cudaMemcpyHostToDevice),
     "sink copy");
  ctx->sinks_set = true;
  return UOCR_OK;
}

static uocr_status step_prologue(uocr_ctx* ctx, int rows) {
  if (rows < 1 || rows > ctx->cfg.max_rows)
    return ctx->fail(UOCR_E_INVALID_ARG, "rows %d outside [1, max_rows = %d]", rows, ctx->cfg.max_rows);
  uocr_status s = check_complete(ctx);
  if (s != UOCR_OK) return s;
  CK(cudaEventRecord(ctx->ev_in, ctx->ust), "event record");
  CK(cudaStreamWaitEvent(ctx->st, ctx->ev_in, 0), "stream wait");
  return UOCR_OK;
}

static uocr_status step_epilogue(uocr_ctx* ctx) {
  CK(cudaEventRecord(ctx->ev_out, ctx->st), "event record");
  CK(cudaStreamWaitEvent(ctx->ust, ctx->ev_out, 0), "stream wait");
  return UOCR_OK;
}

uocr_status uocr_decode_step(uocr_ctx* ctx, int32_t rows, const int32_t* token_ids, const int32_t* positions,
                             int32_t* next_ids, float* logits) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (ctx->cfg.vocab <= 0) return ctx->fail(UOCR_E_STATE, "decode_step needs a vocabulary (use decode_step_embeds)");
  if (!token_ids || !positions || !next_ids) return ctx->fail(UOCR_E_INVALID_ARG, "NULL device pointer");
  uocr_status s = step_prologue(ctx, rows);
  if (s != UOCR_OK) return s;
  CK(cudaMemcpyAsync(ctx->ids_buf, token_ids, rows * 4, cudaMemcpyDeviceToDevice, ctx->st), "ids copy");
  CK(cudaMemcpyAsync(ctx->pos_buf, positions, rows * 4, cudaMemcpyDeviceToDevice, ctx->st), "positions copy");
  s = run_step(ctx, StepShape{rows, true, true, logits != nullptr, false});
  if (s != UOCR_OK) return s;
  CK(cudaMemcpyAsync(next_ids, ctx->next_ids, rows * 4, cudaMemcpyDeviceToDevice, ctx->st), "ids copy");
  if (logits)
    CK(cudaMemcpyAsync(logits, ctx->logits, (size_t)rows * ctx->cfg.vocab * 4, cudaMemcpyDeviceToDevice, ctx->st),
       "logits copy");
  return step_epilogue(ctx);
}

uocr_status uocr_decode_step_embeds(uocr_ctx* ctx, int32_t rows, const uint16_t* x, const int32_t* positions,
                                    float* y, uint16_t* y_f16, int32_t* next_ids, float* logits) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (!x || !positions) return ctx->fail(UOCR_E_INVALID_ARG, "NULL device pointer");
  const bool lm = next_ids != nullptr || logits != nullptr;
  if (lm && ctx->cfg.vocab <= 0) return ctx->fail(UOCR_E_STATE, "next_ids/logits need a vocabulary");
  uocr_status s = step_prologue(ctx, rows);
  if (s != UOCR_OK) return s;
  const int H = ctx->cfg.hidden;
  CK(cudaMemcpyAsync(ctx->x_in, x, (size_t)rows * H * 2, cudaMemcpyDeviceToDevice, ctx->st), "x copy");
  CK(cudaMemcpyAsync(ctx->pos_buf, positions, rows * 4, cudaMemcpyDeviceToDevice, ctx->st), "positions copy");
  s = run_step(ctx, StepShape{rows, false, lm, logits != nullptr, false});
  if (s != UOCR_OK) return s;
  const float* last = ctx->hid + (size_t)2 * ctx->cfg.n_layers * ctx->TC() * H;
  if (y) CK(cudaMemcpyAsync(y, last, (size_t)rows * H * 4, cudaMemcpyDeviceToDevice, ctx->st), "y copy");
  if (y_f16) CK(launch_f32_to_f16(last, reinterpret_cast<__half*>(y_f16), (long long)rows * H, ctx->st), "y_f16");
  if (next_ids) CK(cudaMemcpyAsync(next_ids, ctx->next_ids, rows * 4, cudaMemcpyDeviceToDevice, ctx->st), "ids copy");
  if (logits)
    CK(cudaMemcpyAsync(logits, ctx->logits, (size_t)rows * ctx->cfg.vocab * 4, cudaMemcpyDeviceToDevice, ctx->st),
       "logits copy");
  return step_epilogue(ctx);
}

uocr_status uocr_decode_step_host(uocr_ctx* ctx, int32_t rows, const int32_t* token_ids, const int32_t* positions,
                                  int32_t* next_ids) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (ctx->cfg.vocab <= 0) return ctx->fail(UOCR_E_STATE, "decode_step_host needs a vocabulary");
  if (!token_ids || !positions || !next_ids) return ctx->fail(UOCR_E_INVALID_ARG, "NULL host pointer");
  if (rows < 1 || rows > ctx->cfg.max_rows) return ctx->fail(UOCR_E_INVALID_ARG, "rows out of range");
  uocr_status s = check_complete(ctx);
  if (s != UOCR_OK) return s;
  CK(cudaMemcpyAsync(ctx->ids_buf, token_ids, rows * 4, cudaMemcpyHostToDevice, ctx->st), "ids copy");
  CK(cudaMemcpyAsync(ctx->pos_buf, positions, rows * 4, cudaMemcpyHostToDevice, ctx->st), "positions copy");
  s = run_step(ctx, StepShape{rows, true, true, false, false});
  if (s != UOCR_OK) return s;
  CK(cudaMemcpyAsync(next_ids, ctx->next_ids, rows * 4, cudaMemcpyDeviceToHost, ctx->st), "ids copy");
  CK(cudaStreamSynchronize(ctx->st), "step");
  return UOCR_OK;
}

uocr_status uocr_prefill(uocr_ctx* ctx, int32_t row, const int32_t* token_ids, const uint16_t* x, int32_t n,
                         int32_t start_pos, int32_t* next_id, float* logits) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  const uocr_config& c = ctx->cfg;
  if ((token_ids == nullptr) == (x == nullptr))
    return ctx->fail(UOCR_E_INVALID_ARG, "prefill: give exactly one of token_ids and x");
  if (token_ids && c.vocab <= 0) return ctx->fail(UOCR_E_STATE, "prefill from token ids needs a vocabulary");
  if ((next_id || logits) && c.vocab <= 0) return ctx->fail(UOCR_E_STATE, "next_id/logits need a vocabulary");
  if (row < 0 || row >= c.max_rows) return ctx->fail(UOCR_E_INVALID_ARG, "prefill: row %d outside [0, %d)", row,
                                                     c.max_rows);
  if (n < 1 || start_pos < 0 || (long long)start_pos + n > (long long)ctx->SL)
    return ctx->fail(UOCR_E_INVALID_ARG,
                     "prefill: positions [%d, %d) must lie in [0, prefix_len + ring_len = %d) (no ring wrap)",
                     start_pos, start_pos + n, ctx->SL);
  uocr_status s = check_complete(ctx);
  if (s != UOCR_OK) return s;
  CK(cudaEventRecord(ctx->ev_in, ctx->ust), "event record");
  CK(cudaStreamWaitEvent(ctx->st, ctx->ev_in, 0), "stream wait");
  const int H = c.hidden, TC = ctx->TC();
  for (int off = 0; off < n; off += TC) {
    const int m = n - off < TC ? n - off : TC;
    const bool last = off + m == n;
    if (token_ids)
      CK(cudaMemcpyAsync(ctx->ids_buf, token_ids + off, (size_t)m * 4, cudaMemcpyDeviceToDevice, ctx->st), "ids copy");
    else
      CK(cudaMemcpyAsync(ctx->x_in, x + (size_t)off * H, (size_t)m * H * 2, cudaMemcpyDeviceToDevice, ctx->st),
         "x copy");
    StepShape sh{m, token_ids != nullptr, last && (next_id || logits), last && logits != nullptr, false};
    sh.prefill = true;
    sh.kv_row = row;
    sh.pos_base = start_pos + off;
    s = enqueue_step(ctx, sh, nullptr);
    if (s != UOCR_OK) return s;
  }
  if (next_id) CK(cudaMemcpyAsync(next_id, ctx->next_ids, 4, cudaMemcpyDeviceToDevice, ctx->st), "id copy");
  if (logits)
    CK(cudaMemcpyAsync(logits, ctx->logits, (size_t)c.vocab * 4, cudaMemcpyDeviceToDevice, ctx->st), "logits copy");
  return step_epilogue(ctx);
}

uocr_status uocr_project(uocr_ctx* ctx, int32_t n, const uint16_t* feats, uint16_t* out) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  const uocr_config& c = ctx->cfg;
  if (c.proj_in <= 0) return ctx->fail(UOCR_E_STATE, "project: the config has no projector (proj_in = 0)");
  if (!ctx->loaded.count({UOCR_T_PROJ, 0, 0}) || !ctx->loaded.count({UOCR_T_PROJ_BIAS, 0, 0}))
    return ctx->fail(UOCR_E_STATE, "project: the projector weight and bias have not been loaded");
  if (!feats || !out || n < 1) return ctx->fail(UOCR_E_INVALID_ARG, "project: NULL pointer or n < 1");
  CK(cudaEventRecord(ctx->ev_in, ctx->ust), "event record");
  CK(cudaStreamWaitEvent(ctx->st, ctx->ev_in, 0), "stream wait");
  const int tg = (n + 15) / 16;  // token groups of 16 features (two n-tiles each)
  int gx = ctx->gemv_ctas_per_sm * ctx->n_sm / tg;
  gx = gx < 1 ? 1 : gx > ctx->proj.n_slabs ? ctx->proj.n_slabs : gx;
  GemvArgs pa{};
  pa.w = ctx->proj.view();
  pa.sp = plan_stream(2, ctx->proj.fmt, c.proj_in);
  pa.ntok = n;
  pa.xh = reinterpret_cast<const __half*>(feats);
  pa.ld_src = c.proj_in;
  pa.out_h = reinterpret_cast<__half*>(out);
  pa.ld_out = c.hidden;
  pa.bias = ctx->proj_b;
  pa.status = ctx->status;
  CK(launch_gemv(ctx->proj.fmt, SRC_F16, EPI_BIAS_F16, pa, gx, tg, ctx->st, false), "projector launch");
  return step_epilogue(ctx);
}

uocr_status uocr_debug_wait_probe(uocr_ctx* ctx, int32_t issue_copy) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  // the 16-byte source is the (256-byte aligned) history buffer of the arena
  CK(launch_wait_probe(ctx->hist, issue_copy ? 1 : 0, ctx->status, ctx->st), "wait probe launch");
  return UOCR_OK;
}

uocr_status uocr_generate(uocr_ctx* ctx, int32_t rows, const int32_t* token_ids, const int32_t* positions,
                          int32_t n_steps, int32_t* out_ids) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (ctx->cfg.vocab <= 0) return ctx->fail(UOCR_E_STATE, "generate needs a vocabulary");
  if (!token_ids || !positions || !out_ids || n_steps < 0)
    return ctx->fail(UOCR_E_INVALID_ARG, "NULL device pointer or negative step count");
  uocr_status s = step_prologue(ctx, rows);
  if (s != UOCR_OK) return s;
  CK(cudaMemcpyAsync(ctx->ids_buf, token_ids, rows * 4, cudaMemcpyDeviceToDevice, ctx->st), "ids copy");
  CK(cudaMemcpyAsync(ctx->pos_buf, positions, rows * 4, cudaMemcpyDeviceToDevice, ctx->st), "positions copy");
  for (int done = 0; done < n_steps;) {
    const int n = n_steps - done < kHistCap ? n_steps - done : kHistCap;
    CK(cudaMemsetAsync(ctx->hist_ctr, 0, 4, ctx->st), "history reset");
    for (int i = 0; i < n; ++i) {
      s = run_step(ctx, StepShape{rows, true, true, false, true});
      if (s != UOCR_OK) return s;
    }
    CK(cudaMemcpyAsync(out_ids + (size_t)done * rows, ctx->hist, (size_t)n * rows * 4, cudaMemcpyDeviceToDevice,
                       ctx->st),
       "history copy");
    done += n;
  }
  return step_epilogue(ctx);
}

uocr_status uocr_kv_reset(uocr_ctx* ctx, int32_t row, int32_t keep_prefix) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  const uocr_config& c = ctx->cfg;
  if (row < -1 || row >= c.max_rows) return ctx->fail(UOCR_E_INVALID_ARG, "row out of range");
  const int r0 = row < 0 ? 0 : row, r1 = row < 0 ? c.max_rows : row + 1;
  const int from = keep_prefix ? c.prefix_len : 0;
  for (int l = 0; l < c.n_layers; ++l)
    for (int r = r0; r < r1; ++r) {
      if (!ctx->kv8) {
        __half* base = ctx->kv + ctx->kv_layer * l + (size_t)r * 2 * c.n_heads * ctx->SL * c.head_dim;
        CK(launch_fill_zero_ring(base, c.n_heads, ctx->SL, c.head_dim, from, ctx->st), "kv reset");
        continue;
      }
      for (int vec = 0; vec < 2 * c.n_heads; ++vec) {  // codes and scales of slots [from, SL)
        const size_t v = (size_t)r * 2 * c.n_heads + vec;
        CK(cudaMemsetAsync(ctx->kv8 + ctx->kv_layer * l + (v * ctx->SL + from) * c.head_dim, 0,
                           (size_t)(ctx->SL - from) * c.head_dim, ctx->st),
           "kv reset");
        CK(cudaMemsetAsync(ctx->kvs + ctx->kvs_layer * l + v * ctx->SLp + from, 0, (size_t)(ctx->SL - from) * 4,
                           ctx->st),
           "kv reset");
      }
    }
  return UOCR_OK;
}

uocr_status uocr_sync(uocr_ctx* ctx) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  CK(cudaStreamSynchronize(ctx->st), "sync");
  int st = 0;
  CK(cudaMemcpy(&st, ctx->status, 4, cudaMemcpyDeviceToHost), "status read");
  if (st) {
    CK(cudaMemset(ctx->status, 0, 4), "status clear");
    if (st & kStatusTimeout)
      return ctx->fail(UOCR_E_TIMEOUT, "a kernel's bounded wait for its asynchronous copies ran out");
    if (st & kStatusToken) return ctx->fail(UOCR_E_TOKEN, "a token id was outside [0, vocab)");
    return ctx->fail(UOCR_E_POSITION, "a position was negative");
  }
  return UOCR_OK;
}

const char* uocr_last_error(uocr_ctx* ctx) {
  if (!ctx) return g_create_err.c_str();
  return ctx->err.c_str();
}

uocr_status uocr_memory_report(uocr_ctx* ctx, uocr_mem_report* out) {
  if (!ctx || !out) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  *out = ctx->rep;
  return UOCR_OK;
}

uocr_status uocr_debug_hidden(uocr_ctx* ctx, int32_t tap, int32_t rows, float* out) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  const uocr_config& c = ctx->cfg;
  if (!out || tap < -1 || tap >= 2 * c.n_layers || rows < 1 || rows > ctx->TC())
    return ctx->fail(UOCR_E_INVALID_ARG, "debug_hidden: bad tap/rows");
  CK(cudaStreamSynchronize(ctx->st), "sync");
  CK(cudaMemcpy(out, ctx->hid + (size_t)(tap + 1) * ctx->TC() * c.hidden, (size_t)rows * c.hidden * 4,
                cudaMemcpyDeviceToHost),
     "hidden read");
  return UOCR_OK;
}

uocr_status uocr_debug_router(uocr_ctx* ctx, int32_t layer, int32_t rows, int32_t* idx, float* w, int32_t* count,
                              int32_t* offset, int32_t* perm) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  const uocr_config& c = ctx->cfg;
  if (layer < 0 || layer >= c.n_layers || ctx->layer_dense(layer) || rows < 1 || rows > ctx->TC())
    return ctx->fail(UOCR_E_INVALID_ARG, "debug_router: not a MoE layer or bad rows");
  CK(cudaStreamSynchronize(ctx->st), "sync");
  const size_t MR = ctx->TC(), k = c.top_k, E = c.n_experts;
  if (idx) CK(cudaMemcpy(idx, ctx->r_idx + layer * MR * k, rows * k * 4, cudaMemcpyDeviceToHost), "router read");
  if (w) CK(cudaMemcpy(w, ctx->r_w + layer * MR * k, rows * k * 4, cudaMemcpyDeviceToHost), "router read");
  if (count) CK(cudaMemcpy(count, ctx->r_count + layer * E, E * 4, cudaMemcpyDeviceToHost), "router read");
  if (offset) CK(cudaMemcpy(offset, ctx->r_offset + layer * (E + 1), (E + 1) * 4, cudaMemcpyDeviceToHost), "router read");
  if (perm) CK(cudaMemcpy(perm, ctx->r_perm + layer * MR * k, rows * k * 4, cudaMemcpyDeviceToHost), "router read");
  return UOCR_OK;
}

uocr_status uocr_debug_router_logits(uocr_ctx* ctx, int32_t layer, int32_t rows, float* logits) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  const uocr_config& c = ctx->cfg;
  if (layer < 0 || layer >= c.n_layers || ctx->layer_dense(layer) || rows < 1 || rows > ctx->TC() || !logits)
    return ctx->fail(UOCR_E_INVALID_ARG, "debug_router_logits: not a MoE layer, bad rows or NULL output");
  CK(cudaStreamSynchronize(ctx->st), "sync");
  const size_t MR = ctx->TC(), E = c.n_experts;
  CK(cudaMemcpy(logits, ctx->r_logits + layer * MR * E, rows * E * 4, cudaMemcpyDeviceToHost), "router read");
  return UOCR_OK;
}

uocr_status uocr_profile(uocr_ctx* ctx, int32_t rows, int32_t input_kind, const int32_t* token_ids,
                         const uint16_t* x, const int32_t* positions, const char** names, float* ms,
                         int32_t* n_inout) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  if (!positions || !names || !ms || !n_inout) return ctx->fail(UOCR_E_INVALID_ARG, "NULL pointer");
  const bool ids = input_kind == 0;
  if (ids && (!token_ids || ctx->cfg.vocab <= 0)) return ctx->fail(UOCR_E_INVALID_ARG, "token ids need a vocabulary");
  if (!ids && !x) return ctx->fail(UOCR_E_INVALID_ARG, "x is NULL");
  uocr_status s = step_prologue(ctx, rows);
  if (s != UOCR_OK) return s;
  if (ids)
    CK(cudaMemcpyAsync(ctx->ids_buf, token_ids, rows * 4, cudaMemcpyDeviceToDevice, ctx->st), "ids copy");
  else
    CK(cudaMemcpyAsync(ctx->x_in, x, (size_t)rows * ctx->cfg.hidden * 2, cudaMemcpyDeviceToDevice, ctx->st), "x copy");
  CK(cudaMemcpyAsync(ctx->pos_buf, positions, rows * 4, cudaMemcpyDeviceToDevice, ctx->st), "positions copy");
  const StepShape sh{rows, ids, ctx->cfg.vocab > 0, false, false};
  // one whole step, so that every buffer a class reads holds a real step's values
  s = enqueue_step(ctx, sh, nullptr);
  if (s != UOCR_OK) return s;
  // then each class alone: its launches of one step (every layer, real arguments,
  // programmatic dependent launch between them) captured in a graph and replayed
  constexpr int kReps = 5;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  CK(cudaEventCreate(&e0), "event");
  CK(cudaEventCreate(&e1), "event");
  int n = 0;
  uocr_status out = UOCR_OK;
  for (const char* cls : kClasses) {
    Prof pf;
    pf.only = cls;
    cudaGraph_t g = nullptr;
    cudaGraphExec_t ge = nullptr;
    cudaError_t e = cudaStreamBeginCapture(ctx->st, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
      out = ctx->cuda(e, "profile capture");
      break;
    }
    s = enqueue_step(ctx, sh, &pf);
    e = cudaStreamEndCapture(ctx->st, &g);
    if (s == UOCR_OK && e != cudaSuccess) s = ctx->cuda(e, "profile capture");
    if (s == UOCR_OK && pf.launches > 0) s = ctx->cuda(cudaGraphInstantiate(&ge, g, 0), "profile instantiate");
    if (g) cudaGraphDestroy(g);
    if (s != UOCR_OK) {
      out = s;
      break;
    }
    if (pf.launches == 0) continue;
    float t = 0.f;
    e = cudaGraphLaunch(ge, ctx->st);  // warm-up replay
    if (e == cudaSuccess) e = cudaEventRecord(e0, ctx->st);
    for (int r = 0; r < kReps && e == cudaSuccess; ++r) e = cudaGraphLaunch(ge, ctx->st);
    if (e == cudaSuccess) e = cudaEventRecord(e1, ctx->st);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, e0, e1);
    cudaGraphExecDestroy(ge);
    if (e != cudaSuccess) {
      out = ctx->cuda(e, "profile replay");
      break;
    }
    if (n < *n_inout) {
      names[n] = cls;
      ms[n] = t / kReps;
    }
    ++n;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (out != UOCR_OK) return out;
  *n_inout = n;
  return step_epilogue(ctx);
}

uocr_status uocr_lm_head_argmax_noalloc(uocr_ctx* ctx, int32_t rows, const float* hidden, int32_t* next_ids,
                                        float* logits, void* stream) {
  if (!ctx) return UOCR_E_INVALID_ARG;
  std::lock_guard<std::mutex> lk(ctx->mu);
  const uocr_config& c = ctx->cfg;
  if (c.vocab <= 0) return ctx->fail(UOCR_E_STATE, "lm_head_argmax_noalloc needs a vocabulary");
  if (!hidden || !next_ids) return ctx->fail(UOCR_E_INVALID_ARG, "NULL device pointer");
  if (rows < 1 || rows > kNoAllocMaxRows)
    return ctx->fail(UOCR_E_INVALID_ARG, "rows %d outside [1, %d], the capacity of the static scratch", rows,
                     kNoAllocMaxRows);
  if (rows > 16 && ctx->lm_tc && c.hidden > kNoAllocMaxHidden)
    return ctx->fail(UOCR_E_INVALID_ARG, "rows > 16 need hidden <= %d (the static scratch)", kNoAllocMaxHidden);
  uocr_status s = check_complete(ctx);
  if (s != UOCR_OK) return s;
  unsigned long long* scratch = nullptr;
  CK(noalloc_scratch(c.device, &scratch), "scratch address");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // launch on the context's device, whatever device the calling thread has current
  int prev = 0;
  CK(cudaGetDevice(&prev), "current device");
  if (prev != c.device) CK(cudaSetDevice(c.device), "set device");
  const uocr_status ls = noalloc_launch(ctx, rows, hidden, next_ids, logits, scratch, st);
  if (prev != c.device) CK(cudaSetDevice(prev), "restore device");
  return ls;
}

}  // extern "C"

static uocr_status noalloc_launch(uocr_ctx* ctx, int rows, const float* hidden, int32_t* next_ids, float* logits,
                                  unsigned long long* scratch, cudaStream_t st) {
  const uocr_config& c = ctx->cfg;
  // the keys and the counter must start at zero; a previous call leaves them zero
  // when it completes, but clear them anyway in case it did not
  CK(cudaMemsetAsync(scratch, 0, sizeof(unsigned long long) * (kNoAllocMaxRows + 1), st), "scratch clear");
  if (rows > 16 && ctx->lm_tc) {  // the kernel the decode step runs at this row count
    TcLmArgs ta{};
    ta.w = ctx->lm_tc;
    ta.xc = reinterpret_cast<uint8_t*>(scratch) + kNoAllocKeysBytes;
    ta.x = hidden;
    ta.ld_x = c.hidden;
    ta.norm_w = ctx->final_norm;
    ta.eps = c.rms_eps;
    ta.K = c.hidden;
    ta.V = c.vocab;
    ta.n_mtiles = ctx->lm_mtiles;
    ta.ntok = rows;
    ta.npad = tc_lm_npad(rows);
    ta.logits = logits;
    ta.keys = scratch;
    ta.counter = reinterpret_cast<int*>(scratch + kNoAllocMaxRows);
    ta.next_ids = next_ids;
    ta.status = ctx->status;
    CK(launch_tc_lm(ta, ctx->n_sm, st, false), "tensor-core lm head launch");
    return UOCR_OK;
  }
  const int nt = rows <= 8 ? 1 : 2;
  const int tg = (rows + 15) / 16;
  int gx = ctx->gemv_ctas_per_sm * ctx->n_sm / tg;  // the grid of the step's LM-head launch
  if (gx < 1) gx = 1;
  if (gx > ctx->lm.n_slabs) gx = ctx->lm.n_slabs;
  GemvArgs la{};
  la.w = ctx->lm.view();
  la.sp = plan_stream(nt, F16, c.hidden);
  la.ntok = rows;
  la.status = ctx->status;
  la.xf = hidden;
  la.ld_src = c.hidden;
  la.norm_w = ctx->final_norm;
  la.eps = c.rms_eps;
  la.out_f = logits;
  la.n_valid = c.vocab;
  la.keys = scratch;
  la.counter = reinterpret_cast<int*>(scratch + kNoAllocMaxRows);
  la.next_ids = next_ids;
  CK(launch_gemv(F16, SRC_NORM, EPI_LOGITS, la, gx, tg, st, false), "lm head launch");
  return UOCR_OK;
}
