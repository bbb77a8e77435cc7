// Kernel argument structs and launcher declarations shared by the host engine
// (engine.cu) and the kernel translation units.  Internal to the library.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "device_common.cuh"

namespace uocr {

// Shared-memory plan of a streaming CTA: the activation tile xs[nt*8][ldx]
// fp16 (ldx = K + 8), the cross-warp reduction buffer (two slabs), a row
// list, a zero row, a kernel-specific region (extra) and the per-warp weight
// rings (kWarps x kRingDepth slots of `slot` bytes).
struct StreamPlan {
  int nt;
  int ldx;
  int slot;
  int xs_off, red_off, rows_off, zero_off, extra_off, ring_off;
  int bytes;
};

StreamPlan plan_stream(int nt, int fmt, int k_stage, int n_rows_list = 0, int extra_bytes = 0);

// Projection inputs: RMSNorm of fp32 rows, or fp16 rows; the _I8 forms
// quantise them to int8 per group of 32 and run the int8 tensor-core product.
// SRC_I8_COPY: the int8 staging of each 16-row token group was written once by
// k_act_quant (GemvArgs::x8) and is copied, not recomputed, by every CTA.
enum Src : int { SRC_NORM = 0, SRC_F16 = 1, SRC_NORM_I8 = 2, SRC_F16_I8 = 3, SRC_I8_COPY = 4 };
enum Epi : int { EPI_QKV = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_LOGITS = 3, EPI_BIAS_F16 = 4 };

struct GemvArgs {
  PMat w;
  StreamPlan sp;
  int ntok;                 // rows of the step
  // source: fp32 residual rows + RMSNorm weight, or fp16 rows
  const float* xf;
  const __half* xh;
  int ld_src;
  const __half* norm_w;
  float eps;
  const uint8_t* x8;        // SRC_I8_COPY: int8 staging blocks, one per token group of 16 rows
  // outputs
  const float* res_in;      // EPI_RESID: out = res_in + W x
  float* out_f;             // EPI_RESID output / EPI_LOGITS logits (nullable)
  __half* out_h;            // EPI_SWIGLU output; EPI_BIAS_F16: out = fp16(W x + bias)
  const __half* bias;       // EPI_BIAS_F16 [rows of W] or nullptr
  int ld_out;
  // EPI_QKV
  const int* pos;
  float* q_out;             // [rows][nh][D]
  __half* kv;               // layer base [rows][2][nh][SL][D]
  const float2* rope;       // [rows][D/2] (cos, sin) of the step's positions
  int nh, D, S, P, R, SL;
  int kv_row0, kv_rstep;    // token t writes cache row kv_row0 + t * kv_rstep (decode: 0, 1; prefill: row, 0)
  float* kv_new;            // INT8 cache: rotated k and v go here in fp32 [tokens][2][nh][D] (k_kv_quant
                            // quantises them into the cache); nullptr: written to the fp16 cache directly
  // EPI_LOGITS
  int n_valid;              // vocab
  unsigned long long* keys; // [rows]
  int* counter;
  int* next_ids;            // [rows]
  int* feed_ids;            // nullable: chain the argmax into the next step's ids
  int* feed_pos;            //           and advance positions by one
  int* hist;                //           history [steps][rows]
  int* hist_ctr;
  int* status;
};

struct RouterArgs {
  PMat w;                   // packed F16 router [E][H]
  StreamPlan sp;
  int ntok, H, E, k;
  const float* h;           // residual after attention [rows][H]
  const __half* norm_w;
  float eps;
  float* logits;            // out: [rows][E]
  // routing (rank 0 of each cluster, one cluster per token group of 16 rows)
  int tg;                   // token groups
  int by_slot;              // records per active slot (1) or per expert id (0)
  int n_units;              // records per token group
  int* idx;                 // out: [rows][k] chosen experts
  float* wts;               // out: [rows][k] renormalised weights
  int4* rec;                // out: [tg][n_units] {expert or -1, 16-row mask, slot bits 0-31, slot bits 32-47}
  int* status;
};

struct ExpertArgs {
  PMat wr;                  // routed, expert e at q + e*q_stride
  PMat ws;                  // shared experts packed as one (n_slabs == 0: none)
  StreamPlan sp;
  int ntok, E, k, H, Ie, Ish;
  int by_slot;              // routed CTAs by active slot (1) or by expert id (0)
  int n_units;              // routed units of the grid: max active experts (by slot) or E
  int cpe, cpes;            // CTAs per routed unit (expert ids), for the shared experts
  int n_rctas;              // routed CTAs of the grid when units are active slots (>= n_units)
  int tg;                   // token groups of 16 rows (blockIdx.y)
  const int4* rec;          // [tg][n_units] routing records written by the router
  const int* idx;           // [rows][k] chosen experts (router)
  const float* wts;         // [rows][k] renormalised weights (router)
  // grouping: written by the gate/up launch (CTA 0, 0) from idx
  int* count;               // [E]
  int* offset;              // [E+1]
  int* perm;                // [rows*k] entries row*k + slot grouped by expert, rows ascending
  int* inv;                 // [rows*k] position of each entry in perm
  const float* h;           // residual after attention [rows][H] (gate/up input, combine residual)
  const __half* norm_w;     // post-attention RMSNorm weight
  float eps;
  uint8_t* act_r;           // routed SwiGLU activations, B-fragment order, 16 tokens per (expert, group)
  uint8_t* act_s;           // shared SwiGLU activations, B-fragment order over rows, K = Ish
  // down + combine
  float* part_r;            // [rows*k][H] per entry row*k + slot
  float* part_s;            // [rows][H]
  float* out;               // layer output residual [rows][H]
  int* status;
};

struct AttnArgs {
  const float* q;           // [rows][nh][D]
  const __half* kv;         // layer base [rows][2][nh][SL][D] (fp16 cache)
  const int8_t* kv8;        // INT8 cache: codes [rows][2][nh][SL][D] (nullptr: fp16 cache)
  const float* kvs;         //             scales [rows][2][nh][SLp]
  int SLp;                  //             scale slots per (row, K|V, head): SL rounded up to 16
  const int* pos;
  __half* out;              // [rows][nh*D]
  const float* sink;        // [nh] or nullptr
  int nh, D, P, R, SL, nsplit, chunk;
  int kv_row0, kv_rstep;    // token t reads cache row kv_row0 + t * kv_rstep
  int early;                // 1: stage the first K/V blocks before waiting for the QKV kernel
                            //    (decode: only the current slot changes, and it is re-read)
  float scale;
  int* status;
};

// Quantise key / value vectors into the INT8 cache: one CTA per (token, K|V,
// head), one thread per dimension.  src: fp32 [tokens][2][nh][D] (the step's
// new keys and values) or fp16 [nh][n][D] per K and V (a written prefix).
struct KvQuantArgs {
  const float* src32;       // [tokens][2][nh][D], or nullptr
  const __half* src16k;     // [nh][n][D] keys when src32 == nullptr
  const __half* src16v;     // [nh][n][D] values
  int8_t* kv8;              // layer base of the codes [rows][2][nh][SL][D]
  float* kvs;               // layer base of the scales [rows][2][nh][SLp]
  const int* pos;           // [tokens] positions (src32), or nullptr: slots slot0 + t
  int slot0;
  int nh, D, P, R, SL, SLp, kv_row0, kv_rstep;
};

struct EmbedArgs {
  const int* ids;           // nullable (hidden-vector input)
  const __half* x;          // [rows][H] when ids == nullptr
  const __half* emb;        // [V][H]
  int* pos;                 // [rows]; written as pos_base + row when pos_base >= 0 (prefill)
  int pos_base;
  float* out;               // [rows][H]
  int H, V;
  // the step's rotary table: rope[row][j] = (cos, sin) of pos * inv_freq[j]
  const double* inv_freq;   // [half_d]
  float2* rope;             // [rows][half_d]
  int half_d;
  int* status;
};

struct PackArgs {
  uint8_t* q;
  uint8_t* s;
  int fmt, n_slabs, U, K;   // packed format
  int group, bb;            // canonical blocks: values and bytes per block
  int map;                  // PackMap
  const uint8_t* src[8];    // canonical blobs on the device
  int src_rows, src_cols;   // shape of each source
  int nsrc;
  int S, D;                 // MAP_QKV: section rows, head dim
  int I;                    // MAP_SWIGLU: rows per source expert; MAP_KCAT: cols per source
};
enum PackMap : int { MAP_IDENT = 0, MAP_QKV = 1, MAP_SWIGLU = 2, MAP_KCAT = 3 };

// The tensor-core LM head (tc_kernels.cu) for steps of 17..64 rows.
struct TcLmArgs {
  const uint8_t* w;          // canonical fp16 tiles [n_mtiles][K/64][128 x 64]
  uint8_t* xc;               // staged rows, canonical [K/64][npad x 64] fp16
  const float* x;            // residual rows [ntok][ld_x] (final RMSNorm input)
  int ld_x;
  const __half* norm_w;      // final norm weight [K]
  float eps;
  int K, V, n_mtiles, ntok, npad;
  float* logits;             // [ntok][V] or nullptr
  unsigned long long* keys;  // [ntok], zero on entry
  int* counter;
  int* next_ids;
  int* feed_ids;             // nullable: chain into the next step (as GemvArgs)
  int* feed_pos;
  int* hist;
  int* hist_ctr;
  int* status;
};
int tc_lm_npad(int rows);
int tc_lm_smem_bytes(int npad);
cudaError_t launch_tc_lm(const TcLmArgs& a, int n_sm, cudaStream_t st, bool pdl);

// Tensor-core expert kernels (steps with more than 16 rows): shared-memory plan
// of one CTA (A stages, resident B operand of b_bytes, producer rings,
// barriers) within smem_limit bytes; stages < 2 means it does not fit.
struct TcxPlan {
  int stages, a_off, b_off, ring_off, bar_off, bytes;
};
TcxPlan tcx_plan(int b_bytes, int smem_limit);
bool tcx_format_ok(int fr, int fs);  // both Q8_0 / Q4_0 codes
constexpr int kTcxRowsRouted = 16;   // token rows of a routed pass (B columns)
constexpr int kTcxRowsShared = 32;   // ... of a shared-expert pass
// mode 0: gate/up + SwiGLU (activations in the canonical layout, per (expert,
// group) slot of 16 rows for routed experts, per pass of 32 rows for the
// shared ones); mode 1: down -> fp32 partials.  Expert-id units only.
cudaError_t launch_tc_expert(int mode, int fr, int fs, const ExpertArgs& a, const TcxPlan& pl, cudaStream_t st,
                             bool pdl);
cudaError_t launch_pack_canon(const void* src_f16, uint8_t* dst, int V, int K, cudaStream_t st);

// Launch with or without programmatic dependent launch (the kernel may start
// while the previous kernel on the stream finishes; it calls
// griddepcontrol.wait before touching anything that kernel produces).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// The same as a thread-block cluster launch of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                  bool pdl, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Allow a kernel the largest dynamic shared memory the device offers beside
// its own static shared memory.
template <typename... KArgs>
cudaError_t allow_max_dyn_smem(void (*kern)(KArgs...)) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa{};
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
  // all of the unified L1/shared array as shared memory: the streaming kernels
  // keep their weight rings there and bypass L1 for the weights
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  return e;
}

// launchers (return the launch error)
// Int8 staging of a projection's input, once per step: one CTA per row of each
// token group of G = a.sp.nt * 8 rows (rows beyond ntok zero), RMSNorm first
// when norm is set; block g of `out` (act_i8_bytes(G, K) bytes) is what the
// GEMV CTAs of token group g stage.  Reads the source fields of `a` (K = a.w.K).
cudaError_t launch_act_quant(int fmt, bool norm, const GemvArgs& a, uint8_t* out, cudaStream_t st, bool pdl);
int attn_ctas_per_sm(int D, bool int8_cache);  // resident attention CTAs per SM (occupancy)
cudaError_t launch_gemv(int fmt, int src, int epi, const GemvArgs& a, int grid_x, int grid_y, cudaStream_t st,
                        bool pdl);
// grid (cluster, token groups); cluster = min(8, router slabs) CTAs per token group
cudaError_t launch_router(const RouterArgs& a, cudaStream_t st, bool pdl);
int router_cluster(int n_slabs);
cudaError_t launch_expert_gateup(int fmt_r, int fmt_s, const ExpertArgs& a, cudaStream_t st, bool pdl);
cudaError_t launch_expert_down(int fmt_r, int fmt_s, const ExpertArgs& a, cudaStream_t st, bool pdl);
cudaError_t launch_expert_combine(const ExpertArgs& a, cudaStream_t st, bool pdl);
cudaError_t launch_attn(const AttnArgs& a, int rows, cudaStream_t st, bool pdl);
cudaError_t launch_embed(const EmbedArgs& a, int rows, cudaStream_t st);
cudaError_t launch_pack(const PackArgs& a, cudaStream_t st);
cudaError_t launch_fill_zero_ring(__half* kv_layer_row, int nh, int SL, int D, int from_slot, cudaStream_t st);
cudaError_t launch_f32_to_f16(const float* src, __half* dst, long long n, cudaStream_t st);
cudaError_t launch_kv_quant(const KvQuantArgs& a, int tokens, cudaStream_t st, bool pdl);
cudaError_t launch_kv_dequant(const int8_t* kv8, const float* kvs, int nh, int D, int SL, int SLp, int slot0, int n,
                              __half* k_out, __half* v_out, cudaStream_t st);
int attn8_smem_bytes(int D);
// A bounded mbarrier wait on a copy of 16 bytes from src that is issued only
// when `issue` is set; a wait that runs out sets kStatusTimeout in *status.
cudaError_t launch_wait_probe(const void* src, int issue, int* status, cudaStream_t st);
cudaError_t init_kernel_attributes();
int attn_smem_bytes(int D);

}  // namespace uocr
