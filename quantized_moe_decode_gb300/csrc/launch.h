// Kernel argument structs and launcher declarations shared by the host engine
// (engine.cu) and the kernel translation units.  Internal to the library.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"

namespace uocr {

// Shared-memory plan of a GEMV-family CTA: activation tile xs[NT*8][ldx]
// fp16 (kc inputs staged at a time), I8ASYM block sums, cross-warp
// reduction buffer and per-token norm factors.
struct StagePlan {
  int nt;        // n-tiles of 8 tokens per CTA (1 or 2)
  int kc;        // inputs staged per chunk (multiple of 64, == K when it fits)
  int ldx;       // kc + 8
  int xsum_off;  // byte offsets into dynamic shared memory
  int red_off;
  int rs_off;
  int rows_off;
  int bytes;
};

StagePlan plan_stage(int nt, int K, int fmt);

enum Src : int { SRC_NORM = 0, SRC_F16 = 1 };
enum Epi : int { EPI_QKV = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_LOGITS = 3 };

struct GemvArgs {
  PMat w;
  StagePlan sp;
  int ntok;                 // rows of the step
  // source: fp32 residual rows + RMSNorm weight, or fp16 rows
  const float* xf;
  const __half* xh;
  int ld_src;
  const __half* norm_w;
  float eps;
  // outputs
  const float* res_in;      // EPI_RESID: out = res_in + W x
  float* out_f;             // EPI_RESID output / EPI_LOGITS logits (nullable)
  __half* out_h;            // EPI_SWIGLU output
  int ld_out;
  // EPI_QKV
  const int* pos;
  float* q_out;             // [rows][nh][D]
  __half* kv;               // layer base [rows][2][nh][SL][D]
  const double* inv_freq;   // [D/2]
  int nh, D, S, P, R, SL;
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
  const __half* w;          // packed F16 router [E][H]
  int n_slabs, U;
  StagePlan sp;
  int ntok, H, E, k;
  const float* h;           // residual after attention [rows][H]
  const __half* norm_w;
  float eps;
  __half* xhat;             // out: normed fp16 rows [rows][H]
  float* logits;            // out: [rows][E]
  int* idx;                 // out: [rows][k]
  float* wts;               // out: [rows][k]
  int* count;               // out: [E]
  int* offset;              // out: [E+1]
  int* perm;                // out: [rows*k]
  int* inv;                 // out: [rows*k] position of entry row*k+slot in perm
  int* active;              // out: [E] experts with count > 0, ascending
  int* n_active;            // out
  int* counter;
};

struct ExpertArgs {
  PMat wr;                  // routed, expert e at q + e*q_stride
  PMat ws;                  // shared experts packed as one (n_slabs == 0: none)
  StagePlan sp;
  int ntok, k, H, Ie, Ish;
  const __half* xhat;       // gate/up input [rows][H]
  const int* count;
  const int* offset;
  const int* perm;
  const int* active;
  const int* n_active;
  __half* act_r;            // [rows*k][Ie]   (gate/up out, down in)
  __half* act_s;            // [rows][Ish]
  // down + combine
  float* part_r;            // [rows*k][H]
  float* part_s;            // [rows][H]
  const float* h;           // residual after attention
  const float* wts;         // [rows][k]
  const int* inv;           // [rows*k]
  float* out;               // layer output residual [rows][H]
  int* slab_counter;        // [H/16]
};

struct AttnArgs {
  const float* q;           // [rows][nh][D]
  const __half* kv;         // layer base [rows][2][nh][SL][D]
  const int* pos;
  float* part;              // [rows][nh][nsplit][D+2]
  int* counter;             // [rows][nh]
  __half* out;              // [rows][nh*D]
  const float* sink;        // [nh] or nullptr
  int nh, D, P, R, SL, nsplit, chunk;
  float scale;
};

struct EmbedArgs {
  const int* ids;           // nullable (hidden-vector input)
  const __half* x;          // [rows][H] when ids == nullptr
  const __half* emb;        // [V][H]
  const int* pos;
  float* out;               // [rows][H]
  int H, V;
  int* status;
};

struct PackArgs {
  uint8_t* q;
  uint8_t* s;
  int fmt, n_slabs, U, K;
  int map;                  // PackMap
  const uint8_t* src[8];    // canonical blobs on the device
  int src_rows, src_cols;   // shape of each source
  int nsrc;
  int S, D;                 // MAP_QKV: section rows, head dim
  int I;                    // MAP_SWIGLU: rows per source expert; MAP_KCAT: cols per source
};
enum PackMap : int { MAP_IDENT = 0, MAP_QKV = 1, MAP_SWIGLU = 2, MAP_KCAT = 3 };

// launchers (return cudaGetLastError())
cudaError_t launch_gemv(int fmt, int src, int epi, const GemvArgs& a, int grid_x, int grid_y, cudaStream_t st);
cudaError_t launch_router(const RouterArgs& a, int grid_y, cudaStream_t st);
cudaError_t launch_expert_gateup(int fmt_r, int fmt_s, const ExpertArgs& a, int grid, cudaStream_t st);
cudaError_t launch_expert_down(int fmt_r, int fmt_s, const ExpertArgs& a, int grid, cudaStream_t st);
cudaError_t launch_attn(const AttnArgs& a, int rows, cudaStream_t st);
cudaError_t launch_embed(const EmbedArgs& a, int rows, cudaStream_t st);
cudaError_t launch_pack(const PackArgs& a, cudaStream_t st);
cudaError_t launch_fill_zero_ring(__half* kv_layer_row, int nh, int SL, int D, int from_slot, cudaStream_t st);
cudaError_t init_kernel_attributes();

}  // namespace uocr
