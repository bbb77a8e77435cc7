// MoE kernels of one decode step.
//
//   router   RMSNorm prologue (the normalised fp16 rows are also written out
//            for the experts) -> fp16 router GEMV (E logits per row); the last
//            CTA to finish takes, per row, the top-k logits (lowest index wins
//            a tie), the softmax weights renormalised over them, then the
//            expert grouping: per-expert counts, exclusive scan, and the
//            permutation of (row, slot) entries grouped by expert ascending,
//            rows ascending, plus the list of experts that received a token.
//   gate/up  one launch over (active expert, slab) items and the shared
//            experts' slabs: each item gathers the rows routed to its expert,
//            streams the expert's gate/up slab once for all of them and writes
//            SwiGLU activations.
//   down     one launch over (active expert, output slab) items and the
//            shared slabs; each item writes fp32 partials; the last item of an
//            output slab (a counter per slab, no waiting) combines them in a
//            fixed order: residual + sum_j w_j * expert_j + shared.
//
// Sources: "Unlimited-OCR on Apple Silicon with C and Metal", "Il decoder e
// il Mixture of Experts" (64 routed experts, top-6, two shared experts;
// compute the routing, group the tokens by expert, run the projections,
// recompose without useless copies) and "Quantizzazione" (dequantisation
// fused into GEMV/GEMM, SwiGLU and the expert combine).
#include <math.h>

#include "launch.h"

namespace uocr {

__device__ __forceinline__ float argmax_key_value(unsigned long long k) {
  const uint32_t u = (uint32_t)(k >> 32);
  const uint32_t b = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(b);
}

// ------------------------------------------------------------------ router
template <int NT>
__global__ void __launch_bounds__(kThreads) k_router(const RouterArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __half* xs = reinterpret_cast<__half*>(smem);
  float* red = reinterpret_cast<float*>(smem + a.sp.red_off);
  float* rs = reinterpret_cast<float*>(smem + a.sp.rs_off);
  __shared__ int s_last;
  __shared__ int s_idx[64 * 8];
  __shared__ int s_cnt[257];

  const int tok0 = blockIdx.y * NT * 8;
  const int ntok = min(a.ntok - tok0, NT * 8);
  const int H = a.H, ldx = a.sp.ldx;
  const float* h = a.h + (size_t)tok0 * H;

  stage_rms(rs, h, H, nullptr, ntok, H, a.eps);
  __syncthreads();
  stage_norm_chunk(xs, ldx, h, H, nullptr, ntok, NT * 8, rs, a.norm_w, 0, H);
  __syncthreads();
  if (blockIdx.x == 0) {  // the experts read these normalised rows
    const int per = H / 8;
    for (int i = threadIdx.x; i < ntok * per; i += kThreads) {
      const int tk = i / per, j = (i - tk * per) * 8;
      *reinterpret_cast<uint4*>(a.xhat + (size_t)(tok0 + tk) * H + j) =
          *reinterpret_cast<const uint4*>(xs + tk * ldx + j);
    }
  }
  for (int s = blockIdx.x; s < a.n_slabs; s += gridDim.x) {
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const uint8_t* wq = reinterpret_cast<const uint8_t*>(a.w) + (size_t)s * a.U * kUnitBytes;
    slab_units<F16, NT>(acc, wq, nullptr, 0, a.U, xs, ldx, 0, nullptr, 0);
    slab_store_partial<NT>(acc, red);
    __syncthreads();
    for (int i = threadIdx.x; i < NT * 64; i += kThreads) {
      const int tok = i >> 3, pg = i & 7;
      if (tok >= ntok) continue;
      float lo, hi;
      slab_sum<NT>(red, tok, pg, lo, hi);
      const int e0 = 16 * s + pg;
      if (e0 < a.E) a.logits[(size_t)(tok0 + tok) * a.E + e0] = lo;
      if (e0 + 8 < a.E) a.logits[(size_t)(tok0 + tok) * a.E + e0 + 8] = hi;
    }
    __syncthreads();
  }

  // ---- the last CTA: top-k, weights, grouping
  if (threadIdx.x == 0) {
    __threadfence();
    const int done = atomicAdd(a.counter, 1);
    s_last = (done == (int)(gridDim.x * gridDim.y) - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = a.ntok, E = a.E, k = a.k;
  for (int r = warp; r < rows; r += kWarps) {
    float v[8];
    bool taken[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane + 32 * j;
      v[j] = e < E ? __ldcg(a.logits + (size_t)r * E + e) : -INFINITY;
      taken[j] = e >= E;
    }
    float l0 = 0.f, wsum = 0.f;
    float lsel[8];
    int isel[8];
    for (int j = 0; j < k; ++j) {
      unsigned long long kb = 0ull;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (!taken[q]) {
          const unsigned long long c = argmax_key(v[q], lane + 32 * q);
          kb = c > kb ? c : kb;
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, kb, o);
        kb = other > kb ? other : kb;
      }
      const int e = argmax_key_index(kb);
      const float le = argmax_key_value(kb);
      if ((e & 31) == lane) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q == (e >> 5)) taken[q] = true;
      }
      if (j == 0) l0 = le;
      isel[j] = e;
      lsel[j] = le;
      wsum += expf(le - l0);
    }
    if (lane == 0) {
      for (int j = 0; j < k; ++j) {
        a.idx[r * k + j] = isel[j];
        a.wts[r * k + j] = expf(lsel[j] - l0) / wsum;
        s_idx[r * k + j] = isel[j];
      }
    }
  }
  __syncthreads();
  const int nent = rows * k;
  for (int e = threadIdx.x; e < E; e += kThreads) {
    int c = 0;
    for (int i = 0; i < nent; ++i) c += (s_idx[i] == e);
    s_cnt[e] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0, na = 0;
    for (int e = 0; e < E; ++e) {
      const int c = s_cnt[e];
      a.count[e] = c;
      a.offset[e] = run;
      if (c > 0) a.active[na++] = e;
      s_cnt[e] = run;  // becomes the exclusive offset
      run += c;
    }
    a.offset[E] = run;
    *a.n_active = na;
    atomicExch(a.counter, 0);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads) {
    int pos = s_cnt[e];
    for (int i = 0; i < nent; ++i) {  // entries i = row*k + slot in row order
      if (s_idx[i] == e) {
        a.perm[pos] = i;
        a.inv[i] = pos;
        ++pos;
      }
    }
  }
}

// ------------------------------------------------------------------ experts
// Item of the gate/up launch: (active expert i, slab) for routed experts,
// then the slabs of the shared experts.
template <int FMT_R, int FMT_S, int NT>
__global__ void __launch_bounds__(kThreads) k_expert_gateup(const ExpertArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __half* xs = reinterpret_cast<__half*>(smem);
  float* xsum = reinterpret_cast<float*>(smem + a.sp.xsum_off);
  float* red = reinterpret_cast<float*>(smem + a.sp.red_off);
  int* srows = reinterpret_cast<int*>(smem + a.sp.rows_off);

  const int n_act = *a.n_active;
  const int items_r = n_act * a.wr.n_slabs;
  const int items = items_r + a.ws.n_slabs;
  const int H = a.H, ldx = a.sp.ldx;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const bool routed = item < items_r;
    int s, cnt, off;
    const uint8_t *wq, *wsc;
    if (routed) {
      const int i = item / a.wr.n_slabs;
      s = item - i * a.wr.n_slabs;
      const int e = a.active[i];
      cnt = a.count[e];
      off = a.offset[e];
      wq = a.wr.q + (size_t)e * a.wr.q_stride + (size_t)s * a.wr.U * kUnitBytes;
      wsc = a.wr.s + (size_t)e * a.wr.s_stride + (size_t)s * a.wr.U * unit_scale_bytes(FMT_R);
    } else {
      s = item - items_r;
      cnt = a.ntok;
      off = 0;
      wq = a.ws.q + (size_t)s * a.ws.U * kUnitBytes;
      wsc = a.ws.s + (size_t)s * a.ws.U * unit_scale_bytes(FMT_S);
    }
    for (int t0 = 0; t0 < cnt; t0 += NT * 8) {
      const int ntok = min(NT * 8, cnt - t0);
      __syncthreads();
      if (threadIdx.x < ntok) srows[threadIdx.x] = routed ? a.perm[off + t0 + threadIdx.x] / a.k : t0 + threadIdx.x;
      __syncthreads();
      stage_f16_chunk(xs, ldx, a.xhat, H, srows, 0, ntok, NT * 8, 0, H);
      const bool i8 = routed ? (FMT_R == I8ASYM) : (FMT_S == I8ASYM);
      if (i8) {
        __syncthreads();
        stage_block_sums(xsum, xs, ldx, NT * 8, H);
      }
      __syncthreads();
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
      if (routed)
        slab_units<FMT_R, NT>(acc, wq, wsc, 0, a.wr.U, xs, ldx, 0, xsum, H / 32);
      else
        slab_units<FMT_S, NT>(acc, wq, wsc, 0, a.ws.U, xs, ldx, 0, xsum, H / 32);
      slab_store_partial<NT>(acc, red);
      __syncthreads();
      for (int i = threadIdx.x; i < NT * 64; i += kThreads) {
        const int tok = i >> 3, pg = i & 7;
        if (tok >= ntok) continue;
        float lo, hi;
        slab_sum<NT>(red, tok, pg, lo, hi);
        const __half v = __float2half_rn(silu(lo) * hi);
        if (routed)
          a.act_r[(size_t)(off + t0 + tok) * a.Ie + 8 * s + pg] = v;
        else
          a.act_s[(size_t)(t0 + tok) * a.Ish + 8 * s + pg] = v;
      }
    }
  }
}

template <int FMT_R, int FMT_S, int NT>
__global__ void __launch_bounds__(kThreads) k_expert_down(const ExpertArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __half* xs = reinterpret_cast<__half*>(smem);
  float* xsum = reinterpret_cast<float*>(smem + a.sp.xsum_off);
  float* red = reinterpret_cast<float*>(smem + a.sp.red_off);
  __shared__ int s_last;

  const int n_act = *a.n_active;
  const int nS = a.H / 16;
  const int items_r = n_act * nS;
  const bool has_shared = a.ws.n_slabs > 0;
  const int items = items_r + (has_shared ? nS : 0);
  const int per_slab = n_act + (has_shared ? 1 : 0);
  const int H = a.H, ldx = a.sp.ldx;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const bool routed = item < items_r;
    int s, cnt, off, K;
    const uint8_t *wq, *wsc;
    const __half* src;
    if (routed) {
      const int i = item / nS;
      s = item - i * nS;
      const int e = a.active[i];
      cnt = a.count[e];
      off = a.offset[e];
      K = a.Ie;
      src = a.act_r;
      wq = a.wr.q + (size_t)e * a.wr.q_stride + (size_t)s * a.wr.U * kUnitBytes;
      wsc = a.wr.s + (size_t)e * a.wr.s_stride + (size_t)s * a.wr.U * unit_scale_bytes(FMT_R);
    } else {
      s = item - items_r;
      cnt = a.ntok;
      off = 0;
      K = a.Ish;
      src = a.act_s;
      wq = a.ws.q + (size_t)s * a.ws.U * kUnitBytes;
      wsc = a.ws.s + (size_t)s * a.ws.U * unit_scale_bytes(FMT_S);
    }
    for (int t0 = 0; t0 < cnt; t0 += NT * 8) {
      const int ntok = min(NT * 8, cnt - t0);
      __syncthreads();
      stage_f16_chunk(xs, ldx, src, K, nullptr, off + t0, ntok, NT * 8, 0, K);
      const bool i8 = routed ? (FMT_R == I8ASYM) : (FMT_S == I8ASYM);
      if (i8) {
        __syncthreads();
        stage_block_sums(xsum, xs, ldx, NT * 8, K);
      }
      __syncthreads();
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
      if (routed)
        slab_units<FMT_R, NT>(acc, wq, wsc, 0, a.wr.U, xs, ldx, 0, xsum, K / 32);
      else
        slab_units<FMT_S, NT>(acc, wq, wsc, 0, a.ws.U, xs, ldx, 0, xsum, K / 32);
      slab_store_partial<NT>(acc, red);
      __syncthreads();
      for (int i = threadIdx.x; i < NT * 64; i += kThreads) {
        const int tok = i >> 3, pg = i & 7;
        if (tok >= ntok) continue;
        float lo, hi;
        slab_sum<NT>(red, tok, pg, lo, hi);
        float* dst = routed ? a.part_r + (size_t)(off + t0 + tok) * H : a.part_s + (size_t)(t0 + tok) * H;
        dst[16 * s + pg] = lo;
        dst[16 * s + pg + 8] = hi;
      }
    }
    // the last item of this output slab combines it
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const int done = atomicAdd(a.slab_counter + s, 1);
      s_last = (done == per_slab - 1);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      for (int i = threadIdx.x; i < a.ntok * 16; i += kThreads) {
        const int r = i >> 4, c = 16 * s + (i & 15);
        float v = a.h[(size_t)r * H + c];
        for (int j = 0; j < a.k; ++j)
          v += a.wts[r * a.k + j] * __ldcg(a.part_r + (size_t)a.inv[r * a.k + j] * H + c);
        if (has_shared) v += __ldcg(a.part_s + (size_t)r * H + c);
        a.out[(size_t)r * H + c] = v;
      }
      if (threadIdx.x == 0) atomicExch(a.slab_counter + s, 0);
    }
  }
}

// ------------------------------------------------------------------ launchers
template <int NT>
static cudaError_t launch_router_nt(const RouterArgs& a, int gy, cudaStream_t st) {
  k_router<NT><<<dim3(a.n_slabs, gy), kThreads, a.sp.bytes, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_router(const RouterArgs& a, int gy, cudaStream_t st) {
  return a.sp.nt == 1 ? launch_router_nt<1>(a, gy, st) : launch_router_nt<2>(a, gy, st);
}

template <int FR, int FS, int NT>
static cudaError_t launch_gu(const ExpertArgs& a, int grid, cudaStream_t st) {
  k_expert_gateup<FR, FS, NT><<<grid, kThreads, a.sp.bytes, st>>>(a);
  return cudaGetLastError();
}
template <int FR, int FS, int NT>
static cudaError_t launch_dn(const ExpertArgs& a, int grid, cudaStream_t st) {
  k_expert_down<FR, FS, NT><<<grid, kThreads, a.sp.bytes, st>>>(a);
  return cudaGetLastError();
}

#define UOCR_EXPERT_DISPATCH(FN)                                                           \
  template <int NT>                                                                        \
  static cudaError_t FN##_nt(int fr, int fs, const ExpertArgs& a, int grid, cudaStream_t st) { \
    if (fr == Q8_0 && fs == Q8_0) return FN<Q8_0, Q8_0, NT>(a, grid, st);                  \
    if (fr == Q4_0 && fs == Q8_0) return FN<Q4_0, Q8_0, NT>(a, grid, st);                  \
    if (fr == Q4_0 && fs == Q4_0) return FN<Q4_0, Q4_0, NT>(a, grid, st);                  \
    if (fr == Q8_0 && fs == Q4_0) return FN<Q8_0, Q4_0, NT>(a, grid, st);                  \
    if (fr == I8ASYM && fs == I8ASYM) return FN<I8ASYM, I8ASYM, NT>(a, grid, st);          \
    return cudaErrorInvalidValue;                                                          \
  }
UOCR_EXPERT_DISPATCH(launch_gu)
UOCR_EXPERT_DISPATCH(launch_dn)
#undef UOCR_EXPERT_DISPATCH

cudaError_t launch_expert_gateup(int fr, int fs, const ExpertArgs& a, int grid, cudaStream_t st) {
  return a.sp.nt == 1 ? launch_gu_nt<1>(fr, fs, a, grid, st) : launch_gu_nt<2>(fr, fs, a, grid, st);
}
cudaError_t launch_expert_down(int fr, int fs, const ExpertArgs& a, int grid, cudaStream_t st) {
  return a.sp.nt == 1 ? launch_dn_nt<1>(fr, fs, a, grid, st) : launch_dn_nt<2>(fr, fs, a, grid, st);
}

template <int FR, int FS, int NT>
static cudaError_t set_expert_attr() {
  const int mx = 200 * 1024;
  cudaError_t e = cudaFuncSetAttribute(k_expert_gateup<FR, FS, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_expert_down<FR, FS, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  return e;
}

cudaError_t init_moe_attributes() {
  const int mx = 200 * 1024;
  cudaError_t e = cudaFuncSetAttribute(k_router<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_router<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
#define UOCR_P(FR, FS)                                  \
  if (e == cudaSuccess) e = set_expert_attr<FR, FS, 1>(); \
  if (e == cudaSuccess) e = set_expert_attr<FR, FS, 2>();
  UOCR_P(Q8_0, Q8_0)
  UOCR_P(Q4_0, Q8_0)
  UOCR_P(Q4_0, Q4_0)
  UOCR_P(Q8_0, Q4_0)
  UOCR_P(I8ASYM, I8ASYM)
#undef UOCR_P
  return e;
}

}  // namespace uocr
