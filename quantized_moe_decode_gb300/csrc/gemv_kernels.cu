// Fused dequant GEMV kernels of the dense projections of one decode step:
//   QKV   RMSNorm prologue -> W_qkv x -> RoPE -> q out, k/v written in place
//         at the cache slot of the position (prefix slot or ring slot);
//   O     attention output -> W_o -> + residual;
//   MLP   RMSNorm -> interleaved gate/up -> SwiGLU -> fp16 activations;
//   down  activations -> W_down -> + residual;
//   LM    final RMSNorm -> fp16 LM head -> fp32 logits (optional store) and a
//         vocab-parallel argmax (per-CTA best -> 64-bit atomicMax -> the last
//         CTA writes the ids).
//
// Sources: "Unlimited-OCR on Apple Silicon with C and Metal" ("Il decoder e
// il Mixture of Experts": KV append, 128-token ring, argmax over the language
// head; "Quantizzazione": dequantisation fused into GEMV/SwiGLU/argmax);
// "Falcon-OCR INT8 OpenVINO IR" intro (the cache is an input written in
// place; only the new token's K/V are produced).
//
// Every CTA stages the (normalised) activations of up to 16 rows in shared
// memory once, then streams the weight slabs it owns; all rows of the step
// share that single weight read ("How it is meant to be run": rows share the
// weight read).
#include "launch.h"

namespace uocr {

StagePlan plan_stage(int nt, int K, int fmt) {
  StagePlan p{};
  p.nt = nt;
  const int ntp = nt * 8;
  const int budget = 80 * 1024;
  int kcmax = budget / (ntp * 2) - 8;
  kcmax = (kcmax / 64) * 64;
  p.kc = K < kcmax ? K : kcmax;
  p.ldx = p.kc + 8;
  int off = ((ntp * p.ldx * 2 + 15) / 16) * 16;
  p.xsum_off = off;
  if (fmt == I8ASYM) off += ntp * (p.kc / 32) * 4;
  p.red_off = off;
  off += kWarps * ntp * 16 * 4;
  p.rs_off = off;
  off += 64 * 4;
  p.rows_off = off;
  off += 64 * 4;
  p.bytes = off;
  return p;
}

template <int FMT, int NT, int SRC>
__device__ __forceinline__ void stage_chunk(const GemvArgs& a, __half* xs, float* xsum, const float* rs, int tok0,
                                            int ntok, int k0, int kc) {
  if constexpr (SRC == SRC_NORM) {
    stage_norm_chunk(xs, a.sp.ldx, a.xf + (size_t)tok0 * a.ld_src, a.ld_src, nullptr, ntok, NT * 8, rs, a.norm_w,
                     k0, kc);
  } else {
    stage_f16_chunk(xs, a.sp.ldx, a.xh, a.ld_src, nullptr, tok0, ntok, NT * 8, k0, kc);
  }
  if constexpr (FMT == I8ASYM) {
    __syncthreads();
    stage_block_sums(xsum, xs, a.sp.ldx, NT * 8, kc);
  }
}

template <int FMT, int NT, int SRC, int EPI>
__global__ void __launch_bounds__(kThreads) k_gemv(const GemvArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __half* xs = reinterpret_cast<__half*>(smem);
  float* xsum = reinterpret_cast<float*>(smem + a.sp.xsum_off);
  float* red = reinterpret_cast<float*>(smem + a.sp.red_off);
  float* rs = reinterpret_cast<float*>(smem + a.sp.rs_off);
  __shared__ int s_last;

  constexpr int KU = unit_k(FMT);
  constexpr int SB = unit_scale_bytes(FMT);
  const int tok0 = blockIdx.y * NT * 8;
  const int ntok = min(a.ntok - tok0, NT * 8);
  const int K = a.w.K, U = a.w.U, kc = a.sp.kc;
  const bool single = (kc >= K);

  if constexpr (SRC == SRC_NORM) {
    stage_rms(rs, a.xf + (size_t)tok0 * a.ld_src, a.ld_src, nullptr, ntok, K, a.eps);
    __syncthreads();
  }
  if (single) {
    stage_chunk<FMT, NT, SRC>(a, xs, xsum, rs, tok0, ntok, 0, K);
    __syncthreads();
  }

  unsigned long long best = 0ull;  // EPI_LOGITS: running argmax key of (token, pg)

  for (int s = blockIdx.x; s < a.w.n_slabs; s += gridDim.x) {
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const uint8_t* wq = a.w.q + (size_t)s * U * kUnitBytes;
    const uint8_t* ws = a.w.s + (size_t)s * U * SB;
    if (single) {
      slab_units<FMT, NT>(acc, wq, ws, 0, U, xs, a.sp.ldx, 0, xsum, K / 32);
    } else {
      for (int k0 = 0; k0 < K; k0 += kc) {
        const int kcc = min(kc, K - k0);
        __syncthreads();
        stage_chunk<FMT, NT, SRC>(a, xs, xsum, rs, tok0, ntok, k0, kcc);
        __syncthreads();
        slab_units<FMT, NT>(acc, wq, ws, k0 / KU, (k0 + kcc) / KU, xs, a.sp.ldx, k0, xsum, kcc / 32);
      }
    }
    slab_store_partial<NT>(acc, red);
    __syncthreads();
    for (int i = threadIdx.x; i < NT * 64; i += kThreads) {
      const int tok = i >> 3, pg = i & 7;
      if (tok >= ntok) continue;
      float lo, hi;
      slab_sum<NT>(red, tok, pg, lo, hi);
      const int gt = tok0 + tok;
      if constexpr (EPI == EPI_RESID) {
        const int c = 16 * s + pg;
        a.out_f[(size_t)gt * a.ld_out + c] = a.res_in[(size_t)gt * a.ld_out + c] + lo;
        a.out_f[(size_t)gt * a.ld_out + c + 8] = a.res_in[(size_t)gt * a.ld_out + c + 8] + hi;
      } else if constexpr (EPI == EPI_SWIGLU) {
        a.out_h[(size_t)gt * a.ld_out + 8 * s + pg] = __float2half_rn(silu(lo) * hi);
      } else if constexpr (EPI == EPI_LOGITS) {
        const int r0 = 16 * s + pg, r1 = r0 + 8;
        if (r0 < a.n_valid) {
          if (a.out_f) a.out_f[(size_t)gt * a.n_valid + r0] = lo;
          const unsigned long long k0 = argmax_key(lo, r0);
          best = k0 > best ? k0 : best;
        }
        if (r1 < a.n_valid) {
          if (a.out_f) a.out_f[(size_t)gt * a.n_valid + r1] = hi;
          const unsigned long long k1 = argmax_key(hi, r1);
          best = k1 > best ? k1 : best;
        }
      } else {  // EPI_QKV
        int p = a.pos[gt];
        if (p < 0) p = 0;  // reported by the embedding kernel
        const int pr = 16 * s + pg;
        const int sec = pr / a.S;
        const int wi = pr - sec * a.S;
        const int head = wi / a.D;
        const int js = (wi - head * a.D) >> 4;
        const int dlo = 8 * js + pg, dhi = (a.D >> 1) + dlo;
        float vlo = lo, vhi = hi;
        if (sec < 2) {
          double ang = (double)p * a.inv_freq[dlo];
          ang -= 6.283185307179586 * rint(ang * 0.15915494309189535);
          float sn, cs;
          sincosf((float)ang, &sn, &cs);
          vlo = lo * cs - hi * sn;
          vhi = hi * cs + lo * sn;
        }
        if (sec == 0) {
          float* qo = a.q_out + ((size_t)gt * a.nh + head) * a.D;
          qo[dlo] = vlo;
          qo[dhi] = vhi;
        } else {
          const int slot = p < a.P ? p : a.P + (p - a.P) % a.R;
          __half* c = a.kv + ((((size_t)gt * 2 + (sec - 1)) * a.nh + head) * a.SL + slot) * a.D;
          c[dlo] = __float2half_rn(vlo);
          c[dhi] = __float2half_rn(vhi);
        }
      }
    }
    __syncthreads();
  }

  if constexpr (EPI == EPI_LOGITS) {
    // best over the 8 threads (consecutive lanes) of each token, then one atomic per token
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    const int tok = threadIdx.x >> 3;
    if ((threadIdx.x & 7) == 0 && tok < ntok && best != 0ull) atomicMax(a.keys + tok0 + tok, best);
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const int done = atomicAdd(a.counter, 1);
      s_last = (done == (int)(gridDim.x * gridDim.y) - 1);
    }
    __syncthreads();
    if (s_last && threadIdx.x == 0) {
      __threadfence();
      const int step = a.hist ? *a.hist_ctr : 0;
      for (int t = 0; t < a.ntok; ++t) {
        const unsigned long long key = atomicExch(a.keys + t, 0ull);
        const int id = argmax_key_index(key);
        a.next_ids[t] = id;
        if (a.feed_ids) {
          a.feed_ids[t] = id;
          a.feed_pos[t] += 1;
        }
        if (a.hist) a.hist[(size_t)step * a.ntok + t] = id;
      }
      if (a.hist) *a.hist_ctr = step + 1;
      atomicExch(a.counter, 0);
    }
  }
}

template <int FMT, int NT, int SRC, int EPI>
static cudaError_t launch_one(const GemvArgs& a, int gx, int gy, cudaStream_t st) {
  k_gemv<FMT, NT, SRC, EPI><<<dim3(gx, gy), kThreads, a.sp.bytes, st>>>(a);
  return cudaGetLastError();
}

template <int FMT, int NT>
static cudaError_t dispatch_epi(int src, int epi, const GemvArgs& a, int gx, int gy, cudaStream_t st) {
  if (src == SRC_NORM && epi == EPI_QKV) return launch_one<FMT, NT, SRC_NORM, EPI_QKV>(a, gx, gy, st);
  if (src == SRC_F16 && epi == EPI_RESID) return launch_one<FMT, NT, SRC_F16, EPI_RESID>(a, gx, gy, st);
  if (src == SRC_NORM && epi == EPI_SWIGLU) return launch_one<FMT, NT, SRC_NORM, EPI_SWIGLU>(a, gx, gy, st);
  if constexpr (FMT == F16) {
    if (src == SRC_NORM && epi == EPI_LOGITS) return launch_one<FMT, NT, SRC_NORM, EPI_LOGITS>(a, gx, gy, st);
  }
  return cudaErrorInvalidValue;
}

template <int NT>
static cudaError_t dispatch_fmt(int fmt, int src, int epi, const GemvArgs& a, int gx, int gy, cudaStream_t st) {
  switch (fmt) {
    case F16: return dispatch_epi<F16, NT>(src, epi, a, gx, gy, st);
    case Q8_0: return dispatch_epi<Q8_0, NT>(src, epi, a, gx, gy, st);
    case Q4_0: return dispatch_epi<Q4_0, NT>(src, epi, a, gx, gy, st);
    case I8ASYM: return dispatch_epi<I8ASYM, NT>(src, epi, a, gx, gy, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemv(int fmt, int src, int epi, const GemvArgs& a, int gx, int gy, cudaStream_t st) {
  if (a.sp.nt == 1) return dispatch_fmt<1>(fmt, src, epi, a, gx, gy, st);
  if (a.sp.nt == 2) return dispatch_fmt<2>(fmt, src, epi, a, gx, gy, st);
  return cudaErrorInvalidValue;
}

template <int FMT, int NT>
static cudaError_t set_attr_fmt() {
  const int mx = 200 * 1024;
  cudaError_t e = cudaSuccess;
#define UOCR_SET(SRC_, EPI_)                                                                                    \
  if (e == cudaSuccess)                                                                                         \
    e = cudaFuncSetAttribute(k_gemv<FMT, NT, SRC_, EPI_>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  UOCR_SET(SRC_NORM, EPI_QKV)
  UOCR_SET(SRC_F16, EPI_RESID)
  UOCR_SET(SRC_NORM, EPI_SWIGLU)
  if constexpr (FMT == F16) {
    UOCR_SET(SRC_NORM, EPI_LOGITS)
  }
#undef UOCR_SET
  return e;
}

cudaError_t init_gemv_attributes() {
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess) e = set_attr_fmt<F16, 1>();
  if (e == cudaSuccess) e = set_attr_fmt<Q8_0, 1>();
  if (e == cudaSuccess) e = set_attr_fmt<Q4_0, 1>();
  if (e == cudaSuccess) e = set_attr_fmt<I8ASYM, 1>();
  if (e == cudaSuccess) e = set_attr_fmt<F16, 2>();
  if (e == cudaSuccess) e = set_attr_fmt<Q8_0, 2>();
  if (e == cudaSuccess) e = set_attr_fmt<Q4_0, 2>();
  if (e == cudaSuccess) e = set_attr_fmt<I8ASYM, 2>();
  return e;
}

}  // namespace uocr
