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
// place; only the new token's K/V are produced); "How it is meant to be run"
// (the rows of a step share one read of the weights).
//
// With dynamic int8 activations ("Falcon-OCR INT8 OpenVINO IR": the linear
// layers' inputs quantised per group of 32) the staged rows are int8 codes with
// fp32 scales and the units run on the int8 tensor cores: below 4 rows every
// CTA quantises its rows while staging them (the _I8 sources); from 4 rows
// k_act_quant writes each token group's staging once and the CTAs copy it
// (SRC_I8_COPY).
//
// Each persistent CTA owns slabs blockIdx.x, +gridDim.x, ...; each warp streams
// its units through its own shared-memory ring filled by 16-byte cp.async
// copies, the first ones issued before the CTA waits for the kernel that
// produces its activations.  Up to 16 rows (one token group) share each
// weight read.
#include "launch.h"

namespace uocr {

static int round16(int x) { return (x + 15) / 16 * 16; }

StreamPlan plan_stream(int nt, int fmt, int k_stage, int n_rows_list, int extra_bytes) {
  StreamPlan p{};
  p.nt = nt;
  p.ldx = k_stage > 0 ? k_stage + 8 : 0;
  p.slot = fmt == F16 ? 1024 : 768;
  int off = 0;
  p.xs_off = off;
  off += k_stage > 0 ? round16(nt * 8 * p.ldx * 2) : 0;
  p.red_off = off;
  off += 2 * kWarps * nt * 8 * 16 * 4;  // per-round partials, double-buffered (red_bytes<NT>)
  p.rows_off = off;
  off += round16(n_rows_list * 4);
  p.zero_off = off;
  off += 64;
  p.extra_off = off;
  off += round16(extra_bytes);
  off = (off + 127) / 128 * 128;
  p.ring_off = off;
  off += kWarps * kRingDepth * p.slot;
  p.bytes = off;
  return p;
}

template <int FMT, int NT, int SRC, int EPI>
__global__ void __launch_bounds__(kThreads, kMinBlocks) k_gemv(const GemvArgs a) {
  constexpr bool A8 = SRC == SRC_NORM_I8 || SRC == SRC_F16_I8 || SRC == SRC_I8_COPY;
  constexpr bool NORM = SRC == SRC_NORM || SRC == SRC_NORM_I8;
  extern __shared__ __align__(128) unsigned char smem[];
  const StreamPlan& p = a.sp;
  __shared__ int s_last;
  __shared__ unsigned long long s_best[NT * 8];  // EPI_LOGITS: argmax key per token of this CTA
  __half* xs = reinterpret_cast<__half*>(smem + p.xs_off);
  float* red = reinterpret_cast<float*>(smem + p.red_off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + p.ring_off + (size_t)warp * kRingDepth * p.slot;

  if (!(kPdlLate & PDL_GEMV)) pdl_launch_dependents();
  const int tok0 = blockIdx.y * NT * 8;
  const int ntok = min(a.ntok - tok0, NT * 8);
  const int K = a.w.K;
  const int my_slabs = ((int)blockIdx.x < a.w.n_slabs) ? (a.w.n_slabs - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const SlabWork w = slab_work(blockIdx.x, gridDim.x, my_slabs, a.w.U);
  // the weights do not depend on the previous kernel: start streaming them now
  UnitStream<FMT> us;
  us.start(a.w.q, a.w.s, w);
  us.prefetch(ring, p.slot, w, lane);
  NormW nw;
  if constexpr (SRC == SRC_NORM) load_norm_w(nw, a.norm_w, K);
  (void)nw;

  pdl_wait();  // activations come from the previous kernel
  int* s_pos = reinterpret_cast<int*>(smem + p.rows_off);
  float2* s_rope = reinterpret_cast<float2*>(smem + p.extra_off);  // [NT*8][D/2] (cos, sin)
  if constexpr (EPI == EPI_QKV) {
    for (int i = threadIdx.x; i < ntok; i += blockDim.x) s_pos[i] = max(a.pos[tok0 + i], 0);
    for (int i = threadIdx.x; i < ntok * (a.D / 2); i += blockDim.x) s_rope[i] = a.rope[(size_t)tok0 * (a.D / 2) + i];
  }
  if constexpr (EPI == EPI_LOGITS) {
    if (threadIdx.x < NT * 8) s_best[threadIdx.x] = 0ull;
  }
  if constexpr (SRC == SRC_I8_COPY) {  // written once by k_act_quant for this token group
    stage_bytes(smem + p.xs_off, a.x8 + (size_t)blockIdx.y * act_i8_bytes(NT * 8, K), act_i8_bytes(NT * 8, K));
  } else if constexpr (A8) {  // the int8 staging fits in the fp16 staging area
    stage_act_i8<FMT, NORM>(smem + p.xs_off, NORM ? a.xf + (size_t)tok0 * a.ld_src : nullptr,
                            NORM ? nullptr : a.xh + (size_t)tok0 * a.ld_src, a.ld_src, ntok, NT * 8, a.norm_w, K, a.eps);
  } else if constexpr (SRC == SRC_NORM) {
    stage_norm_rows(xs, p.ldx, a.xf + (size_t)tok0 * a.ld_src, a.ld_src, ntok, NT * 8, a.norm_w, nw, K, a.eps);
  } else {
    stage_f16(xs, p.ldx, a.xh + (size_t)tok0 * a.ld_src, a.ld_src, ntok, NT * 8, K);
  }
  __syncthreads();

  auto epi = [&](int s, const float* rb, int tid, int nthr) {
    for (int i = tid; i < NT * 64; i += nthr) {
      const int tok = i >> 3, pg = i & 7;
      if (tok >= ntok) continue;
      float lo, hi;
      group_sum<NT>(rb, w.ks, tok, pg, lo, hi);
      const int gt = tok0 + tok;
      if constexpr (EPI == EPI_RESID) {
        const int col = 16 * s + pg;
        a.out_f[(size_t)gt * a.ld_out + col] = a.res_in[(size_t)gt * a.ld_out + col] + lo;
        a.out_f[(size_t)gt * a.ld_out + col + 8] = a.res_in[(size_t)gt * a.ld_out + col + 8] + hi;
      } else if constexpr (EPI == EPI_SWIGLU) {
        a.out_h[(size_t)gt * a.ld_out + 8 * s + pg] = __float2half_rn(silu(lo) * hi);
      } else if constexpr (EPI == EPI_BIAS_F16) {
        const int col = 16 * s + pg;
        const float b0 = a.bias ? __half2float(a.bias[col]) : 0.f, b1 = a.bias ? __half2float(a.bias[col + 8]) : 0.f;
        a.out_h[(size_t)gt * a.ld_out + col] = __float2half_rn(lo + b0);
        a.out_h[(size_t)gt * a.ld_out + col + 8] = __float2half_rn(hi + b1);
      } else if constexpr (EPI == EPI_LOGITS) {
        const int r0 = 16 * s + pg, r1 = r0 + 8;
        unsigned long long best = 0ull;
        if (r0 < a.n_valid) {
          if (a.out_f) a.out_f[(size_t)gt * a.n_valid + r0] = lo;
          best = argmax_key(lo, r0);
        }
        if (r1 < a.n_valid) {
          if (a.out_f) a.out_f[(size_t)gt * a.n_valid + r1] = hi;
          const unsigned long long k1 = argmax_key(hi, r1);
          best = k1 > best ? k1 : best;
        }
        if (best != 0ull) atomicMax(&s_best[tok], best);
      } else {  // EPI_QKV
        const int pos = s_pos[tok];  // negative positions are reported by the embedding kernel
        const int pr = 16 * s + pg;
        const int sec = pr / a.S;
        const int wi = pr - sec * a.S;
        const int head = wi / a.D;
        const int js = (wi - head * a.D) >> 4;
        const int dlo = 8 * js + pg, dhi = (a.D >> 1) + dlo;
        float vlo = lo, vhi = hi;
        if (sec < 2) {
          const float2 r = s_rope[tok * (a.D / 2) + dlo];  // (cos, sin) of this position's angle
          vlo = lo * r.x - hi * r.y;
          vhi = hi * r.x + lo * r.y;
        }
        if (sec == 0) {
          float* qo = a.q_out + ((size_t)gt * a.nh + head) * a.D;
          qo[dlo] = vlo;
          qo[dhi] = vhi;
        } else if (a.kv_new) {  // INT8 cache: the quantiser writes the slot
          float* kn = a.kv_new + (((size_t)gt * 2 + (sec - 1)) * a.nh + head) * a.D;
          kn[dlo] = vlo;
          kn[dhi] = vhi;
        } else {
          const int slot = pos < a.P ? pos : a.P + (pos - a.P) % a.R;
          const int kvr = a.kv_row0 + gt * a.kv_rstep;
          __half* c_ = a.kv + ((((size_t)kvr * 2 + (sec - 1)) * a.nh + head) * a.SL + slot) * a.D;
          c_[dlo] = __float2half_rn(vlo);
          c_[dhi] = __float2half_rn(vhi);
        }
      }
    }
  };
  if constexpr (A8) {
    const BSmemI8 bp = make_bsmem_i8(smem + p.xs_off, NT * 8, K);
    run_stream<FMT, NT>(us, w, ring, p.slot, red, bp, NT, epi);
  } else {
    const BSmem bp(xs, p.ldx);
    run_stream<FMT, NT>(us, w, ring, p.slot, red, bp, NT, epi);
  }
  if (kPdlLate & PDL_GEMV) pdl_launch_dependents();

  if constexpr (EPI == EPI_LOGITS) {
    __syncthreads();
    if (threadIdx.x < ntok && s_best[threadIdx.x] != 0ull) atomicMax(a.keys + tok0 + threadIdx.x, s_best[threadIdx.x]);
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const int done = atomicAdd(a.counter, 1);
      s_last = (done == (int)(gridDim.x * gridDim.y) - 1);
    }
    __syncthreads();
    if (s_last) {  // the last CTA: one thread per row writes (and chains) the ids
      __threadfence();
      const int step = a.hist ? *a.hist_ctr : 0;
      for (int t = threadIdx.x; t < a.ntok; t += kThreads) {
        const unsigned long long key = atomicExch(a.keys + t, 0ull);
        const int id = argmax_key_index(key);
        a.next_ids[t] = id;
        if (a.feed_ids) {
          a.feed_ids[t] = id;
          a.feed_pos[t] += 1;
        }
        if (a.hist) a.hist[(size_t)step * a.ntok + t] = id;
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        if (a.hist) *a.hist_ctr = step + 1;
        atomicExch(a.counter, 0);
      }
    }
  }
}

// ------------------------------------------------------------------ int8 staging, once per step
// Row blockIdx.x of the G-row token groups (G = 8 or 16, the rows of a GEMV
// CTA): its K inputs (RMSNorm of fp32 rows rounded to fp16 as the fp16 staging
// rounds them, or fp16 rows) quantised per group of 32 into block blockIdx.x / G
// of `out`, in the layout the GEMV CTAs stage (codes at the units' k order,
// scales and code sums [K/32][G]).
template <int FMT, bool NORM>
__global__ void __launch_bounds__(256) k_act_quant(const GemvArgs a, uint8_t* out, int G) {
  pdl_launch_dependents();
  __shared__ float s_part[8];
  const int row = blockIdx.x, tk = row % G;
  const int K = a.w.K, ng = K / 32, ldq = K + 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* base = out + (size_t)(row / G) * act_i8_bytes(G, K);
  uint8_t* xq = base + (size_t)tk * ldq;
  float* xsc = reinterpret_cast<float*>(base + act_i8_codes_bytes(G, K));
  int* xsm = reinterpret_cast<int*>(xsc + ng * G);
  pdl_wait();  // the source rows come from the previous kernel
  if (row >= a.ntok) {  // a padding row of the last token group
    for (int i = threadIdx.x; i < K / 16; i += blockDim.x) *reinterpret_cast<uint4*>(xq + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < ng; i += blockDim.x) {
      xsc[i * G + tk] = 0.f;
      xsm[i * G + tk] = 0;
    }
    return;
  }
  float r = 1.f;
  if constexpr (NORM) {
    const float4* src = reinterpret_cast<const float4*>(a.xf + (size_t)row * a.ld_src);
    float ss = 0.f;
    for (int f = threadIdx.x; f < K / 4; f += blockDim.x) {
      const float4 v = src[f];
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) s_part[warp] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += s_part[w];
    r = rsqrtf(tot / (float)K + a.eps);
  }
  for (int c = warp; c * kActChunk < K; c += blockDim.x >> 5) {  // 256 inputs per warp pass
    const int k0 = c * kActChunk + 8 * lane;
    const bool on = k0 < K;  // whole groups of 32 (K is a multiple of 32)
    float h[8];
    if constexpr (NORM) {
      const float4* src = reinterpret_cast<const float4*>(a.xf + (size_t)row * a.ld_src + k0);
      const float4 x0 = on ? src[0] : make_float4(0.f, 0.f, 0.f, 0.f), x1 = on ? src[1] : make_float4(0.f, 0.f, 0.f, 0.f);
      const uint4 wv = on ? *reinterpret_cast<const uint4*>(a.norm_w + k0) : make_uint4(0u, 0u, 0u, 0u);
      const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const uint32_t wr[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // fp16(x * r * w), the value the fp16 staging stores
        const __half2 wj = u32_h2(wr[j]);
        const float2 f = __half22float2(__floats2half2_rn(xs[2 * j] * r * __low2float(wj), xs[2 * j + 1] * r * __high2float(wj)));
        h[2 * j] = f.x;
        h[2 * j + 1] = f.y;
      }
    } else {
      const uint4 hv = on ? *reinterpret_cast<const uint4*>(a.xh + (size_t)row * a.ld_src + k0) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t hr[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(u32_h2(hr[j]));
        h[2 * j] = f.x;
        h[2 * j + 1] = f.y;
      }
    }
    const int g = k0 >> 5;
    act_i8_group<FMT>(h, on, xq + 32 * g, xsc + g * G + tk, xsm + g * G + tk);
  }
}

cudaError_t launch_act_quant(int fmt, bool norm, const GemvArgs& a, uint8_t* out, cudaStream_t st, bool pdl) {
  const int G = a.sp.nt * 8;  // the rows of one CTA of the GEMV that copies the blocks
  const dim3 grid((a.ntok + G - 1) / G * G);
#define UOCR_AQ(F_)                                                                                  \
  if (fmt == F_)                                                                                     \
    return norm ? launch_kernel(k_act_quant<F_, true>, grid, dim3(256), 0, st, pdl, a, out, G)        \
                : launch_kernel(k_act_quant<F_, false>, grid, dim3(256), 0, st, pdl, a, out, G);
  UOCR_AQ(Q8_0)
  UOCR_AQ(Q4_0)
  UOCR_AQ(I8ASYM)
#undef UOCR_AQ
  return cudaErrorInvalidValue;
}

template <int FMT, int NT, int SRC, int EPI>
static cudaError_t launch_one(const GemvArgs& a, int gx, int gy, cudaStream_t st, bool pdl) {
  return launch_kernel(k_gemv<FMT, NT, SRC, EPI>, dim3(gx, gy), dim3(kThreads), a.sp.bytes, st, pdl, a);
}

template <int FMT, int NT>
static cudaError_t dispatch_epi(int src, int epi, const GemvArgs& a, int gx, int gy, cudaStream_t st, bool pdl) {
  if (src == SRC_NORM && epi == EPI_QKV) return launch_one<FMT, NT, SRC_NORM, EPI_QKV>(a, gx, gy, st, pdl);
  if (src == SRC_F16 && epi == EPI_RESID) return launch_one<FMT, NT, SRC_F16, EPI_RESID>(a, gx, gy, st, pdl);
  if (src == SRC_NORM && epi == EPI_SWIGLU) return launch_one<FMT, NT, SRC_NORM, EPI_SWIGLU>(a, gx, gy, st, pdl);
  if constexpr (FMT != F16) {
    if (src == SRC_I8_COPY && epi == EPI_QKV) return launch_one<FMT, NT, SRC_I8_COPY, EPI_QKV>(a, gx, gy, st, pdl);
    if (src == SRC_I8_COPY && epi == EPI_RESID) return launch_one<FMT, NT, SRC_I8_COPY, EPI_RESID>(a, gx, gy, st, pdl);
    if (src == SRC_I8_COPY && epi == EPI_SWIGLU) return launch_one<FMT, NT, SRC_I8_COPY, EPI_SWIGLU>(a, gx, gy, st, pdl);
  }
  if constexpr (FMT != F16) {
    if (src == SRC_NORM_I8 && epi == EPI_QKV) return launch_one<FMT, NT, SRC_NORM_I8, EPI_QKV>(a, gx, gy, st, pdl);
    if (src == SRC_F16_I8 && epi == EPI_RESID) return launch_one<FMT, NT, SRC_F16_I8, EPI_RESID>(a, gx, gy, st, pdl);
    if (src == SRC_NORM_I8 && epi == EPI_SWIGLU) return launch_one<FMT, NT, SRC_NORM_I8, EPI_SWIGLU>(a, gx, gy, st, pdl);
  }
  if constexpr (NT == 2 && FMT != F16) {
    if (src == SRC_F16 && epi == EPI_BIAS_F16) return launch_one<FMT, NT, SRC_F16, EPI_BIAS_F16>(a, gx, gy, st, pdl);
  }
  if constexpr (FMT == F16) {
    if (src == SRC_NORM && epi == EPI_LOGITS) return launch_one<FMT, NT, SRC_NORM, EPI_LOGITS>(a, gx, gy, st, pdl);
  }
  return cudaErrorInvalidValue;
}

template <int NT>
static cudaError_t dispatch_fmt(int fmt, int src, int epi, const GemvArgs& a, int gx, int gy, cudaStream_t st,
                                bool pdl) {
  switch (fmt) {
    case F16: return dispatch_epi<F16, NT>(src, epi, a, gx, gy, st, pdl);
    case Q8_0: return dispatch_epi<Q8_0, NT>(src, epi, a, gx, gy, st, pdl);
    case Q4_0: return dispatch_epi<Q4_0, NT>(src, epi, a, gx, gy, st, pdl);
    case I8ASYM: return dispatch_epi<I8ASYM, NT>(src, epi, a, gx, gy, st, pdl);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemv(int fmt, int src, int epi, const GemvArgs& a, int gx, int gy, cudaStream_t st, bool pdl) {
  if (a.sp.nt == 1) return dispatch_fmt<1>(fmt, src, epi, a, gx, gy, st, pdl);
  if (a.sp.nt == 2) return dispatch_fmt<2>(fmt, src, epi, a, gx, gy, st, pdl);
  return cudaErrorInvalidValue;
}

template <int FMT, int NT>
static cudaError_t set_attr_fmt() {
  cudaError_t e = cudaSuccess;
#define UOCR_SET(SRC_, EPI_) \
  if (e == cudaSuccess) e = allow_max_dyn_smem(k_gemv<FMT, NT, SRC_, EPI_>);
  UOCR_SET(SRC_NORM, EPI_QKV)
  UOCR_SET(SRC_F16, EPI_RESID)
  UOCR_SET(SRC_NORM, EPI_SWIGLU)
  if constexpr (FMT != F16) {
    UOCR_SET(SRC_I8_COPY, EPI_QKV)
    UOCR_SET(SRC_I8_COPY, EPI_RESID)
    UOCR_SET(SRC_I8_COPY, EPI_SWIGLU)
  }
  if constexpr (FMT != F16) {
    UOCR_SET(SRC_NORM_I8, EPI_QKV)
    UOCR_SET(SRC_F16_I8, EPI_RESID)
    UOCR_SET(SRC_NORM_I8, EPI_SWIGLU)
  }
  if constexpr (NT == 2 && FMT != F16) {
    UOCR_SET(SRC_F16, EPI_BIAS_F16)
  }
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
