// Split-K flash-decoding attention over the prefix + ring KV cache, and the
// small kernels around the step (embedding gather, weight packer, ring reset).
//
// Attention ("Unlimited-OCR on Apple Silicon with C and Metal", "Il decoder e
// il Mixture of Experts": KV append and a 128-token ring for generated
// tokens; "Falcon-OCR INT8 OpenVINO IR", intro: the sink is one more key
// whose logit is the sink and whose value is zero, and the cache is read in
// place).  For a row at position p the valid slots are a contiguous range:
// [0, p] while p < P, else [0, P + min(p - P + 1, R)) (every ring slot
// written for this sequence; softmax does not care about their order).  CTA
// (split, head, row) takes one chunk of that range, staged by TMA bulk copies;
// each warp reads 4*G slots per iteration (D/8 lanes per slot) and keeps an
// online softmax.  The splits of a (row, head) form a thread-block cluster:
// each keeps its partial in shared memory, and after a cluster barrier every
// CTA merges one slice of D from all partials with their log-sum-exp weights
// and the sink, and writes the fp16 output.
#include <cooperative_groups.h>
#include <math.h>

#include "launch.h"

namespace uocr {

// Slots per shared-memory stage: 16 KB of keys and 16 KB of values.
template <int D>
struct AttnCfg {
  static constexpr int SUB = 8192 / D;
  static constexpr int STAGE = 2 * SUB * D * 2;  // K then V
};

int attn_smem_bytes(int D) { return 2 * (2 * (8192 / D) * D * 2) + 64; }

template <int D>
__global__ void __launch_bounds__(UOCR_ATTN_WARPS * 32) k_attn(const AttnArgs a) {
  constexpr int LPS = D / 8;    // lanes per slot
  constexpr int G = 32 / LPS;   // slots per load instruction
  constexpr int SPI = 4 * G;    // slots per warp iteration
  constexpr int NW = UOCR_ATTN_WARPS;
  constexpr int SUB = AttnCfg<D>::SUB, STAGE = AttnCfg<D>::STAGE;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 2 * STAGE);
  __shared__ float sm_m[NW], sm_l[NW];
  __shared__ float sm_acc[NW][D];
  __shared__ float s_part[D + 2];

  const int split = blockIdx.x, head = blockIdx.y, row = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPS, li = lane % LPS;
  // positions come from a copy that completed before the step's first kernel
  int p = a.pos[row];
  if (p < 0) p = 0;
  const int n_valid = (p < a.P) ? p + 1 : a.P + min(p - a.P + 1, a.R);
  const int s_begin = split * a.chunk;
  const int s_end = min(n_valid, s_begin + a.chunk);
  const int n_sub = s_end > s_begin ? (s_end - s_begin + SUB - 1) / SUB : 0;
  const int kvr = a.kv_row0 + row * a.kv_rstep;
  const __half* Kg = a.kv + (((size_t)kvr * 2 + 0) * a.nh + head) * (size_t)a.SL * D;
  const __half* Vg = a.kv + (((size_t)kvr * 2 + 1) * a.nh + head) * (size_t)a.SL * D;
  auto issue = [&](int sb) {
    const int s0 = s_begin + sb * SUB, n = min(SUB, s_end - s0);
    uint8_t* st = smem + (sb & 1) * STAGE;
    uint64_t* b = bar + (sb & 1);
    mbar_expect_tx(b, 2u * n * D * 2);
    bulk_g2s(st, Kg + (size_t)s0 * D, n * D * 2, b);
    bulk_g2s(st + SUB * D * 2, Vg + (size_t)s0 * D, n * D * 2, b);
  };
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_init(bar + 1, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // decode: every slot but the current token's was written by earlier steps, so
  // stream them now (the current slot is re-read below); a prefill chunk writes
  // many slots, so its copies start once the QKV kernel has finished
  if (a.early && threadIdx.x == 0)
    for (int sb = 0; sb < n_sub && sb < 2; ++sb) issue(sb);
  if (!(kPdlLate & PDL_ATTN)) pdl_launch_dependents();
  pdl_wait();  // q and the current slot come from the QKV kernel
  if (!a.early && threadIdx.x == 0)
    for (int sb = 0; sb < n_sub && sb < 2; ++sb) issue(sb);

  float qv[8];
  {
    const float* qp = a.q + ((size_t)row * a.nh + head) * D + 8 * li;
#pragma unroll
    for (int i = 0; i < 8; ++i) qv[i] = qp[i] * a.scale;
  }
  const int cur = p < a.P ? p : a.P + (p - a.P) % a.R;

  float m = -INFINITY, l = 0.f;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;

  for (int sb = 0; sb < n_sub; ++sb) {
    const int s0 = s_begin + sb * SUB, n = min(SUB, s_end - s0);
    int bad = 0;
    if (threadIdx.x == 0) {
      bad = !mbar_wait(bar + (sb & 1), (uint32_t)((sb >> 1) & 1));
      if (bad) atomicOr(a.status, kStatusTimeout);
    }
    if (__syncthreads_or(bad)) {
      // the status word reports it; wait (bounded) for the copy still in flight, then
      // join the cluster merge with what has been accumulated
      if (threadIdx.x == 0 && sb + 1 < n_sub) mbar_wait(bar + ((sb + 1) & 1), (uint32_t)(((sb + 1) >> 1) & 1));
      break;
    }
    const __half* Ks = reinterpret_cast<const __half*>(smem + (sb & 1) * STAGE);
    const __half* Vs = Ks + SUB * D;
    if (cur >= s0 && cur < s0 + n) {  // the row this step just wrote
      for (int i = threadIdx.x; i < D / 8; i += blockDim.x) {
        *reinterpret_cast<uint4*>(const_cast<__half*>(Ks) + (cur - s0) * D + 8 * i) =
            *reinterpret_cast<const uint4*>(Kg + (size_t)cur * D + 8 * i);
        *reinterpret_cast<uint4*>(const_cast<__half*>(Vs) + (cur - s0) * D + 8 * i) =
            *reinterpret_cast<const uint4*>(Vg + (size_t)cur * D + 8 * i);
      }
      __syncthreads();
    }
    for (int base = warp * SPI; base < n; base += NW * SPI) {
      uint4 kr[4], vr[4];
      bool ok[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int slot = base + j * G + grp;
        ok[j] = slot < n;
        if (ok[j]) {
          kr[j] = lds128(Ks + slot * D + 8 * li);
          vr[j] = lds128(Vs + slot * D + 8 * li);
        } else {
          kr[j] = make_uint4(0u, 0u, 0u, 0u);
          vr[j] = kr[j];
        }
      }
      float sc[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2* kh = reinterpret_cast<const __half2*>(&kr[j]);
        float d = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(kh[i]);
          d = fmaf(qv[2 * i], f.x, d);
          d = fmaf(qv[2 * i + 1], f.y, d);
        }
#pragma unroll
        for (int o = LPS / 2; o; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        sc[j] = ok[j] ? d : -INFINITY;
      }
      float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
#pragma unroll
      for (int o = LPS; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m, mx);  // finite: slot `base` is valid
      const float corr = __expf(m - m_new);
      float ps = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] *= corr;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float pj = ok[j] ? __expf(sc[j] - m_new) : 0.f;
        ps += pj;
        const __half2* vh = reinterpret_cast<const __half2*>(&vr[j]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(vh[i]);
          acc[2 * i] = fmaf(pj, f.x, acc[2 * i]);
          acc[2 * i + 1] = fmaf(pj, f.y, acc[2 * i + 1]);
        }
      }
#pragma unroll
      for (int o = LPS; o < 32; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l = l * corr + ps;
      m = m_new;
    }
    __syncthreads();  // stage consumed
    if (threadIdx.x == 0 && sb + 2 < n_sub) issue(sb + 2);
  }
  if (kPdlLate & PDL_ATTN) pdl_launch_dependents();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
#pragma unroll
    for (int o = LPS; o < 32; o <<= 1) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
  }
  if (lane == 0) {
    sm_m[warp] = m;
    sm_l[warp] = l;
  }
  if (grp == 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) sm_acc[warp][8 * li + i] = acc[i];
  }
  __syncthreads();

  // CTA merge -> this split's partial {m, l, acc[D]} in shared memory
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w]);
  float wsc[NW];
#pragma unroll
  for (int w = 0; w < NW; ++w) wsc[w] = (M == -INFINITY) ? 0.f : __expf(sm_m[w] - M);
  if (threadIdx.x == 0) {
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) L += sm_l[w] * wsc[w];
    s_part[0] = M;
    s_part[1] = L;
  }
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) v += sm_acc[w][d] * wsc[w];
    s_part[2 + d] = v;
  }
  // The splits of one (row, head) form a thread-block cluster: after the cluster
  // barrier every CTA merges its slice of D from all splits' partials (distributed
  // shared memory) with their log-sum-exp weights and the sink.
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  const int ns = a.nsplit;
  float Mt = a.sink ? a.sink[head] : -INFINITY;
  for (int sp = 0; sp < ns; ++sp) Mt = fmaxf(Mt, cluster.map_shared_rank(s_part, sp)[0]);
  float Lt = a.sink ? __expf(a.sink[head] - Mt) : 0.f;
  for (int sp = 0; sp < ns; ++sp) {
    const float* pp = cluster.map_shared_rank(s_part, sp);
    if (pp[0] != -INFINITY) Lt += pp[1] * __expf(pp[0] - Mt);
  }
  const int d0 = split * D / ns, d1 = (split + 1) * D / ns;
  for (int d = d0 + threadIdx.x; d < d1; d += blockDim.x) {
    float v = 0.f;
    for (int sp = 0; sp < ns; ++sp) {
      const float* pp = cluster.map_shared_rank(s_part, sp);
      if (pp[0] != -INFINITY) v += pp[2 + d] * __expf(pp[0] - Mt);
    }
    a.out[(size_t)row * a.nh * D + head * D + d] = __float2half_rn(v / Lt);
  }
  cluster.sync();  // every CTA keeps its partial until all slices are merged
}

// ------------------------------------------------------------------ INT8 KV cache
// Entries: per (row, K|V, head, slot) D int8 codes and one fp32 scale,
// value = scale * code.  Quantisation (one head vector): s = max|x| / 127 and
// code = round-to-nearest-even(x / s) clamped to [-127, 127], in IEEE fp32; a
// zero vector has s = 0 and zero codes ("Falcon-OCR INT8 OpenVINO IR", "How
// it is meant to be run": an INT8 KV cache; the per-head scale is our reading).

// int8 code byte b of w (as a signed value) in fp32, exactly: the byte + 128 is
// placed in the mantissa of 2^23 (byte permute) and 2^23 + 128 is subtracted.
template <int B>
__device__ __forceinline__ float s8_to_f32(uint32_t u_biased) {
  static_assert(B >= 0 && B < 4, "byte");
  return __uint_as_float(__byte_perm(u_biased, 0x4B000000u, 0x7540 + B)) - 8388736.0f;
}

__global__ void k_kv_quant(const KvQuantArgs a) {
  __shared__ float s_max[8];
  pdl_launch_dependents();
  pdl_wait();  // the new keys and values come from the QKV kernel
  const int t = blockIdx.x, kv = blockIdx.y, head = blockIdx.z, d = threadIdx.x;
  float x = 0.f;  // threads beyond D (head_dim 16: the block is one whole warp) hold zero
  if (d < a.D) {
    if (a.src32) {
      x = a.src32[(((size_t)t * 2 + kv) * a.nh + head) * a.D + d];
    } else {
      const __half* src = kv ? a.src16v : a.src16k;
      x = __half2float(src[((size_t)head * gridDim.x + t) * a.D + d]);
    }
  }
  float m = fabsf(x);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((d & 31) == 0) s_max[d >> 5] = m;
  __syncthreads();
  float amax = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, s_max[w]);
  const float sc = amax / 127.0f;
  int q = 0;
  if (sc > 0.f) q = max(-127, min(127, __float2int_rn(x / sc)));
  int slot;
  if (a.pos) {
    const int p = max(a.pos[t], 0);  // negative positions are reported by the embedding kernel
    slot = p < a.P ? p : a.P + (p - a.P) % a.R;
  } else {
    slot = a.slot0 + t;
  }
  const int kvr = a.kv_row0 + t * a.kv_rstep;
  const size_t vec = ((size_t)kvr * 2 + kv) * a.nh + head;
  if (d < a.D) a.kv8[(vec * a.SL + slot) * a.D + d] = (int8_t)q;
  if (d == 0) a.kvs[vec * a.SLp + slot] = sc;
}

cudaError_t launch_kv_quant(const KvQuantArgs& a, int tokens, cudaStream_t st, bool pdl) {
  return launch_kernel(k_kv_quant, dim3(tokens, 2, a.nh), dim3(a.D < 32 ? 32 : a.D), 0, st, pdl, a);
}

// Cache slots [slot0, slot0 + n) of one (layer, row) as fp16 values s * code:
// k_out / v_out [nh][n][D].
__global__ void k_kv_dequant(const int8_t* kv8, const float* kvs, int nh, int D, int SL, int SLp, int slot0,
                             int n, __half* k_out, __half* v_out) {
  const int t = blockIdx.x, kv = blockIdx.y, head = blockIdx.z, d = threadIdx.x;
  const size_t vec = (size_t)kv * nh + head;
  const float v = kvs[vec * SLp + slot0 + t] * (float)kv8[(vec * SL + slot0 + t) * D + d];
  (kv ? v_out : k_out)[((size_t)head * n + t) * D + d] = __float2half_rn(v);
}

cudaError_t launch_kv_dequant(const int8_t* kv8, const float* kvs, int nh, int D, int SL, int SLp, int slot0, int n,
                              __half* k_out, __half* v_out, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  k_kv_dequant<<<dim3(n, 2, nh), D, 0, st>>>(kv8, kvs, nh, D, SL, SLp, slot0, n, k_out, v_out);
  return cudaGetLastError();
}

// Split-K attention over the INT8 cache: the same structure as k_attn (TMA bulk
// stages, online softmax per warp, cluster merge with the sink), with stages of
// SUB slots holding the key codes, the value codes and both scale runs.  A lane
// reads 16 codes of a slot per load (D/16 lanes per slot); scores are
// s_k * (q . code) and values accumulate (p * s_v) * code, all in fp32.
template <int D>
struct Attn8Cfg {
  static constexpr int SUB = 16384 / D;                // slots per stage (16 KB of key codes)
  static constexpr int CODES = SUB * D;                // bytes of one code block
  static constexpr int STAGE = 2 * CODES + 2 * SUB * 4;  // K codes, V codes, K scales, V scales
};

int attn8_smem_bytes(int D) { return 2 * (2 * 16384 + 2 * (16384 / D) * 4) + 64; }

template <int D>
__global__ void __launch_bounds__(UOCR_ATTN_WARPS * 32) k_attn8(const AttnArgs a) {
  constexpr int LPS = D / 16;   // lanes per slot
  constexpr int G = 32 / LPS;   // slots per load instruction
  constexpr int SPI = 4 * G;    // slots per warp iteration
  constexpr int NW = UOCR_ATTN_WARPS;
  constexpr int SUB = Attn8Cfg<D>::SUB, CODES = Attn8Cfg<D>::CODES, STAGE = Attn8Cfg<D>::STAGE;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 2 * STAGE);
  __shared__ float sm_m[NW], sm_l[NW];
  __shared__ float sm_acc[NW][D];
  __shared__ float s_part[D + 2];

  const int split = blockIdx.x, head = blockIdx.y, row = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPS, li = lane % LPS;
  int p = a.pos[row];
  if (p < 0) p = 0;
  const int n_valid = (p < a.P) ? p + 1 : a.P + min(p - a.P + 1, a.R);
  const int s_begin = split * a.chunk;  // a multiple of 16
  const int s_end = min(n_valid, s_begin + a.chunk);
  const int n_sub = s_end > s_begin ? (s_end - s_begin + SUB - 1) / SUB : 0;
  const int kvr = a.kv_row0 + row * a.kv_rstep;
  const size_t kvec = ((size_t)kvr * 2 + 0) * a.nh + head, vvec = ((size_t)kvr * 2 + 1) * a.nh + head;
  const int8_t* Kg = a.kv8 + kvec * a.SL * D;
  const int8_t* Vg = a.kv8 + vvec * a.SL * D;
  const float* KSg = a.kvs + kvec * a.SLp;
  const float* VSg = a.kvs + vvec * a.SLp;
  auto issue = [&](int sb) {
    const int s0 = s_begin + sb * SUB, n = min(SUB, s_end - s0);
    const int n4 = (n + 3) & ~3;  // scale runs in whole 16-byte pieces (SLp covers the round-up)
    uint8_t* st = smem + (sb & 1) * STAGE;
    uint64_t* b = bar + (sb & 1);
    mbar_expect_tx(b, 2u * n * D + 2u * n4 * 4);
    bulk_g2s(st, Kg + (size_t)s0 * D, n * D, b);
    bulk_g2s(st + CODES, Vg + (size_t)s0 * D, n * D, b);
    bulk_g2s(st + 2 * CODES, KSg + s0, n4 * 4, b);
    bulk_g2s(st + 2 * CODES + SUB * 4, VSg + s0, n4 * 4, b);
  };
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_init(bar + 1, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (a.early && threadIdx.x == 0)
    for (int sb = 0; sb < n_sub && sb < 2; ++sb) issue(sb);
  if (!(kPdlLate & PDL_ATTN)) pdl_launch_dependents();
  pdl_wait();  // q and the current slot come from the QKV and quantiser kernels
  if (!a.early && threadIdx.x == 0)
    for (int sb = 0; sb < n_sub && sb < 2; ++sb) issue(sb);

  float qv[16];
  {
    const float* qp = a.q + ((size_t)row * a.nh + head) * D + 16 * li;
#pragma unroll
    for (int i = 0; i < 16; ++i) qv[i] = qp[i] * a.scale;
  }
  const int cur = p < a.P ? p : a.P + (p - a.P) % a.R;

  float m = -INFINITY, l = 0.f;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;

  for (int sb = 0; sb < n_sub; ++sb) {
    const int s0 = s_begin + sb * SUB, n = min(SUB, s_end - s0);
    int bad = 0;
    if (threadIdx.x == 0) {
      bad = !mbar_wait(bar + (sb & 1), (uint32_t)((sb >> 1) & 1));
      if (bad) atomicOr(a.status, kStatusTimeout);
    }
    if (__syncthreads_or(bad)) {
      if (threadIdx.x == 0 && sb + 1 < n_sub) mbar_wait(bar + ((sb + 1) & 1), (uint32_t)(((sb + 1) >> 1) & 1));
      break;
    }
    uint8_t* stg = smem + (sb & 1) * STAGE;
    const int8_t* Ks = reinterpret_cast<const int8_t*>(stg);
    const int8_t* Vs = Ks + CODES;
    float* KSs = reinterpret_cast<float*>(stg + 2 * CODES);
    float* VSs = KSs + SUB;
    if (a.early && cur >= s0 && cur < s0 + n) {  // the slot this step just wrote
      for (int i = threadIdx.x; i < D / 16; i += blockDim.x) {
        reinterpret_cast<uint4*>(stg + (size_t)(cur - s0) * D)[i] = reinterpret_cast<const uint4*>(Kg + (size_t)cur * D)[i];
        reinterpret_cast<uint4*>(stg + CODES + (size_t)(cur - s0) * D)[i] =
            reinterpret_cast<const uint4*>(Vg + (size_t)cur * D)[i];
      }
      if (threadIdx.x == 0) {
        KSs[cur - s0] = KSg[cur];
        VSs[cur - s0] = VSg[cur];
      }
      __syncthreads();
    }
    for (int base = warp * SPI; base < n; base += NW * SPI) {
      uint4 kr[4], vr[4];
      float ks[4], vs[4];
      bool ok[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int slot = base + j * G + grp;
        ok[j] = slot < n;
        if (ok[j]) {
          kr[j] = lds128(Ks + slot * D + 16 * li);
          vr[j] = lds128(Vs + slot * D + 16 * li);
          ks[j] = KSs[slot];
          vs[j] = VSs[slot];
        } else {
          kr[j] = make_uint4(0u, 0u, 0u, 0u);
          vr[j] = kr[j];
          ks[j] = 0.f;
          vs[j] = 0.f;
        }
      }
      float sc[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t w[4] = {kr[j].x ^ 0x80808080u, kr[j].y ^ 0x80808080u, kr[j].z ^ 0x80808080u,
                               kr[j].w ^ 0x80808080u};
        float d = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          d = fmaf(qv[4 * i + 0], s8_to_f32<0>(w[i]), d);
          d = fmaf(qv[4 * i + 1], s8_to_f32<1>(w[i]), d);
          d = fmaf(qv[4 * i + 2], s8_to_f32<2>(w[i]), d);
          d = fmaf(qv[4 * i + 3], s8_to_f32<3>(w[i]), d);
        }
#pragma unroll
        for (int o = LPS / 2; o; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        sc[j] = ok[j] ? d * ks[j] : -INFINITY;
      }
      float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
#pragma unroll
      for (int o = LPS; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m, mx);  // finite: slot `base` is valid
      const float corr = __expf(m - m_new);
      float ps = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] *= corr;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float pj = ok[j] ? __expf(sc[j] - m_new) : 0.f;
        ps += pj;
        const float pv = pj * vs[j];
        const uint32_t w[4] = {vr[j].x ^ 0x80808080u, vr[j].y ^ 0x80808080u, vr[j].z ^ 0x80808080u,
                               vr[j].w ^ 0x80808080u};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[4 * i + 0] = fmaf(pv, s8_to_f32<0>(w[i]), acc[4 * i + 0]);
          acc[4 * i + 1] = fmaf(pv, s8_to_f32<1>(w[i]), acc[4 * i + 1]);
          acc[4 * i + 2] = fmaf(pv, s8_to_f32<2>(w[i]), acc[4 * i + 2]);
          acc[4 * i + 3] = fmaf(pv, s8_to_f32<3>(w[i]), acc[4 * i + 3]);
        }
      }
#pragma unroll
      for (int o = LPS; o < 32; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l = l * corr + ps;
      m = m_new;
    }
    __syncthreads();  // stage consumed
    if (threadIdx.x == 0 && sb + 2 < n_sub) issue(sb + 2);
  }
  if (kPdlLate & PDL_ATTN) pdl_launch_dependents();
#pragma unroll
  for (int i = 0; i < 16; ++i) {
#pragma unroll
    for (int o = LPS; o < 32; o <<= 1) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
  }
  if (lane == 0) {
    sm_m[warp] = m;
    sm_l[warp] = l;
  }
  if (grp == 0) {
#pragma unroll
    for (int i = 0; i < 16; ++i) sm_acc[warp][16 * li + i] = acc[i];
  }
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w]);
  float wsc[NW];
#pragma unroll
  for (int w = 0; w < NW; ++w) wsc[w] = (M == -INFINITY) ? 0.f : __expf(sm_m[w] - M);
  if (threadIdx.x == 0) {
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) L += sm_l[w] * wsc[w];
    s_part[0] = M;
    s_part[1] = L;
  }
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) v += sm_acc[w][d] * wsc[w];
    s_part[2 + d] = v;
  }
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  const int ns = a.nsplit;
  float Mt = a.sink ? a.sink[head] : -INFINITY;
  for (int sp = 0; sp < ns; ++sp) Mt = fmaxf(Mt, cluster.map_shared_rank(s_part, sp)[0]);
  float Lt = a.sink ? __expf(a.sink[head] - Mt) : 0.f;
  for (int sp = 0; sp < ns; ++sp) {
    const float* pp = cluster.map_shared_rank(s_part, sp);
    if (pp[0] != -INFINITY) Lt += pp[1] * __expf(pp[0] - Mt);
  }
  const int d0 = split * D / ns, d1 = (split + 1) * D / ns;
  for (int d = d0 + threadIdx.x; d < d1; d += blockDim.x) {
    float v = 0.f;
    for (int sp = 0; sp < ns; ++sp) {
      const float* pp = cluster.map_shared_rank(s_part, sp);
      if (pp[0] != -INFINITY) v += pp[2 + d] * __expf(pp[0] - Mt);
    }
    a.out[(size_t)row * a.nh * D + head * D + d] = __float2half_rn(v / Lt);
  }
  cluster.sync();
}

cudaError_t launch_attn(const AttnArgs& a, int rows, cudaStream_t st, bool pdl) {
  const dim3 grid(a.nsplit, a.nh, rows);
  if (a.kv8) {
    const size_t sm8 = attn8_smem_bytes(a.D);
    switch (a.D) {
      case 16: return launch_kernel_cluster(k_attn8<16>, grid, dim3(UOCR_ATTN_WARPS * 32), sm8, st, pdl, a.nsplit, a);
      case 32: return launch_kernel_cluster(k_attn8<32>, grid, dim3(UOCR_ATTN_WARPS * 32), sm8, st, pdl, a.nsplit, a);
      case 64: return launch_kernel_cluster(k_attn8<64>, grid, dim3(UOCR_ATTN_WARPS * 32), sm8, st, pdl, a.nsplit, a);
      case 128: return launch_kernel_cluster(k_attn8<128>, grid, dim3(UOCR_ATTN_WARPS * 32), sm8, st, pdl, a.nsplit, a);
      case 256: return launch_kernel_cluster(k_attn8<256>, grid, dim3(UOCR_ATTN_WARPS * 32), sm8, st, pdl, a.nsplit, a);
    }
    return cudaErrorInvalidValue;
  }
  const size_t sm = attn_smem_bytes(a.D);
  switch (a.D) {
    case 16: return launch_kernel_cluster(k_attn<16>, grid, dim3(UOCR_ATTN_WARPS * 32), sm, st, pdl, a.nsplit, a);
    case 32: return launch_kernel_cluster(k_attn<32>, grid, dim3(UOCR_ATTN_WARPS * 32), sm, st, pdl, a.nsplit, a);
    case 64: return launch_kernel_cluster(k_attn<64>, grid, dim3(UOCR_ATTN_WARPS * 32), sm, st, pdl, a.nsplit, a);
    case 128: return launch_kernel_cluster(k_attn<128>, grid, dim3(UOCR_ATTN_WARPS * 32), sm, st, pdl, a.nsplit, a);
    case 256: return launch_kernel_cluster(k_attn<256>, grid, dim3(UOCR_ATTN_WARPS * 32), sm, st, pdl, a.nsplit, a);
  }
  return cudaErrorInvalidValue;
}

// Attention CTAs of one launch that fit on an SM at once (shared memory bound).
int attn_ctas_per_sm(int D, bool int8_cache) {
  int n = 0;
  cudaError_t e = cudaSuccess;
#define UOCR_OCC(K_, SM_) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, K_, UOCR_ATTN_WARPS * 32, SM_);
  if (int8_cache) {
    switch (D) {
      case 16: UOCR_OCC(k_attn8<16>, attn8_smem_bytes(16)) break;
      case 32: UOCR_OCC(k_attn8<32>, attn8_smem_bytes(32)) break;
      case 64: UOCR_OCC(k_attn8<64>, attn8_smem_bytes(64)) break;
      case 128: UOCR_OCC(k_attn8<128>, attn8_smem_bytes(128)) break;
      default: UOCR_OCC(k_attn8<256>, attn8_smem_bytes(256)) break;
    }
  } else {
    switch (D) {
      case 16: UOCR_OCC(k_attn<16>, attn_smem_bytes(16)) break;
      case 32: UOCR_OCC(k_attn<32>, attn_smem_bytes(32)) break;
      case 64: UOCR_OCC(k_attn<64>, attn_smem_bytes(64)) break;
      case 128: UOCR_OCC(k_attn<128>, attn_smem_bytes(128)) break;
      default: UOCR_OCC(k_attn<256>, attn_smem_bytes(256)) break;
    }
  }
#undef UOCR_OCC
  return e == cudaSuccess && n > 0 ? n : 1;
}

static cudaError_t init_attn_attributes() {
  cudaError_t e = cudaSuccess;
#define UOCR_A(D_) \
  if (e == cudaSuccess) e = allow_max_dyn_smem(k_attn<D_>);
  UOCR_A(16) UOCR_A(32) UOCR_A(64) UOCR_A(128) UOCR_A(256)
#undef UOCR_A
#define UOCR_A8(D_) \
  if (e == cudaSuccess) e = allow_max_dyn_smem(k_attn8<D_>);
  UOCR_A8(16) UOCR_A8(32) UOCR_A8(64) UOCR_A8(128) UOCR_A8(256)
#undef UOCR_A8
  return e;
}

// ------------------------------------------------------------------ embedding
// Token ids -> fp16 embedding row, or the given fp16 hidden vectors, widened
// into the fp32 residual stream; validates ids and positions.
__global__ void k_embed(const EmbedArgs a) {
  pdl_launch_dependents();  // the next kernel may start streaming its weights
  const int row = blockIdx.x;
  const __half* src;
  if (a.ids) {
    int id = a.ids[row];
    if (id < 0 || id >= a.V) {
      if (threadIdx.x == 0) atomicOr(a.status, kStatusToken);
      id = 0;
    }
    src = a.emb + (size_t)id * a.H;
  } else {
    src = a.x + (size_t)row * a.H;
  }
  if (a.pos_base >= 0) {  // prefill: consecutive positions from pos_base
    if (threadIdx.x == 0) a.pos[row] = a.pos_base + row;
    __syncthreads();
  }
  if (threadIdx.x == 0 && a.pos[row] < 0) atomicOr(a.status, kStatusPosition);
  for (int k = threadIdx.x * 2; k < a.H; k += blockDim.x * 2) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(src + k));
    a.out[(size_t)row * a.H + k] = f.x;
    a.out[(size_t)row * a.H + k + 1] = f.y;
  }
  // rotary angles of this row's position (rotate-half RoPE): the angle is formed
  // and reduced modulo 2 pi in double precision, then its cosine and sine in float
  const int pos = max(a.pos[row], 0);
  for (int j = threadIdx.x; j < a.half_d; j += blockDim.x) {
    double ang = (double)pos * a.inv_freq[j];
    ang -= 6.283185307179586 * rint(ang * 0.15915494309189535);
    float sn, cs;
    sincosf((float)ang, &sn, &cs);
    a.rope[(size_t)row * a.half_d + j] = make_float2(cs, sn);
  }
}

cudaError_t launch_embed(const EmbedArgs& a, int rows, cudaStream_t st) {
  k_embed<<<rows, 256, 0, st>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ packer
// Canonical blocks -> fragment-ordered device layout (see device_common.cuh).
// One thread per (slab, unit, lane); packed row pr maps to (source, row) by
// the matrix's row map: identity, Q/K/V sections with the rotary pairs (i,
// i + D/2) placed in rows g and g + 8 of one slab, interleaved gate/up rows
// (gate in rows 0..7 of a slab, up in 8..15) over one or more experts, or
// column concatenation of several experts (shared down projections).
struct PackSrcRef {
  int src;  // -1: zero padding
  int row;
};

__device__ __forceinline__ PackSrcRef pack_row(const PackArgs& a, int pr) {
  PackSrcRef r{-1, 0};
  switch (a.map) {
    case MAP_IDENT:
    case MAP_KCAT:
      if (pr < a.src_rows) r = {0, pr};
      break;
    case MAP_QKV: {
      const int sec = pr / a.S, w = pr - sec * a.S;
      const int head = w / a.D, wi = w - head * a.D;
      const int js = wi >> 4, j = wi & 15;
      const int dim = j < 8 ? 8 * js + j : (a.D >> 1) + 8 * js + (j - 8);
      if (sec < a.nsrc) r = {sec, head * a.D + dim};
      break;
    }
    case MAP_SWIGLU: {
      const int s = pr >> 4, j = pr & 15;
      const int gr = 8 * s + (j & 7);
      const int ex = gr / a.I;
      const int src = 2 * ex + (j < 8 ? 0 : 1);
      if (src < a.nsrc) r = {src, gr - ex * a.I};
      break;
    }
  }
  return r;
}

// code and scale fetch from canonical blocks; k is the packed column
struct Code {
  const uint8_t* blk;
  int j;
};

__device__ __forceinline__ Code locate(const PackArgs& a, PackSrcRef r, int k) {
  int src = r.src, kk = k;
  if (a.map == MAP_KCAT) {
    src = k / a.I;
    kk = k - src * a.I;
  }
  const uint8_t* blk = a.src[src] + ((size_t)r.row * (a.src_cols / a.group) + kk / a.group) * a.bb;
  return Code{blk, kk % a.group};
}

__device__ __forceinline__ uint32_t get_code(const PackArgs& a, PackSrcRef r, int k) {
  if (r.src < 0) return a.fmt == Q4_0 ? 8u : 0u;
  const Code c = locate(a, r, k);
  if (a.fmt == Q8_0) return c.blk[2 + c.j];
  if (a.fmt == Q4_0) {  // element j < group/2: low nibble of byte j, else high nibble of byte j - group/2
    const int half = a.group / 2;
    return c.j < half ? (c.blk[2 + c.j] & 0xF) : (c.blk[2 + c.j - half] >> 4);
  }
  return c.blk[4 + c.j];  // I8ASYM
}

__device__ __forceinline__ uint16_t get_half(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

__device__ __forceinline__ uint16_t get_f16(const PackArgs& a, PackSrcRef r, int k) {
  if (r.src < 0) return 0;
  int src = r.src, kk = k;
  if (a.map == MAP_KCAT) {
    src = k / a.I;
    kk = k - src * a.I;
  }
  return get_half(a.src[src] + ((size_t)r.row * a.src_cols + kk) * 2);
}

__device__ __forceinline__ uint16_t get_scale(const PackArgs& a, PackSrcRef r, int k, int which) {
  if (r.src < 0) return 0;
  const Code c = locate(a, r, k);
  return get_half(c.blk + 2 * which);
}

__global__ void k_pack(const PackArgs a) {
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long total = (long long)a.n_slabs * a.U * 32;
  if (gid >= total) return;
  const int lane = (int)(gid & 31);
  const long long su = gid >> 5;
  const int u = (int)(su % a.U);
  const int slab = (int)(su / a.U);
  const int g = lane >> 2, t = lane & 3;
  const PackSrcRef r0 = pack_row(a, 16 * slab + g);
  const PackSrcRef r1 = pack_row(a, 16 * slab + g + 8);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  if (a.fmt == F16) {
    // unit u (32 inputs) = two 512-byte halves of 16 inputs each; thread handles half u % 2
    const int kk = (u >> 1) * 32 + (u & 1) * 16 + 2 * t;
    w[0] = get_f16(a, r0, kk) | ((uint32_t)get_f16(a, r0, kk + 1) << 16);
    w[1] = get_f16(a, r1, kk) | ((uint32_t)get_f16(a, r1, kk + 1) << 16);
    w[2] = get_f16(a, r0, kk + 8) | ((uint32_t)get_f16(a, r0, kk + 9) << 16);
    w[3] = get_f16(a, r1, kk + 8) | ((uint32_t)get_f16(a, r1, kk + 9) << 16);
  } else if (a.fmt == Q4_0) {
    for (int ks = 0; ks < 4; ++ks) {
      const int kk = u * 64 + 16 * ks + 2 * t;
      const uint32_t c0 = get_code(a, r0, kk), c1 = get_code(a, r0, kk + 1);
      const uint32_t c2 = get_code(a, r1, kk), c3 = get_code(a, r1, kk + 1);
      const uint32_t c4 = get_code(a, r0, kk + 8), c5 = get_code(a, r0, kk + 9);
      const uint32_t c6 = get_code(a, r1, kk + 8), c7 = get_code(a, r1, kk + 9);
      w[ks] = c0 | (c2 << 4) | (c4 << 8) | (c6 << 12) | (c1 << 16) | (c3 << 20) | (c5 << 24) | (c7 << 28);
    }
  } else {  // Q8_0, I8ASYM: byte order a0..a7 per k-step
    for (int ks = 0; ks < 2; ++ks) {
      const int kk = u * 32 + 16 * ks + 2 * t;
      const uint32_t c0 = get_code(a, r0, kk), c1 = get_code(a, r0, kk + 1);
      const uint32_t c2 = get_code(a, r1, kk), c3 = get_code(a, r1, kk + 1);
      const uint32_t c4 = get_code(a, r0, kk + 8), c5 = get_code(a, r0, kk + 9);
      const uint32_t c6 = get_code(a, r1, kk + 8), c7 = get_code(a, r1, kk + 9);
      w[2 * ks] = c0 | (c1 << 8) | (c2 << 16) | (c3 << 24);
      w[2 * ks + 1] = c4 | (c5 << 8) | (c6 << 16) | (c7 << 24);
    }
  }
  // F16: a.U counts 16-input halves here (two per 1024-byte unit); others: 512-byte units
  uint4* dst = reinterpret_cast<uint4*>(a.q + ((size_t)slab * a.U + u) * 512 + lane * 16);
  *dst = make_uint4(w[0], w[1], w[2], w[3]);
  if (t == 0 && a.fmt != F16) {
    const size_t unit = (size_t)slab * a.U + u;
    if (a.fmt == Q8_0) {
      uint16_t* sp = reinterpret_cast<uint16_t*>(a.s + unit * 32 + g * 4);
      sp[0] = get_scale(a, r0, u * 32, 0);
      sp[1] = get_scale(a, r1, u * 32, 0);
    } else if (a.fmt == Q4_0) {
      uint16_t* sp = reinterpret_cast<uint16_t*>(a.s + unit * 64 + g * 8);
      sp[0] = get_scale(a, r0, u * 64, 0);
      sp[1] = get_scale(a, r1, u * 64, 0);
      sp[2] = get_scale(a, r0, u * 64 + 32, 0);
      sp[3] = get_scale(a, r1, u * 64 + 32, 0);
    } else {
      uint16_t* sp = reinterpret_cast<uint16_t*>(a.s + unit * 64 + g * 8);
      sp[0] = get_scale(a, r0, u * 32, 0);
      sp[1] = get_scale(a, r1, u * 32, 0);
      sp[2] = get_scale(a, r0, u * 32, 1);
      sp[3] = get_scale(a, r1, u * 32, 1);
    }
  }
}

cudaError_t launch_pack(const PackArgs& a, cudaStream_t st) {
  const long long total = (long long)a.n_slabs * a.U * 32;
  const int blocks = (int)((total + 255) / 256);
  k_pack<<<blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ fp32 -> fp16
__global__ void k_f32_to_f16(const float* src, __half* dst, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    dst[i] = __float2half_rn(src[i]);
}

cudaError_t launch_f32_to_f16(const float* src, __half* dst, long long n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const long long b = (n + 255) / 256;
  k_f32_to_f16<<<(int)(b < 1024 ? b : 1024), 256, 0, st>>>(src, dst, n);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ bounded-wait probe
// The pattern every TMA wait of the step follows (arm the barrier with the
// bytes expected, issue the copy, poll with an iteration limit, report a
// timeout through the status word), with a short limit and the copy issued
// only when `issue` is set: without it the barrier's phase never completes
// and the wait must give up and report.  No copy is left in flight either way.
constexpr uint32_t kProbeSpinLimit = 1u << 12;

__global__ void k_wait_probe(const void* src, int issue, int* status) {
  __shared__ __align__(16) unsigned char buf[16];
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  mbar_expect_tx(&bar, 16);
  if (issue) bulk_g2s(buf, src, 16, &bar);
  if (!mbar_wait<kProbeSpinLimit>(&bar, 0)) atomicOr(status, kStatusTimeout);
}

cudaError_t launch_wait_probe(const void* src, int issue, int* status, cudaStream_t st) {
  k_wait_probe<<<1, 32, 0, st>>>(src, issue, status);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ reset
__global__ void k_zero_slots(__half* base, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    base[i] = __float2half_rn(0.f);
}

// Zero slots [from_slot, SL) of every head of both K and V of one (layer, row).
cudaError_t launch_fill_zero_ring(__half* kv_layer_row, int nh, int SL, int D, int from_slot, cudaStream_t st) {
  for (int kvh = 0; kvh < 2 * nh; ++kvh) {
    __half* b = kv_layer_row + ((size_t)kvh * SL + from_slot) * D;
    const long long n = (long long)(SL - from_slot) * D;
    if (n <= 0) continue;
    k_zero_slots<<<(int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024), 256, 0, st>>>(b, n);
  }
  return cudaGetLastError();
}

cudaError_t init_gemv_attributes();
cudaError_t init_moe_attributes();
cudaError_t init_tc_attributes();
cudaError_t init_tc_expert_attributes();

cudaError_t init_kernel_attributes() {
  cudaError_t e = init_gemv_attributes();
  if (e == cudaSuccess) e = init_moe_attributes();
  if (e == cudaSuccess) e = init_attn_attributes();
  if (e == cudaSuccess) e = init_tc_attributes();
  if (e == cudaSuccess) e = init_tc_expert_attributes();
  return e;
}

}  // namespace uocr
