// Device-side building blocks shared by the decode-step kernels (sm_103a).
//
// Weight layout ("packed"): a matrix W[N][K] is cut into slabs of 16 output
// rows; a slab is cut into units of 16 rows x KU inputs, KU = 32 (Q8_0,
// I8ASYM), 64 (Q4_0) or 16 (F16).  A unit is 512 bytes of codes stored in the
// register order of the m16n8k16 tensor-core A fragment, so lane L of a warp
// loads bytes [16L, 16L+16) of the unit with one 128-bit load and holds its
// fragment(s) without any shuffle.  Scales live in a separate plane, per unit
// and per fragment row group g = lane/4: Q8_0 {d[g], d[g+8]} (4 B),
// Q4_0 {d[g][b0], d[g+8][b0], d[g][b1], d[g+8][b1]} (8 B),
// I8ASYM {s[g], s[g+8], z[g], z[g+8]} (8 B).
//
// Dequantisation ("Unlimited-OCR on Apple Silicon with C and Metal",
// "Quantizzazione": no full fp16 copy of the weights, dequantise inside the
// matmul).  Integer codes become exact fp16 integers with the exponent-bias
// method (OR the code into the mantissa of 1024 and subtract the bias), the
// tensor core multiplies them with fp16 activations accumulating in fp32,
// and the block scale is applied to the fp32 block sum, so no weight value is
// ever rounded.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace uocr {

enum Fmt : int { F16 = 0, Q8_0 = 1, Q4_0 = 2, I8ASYM = 3 };

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kUnitBytes = 512;

__host__ __device__ constexpr int unit_k(int fmt) { return fmt == Q4_0 ? 64 : (fmt == F16 ? 16 : 32); }
__host__ __device__ constexpr int unit_scale_bytes(int fmt) {
  return fmt == Q8_0 ? 32 : (fmt == F16 ? 0 : 64);
}

// A packed matrix as the kernels see it.
struct PMat {
  const uint8_t* q;   // slabs * U * 512 bytes
  const uint8_t* s;   // slabs * U * unit_scale_bytes
  int n_slabs;        // ceil(N_packed / 16)
  int U;              // units per slab = K / unit_k
  int K;
  long long q_stride; // bytes between consecutive experts (expert arrays)
  long long s_stride;
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;  // (a & b) | c
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}

__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], const void* p) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(a));
}

__device__ __forceinline__ uint32_t h2_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ __half2 h2_bits(uint16_t b) {
  return __halves2half2(__ushort_as_half(b), __ushort_as_half(b));
}

// ------------------------------------------------------------------ code -> fp16
// Q8_0: bytes (b0 b1 b2 b3) of signed codes -> (b0,b1), (b2,b3) as fp16 pairs.
__device__ __forceinline__ void dq_s8x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;                // code + 128, unsigned
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);  // fp16 1024 + u0, 1024 + u1
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = h2_bits(0x6480);              // 1152 = 1024 + 128
  lo = h2_u32(__hsub2(u32_h2(a), bias));
  hi = h2_u32(__hsub2(u32_h2(b), bias));
}

// I8ASYM: unsigned codes -> fp16 pairs (exact integers 0..255).
__device__ __forceinline__ void dq_u8x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t a = __byte_perm(w, 0x64646464u, 0x4140);
  const uint32_t b = __byte_perm(w, 0x64646464u, 0x4342);
  const __half2 bias = h2_bits(0x6400);              // 1024
  lo = h2_u32(__hsub2(u32_h2(a), bias));
  hi = h2_u32(__hsub2(u32_h2(b), bias));
}

// Q4_0: one 32-bit word = the 8 codes of one k-step fragment, nibble positions
// a0@0 a2@4 a4@8 a6@12 a1@16 a3@20 a5@24 a7@28; returns the four A registers
// (a0,a1) (a2,a3) (a4,a5) (a6,a7) as fp16 pairs of (code - 8).
__device__ __forceinline__ void dq_q4(uint32_t w, uint32_t (&r)[4]) {
  const uint32_t x0 = lop_and_or(w, 0x000F000Fu, 0x64006400u);        // 1024 + n
  const uint32_t x1 = lop_and_or(w, 0x00F000F0u, 0x64006400u);        // 1024 + 16 n
  const uint32_t w8 = w >> 8;
  const uint32_t x2 = lop_and_or(w8, 0x000F000Fu, 0x64006400u);
  const uint32_t x3 = lop_and_or(w8, 0x00F000F0u, 0x64006400u);
  const __half2 k1032 = h2_bits(0x6408);   // 1024 + 8
  const __half2 k1_16 = h2_bits(0x2C00);   // 1/16
  const __half2 km72 = h2_bits(0xD480);    // -(64 + 8)
  r[0] = h2_u32(__hsub2(u32_h2(x0), k1032));
  r[1] = h2_u32(__hfma2(u32_h2(x1), k1_16, km72));
  r[2] = h2_u32(__hsub2(u32_h2(x2), k1032));
  r[3] = h2_u32(__hfma2(u32_h2(x3), k1_16, km72));
}

__device__ __forceinline__ float half_lo(uint32_t u) { return __half2float(__ushort_as_half((uint16_t)(u & 0xFFFF))); }
__device__ __forceinline__ float half_hi(uint32_t u) { return __half2float(__ushort_as_half((uint16_t)(u >> 16))); }

// ------------------------------------------------------------------ slab compute
// Shared-memory activation tile: xs[NT*8 tokens][ldx] fp16, ldx = kc + 8
// (the +8 makes every 8-row ldmatrix phase hit 32 distinct banks).
//
// acc[nt][0..3] follows the m16n8 C fragment: (row g, token 2t), (g, 2t+1),
// (g+8, 2t), (g+8, 2t+1) of n-tile nt.

template <int FMT>
__device__ __forceinline__ uint2 load_scales(const uint8_t* __restrict__ ws, int u, int g) {
  if constexpr (FMT == Q8_0) {
    uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(ws + (size_t)u * 32 + g * 4));
    return make_uint2(v, 0u);
  } else if constexpr (FMT == Q4_0 || FMT == I8ASYM) {
    return __ldg(reinterpret_cast<const uint2*>(ws + (size_t)u * 64 + g * 8));
  } else {
    return make_uint2(0u, 0u);
  }
}

// One unit (16 rows x unit_k(FMT) inputs) against every n-tile.
// xs_k: &xs[0][k_local] where k_local is the unit's first input within the
// staged chunk; xsum: per-token block sums of the staged activations
// [NT*8][nblk_chunk] (I8ASYM only), blk = the unit's block within the chunk.
template <int FMT, int NT>
__device__ __forceinline__ void unit_mma(float (&acc)[NT][4], uint4 q, uint2 sc, const __half* xs_k, int ldx,
                                         const float* xsum, int nblk, int blk, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int r8 = lane & 7, mi = lane >> 3;
  if constexpr (FMT == F16) {
    const uint32_t A[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      uint32_t B[2];
      ldsm_x2(B, xs_k + (nt * 8 + r8) * ldx + 8 * (mi & 1));
      mma_16816(acc[nt], A, B[0], B[1]);
    }
  } else if constexpr (FMT == Q8_0 || FMT == I8ASYM) {
    uint32_t A0[4], A1[4];
    if constexpr (FMT == Q8_0) {
      dq_s8x4(q.x, A0[0], A0[1]);
      dq_s8x4(q.y, A0[2], A0[3]);
      dq_s8x4(q.z, A1[0], A1[1]);
      dq_s8x4(q.w, A1[2], A1[3]);
    } else {
      dq_u8x4(q.x, A0[0], A0[1]);
      dq_u8x4(q.y, A0[2], A0[3]);
      dq_u8x4(q.z, A1[0], A1[1]);
      dq_u8x4(q.w, A1[2], A1[3]);
    }
    const float d_lo = half_lo(sc.x), d_hi = half_hi(sc.x);
    float z_lo = 0.f, z_hi = 0.f;
    if constexpr (FMT == I8ASYM) {
      z_lo = half_lo(sc.y);
      z_hi = half_hi(sc.y);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      uint32_t B[4];
      ldsm_x4(B, xs_k + (nt * 8 + r8) * ldx + 8 * mi);
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      mma_16816(c, A0, B[0], B[1]);
      mma_16816(c, A1, B[2], B[3]);
      if constexpr (FMT == I8ASYM) {
        const float s0 = xsum[(nt * 8 + 2 * t) * nblk + blk];
        const float s1 = xsum[(nt * 8 + 2 * t + 1) * nblk + blk];
        c[0] -= z_lo * s0;
        c[1] -= z_lo * s1;
        c[2] -= z_hi * s0;
        c[3] -= z_hi * s1;
      }
      acc[nt][0] = fmaf(d_lo, c[0], acc[nt][0]);
      acc[nt][1] = fmaf(d_lo, c[1], acc[nt][1]);
      acc[nt][2] = fmaf(d_hi, c[2], acc[nt][2]);
      acc[nt][3] = fmaf(d_hi, c[3], acc[nt][3]);
    }
  } else {  // Q4_0: 4 k-steps, 2 blocks
    uint32_t A[4][4];
    dq_q4(q.x, A[0]);
    dq_q4(q.y, A[1]);
    dq_q4(q.z, A[2]);
    dq_q4(q.w, A[3]);
    const float d0_lo = half_lo(sc.x), d0_hi = half_hi(sc.x);
    const float d1_lo = half_lo(sc.y), d1_hi = half_hi(sc.y);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      uint32_t B0[4], B1[4];
      ldsm_x4(B0, xs_k + (nt * 8 + r8) * ldx + 8 * mi);
      ldsm_x4(B1, xs_k + (nt * 8 + r8) * ldx + 32 + 8 * mi);
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      mma_16816(c, A[0], B0[0], B0[1]);
      mma_16816(c, A[1], B0[2], B0[3]);
      acc[nt][0] = fmaf(d0_lo, c[0], acc[nt][0]);
      acc[nt][1] = fmaf(d0_lo, c[1], acc[nt][1]);
      acc[nt][2] = fmaf(d0_hi, c[2], acc[nt][2]);
      acc[nt][3] = fmaf(d0_hi, c[3], acc[nt][3]);
      float e[4] = {0.f, 0.f, 0.f, 0.f};
      mma_16816(e, A[2], B1[0], B1[1]);
      mma_16816(e, A[3], B1[2], B1[3]);
      acc[nt][0] = fmaf(d1_lo, e[0], acc[nt][0]);
      acc[nt][1] = fmaf(d1_lo, e[1], acc[nt][1]);
      acc[nt][2] = fmaf(d1_hi, e[2], acc[nt][2]);
      acc[nt][3] = fmaf(d1_hi, e[3], acc[nt][3]);
    }
  }
}

// Units [u_begin, u_end) of one slab, split across the CTA's warps
// (warp w takes units u_begin + w, + w + kWarps, ...; consecutive warps read
// consecutive 512-byte units), with UNR units of loads in flight per warp.
// k_chunk0: input index of xs column 0.
template <int FMT, int NT>
__device__ __forceinline__ void slab_units(float (&acc)[NT][4], const uint8_t* __restrict__ wq,
                                           const uint8_t* __restrict__ ws, int u_begin, int u_end,
                                           const __half* xs, int ldx, int k_chunk0, const float* xsum,
                                           int nblk) {
  constexpr int KU = unit_k(FMT);
  constexpr int UNR = (FMT == F16) ? 8 : 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2;
  for (int u0 = u_begin + warp; u0 < u_end; u0 += kWarps * UNR) {
    uint4 q[UNR];
    uint2 s[UNR];
#pragma unroll
    for (int i = 0; i < UNR; ++i) {
      const int u = u0 + i * kWarps;
      if (u < u_end) {
        q[i] = ldg_stream(wq + (size_t)u * kUnitBytes + lane * 16);
        s[i] = load_scales<FMT>(ws, u, g);
      }
    }
#pragma unroll
    for (int i = 0; i < UNR; ++i) {
      const int u = u0 + i * kWarps;
      if (u < u_end) {
        const int kl = u * KU - k_chunk0;
        unit_mma<FMT, NT>(acc, q[i], s[i], xs + kl, ldx, xsum, nblk, kl / 32, lane);
      }
    }
  }
}

// Cross-warp reduction: red[kWarps][NT*8][16] fp32 in shared memory.
template <int NT>
__device__ __forceinline__ void slab_store_partial(const float (&acc)[NT][4], float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  float* r = red + warp * (NT * 8 * 16);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int tok = nt * 8 + 2 * t;
    r[tok * 16 + g] = acc[nt][0];
    r[(tok + 1) * 16 + g] = acc[nt][1];
    r[tok * 16 + g + 8] = acc[nt][2];
    r[(tok + 1) * 16 + g + 8] = acc[nt][3];
  }
}

template <int NT>
__device__ __forceinline__ void slab_sum(const float* red, int tok, int pg, float& lo, float& hi) {
  lo = 0.f;
  hi = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    lo += red[w * (NT * 8 * 16) + tok * 16 + pg];
    hi += red[w * (NT * 8 * 16) + tok * 16 + pg + 8];
  }
}

// ------------------------------------------------------------------ staging
// Per-token RMSNorm factor 1/sqrt(mean(x^2)+eps) of fp32 rows (one warp per token).
__device__ __forceinline__ void stage_rms(float* rs, const float* x, int ldx_g, const int* rows, int ntok,
                                          int K, float eps) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int tk = warp; tk < ntok; tk += kWarps) {
    const float* xr = x + (size_t)(rows ? rows[tk] : tk) * ldx_g;
    float ss = 0.f;
    for (int k = lane * 4; k < K; k += 128) {
      const float4 v = *reinterpret_cast<const float4*>(xr + k);
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) rs[tk] = rsqrtf(ss / (float)K + eps);
  }
}

// xs[tk][j] = fp16(x[row(tk)][k0 + j] * rs[tk] * w[k0 + j]) for j < kc; rows tk >= ntok are zero.
__device__ __forceinline__ void stage_norm_chunk(__half* xs, int ldx, const float* x, int ldx_g, const int* rows,
                                                 int ntok, int ntok_pad, const float* rs, const __half* w, int k0,
                                                 int kc) {
  const int per_row = kc / 4;
  for (int i = threadIdx.x; i < ntok_pad * per_row; i += kThreads) {
    const int tk = i / per_row, j = (i - tk * per_row) * 4;
    __half2 o0, o1;
    if (tk < ntok) {
      const float* xr = x + (size_t)(rows ? rows[tk] : tk) * ldx_g + k0 + j;
      const float4 v = *reinterpret_cast<const float4*>(xr);
      const float r = rs[tk];
      const __half2 w0 = *reinterpret_cast<const __half2*>(w + k0 + j);
      const __half2 w1 = *reinterpret_cast<const __half2*>(w + k0 + j + 2);
      o0 = __floats2half2_rn(v.x * r * __low2float(w0), v.y * r * __high2float(w0));
      o1 = __floats2half2_rn(v.z * r * __low2float(w1), v.w * r * __high2float(w1));
    } else {
      o0 = __float2half2_rn(0.f);
      o1 = o0;
    }
    __half2* d = reinterpret_cast<__half2*>(xs + tk * ldx + j);
    d[0] = o0;
    d[1] = o1;
  }
}

// xs[tk][j] = src[row(tk)][k0 + j] (fp16), rows tk >= ntok zero.  kc % 8 == 0.
__device__ __forceinline__ void stage_f16_chunk(__half* xs, int ldx, const __half* src, int lds, const int* rows,
                                                int row0, int ntok, int ntok_pad, int k0, int kc) {
  const int per_row = kc / 8;
  for (int i = threadIdx.x; i < ntok_pad * per_row; i += kThreads) {
    const int tk = i / per_row, j = (i - tk * per_row) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (tk < ntok) {
      const int r = rows ? rows[tk] : row0 + tk;
      v = *reinterpret_cast<const uint4*>(src + (size_t)r * lds + k0 + j);
    }
    *reinterpret_cast<uint4*>(xs + tk * ldx + j) = v;
  }
}

// Per-token sums of each 32-input block of the staged chunk (I8ASYM zero points).
__device__ __forceinline__ void stage_block_sums(float* xsum, const __half* xs, int ldx, int ntok_pad, int kc) {
  const int nblk = kc / 32;
  for (int i = threadIdx.x; i < ntok_pad * nblk; i += kThreads) {
    const int tk = i / nblk, b = i - tk * nblk;
    const __half2* p = reinterpret_cast<const __half2*>(xs + tk * ldx + b * 32);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float2 f = __half22float2(p[j]);
      s += f.x + f.y;
    }
    xsum[i] = s;
  }
}

// ------------------------------------------------------------------ misc
__device__ __forceinline__ float silu(float z) { return z / (1.f + __expf(-z)); }

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}
__device__ __forceinline__ int argmax_key_index(unsigned long long k) {
  return (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
}

// Device status bits (reported by uocr_sync).
constexpr int kStatusToken = 1;
constexpr int kStatusPosition = 2;

}  // namespace uocr
