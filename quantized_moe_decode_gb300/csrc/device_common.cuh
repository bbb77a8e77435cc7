// Device-side building blocks shared by the decode-step kernels (sm_103a).
//
// Weight layout ("packed"): a matrix W[N][K] is cut into slabs of 16 output
// rows; a slab is cut into units of 16 rows x KU inputs, KU = 32 (Q8_0,
// I8ASYM, F16) or 64 (Q4_0).  A unit holds the codes in the register order of
// the m16n8k16 tensor-core A fragment: lane L reads bytes [16L, 16L+16) of
// each 512-byte quarter (one quarter for the 8-bit and 4-bit formats, two for
// fp16) and holds its fragments without any shuffle.  Scales live in a
// separate plane, per unit and per fragment row group g = lane/4:
// Q8_0 {d[g], d[g+8]} (4 B), Q4_0 {d[g][b0], d[g+8][b0], d[g][b1], d[g+8][b1]}
// (8 B), I8ASYM {s[g], s[g+8], z[g], z[g+8]} (8 B).
//
// Dequantisation ("Unlimited-OCR on Apple Silicon with C and Metal",
// "Quantizzazione": no full fp16 copy of the weights, dequantise inside the
// matmul).  Integer codes become exact fp16 integers with the exponent-bias
// method (OR the code into the mantissa of 1024 and subtract the bias), the
// tensor core multiplies them with fp16 activations accumulating in fp32,
// and the block scale is applied to the fp32 block sum, so no weight value is
// ever rounded.
//
// Weight streaming: in every GEMV-like kernel each warp streams its own
// units through a private shared-memory ring with 16-byte cp.async copies
// (D units in flight per warp; on GB300 ordinary loads reach the HBM peak
// with ~64 KB in flight per SM, while one-dimensional bulk copies need about
// three times as much).  Kernels are chained with programmatic dependent
// launch: a kernel's first weight copies are issued before it waits for the
// kernel that produces its activations.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

namespace uocr {

enum Fmt : int { F16 = 0, Q8_0 = 1, Q4_0 = 2, I8ASYM = 3 };

// Streaming CTAs: kWarps warps, each streaming its own weight units.
constexpr int kWarps = 8;
constexpr int kConsumers = kWarps * 32;
constexpr int kThreads = kConsumers;
// Build-time tuning (defaults are the measured best on GB300):
//   UOCR_RING_DEPTH  units in flight per warp (weight ring slots)
//   UOCR_MIN_BLOCKS  minimum resident CTAs per SM asked of the compiler
//   UOCR_UNROLL      units consumed per step of the inner loop (1 or 2)
#ifndef UOCR_RING_DEPTH
#define UOCR_RING_DEPTH 5
#endif
#ifndef UOCR_MIN_BLOCKS
#define UOCR_MIN_BLOCKS 2
#endif
#ifndef UOCR_UNROLL
#define UOCR_UNROLL 1
#endif
//   UOCR_PDL_LATE    kernels that let their dependents launch only after their
//                    weight stream instead of at their start (bit mask:
//                    1 GEMV, 2 router, 4 expert kernels, 8 attention)
//   UOCR_KS_MAX      most warps that share one slab (8, 4, 2 or 1)
#ifndef UOCR_KS_MAX
#define UOCR_KS_MAX 8
#endif
//   UOCR_WARM_TOPK   1 = the router runs its top-k once before waiting (code warm-up)
#ifndef UOCR_WARM_TOPK
#define UOCR_WARM_TOPK 1
#endif
//   UOCR_ATTN_WARPS  warps per attention CTA (4 or 8)
#ifndef UOCR_ATTN_WARPS
#define UOCR_ATTN_WARPS 4
#endif
//   UOCR_COMBINE_B   outputs per thread per batch of loads in the expert combine
//                    (fewer when more CTAs per SM leave fewer registers per thread)
#ifndef UOCR_COMBINE_B
#if UOCR_MIN_BLOCKS >= 3
#define UOCR_COMBINE_B 3
#else
#define UOCR_COMBINE_B 6
#endif
#endif
#ifndef UOCR_PDL_LATE
#define UOCR_PDL_LATE 8
#endif
constexpr int kRingDepth = UOCR_RING_DEPTH;
constexpr int kMinBlocks = UOCR_MIN_BLOCKS;
constexpr int kUnroll = UOCR_UNROLL;
constexpr int kPdlLate = UOCR_PDL_LATE;
constexpr int kKsMax = UOCR_KS_MAX;
constexpr int kWarmTopk = UOCR_WARM_TOPK;
enum PdlKernel : int { PDL_GEMV = 1, PDL_ROUTER = 2, PDL_EXPERT = 4, PDL_ATTN = 8 };
static_assert(kRingDepth >= 2 && kRingDepth <= 16, "ring depth");
static_assert(kUnroll == 1 || kUnroll == 2, "unroll");
constexpr int kSlotBytes = 1024;         // codes (512 or 1024) + lane-private scales (32 x 8 B)

__host__ __device__ constexpr int unit_k(int fmt) { return fmt == Q4_0 ? 64 : 32; }
__host__ __device__ constexpr int unit_bytes(int fmt) { return fmt == F16 ? 1024 : 512; }
__host__ __device__ constexpr int unit_scale_bytes(int fmt) {
  return fmt == Q8_0 ? 32 : (fmt == F16 ? 0 : 64);
}

// A packed matrix as the kernels see it.
struct PMat {
  const uint8_t* q;   // slabs * U * unit_bytes
  const uint8_t* s;   // slabs * U * unit_scale_bytes
  int n_slabs;        // ceil(N_packed / 16)
  int U;              // units per slab = K / unit_k
  int K;
  long long q_stride; // bytes between consecutive experts (expert arrays)
  long long s_stride;
};

// Device status bits (reported by uocr_sync).
constexpr int kStatusToken = 1;
constexpr int kStatusPosition = 2;
constexpr int kStatusTimeout = 4;

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

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

// d = a * b (a zero accumulator operand instead of a zeroed register quad)
__device__ __forceinline__ void mma_16816_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  const float z = 0.f;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}

// int8 tensor-core MMA, m16n8k32, int32 accumulate from zero: A signed or
// unsigned bytes (ASIGNED), B signed bytes.
template <bool ASIGNED>
__device__ __forceinline__ void mma_i8_z(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  const int z = 0;
  if constexpr (ASIGNED)
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(z));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(z));
}

__device__ __forceinline__ void ldsm_x2(uint32_t& r0, uint32_t& r1, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(smem_u32(p)));
  return r;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ---- per-thread asynchronous copies (cp.async)
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---- mbarrier + bulk copy
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same with a suspend-time hint: the thread sleeps until the phase
// completes or about `ns` nanoseconds pass (waits that can last microseconds
// leave the issue slots to the warps doing the work).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// Bounded wait: false after kSpinLimit polls (each poll may suspend briefly).
constexpr uint32_t kSpinLimit = 1u << 22;
template <uint32_t Limit = kSpinLimit>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < Limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Bounded sleeping wait: false after Limit polls of up to `ns` each.
template <uint32_t Limit = (1u << 16)>
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  for (uint32_t i = 0; i < Limit; ++i)
    if (mbar_try_wait_sleep(bar, parity, ns)) return true;
  return false;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ---- programmatic dependent launch
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t h2_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ __half2 h2_bits(uint16_t b) {
  return __halves2half2(__ushort_as_half(b), __ushort_as_half(b));
}

// ------------------------------------------------------------------ code -> fp16
// Q8_0: bytes (b0 b1 b2 b3) of signed codes -> (b0,b1), (b2,b3) as fp16 pairs.
__device__ __forceinline__ void dq_s8x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;                      // code + 128, unsigned
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);  // fp16 1024 + u0, 1024 + u1
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = h2_bits(0x6480);                    // 1152 = 1024 + 128
  lo = h2_u32(__hsub2(u32_h2(a), bias));
  hi = h2_u32(__hsub2(u32_h2(b), bias));
}

// I8ASYM: unsigned codes -> fp16 pairs (exact integers 0..255).
__device__ __forceinline__ void dq_u8x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t a = __byte_perm(w, 0x64646464u, 0x4140);
  const uint32_t b = __byte_perm(w, 0x64646464u, 0x4342);
  const __half2 bias = h2_bits(0x6400);  // 1024
  lo = h2_u32(__hsub2(u32_h2(a), bias));
  hi = h2_u32(__hsub2(u32_h2(b), bias));
}

// Q4_0: one 32-bit word = the 8 codes of one k-step fragment, nibble positions
// a0@0 a2@4 a4@8 a6@12 a1@16 a3@20 a5@24 a7@28; returns the four A registers
// (a0,a1) (a2,a3) (a4,a5) (a6,a7) as fp16 pairs of (code - 8).
__device__ __forceinline__ void dq_q4(uint32_t w, uint32_t (&r)[4]) {
  const uint32_t x0 = lop_and_or(w, 0x000F000Fu, 0x64006400u);  // 1024 + n
  const uint32_t x1 = lop_and_or(w, 0x00F000F0u, 0x64006400u);  // 1024 + 16 n
  const uint32_t w8 = w >> 8;
  const uint32_t x2 = lop_and_or(w8, 0x000F000Fu, 0x64006400u);
  const uint32_t x3 = lop_and_or(w8, 0x00F000F0u, 0x64006400u);
  const __half2 k1032 = h2_bits(0x6408);  // 1024 + 8
  const __half2 k1_16 = h2_bits(0x2C00);  // 1/16
  const __half2 km72 = h2_bits(0xD480);   // -(64 + 8)
  r[0] = h2_u32(__hsub2(u32_h2(x0), k1032));
  r[1] = h2_u32(__hfma2(u32_h2(x1), k1_16, km72));
  r[2] = h2_u32(__hsub2(u32_h2(x2), k1032));
  r[3] = h2_u32(__hfma2(u32_h2(x3), k1_16, km72));
}

__device__ __forceinline__ float half_lo(uint32_t u) { return __half2float(__ushort_as_half((uint16_t)(u & 0xFFFF))); }
__device__ __forceinline__ float half_hi(uint32_t u) { return __half2float(__ushort_as_half((uint16_t)(u >> 16))); }

// ------------------------------------------------------------------ B operands
// A B provider returns, for n-tile nt and the 32 inputs starting at kk, the
// four B registers of two k-steps: (k 2t..2t+1, token g), (k 2t+8.., g),
// (k 16+2t.., g), (k 24+2t.., g).

// Activations staged in shared memory xs[row][ldx] (fp16), contiguous tokens.
struct BSmem {
  const __half* base;  // this lane's ldmatrix row address at kk = 0, n-tile 0
  int nt_stride;       // halves between n-tiles (8 rows)
  __device__ __forceinline__ BSmem(const __half* xs, int ldx)
      : base(xs + (threadIdx.x & 7) * ldx + 8 * ((threadIdx.x & 31) >> 3)), nt_stride(8 * ldx) {}
  __device__ __forceinline__ void operator()(int nt, int kk, int, uint32_t (&b)[4]) const {
    ldsm_x4(b, base + nt * nt_stride + kk);
  }
};

// Activations staged in shared memory, tokens gathered through a row list
// (rows[] holds the staged row of each token of the item, -1 = padding).
struct BSmemGather {
  const __half* xs;
  int ldx;
  const int* rows;  // [n-tiles * 8]
  const __half* zero;  // a zero row of at least 32 halves (padding tokens)
  __device__ __forceinline__ void operator()(int nt, int kk, int lane, uint32_t (&b)[4]) const {
    const int r = rows[nt * 8 + (lane & 7)];
    const __half* p = r >= 0 ? xs + r * ldx + kk + 8 * (lane >> 3) : zero + 8 * (lane >> 3);
    ldsm_x4(b, p);
  }
};

// Activations in global memory already in B-fragment order: for tile tl of 8
// tokens and 32-input unit u, lane L's 16 bytes at ((tl*K32 + u)*32 + L)*16.
struct BGlobalFrag {
  const uint8_t* base;  // first tile of this item
  int k32;              // K / 32
  __device__ __forceinline__ void operator()(int nt, int kk, int lane, uint32_t (&b)[4]) const {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(base + (((size_t)nt * k32 + (kk >> 5)) * 32 + lane) * 16));
    b[0] = v.x;
    b[1] = v.y;
    b[2] = v.z;
    b[3] = v.w;
  }
};

// Activations in shared memory in B-fragment order (a copy of the global
// layout below): lane L's 16 bytes at ((tl*K32 + u)*32 + L)*16.
struct BSmemFrag {
  const uint8_t* base;
  int k32;
  __device__ __forceinline__ void operator()(int nt, int kk, int lane, uint32_t (&b)[4]) const {
    const uint4 v = lds128(base + (((size_t)nt * k32 + (kk >> 5)) * 32 + lane) * 16);
    b[0] = v.x;
    b[1] = v.y;
    b[2] = v.z;
    b[3] = v.w;
  }
};

// Byte offset of activation (token n of tile tl, input i) in B-fragment order.
__host__ __device__ __forceinline__ size_t bfrag_offset(int tl, int n, int i, int k32) {
  const int u = i >> 5, kk = i & 31;
  const int ks = kk >> 4, kw = kk & 15;
  const int hi8 = kw >> 3, t = (kw & 7) >> 1, hf = kw & 1;
  const int lane = n * 4 + t;
  return (((size_t)tl * k32 + u) * 32 + lane) * 16 + (ks * 2 + hi8) * 4 + hf * 2;
}

// Sum of the 32 inputs of the current block for tokens 2t and 2t+1 of an
// n-tile, from the B registers the lanes already hold (I8ASYM zero points).
__device__ __forceinline__ void block_sums(const uint32_t (&b)[4], int lane, float& s0, float& s1) {
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(u32_h2(b[i]));
    s += f.x + f.y;
  }
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  s += __shfl_xor_sync(0xffffffffu, s, 2);  // token g's block sum in every lane of group g
  const int t = lane & 3;
  s0 = __shfl_sync(0xffffffffu, s, (2 * t) * 4);
  s1 = __shfl_sync(0xffffffffu, s, (2 * t + 1) * 4);
}

// ------------------------------------------------------------------ unit compute
// One unit from shared memory (`a` = the unit's bytes, `sc` = this lane's own
// copy of its row group's scale entry) against NT n-tiles of B.
// acc[nt][0..3] follows the m16n8 C fragment: (row g, token 2t), (g, 2t+1),
// (g+8, 2t), (g+8, 2t+1).
template <int FMT, int NT, class BP>
__device__ __forceinline__ void unit_mma(float (&acc)[NT][4], const uint8_t* a, const uint8_t* sc, const BP& bp,
                                         int kk, int lane, int nt_used) {
  if constexpr (FMT == F16) {
    const uint4 q0 = lds128(a + lane * 16);
    const uint4 q1 = lds128(a + 512 + lane * 16);
    const uint32_t A0[4] = {q0.x, q0.y, q0.z, q0.w};
    const uint32_t A1[4] = {q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (NT == 1 || nt < nt_used) {
        uint32_t B[4];
        bp(nt, kk, lane, B);
        mma_16816(acc[nt], A0, B[0], B[1]);
        mma_16816(acc[nt], A1, B[2], B[3]);
      }
    }
  } else if constexpr (FMT == Q8_0 || FMT == I8ASYM) {
    const uint4 q = lds128(a + lane * 16);
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
    float d_lo, d_hi, z_lo = 0.f, z_hi = 0.f;
    if constexpr (FMT == Q8_0) {
      const uint32_t s = *reinterpret_cast<const uint32_t*>(sc);
      d_lo = half_lo(s);
      d_hi = half_hi(s);
    } else {
      const uint2 s = *reinterpret_cast<const uint2*>(sc);
      d_lo = half_lo(s.x);
      d_hi = half_hi(s.x);
      z_lo = half_lo(s.y);
      z_hi = half_hi(s.y);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (NT == 1 || nt < nt_used) {
        uint32_t B[4];
        bp(nt, kk, lane, B);
        float c[4];
        mma_16816_z(c, A0, B[0], B[1]);
        mma_16816(c, A1, B[2], B[3]);
        if constexpr (FMT == I8ASYM) {
          float s0, s1;
          block_sums(B, lane, s0, s1);
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
    }
  } else {  // Q4_0: 4 k-steps, 2 blocks
    const uint4 q = lds128(a + lane * 16);
    uint32_t A[4][4];
    dq_q4(q.x, A[0]);
    dq_q4(q.y, A[1]);
    dq_q4(q.z, A[2]);
    dq_q4(q.w, A[3]);
    const uint2 s = *reinterpret_cast<const uint2*>(sc);
    const float d0_lo = half_lo(s.x), d0_hi = half_hi(s.x);
    const float d1_lo = half_lo(s.y), d1_hi = half_hi(s.y);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (NT == 1 || nt < nt_used) {
        uint32_t B0[4], B1[4];
        bp(nt, kk, lane, B0);
        bp(nt, kk + 32, lane, B1);
        float c[4];
        mma_16816_z(c, A[0], B0[0], B0[1]);
        mma_16816(c, A[1], B0[2], B0[3]);
        acc[nt][0] = fmaf(d0_lo, c[0], acc[nt][0]);
        acc[nt][1] = fmaf(d0_lo, c[1], acc[nt][1]);
        acc[nt][2] = fmaf(d0_hi, c[2], acc[nt][2]);
        acc[nt][3] = fmaf(d0_hi, c[3], acc[nt][3]);
        float e[4];
        mma_16816_z(e, A[2], B1[0], B1[1]);
        mma_16816(e, A[3], B1[2], B1[3]);
        acc[nt][0] = fmaf(d1_lo, e[0], acc[nt][0]);
        acc[nt][1] = fmaf(d1_lo, e[1], acc[nt][1]);
        acc[nt][2] = fmaf(d1_hi, e[2], acc[nt][2]);
        acc[nt][3] = fmaf(d1_hi, e[3], acc[nt][3]);
      }
    }
  }
}

// ------------------------------------------------------------------ int8 activations
// Dynamic int8 activations ("Falcon-OCR INT8 OpenVINO IR": the linear layers'
// inputs are quantised dynamically in groups of 32): each group of 32 inputs
// of a row has a scale s = max|x| / 127 and codes round(x / s), and the
// product runs on the int8 tensor cores (m16n8k32, exact int32 per group).
//
// The k order inside a group: lane (g, t) of a packed 8-bit unit holds, per
// row, the codes of k = 2t, 2t+1, 2t+8, 2t+9 (and 16 + the same); a Q4_0 word's
// low / high nibbles give k = 2t, 2t+8, 2t+1, 2t+9.  The int8 A fragment wants
// "virtual" k = 4t .. 4t+3 (and 16 + the same), so virtual position v stands
// for the real k those bytes hold, and the activation codes of a group are
// staged at the same virtual positions: the sum over k is unchanged.
template <int FMT>
__host__ __device__ __forceinline__ int act_vpos(int k) {  // real k (0..31) -> virtual position
  const int h = k & 16, kk = k & 15;
  const int hi8 = kk >> 3, t = (kk & 7) >> 1, odd = kk & 1;
  const int j = FMT == Q4_0 ? (odd ? 2 : 0) + hi8 : hi8 * 2 + odd;
  return h + 4 * t + j;
}

// Activation codes staged in shared memory: xq[row][ldq] int8 (ldq = K + 16;
// groups of 32 in virtual order), scales sc[group][ldr] fp32 and code sums
// sm[group][ldr] int32 (ldr = the padded row count; rows 2t, 2t+1 adjacent).
struct BSmemI8 {
  const uint8_t* lane_base;  // this lane's ldmatrix row address at k = 0, n-tile 0
  int nt_stride;             // bytes between n-tiles (8 rows)
  const float* sc;
  const int* sm;
  int ldr;
  __device__ __forceinline__ BSmemI8(const int8_t* xq, int ldq, const float* sc_, const int* sm_, int ldr_)
      : lane_base(reinterpret_cast<const uint8_t*>(xq) + (threadIdx.x & 7) * ldq + 16 * ((threadIdx.x & 31) >> 3)),
        nt_stride(8 * ldq),
        sc(sc_),
        sm(sm_),
        ldr(ldr_) {}
};

__device__ __forceinline__ BSmemI8 make_bsmem_i8(const uint8_t* base, int ntok_pad, int K) {
  const float* sc = reinterpret_cast<const float*>(base + ntok_pad * (K + 16));
  return BSmemI8(reinterpret_cast<const int8_t*>(base), K + 16, sc, reinterpret_cast<const int*>(sc + (K / 32) * ntok_pad),
                 ntok_pad);
}

// Bytes of the int8 staging of ntok_pad rows of K inputs (codes, scales, sums).
__host__ __device__ __forceinline__ int act_i8_codes_bytes(int ntok_pad, int K) { return ntok_pad * (K + 16); }
__host__ __device__ __forceinline__ int act_i8_bytes(int ntok_pad, int K) {
  return act_i8_codes_bytes(ntok_pad, K) + 2 * (K / 32) * ntok_pad * 4;
}

// One unit against int8 activations: Q8_0 / I8ASYM units hold one group of 32,
// Q4_0 units two.  acc[nt][i] follows the C fragment as in unit_mma.
template <int FMT, int NT>
__device__ __forceinline__ void unit_mma_i8(float (&acc)[NT][4], const uint8_t* a, const uint8_t* scp,
                                            const BSmemI8& bp, int kk, int lane, int nt_used) {
  static_assert(FMT == Q8_0 || FMT == Q4_0 || FMT == I8ASYM, "int8 activations need 8- or 4-bit weight codes");
  const uint4 q = lds128(a + lane * 16);
  const int t = lane & 3;
  if constexpr (FMT == Q8_0 || FMT == I8ASYM) {
    const uint32_t A[4] = {__byte_perm(q.x, q.y, 0x5410), __byte_perm(q.x, q.y, 0x7632),
                           __byte_perm(q.z, q.w, 0x5410), __byte_perm(q.z, q.w, 0x7632)};
    float d_lo, d_hi, z_lo = 0.f, z_hi = 0.f;
    if constexpr (FMT == Q8_0) {
      const uint32_t sv = *reinterpret_cast<const uint32_t*>(scp);
      d_lo = half_lo(sv);
      d_hi = half_hi(sv);
    } else {
      const uint2 sv = *reinterpret_cast<const uint2*>(scp);
      d_lo = half_lo(sv.x);
      d_hi = half_hi(sv.x);
      z_lo = half_lo(sv.y);
      z_hi = half_hi(sv.y);
    }
    const int grp = kk >> 5;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (NT == 1 || nt < nt_used) {
        uint32_t b0, b1;
        ldsm_x2(b0, b1, bp.lane_base + nt * bp.nt_stride + kk);
        int c[4];
        mma_i8_z<FMT == Q8_0>(c, A, b0, b1);
        const int ix = grp * bp.ldr + nt * 8 + 2 * t;  // rows 2t, 2t+1 of the n-tile
        const float2 sx = *reinterpret_cast<const float2*>(bp.sc + ix);
        float c0 = (float)c[0], c1 = (float)c[1], c2 = (float)c[2], c3 = (float)c[3];
        if constexpr (FMT == I8ASYM) {  // sum (q - z) x = sum q x - z sum x
          const int2 m = *reinterpret_cast<const int2*>(bp.sm + ix);
          c0 = fmaf(-z_lo, (float)m.x, c0);
          c1 = fmaf(-z_lo, (float)m.y, c1);
          c2 = fmaf(-z_hi, (float)m.x, c2);
          c3 = fmaf(-z_hi, (float)m.y, c3);
        }
        acc[nt][0] = fmaf(d_lo * sx.x, c0, acc[nt][0]);
        acc[nt][1] = fmaf(d_lo * sx.y, c1, acc[nt][1]);
        acc[nt][2] = fmaf(d_hi * sx.x, c2, acc[nt][2]);
        acc[nt][3] = fmaf(d_hi * sx.y, c3, acc[nt][3]);
      }
    }
  } else {  // Q4_0: groups kk/32 and kk/32 + 1, unsigned nibbles, sum (q - 8) x = sum q x - 8 sum x
    const uint32_t m4 = 0x0F0F0F0Fu;
    const uint32_t A0[4] = {q.x & m4, (q.x >> 4) & m4, q.y & m4, (q.y >> 4) & m4};
    const uint32_t A1[4] = {q.z & m4, (q.z >> 4) & m4, q.w & m4, (q.w >> 4) & m4};
    const uint2 sv = *reinterpret_cast<const uint2*>(scp);
    const float d0_lo = half_lo(sv.x), d0_hi = half_hi(sv.x), d1_lo = half_lo(sv.y), d1_hi = half_hi(sv.y);
    const int grp = kk >> 5;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (NT == 1 || nt < nt_used) {
        uint32_t B[4];
        ldsm_x4(B, bp.lane_base + nt * bp.nt_stride + kk);
        int c[4], e[4];
        mma_i8_z<false>(c, A0, B[0], B[1]);
        mma_i8_z<false>(e, A1, B[2], B[3]);
        const int ix = grp * bp.ldr + nt * 8 + 2 * t;  // group grp, rows 2t, 2t+1; group grp+1 at + ldr
        const float2 sx = *reinterpret_cast<const float2*>(bp.sc + ix);
        const float2 sy = *reinterpret_cast<const float2*>(bp.sc + ix + bp.ldr);
        const int2 mx = *reinterpret_cast<const int2*>(bp.sm + ix);
        const int2 my = *reinterpret_cast<const int2*>(bp.sm + ix + bp.ldr);
        // int32 exact: |sum q x| <= 15 * 127 * 32
        const float c0 = (float)(c[0] - 8 * mx.x), c1 = (float)(c[1] - 8 * mx.y);
        const float c2 = (float)(c[2] - 8 * mx.x), c3 = (float)(c[3] - 8 * mx.y);
        const float e0 = (float)(e[0] - 8 * my.x), e1 = (float)(e[1] - 8 * my.y);
        const float e2 = (float)(e[2] - 8 * my.x), e3 = (float)(e[3] - 8 * my.y);
        acc[nt][0] = fmaf(d0_lo * sx.x, c0, fmaf(d1_lo * sy.x, e0, acc[nt][0]));
        acc[nt][1] = fmaf(d0_lo * sx.y, c1, fmaf(d1_lo * sy.y, e1, acc[nt][1]));
        acc[nt][2] = fmaf(d0_hi * sx.x, c2, fmaf(d1_hi * sy.x, e2, acc[nt][2]));
        acc[nt][3] = fmaf(d0_hi * sx.y, c3, fmaf(d1_hi * sy.y, e3, acc[nt][3]));
      }
    }
  }
}

// A unit against whichever activations the B provider stages.
template <int FMT, int NT, class BP>
__device__ __forceinline__ void unit_any(float (&acc)[NT][4], const uint8_t* a, const uint8_t* sc, const BP& bp, int kk,
                                         int lane, int nt_used) {
  if constexpr (std::is_same<BP, BSmemI8>::value)
    unit_mma_i8<FMT, NT>(acc, a, sc, bp, kk, lane, nt_used);
  else
    unit_mma<FMT, NT>(acc, a, sc, bp, kk, lane, nt_used);
}

// Codes of one group of 32 inputs held by 4 lanes (lane q = lane & 3 holds the
// inputs 8q .. 8q+7 as P0 = codes 0..3, P1 = codes 4..7) -> the 8 bytes this
// lane stores at virtual offset 16 (q >> 1) + 8 (q & 1): the even lane of a
// pair builds virtual words 0-1 of its half, the odd lane words 2-3, each from
// its own and its partner's codes (word t = real 2t, 2t+1, 2t+8, 2t+9 for
// 8-bit codes; 2t, 2t+8, 2t+1, 2t+9 for Q4_0; see act_vpos).
template <int FMT>
__device__ __forceinline__ uint2 act_i8_words(uint32_t P0, uint32_t P1, int q) {
  const bool odd = q & 1;
  const uint32_t mine = odd ? P1 : P0;
  const uint32_t other = __shfl_xor_sync(0xffffffffu, odd ? P0 : P1, 1);
  const uint32_t lo = odd ? other : mine, hi = odd ? mine : other;  // even lane's codes, odd lane's codes
  constexpr uint32_t s0 = FMT == Q4_0 ? 0x5140u : 0x5410u, s1 = FMT == Q4_0 ? 0x7362u : 0x7632u;
  return make_uint2(__byte_perm(lo, hi, s0), __byte_perm(lo, hi, s1));
}

// round-half-even(x / s) of the IEEE quotient: the rare inputs within 2^-12 of
// a half-integer (kept out of line so that the staging code stays small)
static __device__ __noinline__ float act_i8_exact_code(float x, float s) { return rintf(x / s); }

// Quantise 8 consecutive inputs (lane q of a 4-lane group of 32) and store the
// group's codes, scale and code sum.  on: the lane's group lies inside the row
// (whole groups only, so the 4 lanes agree).
template <int FMT>
__device__ __forceinline__ void act_i8_group(const float (&h)[8], bool on, uint8_t* gq, float* gsc, int* gsm) {
  const int q = threadIdx.x & 3;
  float m = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(h[e]));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  // fp32 decisions: code = round-half-even(x / s) of the IEEE quotient.  x * (1/s)
  // lies within 3 ulp(127) < 2^-12 of that quotient, so wherever it is farther
  // than 2^-12 from a half-integer both round to the same code; the rest take
  // the exact divide.
  const float sc = m / 127.0f;
  const float inv = sc > 0.f ? 1.0f / sc : 0.f;
  uint32_t P[2] = {0u, 0u};
  int cs = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float y = h[e] * inv;
    float cf = rintf(y);
    if (fabsf(y - cf) > 0.5f - 0x1p-12f) cf = act_i8_exact_code(h[e], sc);
    const int c = max(-127, min(127, (int)cf));
    cs += c;
    P[e >> 2] |= (uint32_t)(c & 0xFF) << (8 * (e & 3));
  }
  cs += __shfl_xor_sync(0xffffffffu, cs, 1);
  cs += __shfl_xor_sync(0xffffffffu, cs, 2);
  const uint2 wds = act_i8_words<FMT>(P[0], P[1], q);
  if (on) {
    *reinterpret_cast<uint2*>(gq + 16 * (q >> 1) + 8 * (q & 1)) = wds;
    if (q == 0) {
      *gsc = sc;
      *gsm = cs;
    }
  }
}

// Rows tk < ntok of the CTA's token group quantised per group of 32 into the
// layout of BSmemI8 at `base` (codes, then scales, then sums; ldr = ntok_pad);
// rows ntok..ntok_pad hold zero codes and scales.  NORM: RMSNorm of fp32 rows
// (weight w) rounded to fp16 as the fp16 staging rounds them; else fp16 rows.
// All warps share the (row, 256-input chunk) items, two in flight per warp, so
// a single row costs one load latency per pass, not one per 128 inputs.
constexpr int kActChunk = 256;
constexpr int kActMaxChunks = 32;  // K <= 8192
template <int FMT, bool NORM>
__device__ __forceinline__ void stage_act_i8(uint8_t* base, const float* xf, const __half* xh, int lds, int ntok,
                                             int ntok_pad, const __half* w, int K, float eps) {
  __shared__ float s_part[16 * kActMaxChunks];  // per (row, chunk) sums of squares (NORM)
  __shared__ float s_r[16];                     // per row 1 / rms (NORM)
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5, lane = threadIdx.x & 31;
  const int ng = K / 32, ldq = K + 16, nch = (K + kActChunk - 1) / kActChunk;
  uint8_t* xq = base;
  float* xsc = reinterpret_cast<float*>(base + act_i8_codes_bytes(ntok_pad, K));
  int* xsm = reinterpret_cast<int*>(xsc + ng * ntok_pad);
  for (int tk = ntok + warp; tk < ntok_pad; tk += nw) {  // padding rows
    for (int i = lane; i < K / 16; i += 32) *reinterpret_cast<uint4*>(xq + tk * ldq + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
    for (int i = lane; i < ng; i += 32) {
      xsc[i * ntok_pad + tk] = 0.f;
      xsm[i * ntok_pad + tk] = 0;
    }
  }
  const int items = ntok * nch;
  constexpr int NI = NORM ? 4 : 8;  // items in flight per warp
  if constexpr (NORM) {
    for (int i0 = warp; i0 < items; i0 += NI * nw) {
      float4 v[NI][2];
#pragma unroll
      for (int u = 0; u < NI; ++u) {
        const int it = i0 + u * nw, tk = it / nch, k0 = (it - tk * nch) * kActChunk + 8 * lane;
        const bool on = it < items && k0 < K;
        const float4* src = reinterpret_cast<const float4*>(xf + (size_t)tk * lds + k0);
        v[u][0] = on ? src[0] : make_float4(0.f, 0.f, 0.f, 0.f);
        v[u][1] = on ? src[1] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < NI; ++u) {
        const int it = i0 + u * nw;
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) ss += v[u][j].x * v[u][j].x + v[u][j].y * v[u][j].y + v[u][j].z * v[u][j].z + v[u][j].w * v[u][j].w;
#pragma unroll
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0 && it < items) s_part[(it / nch) * kActMaxChunks + it % nch] = ss;
      }
    }
    __syncthreads();
    if ((int)threadIdx.x < ntok) {
      float ss = 0.f;
      for (int c = 0; c < nch; ++c) ss += s_part[threadIdx.x * kActMaxChunks + c];
      s_r[threadIdx.x] = rsqrtf(ss / (float)K + eps);
    }
    __syncthreads();
  }
  for (int i0 = warp; i0 < items; i0 += NI * nw) {
    // raw loads of all NI items first (one latency per pass), then quantise
    uint4 raw[NI][NORM ? 3 : 1];
#pragma unroll
    for (int u = 0; u < NI; ++u) {
      const int it = i0 + u * nw, tk = it / nch, k0 = (it - tk * nch) * kActChunk + 8 * lane;
      const bool on = it < items && k0 < K;
      if constexpr (NORM) {
        const uint4* src = reinterpret_cast<const uint4*>(xf + (size_t)tk * lds + k0);
        raw[u][0] = on ? src[0] : make_uint4(0u, 0u, 0u, 0u);
        raw[u][1] = on ? src[1] : make_uint4(0u, 0u, 0u, 0u);
        raw[u][2] = on ? *reinterpret_cast<const uint4*>(w + k0) : make_uint4(0u, 0u, 0u, 0u);
      } else {
        raw[u][0] = on ? *reinterpret_cast<const uint4*>(xh + (size_t)tk * lds + k0) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    // one item at a time through a rotating window (raw[0] is the current item), in a
    // rolled loop: the quantiser's code is run once per CTA from a cold instruction cache
#pragma unroll 1
    for (int u = 0; u < NI; ++u) {
      const int it = i0 + u * nw, tk = it / nch, k0 = (it - tk * nch) * kActChunk + 8 * lane;
      if (it >= items) break;  // warp-uniform: no later item of this pass is valid either
      const bool on = k0 < K;
      float h[8];
      if constexpr (NORM) {
        const uint32_t xr[8] = {raw[0][0].x, raw[0][0].y, raw[0][0].z, raw[0][0].w,
                                raw[0][1].x, raw[0][1].y, raw[0][1].z, raw[0][1].w};
        const uint32_t wr[4] = {raw[0][2].x, raw[0][2].y, raw[0][2].z, raw[0][2].w};
        const float r = on ? s_r[tk] : 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // fp16(x * r * w), the value the fp16 staging stores
          const __half2 wj = u32_h2(wr[j]);
          const float2 f = __half22float2(__floats2half2_rn(__uint_as_float(xr[2 * j]) * r * __low2float(wj),
                                                            __uint_as_float(xr[2 * j + 1]) * r * __high2float(wj)));
          h[2 * j] = f.x;
          h[2 * j + 1] = f.y;
        }
      } else {
        const uint32_t hr[4] = {raw[0][0].x, raw[0][0].y, raw[0][0].z, raw[0][0].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __half22float2(u32_h2(hr[j]));
          h[2 * j] = f.x;
          h[2 * j + 1] = f.y;
        }
      }
      const int g = k0 >> 5;  // group of 32 (the 4 lanes of this group agree on `on`)
      act_i8_group<FMT>(h, on, xq + tk * ldq + 32 * g, xsc + g * ntok_pad + tk, xsm + g * ntok_pad + tk);
#pragma unroll
      for (int j = 0; j + 1 < NI; ++j) {
#pragma unroll
        for (int c = 0; c < (NORM ? 3 : 1); ++c) raw[j][c] = raw[j + 1][c];
      }
    }
  }
}

template <int NT>
__device__ __forceinline__ void zero_acc(float (&acc)[NT][4]) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
}

// ------------------------------------------------------------------ warp weight streams
// Ring slot layout: codes at [0, unit_bytes), then this lane's scale entry at
// 512 + 8*lane (the 8-bit and 4-bit formats only).  Every byte of a slot is
// written and read by the same lane, so a slot needs no barrier.

// How a CTA's slabs are shared by its warps.  The CTA owns the slabs
// first + m*stride, m in [0, n).  Its kWarps warps form G = kWarps/ks groups
// of ks warps, ks the largest of 8, 4, 2, 1 dividing U, so that every warp
// gets the same number of units: group j takes m = j, j + G, ... (one slab
// per round) and warp r of the group the units [r*uw, (r+1)*uw) of each, uw =
// U/ks.  Only the ks warps of a group meet at a barrier, once per round.
struct SlabWork {
  int first, stride, n, U;
  int ks, uw, G, grp, rank;
};
__host__ __device__ __forceinline__ int warps_per_slab(int U) {
  const int ks = (U & 7) == 0 ? 8 : (U & 3) == 0 ? 4 : (U & 1) == 0 ? 2 : 1;
  return ks < kKsMax ? ks : kKsMax;
}
__device__ __forceinline__ SlabWork slab_work(int first, int stride, int n, int U) {
  SlabWork w;
  w.first = first;
  w.stride = stride;
  w.n = n;
  w.U = U;
  w.ks = warps_per_slab(U);
  w.uw = U / w.ks;
  w.G = kWarps / w.ks;
  const int warp = threadIdx.x >> 5;
  w.grp = warp / w.ks;
  w.rank = warp - w.grp * w.ks;
  return w;
}

// The units a warp fetches, in the order it consumes them: for each of its
// group's slabs (first + m*stride, m = grp, grp + G, ...) the run of uw units
// starting at rank*uw.  UOCR_STREAM_PTR selects how a unit's address is formed:
// 1 = this lane's code and scale pointers advance by one unit per fetch and are
// recomputed only when the run moves to the next slab; 0 = the unit index is
// recomputed from the warp-uniform counters at every fetch.
#ifndef UOCR_STREAM_PTR
#define UOCR_STREAM_PTR 1
#endif
template <int FMT>
struct UnitStream {
  static constexpr int UB = unit_bytes(FMT);
  static constexpr int SB = unit_scale_bytes(FMT);
  static constexpr int SE = FMT == Q8_0 ? 4 : 8;  // bytes of a lane's scale entry
  const uint8_t* q;
  const uint8_t* sc;
  const uint8_t* qp;  // this lane's next code bytes / scale entry (UOCR_STREAM_PTR)
  const uint8_t* sp;
  int m, i;
  int first, stride, n, U, uw, G, rank;
  __device__ __forceinline__ void set_run(int lane) {
    const size_t unit0 = (size_t)(first + m * stride) * U + rank * uw;
    qp = q + unit0 * UB + lane * 16;
    sp = sc + unit0 * SB + (lane >> 2) * SE;
  }
  __device__ __forceinline__ void start(const uint8_t* q_, const uint8_t* sc_, const SlabWork& w) {
    q = q_;
    sc = sc_;
    first = w.first;
    stride = w.stride;
    n = w.n;
    U = w.U;
    uw = w.uw;
    G = w.G;
    rank = w.rank;
    m = w.grp;
    i = 0;
    if (UOCR_STREAM_PTR && m < n) set_run(threadIdx.x & 31);
  }
  __device__ __forceinline__ void fetch_next(uint8_t* slot, int lane) {
    if (m < n) {
#if UOCR_STREAM_PTR
      cp_async16(slot + lane * 16, qp);
      if constexpr (FMT == F16) {
        cp_async16(slot + 512 + lane * 16, qp + 512);
      } else if constexpr (FMT == Q8_0) {
        cp_async4(slot + 512 + lane * 8, sp);
      } else {
        cp_async8(slot + 512 + lane * 8, sp);
      }
      qp += UB;
      sp += SB;
      if (++i == uw) {
        i = 0;
        m += G;
        if (m < n) set_run(lane);
      }
#else
      const size_t unit = (size_t)(first + m * stride) * U + rank * uw + i;
      const uint8_t* qu = q + unit * UB;
      cp_async16(slot + lane * 16, qu + lane * 16);
      if constexpr (FMT == F16) {
        cp_async16(slot + 512 + lane * 16, qu + 512 + lane * 16);
      } else {
        if constexpr (FMT == Q8_0)
          cp_async4(slot + 512 + lane * 8, sc + unit * SB + (lane >> 2) * SE);
        else
          cp_async8(slot + 512 + lane * 8, sc + unit * SB + (lane >> 2) * SE);
      }
      if (++i == uw) {
        i = 0;
        m += G;
      }
#endif
    }
    cp_commit();  // one group per call, empty or not, keeps the wait counts uniform
  }
  // the first kRingDepth units (weights only: may run before griddepcontrol.wait)
  __device__ __forceinline__ void prefetch(uint8_t* ring, int slot_bytes, const SlabWork&, int lane) {
#pragma unroll
    for (int d = 0; d < kRingDepth; ++d) fetch_next(ring + d * slot_bytes, lane);
  }
};

__device__ __forceinline__ void group_sync(int grp, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(grp + 1), "r"(nthreads) : "memory");
}

// Shared memory of the per-round partials: [G][2][ks][NT*8][16] fp32 =
// 2*kWarps*NT*512 bytes for any ks.
template <int NT>
constexpr int red_bytes() { return 2 * kWarps * NT * 8 * 16 * 4; }

// lo/hi = sum over the ks partials of (token tok, rows pg and pg+8).
template <int NT>
__device__ __forceinline__ void group_sum(const float* rb, int ks, int tok, int pg, float& lo, float& hi) {
  lo = 0.f;
  hi = 0.f;
  for (int r = 0; r < ks; ++r) {
    lo += rb[r * (NT * 128) + tok * 16 + pg];
    hi += rb[r * (NT * 128) + tok * 16 + pg + 8];
  }
}

// Stream the CTA's slabs through the warp rings (the first kRingDepth units
// already issued by us.prefetch).  After each round the group's threads call
// epi(slab, rb, tid, nthreads): rb holds the ks partials of the slab; thread
// tid of nthreads = 32*ks takes items tid, tid + nthreads, ... of NT*64.
template <int FMT, int NT, class BP, class Epi>
__device__ __forceinline__ void run_stream(UnitStream<FMT>& us, const SlabWork& w, uint8_t* ring, int slot_bytes,
                                           float* red, const BP& bp, int nt_used, const Epi& epi) {
  constexpr int KU = unit_k(FMT);
  const int lane = threadIdx.x & 31;
  const int nthr = w.ks * 32, tid = threadIdx.x - w.grp * nthr;
  float* gred = red + (size_t)w.grp * 2 * w.ks * (NT * 128);
  float acc[NT][4];
  int si = 0, par = 0;  // ring slot of the next unit to consume; round parity
  auto next_slot = [&]() {
    uint8_t* sl = ring + si * slot_bytes;
    si = si + 1 == kRingDepth ? 0 : si + 1;
    return sl;
  };
  for (int m = w.grp; m < w.n; m += w.G, par ^= 1) {
    zero_acc<NT>(acc);
    const int k0 = w.rank * w.uw;
    int i = 0;
    if constexpr (kUnroll == 2) {
      for (; i + 1 < w.uw; i += 2) {
        cp_wait<kRingDepth - 2>();  // units i and i+1 have landed (this lane's bytes)
        uint8_t* s0 = next_slot();
        uint8_t* s1 = next_slot();
        unit_any<FMT, NT>(acc, s0, s0 + 512 + lane * 8, bp, (k0 + i) * KU, lane, nt_used);
        unit_any<FMT, NT>(acc, s1, s1 + 512 + lane * 8, bp, (k0 + i + 1) * KU, lane, nt_used);
        us.fetch_next(s0, lane);  // refill both with the units kRingDepth ahead
        us.fetch_next(s1, lane);
      }
    }
    for (; i < w.uw; ++i) {
      cp_wait<kRingDepth - 1>();  // unit i has landed (this lane's bytes)
      uint8_t* s0 = next_slot();
      unit_any<FMT, NT>(acc, s0, s0 + 512 + lane * 8, bp, (k0 + i) * KU, lane, nt_used);
      us.fetch_next(s0, lane);  // refill it with the unit kRingDepth ahead
    }
    float* rb = gred + par * w.ks * (NT * 128);
    {
      const int g = lane >> 2, t = lane & 3;
      float* r = rb + w.rank * (NT * 128);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tok = nt * 8 + 2 * t;
        r[tok * 16 + g] = acc[nt][0];
        r[(tok + 1) * 16 + g] = acc[nt][1];
        r[tok * 16 + g + 8] = acc[nt][2];
        r[(tok + 1) * 16 + g + 8] = acc[nt][3];
      }
    }
    group_sync(w.grp, nthr);
    epi(w.first + m * w.stride, rb, tid, nthr);
  }
  cp_wait<0>();
}

// ------------------------------------------------------------------ staging
// All staging loops load first and compute afterwards so that one L2/HBM
// latency, not one per element, is paid per batch.

// One warp: dst[:] = fp16(src[:] * rsqrt(mean(src^2) + eps) * w[:]).  A row of
// up to 32*4*kNormRegs values (1280 for the decoders here) is held in
// registers; longer rows are read twice.
constexpr int kNormRegs = 10;

// This lane's norm weights for the register path (elements 4f..4f+3 for f =
// lane + 32 i).  The norm weights never change during a step, so kernels load
// them before griddepcontrol.wait and the staging after it waits for the
// activations alone.
struct NormW {
  uint2 v[kNormRegs];
};
__device__ __forceinline__ void load_norm_w(NormW& nw, const __half* w, int K) {
  const int lane = threadIdx.x & 31, n4 = K / 4;
#pragma unroll
  for (int i = 0; i < kNormRegs; ++i)
    nw.v[i] = (n4 <= kNormRegs * 32 && lane + 32 * i < n4) ? *reinterpret_cast<const uint2*>(w + 4 * (lane + 32 * i))
                                                           : make_uint2(0u, 0u);
}

__device__ __forceinline__ void stage_norm_rows_one(__half* dst, const float* srcf, const __half* w, const NormW& nw,
                                                    int K, float eps) {
  const int lane = threadIdx.x & 31;
  const int n4 = K / 4;
  const float4* src = reinterpret_cast<const float4*>(srcf);
  auto store_w = [&](int f, const float4& v, float r, uint2 wv) {
    const __half2 w0 = u32_h2(wv.x), w1 = u32_h2(wv.y);
    __half2* d = reinterpret_cast<__half2*>(dst + 4 * f);
    d[0] = __floats2half2_rn(v.x * r * __low2float(w0), v.y * r * __high2float(w0));
    d[1] = __floats2half2_rn(v.z * r * __low2float(w1), v.w * r * __high2float(w1));
  };
  auto store = [&](int f, const float4& v, float r) {
    store_w(f, v, r, *reinterpret_cast<const uint2*>(w + 4 * f));
  };
  if (n4 <= kNormRegs * 32) {
    float4 v[kNormRegs];
#pragma unroll
    for (int i = 0; i < kNormRegs; ++i) v[i] = (lane + 32 * i < n4) ? src[lane + 32 * i] : make_float4(0.f, 0.f, 0.f, 0.f);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kNormRegs; ++i) ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(ss / (float)K + eps);
#pragma unroll
    for (int i = 0; i < kNormRegs; ++i)
      if (lane + 32 * i < n4) store_w(lane + 32 * i, v[i], r, nw.v[i]);
  } else {
    float ss = 0.f;
    for (int f0 = 0; f0 < n4; f0 += 8 * 32) {
      float4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = (f0 + lane + 32 * i < n4) ? src[f0 + lane + 32 * i] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(ss / (float)K + eps);
    for (int f0 = 0; f0 < n4; f0 += 8 * 32) {
      float4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = (f0 + lane + 32 * i < n4) ? src[f0 + lane + 32 * i] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (f0 + lane + 32 * i < n4) store(f0 + lane + 32 * i, v[i], r);
    }
  }
}

// xs[tk][:] = normalised x[tk][:] for tk < ntok, zero rows up to ntok_pad (one warp per row).
__device__ __forceinline__ void stage_norm_rows(__half* xs, int ldx, const float* x, int ldx_g, int ntok, int ntok_pad,
                                                const __half* w, const NormW& nwr, int K, float eps) {
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int tk = warp; tk < ntok_pad; tk += nw) {
    if (tk < ntok)
      stage_norm_rows_one(xs + tk * ldx, x + (size_t)tk * ldx_g, w, nwr, K, eps);
    else
      for (int i = (threadIdx.x & 31); i < K / 8; i += 32)
        *reinterpret_cast<uint4*>(xs + tk * ldx + 8 * i) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// stage_norm_rows over gathered rows: xs[t] = norm(x[rows[t]]) for t < ntok.
__device__ __forceinline__ void stage_norm_gather(__half* xs, int ldx, const float* x, int ldx_g, const int* rows,
                                                  int ntok, int ntok_pad, const __half* w, const NormW& nwr, int K,
                                                  float eps) {
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int tk = warp; tk < ntok_pad; tk += nw) {
    // one row at a time through the contiguous routine (it handles zero padding)
    if (tk < ntok)
      stage_norm_rows_one(xs + tk * ldx, x + (size_t)rows[tk] * ldx_g, w, nwr, K, eps);
    else
      for (int i = (threadIdx.x & 31); i < K / 8; i += 32)
        *reinterpret_cast<uint4*>(xs + tk * ldx + 8 * i) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// dst[0, bytes) = src[0, bytes) (16-byte multiples), batched loads.
__device__ __forceinline__ void stage_bytes(uint8_t* dst, const uint8_t* src, int bytes) {
  const int n = bytes / 16;
  for (int i0 = threadIdx.x; i0 < n; i0 += 8 * blockDim.x) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      v[u] = i < n ? reinterpret_cast<const uint4*>(src)[i] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < n) reinterpret_cast<uint4*>(dst)[i] = v[u];
    }
  }
}

// xs[tk][j] = src[tk][j] (fp16), rows tk in [ntok, ntok_pad) zero.  K % 8 == 0.
__device__ __forceinline__ void stage_f16(__half* xs, int ldx, const __half* src, int lds, int ntok, int ntok_pad,
                                          int K) {
  const int per_row = K / 8;
  const int total = ntok_pad * per_row;
  for (int i0 = threadIdx.x; i0 < total; i0 += 8 * blockDim.x) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      const int tk = i / per_row, j = (i - tk * per_row) * 8;
      v[u] = (i < total && tk < ntok) ? *reinterpret_cast<const uint4*>(src + (size_t)tk * lds + j)
                                      : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < total) {
        const int tk = i / per_row, j = (i - tk * per_row) * 8;
        *reinterpret_cast<uint4*>(xs + tk * ldx + j) = v[u];
      }
    }
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

}  // namespace uocr
