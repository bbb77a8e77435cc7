// Tensor-core (tcgen05) expert kernels for steps with more than 16 rows.
//
// The fragment-GEMV expert kernels spend most of their issue slots on the
// product itself (B-fragment loads, one mma.sync per 8 tokens, per-block scale
// FMAs).  Here the SM only dequantises: the product runs on the tensor core.
//
//   * The CTA takes the same work as the GEMV kernels (a routed expert and a
//     part of its slabs, or a part of the shared experts) in 128-row tiles of
//     8 slabs.  Warp w < 8 streams the units of slab w of every tile through
//     its own cp.async ring, dequantises each unit with its block scale folded
//     in (value = fp16(d * q), or fp16(d * (q - 8)) for Q4_0: one rounding of
//     the exact product) and stores it in the canonical K-major layout of a
//     128 x 64 A tile (one stage of an S-stage ring, full / empty mbarriers).
//   * The token rows of a pass (16 for a routed expert, 32 for the shared
//     experts) stay resident as the B operand: gate/up stages them normalised
//     (the same fp16 values as the GEMV path); down copies the SwiGLU
//     activations gate/up wrote in the same layout.
//   * Warp 12 (one lane) issues tcgen05.mma (M = 128, N = 16 or 32, K = 16,
//     fp16 x fp16 -> fp32) into one of two TMEM accumulators; warps 8..11 read
//     a finished accumulator (each its 32-lane quadrant = 32 weight rows) and
//     write SwiGLU activations (gate rows 0..7 and up rows 8..15 of a slab sit
//     8 lanes apart) or the fp32 partials the combine kernel sums.
//
// Measured on the 64-row decode step this path is slower than the fragment-
// GEMV kernels (gate/up 71 us against 44 us per layer): with about six rows per
// routed expert, dequantising into shared memory (a multiply and a store per
// pair of weights) costs the SM about what the mma.sync products cost it, and
// one CTA per SM keeps fewer weight bytes in flight than two GEMV CTAs.  It is
// therefore chosen only on request (the engine's UOCR_TC_EXPERTS=1).
//
// Every mbarrier wait is bounded; a role whose wait gives up sets
// kStatusTimeout and stops, every role still reaches the final barrier, and
// the TMEM is freed after the last MMA has completed.
//
// Sources: "Unlimited-OCR on Apple Silicon with C and Metal", "Il decoder e il
// Mixture of Experts" (routed and shared experts, tokens grouped by expert)
// and "Quantizzazione: Q8 prima, Q4 dove conviene" (GEMM with the
// dequantisation fused in).
#include "moe_common.cuh"
#include "tc_common.cuh"

namespace uocr {

constexpr int kTcxProducers = 8;  // warps 0..7: slab w of each 128-row tile
constexpr int kTcxEpiWarp0 = 8;   // warps 8..11: TMEM lane quadrants 0..3
constexpr int kTcxMmaWarp = 12;
constexpr int kTcxThreads = 13 * 32;
constexpr int kTcxRing = 8;       // weight units in flight per producer warp
constexpr int kTcxSlot = 768;     // a unit's codes (512 B) + lane-private scales (32 x 8 B)
constexpr int kTcxNbRouted = kTcxRowsRouted;
constexpr int kTcxNbShared = kTcxRowsShared;
constexpr int kTcxAccCols = 32;   // TMEM columns of one accumulator
constexpr int kTcxTmemCols = 64;  // two accumulators
constexpr int kTcxMaxStages = 6;
constexpr uint32_t kTcxSleepNs = 2000;  // suspend hint of the pipeline waits (a bounded wait: 2^16 of them)

// Shared-memory plan: A stages, the resident B operand, the producer rings,
// the barriers.
TcxPlan tcx_plan(int b_bytes, int smem_limit) {
  TcxPlan p{};
  const int b = (b_bytes + 1023) / 1024 * 1024;
  const int fixed = b + kTcxProducers * kTcxRing * kTcxSlot + (2 * kTcxMaxStages + 5) * 8 + 16 + 1024;
  int s = (smem_limit - fixed) / kTcTileBytes;
  s = s > kTcxMaxStages ? kTcxMaxStages : s;
  p.stages = s;
  p.a_off = 0;
  p.b_off = s * kTcTileBytes;
  p.ring_off = p.b_off + b;
  p.bar_off = p.ring_off + kTcxProducers * kTcxRing * kTcxSlot;
  p.bytes = p.bar_off + (2 * s + 5) * 8 + 16;
  return p;
}

__device__ __forceinline__ void sts32(uint8_t* p, uint32_t v) { *reinterpret_cast<uint32_t*>(p) = v; }
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t x, __half2 d) { return h2_u32(__hmul2(u32_h2(x), d)); }
__device__ __forceinline__ __half2 half_bcast(uint16_t bits) { return __half2half2(__ushort_as_half(bits)); }

// Unit u of k-block (64 inputs) of slab w of the tile, from its ring slot, into
// the A tile: rows 16 w + g (+ 8), inputs 32 u + 16 s + 2 t (+ 8) (+ 1).
template <int F>
__device__ __forceinline__ void dequant_unit_to_tile(uint8_t* At, const uint8_t* slot, int w, int u, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const uint4 q = lds128(slot + lane * 16);
  uint8_t* base = At + (2 * w) * 1024 + g * 16 + 4 * t;
  if constexpr (F == Q4_0) {  // one unit = the whole k-block: word j = inputs 16 j ..
    const uint2 sv = *reinterpret_cast<const uint2*>(slot + 512 + lane * 8);
    const __half2 d0g = half_bcast((uint16_t)(sv.x & 0xFFFF)), d0h = half_bcast((uint16_t)(sv.x >> 16));
    const __half2 d1g = half_bcast((uint16_t)(sv.y & 0xFFFF)), d1h = half_bcast((uint16_t)(sv.y >> 16));
    const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t r[4];
      dq_q4(wd[j], r);  // (row g, k 2t..), (row g+8, ..), (row g, k 2t+8..), (row g+8, ..), codes - 8
      const __half2 dg = j < 2 ? d0g : d1g, dh = j < 2 ? d0h : d1h;
      uint8_t* p = base + (2 * j) * 128;
      sts32(p, hmul2_u32(r[0], dg));
      sts32(p + 1024, hmul2_u32(r[1], dh));
      sts32(p + 128, hmul2_u32(r[2], dg));
      sts32(p + 1024 + 128, hmul2_u32(r[3], dh));
    }
  } else {  // Q8_0: inputs 32 u .. 32 u + 31; q.x/q.y the first k-step, q.z/q.w the second
    const uint32_t sv = *reinterpret_cast<const uint32_t*>(slot + 512 + lane * 8);
    const __half2 dg = half_bcast((uint16_t)(sv & 0xFFFF)), dh = half_bcast((uint16_t)(sv >> 16));
    const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      uint32_t a0, a1, a2, a3;
      dq_s8x4(wd[2 * s], a0, a1);      // (row g, k 2t..), (row g+8, k 2t..)
      dq_s8x4(wd[2 * s + 1], a2, a3);  // (row g, k 2t+8..), (row g+8, k 2t+8..)
      uint8_t* p = base + (4 * u + 2 * s) * 128;
      sts32(p, hmul2_u32(a0, dg));
      sts32(p + 1024, hmul2_u32(a1, dh));
      sts32(p + 128, hmul2_u32(a2, dg));
      sts32(p + 1024 + 128, hmul2_u32(a3, dh));
    }
  }
}

// B rows j < NB of the pass (gate/up): row src_row(j) of h normalised with the
// post-attention RMSNorm, fp16 as the GEMV path's staging rounds it, in the
// canonical layout (64-input blocks of NB * 128 bytes); rows j >= n are zero.
template <int NB, class RowOf>
__device__ __forceinline__ void stage_b_norm(uint8_t* Bs, const ExpertArgs& a, int n, const RowOf& row_of) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int H = a.H, n8 = H / 8;
  for (int j = warp; j < NB; j += nw) {
    if (j < n) {
      const float4* src = reinterpret_cast<const float4*>(a.h + (size_t)row_of(j) * H);
      float ss = 0.f;
      for (int f = lane; f < H / 4; f += 32) {  // the order of the GEMV path's sum of squares
        const float4 v = src[f];
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float r = rsqrtf(ss / (float)H + a.eps);
      for (int c = lane; c < n8; c += 32) {
        const float4 v0 = src[2 * c], v1 = src[2 * c + 1];
        const uint4 wv = *reinterpret_cast<const uint4*>(a.norm_w + 8 * c);
        const __half2 w0 = u32_h2(wv.x), w1 = u32_h2(wv.y), w2 = u32_h2(wv.z), w3 = u32_h2(wv.w);
        uint4 o;
        o.x = h2_u32(__floats2half2_rn(v0.x * r * __low2float(w0), v0.y * r * __high2float(w0)));
        o.y = h2_u32(__floats2half2_rn(v0.z * r * __low2float(w1), v0.w * r * __high2float(w1)));
        o.z = h2_u32(__floats2half2_rn(v1.x * r * __low2float(w2), v1.y * r * __high2float(w2)));
        o.w = h2_u32(__floats2half2_rn(v1.z * r * __low2float(w3), v1.w * r * __high2float(w3)));
        const int k = 8 * c;
        *reinterpret_cast<uint4*>(Bs + (k >> 6) * (NB * 128) + canon_offset(j, k & 63)) = o;
      }
    } else {
      for (int c = lane; c < n8; c += 32) {
        const int k = 8 * c;
        *reinterpret_cast<uint4*>(Bs + (k >> 6) * (NB * 128) + canon_offset(j, k & 63)) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
}

// Byte offset of activation (token j, input o) in a pass's canonical block.
template <int NB>
__device__ __forceinline__ int act_canon(int j, int o) {
  return (o >> 6) * (NB * 128) + canon_offset(j, o & 63);
}

template <int F, int MODE, bool SH>
__device__ __forceinline__ void tcx_run(const ExpertArgs& a, const TcxPlan& pl, ExpertCta ec, unsigned char* smem,
                                        RouteSmem& rs) {
  constexpr int KU = unit_k(F);
  constexpr int UPB = kTcTileK / KU;  // units per 64-input k-block
  constexpr int NB = SH ? kTcxNbShared : kTcxNbRouted;
  constexpr uint32_t IDESC = idesc_f16(kTcTileRows, NB);
  const int S = pl.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + pl.bar_off);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done = acc_empty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);
  uint8_t* Bs = smem + pl.b_off;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PMat& m = SH ? a.ws : a.wr;
  const int K = MODE == 0 ? a.H : (SH ? a.Ish : a.Ie);
  const int KB = K / kTcTileK, U = K / KU;
  const int n_slabs = MODE == 0 ? m.n_slabs : a.H / 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + s, kTcxProducers);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full + b, 1);
      mbar_init(acc_empty + b, 4);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == kTcxMmaWarp) {
    tmem_alloc(s_tmem, kTcxTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  // ---- this CTA's slabs and the producers' weight streams
  int s0 = 0, s1 = 0;
  const uint8_t* wq = nullptr;
  const uint8_t* wsc = nullptr;
  uint8_t* ring = smem + pl.ring_off + (size_t)(warp < kTcxProducers ? warp : 0) * kTcxRing * kTcxSlot;
  UnitStream<F> us;
  SlabWork sw{};
  const int slab_w = warp;  // producers: slab slab_w of every tile
  auto start_stream = [&]() {  // the units of slabs s0 + slab_w + 8 t, in order
    sw.first = s0 + slab_w;
    sw.stride = 8;
    sw.n = s1 - s0 > slab_w ? (s1 - s0 - slab_w + 7) / 8 : 0;
    sw.U = U;
    sw.ks = 1;
    sw.uw = U;
    sw.G = 1;
    sw.grp = 0;
    sw.rank = 0;
    us.start(wq, wsc, sw);
#pragma unroll 1
    for (int d = 0; d < kTcxRing; ++d) us.fetch_next(ring + d * kTcxSlot, lane);
  };
  bool streaming = false;
  if (SH) {  // the shared experts (and, with expert-id units, the routed expert) need nothing from the router
    part_range(n_slabs, 8, ec.part, ec.parts, s0, s1);
    wq = m.q;
    wsc = m.s;
  } else {
    part_range(n_slabs, 8, ec.part, ec.parts, s0, s1);
    wq = m.q + (size_t)ec.i * m.q_stride;
    wsc = m.s + (size_t)ec.i * m.s_stride;
  }
  if (s0 < s1) {
    if (warp < kTcxProducers) start_stream();
    streaming = true;
  }
  pdl_wait();
  if (MODE == 0 && blockIdx.x == 0) write_grouping(rs, a);

  // ---- this CTA's rows
  int e = -1, ntk = a.ntok;
  if (!SH) {
    if ((int)threadIdx.x < a.tg) rs.grec[threadIdx.x] = __ldcg(a.rec + (size_t)threadIdx.x * a.n_units + ec.i);
    __syncthreads();
    e = rs.grec[0].x;
    for (int g = 1; g < a.tg; ++g) e = e >= 0 ? e : rs.grec[g].x;
    ntk = e >= 0 ? gather_unit_rows(rs, a.tg, a.k) : 0;
  }
  if (s0 >= s1) ntk = 0;  // a part without a tile

  const int ntiles = (s1 - s0 + 7) / 8;
  int it = 0, tl = 0;  // stage iterations and tiles, continued over passes
  bool ok = true, issued = false;
  for (int pass = 0; pass * NB < ntk; ++pass) {
    const int r0 = pass * NB, n = min(NB, ntk - r0);
    if (pass > 0 && warp < kTcxProducers) start_stream();  // the same slabs again (L2-resident by now)
    __syncthreads();  // every MMA of the previous pass has completed (its epilogue has run)
    if constexpr (MODE == 0) {
      if (SH)
        stage_b_norm<NB>(Bs, a, n, [&](int j) { return r0 + j; });
      else
        stage_b_norm<NB>(Bs, a, n, [&](int j) { return rs.rows[r0 + j]; });
    } else {
      const uint8_t* src = SH ? a.act_s + (size_t)pass * NB * a.Ish * 2 : a.act_r + (size_t)(e * a.tg + pass) * NB * a.Ie * 2;
      stage_bytes(Bs, src, NB * K * 2);
    }
    fence_proxy_async_smem();  // the B operand is read by the tensor core
    __syncthreads();

    if (warp < kTcxProducers) {  // ---------------- producers
      int si = 0;
      for (int t = 0; t < ntiles && ok; ++t) {
        const bool mine = s0 + 8 * t + slab_w < s1;
        for (int kb = 0; kb < KB; ++kb) {
          const int itk = it + t * KB + kb, s = itk % S;
          if (itk >= S &&
              !__all_sync(0xffffffffu, (int)mbar_wait_sleep(empty + s, (uint32_t)(((itk / S) - 1) & 1), kTcxSleepNs))) {
            ok = false;
            break;
          }
          uint8_t* At = smem + pl.a_off + (size_t)s * kTcTileBytes;
          if (mine) {
#pragma unroll
            for (int u = 0; u < UPB; ++u) {
              cp_wait<kTcxRing - 1>();  // the unit has landed (this lane's bytes)
              uint8_t* slot = ring + si * kTcxSlot;
              si = si + 1 == kTcxRing ? 0 : si + 1;
              dequant_unit_to_tile<F>(At, slot, slab_w, u, lane);
              us.fetch_next(slot, lane);  // refill the slot kTcxRing units ahead
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(full + s);
        }
      }
    } else if (warp == kTcxMmaWarp) {  // ---------------- MMA issue
      if (lane == 0 && ok) {
        for (int t = 0; t < ntiles && ok; ++t) {
          const int tli = tl + t, buf = tli & 1;
          if (tli >= 2 && !mbar_wait_sleep(acc_empty + buf, (uint32_t)(((tli >> 1) - 1) & 1), kTcxSleepNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(buf * kTcxAccCols);
          for (int kb = 0; kb < KB; ++kb) {
            const int itk = it + t * KB + kb, s = itk % S;
            if (!mbar_wait_sleep(full + s, (uint32_t)((itk / S) & 1), kTcxSleepNs)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint8_t* At = smem + pl.a_off + (size_t)s * kTcTileBytes;
            const uint8_t* Bk = Bs + (size_t)kb * (NB * 128);
#pragma unroll
            for (int ks = 0; ks < kTcTileK / 16; ++ks)
              tc_mma_f16(d, smem_desc(At + ks * 256, 128, 1024), smem_desc(Bk + ks * 256, 128, 1024), IDESC,
                         (kb | ks) != 0);
            tc_commit(empty + s);  // the stage is free once these MMAs have read it
            issued = true;
          }
          if (!ok) break;
          tc_commit(acc_full + buf);
        }
      }
    } else {  // ---------------- epilogue: warps 8..11, TMEM lanes 32 q .. 32 q + 31
      const int qd = warp - kTcxEpiWarp0;
      const int r = 32 * qd + lane, rr = r & 15;
      for (int t = 0; t < ntiles && ok; ++t) {
        const int tli = tl + t, buf = tli & 1;
        if (!__all_sync(0xffffffffu,
                        lane == 0 ? (int)mbar_wait_sleep(acc_full + buf, (uint32_t)((tli >> 1) & 1), kTcxSleepNs) : 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int slab = s0 + 8 * t + (r >> 4);
        uint8_t* act = nullptr;
        if constexpr (MODE == 0)
          act = SH ? a.act_s + (size_t)pass * NB * a.Ish * 2 : a.act_r + (size_t)(e * a.tg + pass) * NB * a.Ie * 2;
        // 16 columns (token rows) at a time: TMEM -> registers -> SwiGLU or partials
#pragma unroll 1
        for (int c0 = 0; c0 < NB; c0 += 16) {
          uint32_t x[16];
          tc_ld16(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(buf * kTcxAccCols + c0), x);
          tc_wait_ld();
          if (c0 + 16 >= NB) {  // the accumulator is in registers: release it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty + buf);
          }
          if constexpr (MODE == 0) {  // SwiGLU: gate row rr < 8, its up row 8 lanes on
            const int o = 8 * slab + rr;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const float g = __uint_as_float(x[jj]);
              const float up = __shfl_down_sync(0xffffffffu, g, 8);
              const int j = c0 + jj;
              if (rr < 8 && slab < s1 && j < n)
                *reinterpret_cast<__half*>(act + act_canon<NB>(j, o)) = __float2half_rn(silu(g) * up);
            }
          } else {
            const int c = 16 * slab + rr;
            if (slab < s1) {
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) {
                const int j = c0 + jj;
                if (j < n) {
                  float* dst = SH ? a.part_s + (size_t)(r0 + j) * a.H : a.part_r + (size_t)rs.ent[r0 + j] * a.H;
                  dst[c] = __uint_as_float(x[jj]);
                }
              }
            }
          }
        }
      }
    }
    it += ntiles * KB;
    tl += ntiles;
  }

  // ---- teardown: copies in flight land, the last MMAs complete, TMEM is freed
  if (warp < kTcxProducers && streaming) cp_wait<0>();
  if (warp == kTcxMmaWarp && lane == 0 && issued) {
    tc_commit(done);
    if (!mbar_wait(done, 0)) ok = false;
  }
  if (!ok && (lane == 0)) atomicOr(a.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == kTcxMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcxTmemCols);
  }
}

template <int FR, int FS, int MODE>
__global__ void __launch_bounds__(kTcxThreads, 1) k_tc_expert(const ExpertArgs a, const TcxPlan pl) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ RouteSmem rs;
  if (!(kPdlLate & PDL_EXPERT)) pdl_launch_dependents();
  const ExpertCta ec = expert_cta(a);
  if (ec.shared)
    tcx_run<FS, MODE, true>(a, pl, ec, smem, rs);
  else
    tcx_run<FR, MODE, false>(a, pl, ec, smem, rs);
  if (kPdlLate & PDL_EXPERT) pdl_launch_dependents();
}

bool tcx_format_ok(int fr, int fs) { return (fr == Q8_0 || fr == Q4_0) && (fs == Q8_0 || fs == Q4_0); }

#define UOCR_TCX_PAIRS(X) X(Q8_0, Q8_0) X(Q4_0, Q8_0) X(Q4_0, Q4_0) X(Q8_0, Q4_0)

cudaError_t launch_tc_expert(int mode, int fr, int fs, const ExpertArgs& a, const TcxPlan& pl, cudaStream_t st,
                             bool pdl) {
  const dim3 grid((a.ws.n_slabs > 0 ? a.cpes : 0) + a.n_units * a.cpe, 1);
#define X(FR_, FS_)                                                                                           \
  if (fr == FR_ && fs == FS_)                                                                                 \
    return mode == 0 ? launch_kernel(k_tc_expert<FR_, FS_, 0>, grid, dim3(kTcxThreads), pl.bytes, st, pdl, a, pl) \
                     : launch_kernel(k_tc_expert<FR_, FS_, 1>, grid, dim3(kTcxThreads), pl.bytes, st, pdl, a, pl);
  UOCR_TCX_PAIRS(X)
#undef X
  return cudaErrorInvalidValue;
}

cudaError_t init_tc_expert_attributes() {
  cudaError_t e = cudaSuccess;
#define X(FR_, FS_)                                                     \
  if (e == cudaSuccess) e = allow_max_dyn_smem(k_tc_expert<FR_, FS_, 0>); \
  if (e == cudaSuccess) e = allow_max_dyn_smem(k_tc_expert<FR_, FS_, 1>);
  UOCR_TCX_PAIRS(X)
#undef X
  return e;
}

}  // namespace uocr
