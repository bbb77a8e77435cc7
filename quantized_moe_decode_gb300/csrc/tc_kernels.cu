// Tensor-core (tcgen05) LM head for steps with more than 16 rows.
//
// At 17..64 rows the LM head is a dense contraction (logits = W x for V = 102400
// fp16 rows, H inputs, N rows of the step), and the fragment-ordered GEMV
// streams W once per 16-row token group.  Here every weight tile is read once
// for all the step's rows:
//
//   * W is packed a second time, in the canonical K-major layout of the tensor
//     core's shared-memory operands without swizzle: tiles of 128 rows x 64
//     inputs (16 KB), element (r, k) of a tile at
//     (r/8)*1024 + (k/8)*128 + (r%8)*16 + (k%8)*2 bytes (8-row x 16-byte core
//     matrices; 128 bytes between core matrices along K, 1024 along M); tile
//     (m, kb) at ((m * KB) + kb) * 16 KB, so one 1-D TMA bulk copy moves a tile.
//   * k_lm_stage writes the final-normalised rows (fp16) in the same layout,
//     NPAD rows per 64-input block (rows beyond the step's are zero).
//   * k_tc_lm: one CTA per SM walks M tiles.  Warp 4 (one lane) streams
//     (weight tile, activation block) pairs into an S-stage ring with bulk
//     copies on full/empty mbarriers; warp 5 (one lane) issues tcgen05.mma
//     (M = 128, N = NPAD, K = 16, fp16 x fp16 -> fp32) into one of two TMEM
//     accumulators; warps 0..3 read the finished accumulator (tcgen05.ld, each
//     warp its 32-lane quadrant = 32 vocabulary rows), store logits on request
//     and keep each token's best (logit, lowest index) key; the last CTA to
//     finish writes the ids, as the GEMV path does.
//
// Every mbarrier wait is bounded; a wait that gives up sets kStatusTimeout and
// its role stops, so every role reaches the final barrier and the TMEM is freed.
//
// Source: "Unlimited-OCR on Apple Silicon with C and Metal", "Il decoder e il
// Mixture of Experts" (the decode loop ends in an argmax over the language
// head); "Falcon-OCR INT8 OpenVINO IR", "How it is meant to be run" (the rows of
// a step share one read of the weights).
#include "tc_common.cuh"

namespace uocr {

// ------------------------------------------------------------------ LM-head tiling
// UOCR_TC_SPLIT: bulk copies per 16 KB weight tile (build-time tuning)
#ifndef UOCR_TC_SPLIT
#define UOCR_TC_SPLIT 1
#endif
constexpr int kTcSplit = UOCR_TC_SPLIT;
static_assert(kTcSplit >= 1 && kTcSplit <= 16 && (kTcTileBytes / kTcSplit) % 16 == 0, "tile copy split");

// A weight tile into shared memory in kTcSplit bulk copies on one mbarrier.
__device__ __forceinline__ void tile_g2s(uint8_t* dst, const uint8_t* src, uint64_t* bar) {
#pragma unroll
  for (int c = 0; c < kTcSplit; ++c)
    bulk_g2s(dst + c * (kTcTileBytes / kTcSplit), src + c * (kTcTileBytes / kTcSplit), kTcTileBytes / kTcSplit, bar);
}
constexpr int kTcThreads = 192;                           // 4 epilogue warps, producer, MMA
constexpr int kTcSmemBudget = 200 * 1024;                 // stage ring (the rest: barriers, per-warp bests)

__host__ __device__ constexpr int tc_block_b_bytes(int npad) { return npad * kTcTileK * 2; }
__host__ __device__ constexpr int tc_stages(int npad) {
  return kTcSmemBudget / (kTcTileBytes + tc_block_b_bytes(npad)) < 12 ? kTcSmemBudget / (kTcTileBytes + tc_block_b_bytes(npad))
                                                                    : 12;
}

// ------------------------------------------------------------------ packer
// Row-major fp16 W [V][K] -> canonical tiles; rows >= V are zero.  One thread
// per 16-byte chunk (8 inputs of one row).
__global__ void k_pack_canon(const __half* src, uint8_t* dst, int V, int K, int n_mtiles) {
  const int KB = K / kTcTileK;
  const long long total = (long long)n_mtiles * KB * kTcTileRows * 8;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int k8 = (int)(i & 7);
    const int r = (int)((i >> 3) % kTcTileRows);
    const long long tile = (i >> 3) / kTcTileRows;  // m * KB + kb
    const int kb = (int)(tile % KB);
    const int m = (int)(tile / KB);
    const int row = m * kTcTileRows + r;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < V) v = *reinterpret_cast<const uint4*>(src + (size_t)row * K + kb * kTcTileK + k8 * 8);
    *reinterpret_cast<uint4*>(dst + tile * kTcTileBytes + canon_offset(r, k8 * 8)) = v;
  }
}

cudaError_t launch_pack_canon(const void* src_f16, uint8_t* dst, int V, int K, cudaStream_t st) {
  const int n_mtiles = (V + kTcTileRows - 1) / kTcTileRows;
  const long long total = (long long)n_mtiles * (K / kTcTileK) * kTcTileRows * 8;
  const long long blocks = (total + 255) / 256;
  k_pack_canon<<<(int)(blocks < 65535 ? blocks : 65535), 256, 0, st>>>(reinterpret_cast<const __half*>(src_f16), dst,
                                                                        V, K, n_mtiles);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ activation staging
// Block t: row t of the step (t < ntok) final-normalised to fp16, or zeros,
// written in the canonical layout: block kb holds inputs [64 kb, 64 kb + 64)
// of all NPAD rows (NPAD * 128 bytes).
__global__ void __launch_bounds__(256) k_lm_stage(const TcLmArgs a) {
  pdl_launch_dependents();
  const int t = blockIdx.x, K = a.K;
  const int warp = threadIdx.x >> 5;
  __shared__ float s_part[8];
  pdl_wait();  // the residual rows come from the previous kernel
  float ss = 0.f;
  if (t < a.ntok)
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
      const float v = a.x[(size_t)t * a.ld_x + k];
      ss += v * v;
    }
#pragma unroll
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) s_part[warp] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += s_part[w];
  const float r = rsqrtf(tot / (float)K + a.eps);
  const int bb = tc_block_b_bytes(a.npad);
  for (int k2 = threadIdx.x; k2 < K / 2; k2 += blockDim.x) {
    const int k = 2 * k2;
    __half2 h = __floats2half2_rn(0.f, 0.f);
    if (t < a.ntok) {
      const float x0 = a.x[(size_t)t * a.ld_x + k], x1 = a.x[(size_t)t * a.ld_x + k + 1];
      h = __floats2half2_rn(x0 * r * __half2float(a.norm_w[k]), x1 * r * __half2float(a.norm_w[k + 1]));
    }
    *reinterpret_cast<__half2*>(a.xc + (size_t)(k / kTcTileK) * bb + canon_offset(t, k % kTcTileK)) = h;
  }
}

// ------------------------------------------------------------------ the tensor-core LM head
template <int NPAD>
__global__ void __launch_bounds__(kTcThreads, 1) k_tc_lm(const TcLmArgs a) {
  constexpr int S = tc_stages(NPAD);
  constexpr int BB = tc_block_b_bytes(NPAD);
  constexpr int STAGE = kTcTileBytes + BB;
  constexpr int NCOLS = 2 * NPAD < 32 ? 32 : 2 * NPAD;  // two accumulators, a power of two
  constexpr uint32_t IDESC = idesc_f16(kTcTileRows, NPAD);
  static_assert(NPAD % 16 == 0 && NPAD >= 16 && NPAD <= 128, "N of the MMA");
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * STAGE);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done = acc_empty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);
  __shared__ unsigned long long s_best[4][NPAD];
  __shared__ float s_tr[4][32][33];  // per epilogue warp: a 32 x 32 chunk transposed (padded: no bank conflicts)
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = a.K / kTcTileK;
  const int n_mt = a.n_mtiles;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full + b, 1);
      mbar_init(acc_empty + b, 4);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < 4 * NPAD; i += blockDim.x) (&s_best[0][0])[i] = 0ull;
  if (warp == 5) {
    tmem_alloc(s_tmem, NCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  pdl_launch_dependents();

  if (warp == 4) {  // ---------------- producer
    if (lane == 0) {
      const int my_tiles = blockIdx.x < n_mt ? (n_mt - 1 - blockIdx.x) / gridDim.x + 1 : 0;
      const int total = my_tiles * KB;
      const int pre = total < S ? total : S;
      auto tile_of = [&](int i) { return (size_t)(blockIdx.x + (i / KB) * gridDim.x) * KB + (i % KB); };
      // the weight tiles do not depend on the previous kernel: the first S go out now
      for (int i = 0; i < pre; ++i) {
        mbar_expect_tx(full + i, (uint32_t)STAGE);
        tile_g2s(smem + i * STAGE, a.w + tile_of(i) * kTcTileBytes, full + i);
      }
      pdl_wait();  // the staged activations come from k_lm_stage
      for (int i = 0; i < pre; ++i)
        bulk_g2s(smem + i * STAGE + kTcTileBytes, a.xc + (size_t)(i % KB) * BB, BB, full + i);
      bool ok = true;
      for (int it = pre; it < total; ++it) {
        const int s = it % S;
        if (!mbar_wait(empty + s, (uint32_t)(((it / S) - 1) & 1))) {
          ok = false;
          break;
        }
        uint8_t* st = smem + s * STAGE;
        mbar_expect_tx(full + s, (uint32_t)STAGE);
        tile_g2s(st, a.w + tile_of(it) * kTcTileBytes, full + s);
        bulk_g2s(st + kTcTileBytes, a.xc + (size_t)(it % KB) * BB, BB, full + s);
      }
      // every copy issued has landed before the CTA can leave (bounded)
      const int issued = ok ? total : 0;
      for (int i = issued > S ? issued - S : 0; i < issued; ++i)
        if (!mbar_wait(full + (i % S), (uint32_t)((i / S) & 1))) ok = false;
      if (!ok) atomicOr(a.status, kStatusTimeout);
    }
  } else if (warp == 5) {  // ---------------- MMA issue
    if (lane == 0) {
      int it = 0, tl = 0;
      bool ok = true;
      for (int mt = blockIdx.x; mt < n_mt && ok; mt += gridDim.x, ++tl) {
        const int buf = tl & 1;
        if (tl >= 2 && !mbar_wait(acc_empty + buf, (uint32_t)(((tl >> 1) - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * NPAD);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % S;
          if (!mbar_wait(full + s, (uint32_t)((it / S) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* st = smem + s * STAGE;
#pragma unroll
          for (int ks = 0; ks < kTcTileK / 16; ++ks)
            tc_mma_f16(d, smem_desc(st + ks * 256, 128, 1024), smem_desc(st + kTcTileBytes + ks * 256, 128, 1024),
                       IDESC, (kb | ks) != 0);
          tc_commit(empty + s);  // the stage is free once these MMAs have read it
        }
        if (!ok) break;
        tc_commit(acc_full + buf);
      }
      // no MMA may still be running when the TMEM is freed: wait (bounded) for the last ones
      tc_commit(done);
      if (!mbar_wait(done, 0)) ok = false;
      if (!ok) atomicOr(a.status, kStatusTimeout);
    }
  } else {  // ---------------- epilogue: warps 0..3, TMEM lanes 32 w .. 32 w + 31
    pdl_wait();
    int tl = 0;
    for (int mt = blockIdx.x; mt < n_mt; mt += gridDim.x, ++tl) {
      const int buf = tl & 1;
      const int ok = lane == 0 ? (int)mbar_wait(acc_full + buf, (uint32_t)((tl >> 1) & 1)) : 1;
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) atomicOr(a.status, kStatusTimeout);
        break;
      }
      tc_fence_after();
      const int row0 = mt * kTcTileRows + warp * 32, row = row0 + lane;
#pragma unroll 1
      for (int c = 0; c < NPAD / 32; ++c) {
        uint32_t r[32];
        tc_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(buf * NPAD + c * 32), r);
        tc_wait_ld();
        if (c == NPAD / 32 - 1) {  // the whole accumulator is in registers: the MMA may reuse it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty + buf);
        }
        // lane = vocabulary row: store the logits on request, then pass the chunk
        // through shared memory so that lane = token scans its 32 rows
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int tok = c * 32 + j;
          if (a.logits && tok < a.ntok && row < a.V) a.logits[(size_t)tok * a.V + row] = __uint_as_float(r[j]);
          s_tr[warp][j][lane] = __uint_as_float(r[j]);
        }
        __syncwarp();
        const int tok = c * 32 + lane;
        if (tok < a.ntok) {
          unsigned long long best = s_best[warp][tok];  // this lane's token: no other thread writes it
#pragma unroll 8
          for (int rr = 0; rr < 32; ++rr) {
            if (row0 + rr < a.V) {
              const unsigned long long key = argmax_key(s_tr[warp][lane][rr], row0 + rr);
              best = key > best ? key : best;
            }
          }
          s_best[warp][tok] = best;
        }
        __syncwarp();  // the chunk buffer is free for the next chunk
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, NCOLS);
  }
  // this CTA's best per row of the step -> the global keys; the last CTA writes the ids
  for (int t = threadIdx.x; t < a.ntok; t += blockDim.x) {
    unsigned long long k = s_best[0][t];
    for (int w = 1; w < 4; ++w) k = s_best[w][t] > k ? s_best[w][t] : k;
    if (k) atomicMax(a.keys + t, k);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int done = atomicAdd(a.counter, 1);
    s_last = done == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    const int step = a.hist ? *a.hist_ctr : 0;
    for (int t = threadIdx.x; t < a.ntok; t += blockDim.x) {
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

int tc_lm_npad(int rows) { return rows <= 32 ? 32 : 64; }

int tc_lm_smem_bytes(int npad) {
  const int S = tc_stages(npad);
  return S * (kTcTileBytes + tc_block_b_bytes(npad)) + (2 * S + 5) * 8 + 16;
}

cudaError_t launch_tc_lm(const TcLmArgs& a, int n_sm, cudaStream_t st, bool pdl) {
  const int gx = a.n_mtiles < n_sm ? a.n_mtiles : n_sm;
  cudaError_t e = launch_kernel(k_lm_stage, dim3(a.npad), dim3(256), 0, st, pdl, a);
  if (e != cudaSuccess) return e;
  if (a.npad == 32) return launch_kernel(k_tc_lm<32>, dim3(gx), dim3(kTcThreads), tc_lm_smem_bytes(32), st, pdl, a);
  if (a.npad == 64) return launch_kernel(k_tc_lm<64>, dim3(gx), dim3(kTcThreads), tc_lm_smem_bytes(64), st, pdl, a);
  return cudaErrorInvalidValue;
}

cudaError_t init_tc_attributes() {
  cudaError_t e = cudaFuncSetAttribute(k_tc_lm<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, tc_lm_smem_bytes(32));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_tc_lm<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, tc_lm_smem_bytes(64));
  return e;
}

}  // namespace uocr
