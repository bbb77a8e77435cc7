// MoE kernels of one decode step.
//
//   router   one thread-block cluster per token group of 16 rows: its CTAs
//            share the E/16 slabs of the fp16 router GEMV (RMSNorm prologue)
//            and keep their logits in shared memory; after a cluster barrier
//            each rank takes a share of the rows (row r by rank r % cluster
//            size), reads all E logits of the row through distributed shared
//            memory, takes the top-k (lowest index wins a tie) and the softmax
//            weights renormalised over them, and ORs the choices into rank 0's
//            per-expert masks (remote atomics, then a cluster-scope release
//            fence); after a second barrier rank 0 writes one record per
//            routed unit (active slot or expert id): the expert, the rows of
//            the group that chose it (its segment of the token grouping, a
//            16-bit mask) and each row's slot in its top-k (3 bits per row).
//   gate/up  shared-expert CTAs first (they need nothing from the router),
//            then routed CTAs, one per (unit, part of the expert's slabs).  A
//            routed CTA reads its unit's record of every token group, gathers
//            the unit's rows over the whole step, stages them (16 per pass),
//            streams the expert's gate/up slabs once per pass and writes SwiGLU
//            activations in the B-fragment order the down projection reads
//            directly.  CTA 0 also writes the grouping arrays (count, offset,
//            perm, inv) from the router's choices.
//   down     the same CTA layout; it streams the expert's down slabs and
//            writes fp32 partials per (row, slot) and per row for the shared
//            experts.
//   combine  one thread per output: residual + sum_j w_j * expert_j (slot
//            order) + shared, in the same fixed order for every row.
//
// Routed units are expert ids when most experts are expected to receive a
// token (the CTA streams the head of its expert's weights before the routing
// is known, into bandwidth the router leaves idle), else active slots (few
// rows: unit i is the i-th expert that received a token).
//
// Sources: "Unlimited-OCR on Apple Silicon with C and Metal", "Il decoder e
// il Mixture of Experts" (64 routed experts, top-6, two shared experts;
// compute the routing, group the tokens by expert, run the projections,
// recompose without useless copies) and "Quantizzazione" (dequantisation
// fused into GEMV/GEMM, SwiGLU and the expert combine).
#include <cooperative_groups.h>
#include <math.h>

#include <type_traits>

#include "moe_common.cuh"

namespace uocr {

// ------------------------------------------------------------------ routing
// One warp, one row: the E <= 256 logits (8 per lane).
struct RowLogits {
  float v[8];
};
__device__ __forceinline__ void topk_load(RowLogits& rl, const float* lg, int E, int lane) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int e = lane + 32 * q;
    rl.v[q] = e < E ? __ldcg(lg + e) : -INFINITY;
  }
}
// Top-k by logit, lowest index first among equal logits, by ranking: the
// rank of logit e is the number of logits that beat it (greater, or equal
// with a lower index); e is chosen iff rank < k, and its slot is its rank.
// All lanes compare their QN logits (experts lane + 32q) against every logit
// broadcast from the other lanes: independent work, no serial argmax rounds.
// Weights: exp(l_e - l_max) / sum over the chosen of exp(l - l_max).
// Returns, per held logit q, its rank (>= k: not chosen) and weight.
template <int QN>
__device__ __forceinline__ void topk_rank(const RowLogits& rl, int E, int k, int lane, int (&rank)[QN],
                                          float (&wt)[QN]) {
#pragma unroll
  for (int q = 0; q < QN; ++q) rank[q] = 0;
#pragma unroll 4
  for (int src = 0; src < 32; ++src) {  // the router warms this code up before it waits
#pragma unroll
    for (int qs = 0; qs < QN; ++qs) {
      const float o = __shfl_sync(0xffffffffu, rl.v[qs], src);
      const int eo = src + 32 * qs;
#pragma unroll
      for (int q = 0; q < QN; ++q) {
        const int em = lane + 32 * q;
        rank[q] += (o > rl.v[q]) || (o == rl.v[q] && eo < em);
      }
    }
  }
  float mx = -INFINITY;
#pragma unroll
  for (int q = 0; q < QN; ++q) mx = fmaxf(mx, rl.v[q]);
#pragma unroll
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float ex[QN], sum = 0.f;
#pragma unroll
  for (int q = 0; q < QN; ++q) {
    ex[q] = (rank[q] < k && lane + 32 * q < E) ? expf(rl.v[q] - mx) : 0.f;
    sum += ex[q];
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
#pragma unroll
  for (int q = 0; q < QN; ++q) wt[q] = ex[q] / sum;
}

// ------------------------------------------------------------------ router
template <int NT>
__global__ void __launch_bounds__(kThreads, 1) k_router(const RouterArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float s_lg[16][256];             // this CTA's logits, by expert index
  __shared__ unsigned s_mask[256];            // rank 0: rows of the group that chose expert e
  __shared__ unsigned long long s_jbits[256]; // rank 0: 3-bit slot of each such row
  __shared__ int4 s_scan[kWarps];
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const StreamPlan& p = a.sp;
  __half* xs = reinterpret_cast<__half*>(smem + p.xs_off);
  float* red = reinterpret_cast<float*>(smem + p.red_off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + p.ring_off + (size_t)warp * kRingDepth * p.slot;

  if (!(kPdlLate & PDL_ROUTER)) pdl_launch_dependents();
  const int cs = gridDim.x, rank = blockIdx.x;  // the cluster spans x
  const int g = blockIdx.y, tok0 = g * 16;
  const int ntok = min(a.ntok - tok0, NT * 8);
  const int H = a.H, E = a.E;
  const int my_slabs = (rank < a.w.n_slabs) ? (a.w.n_slabs - 1 - rank) / cs + 1 : 0;
  const SlabWork w = slab_work(rank, cs, my_slabs, a.w.U);
  UnitStream<F16> us;
  us.start(a.w.q, a.w.s, w);
  us.prefetch(ring, p.slot, w, lane);
  if (kWarmTopk && E <= 64) {
    // run the top-k once on placeholder logits while the previous kernel drains:
    // it pulls the (once-per-launch, otherwise cold) code into the instruction cache
    RowLogits rl;
#pragma unroll
    for (int q = 0; q < 8; ++q) rl.v[q] = (float)((lane * 37 + q * 11) & 63);
    int rk[2];
    float wt[2];
    topk_rank<2>(rl, E, a.k, lane, rk, wt);
    if (wt[0] < -1.f) s_mask[lane] = (unsigned)rk[0];  // never true; keeps the work
  }
  NormW nw;
  load_norm_w(nw, a.norm_w, H);
  if (rank == 0)  // every rank ORs its rows' choices into rank 0's masks (cleared before the first cluster barrier)
    for (int e = threadIdx.x; e < E; e += kThreads) {
      s_mask[e] = 0u;
      s_jbits[e] = 0ull;
    }
  pdl_wait();
  stage_norm_rows(xs, p.ldx, a.h + (size_t)tok0 * H, H, ntok, NT * 8, a.norm_w, nw, H, a.eps);
  __syncthreads();
  const BSmem bp(xs, p.ldx);
  auto epi = [&](int sl, const float* rb, int tid, int nthr) {
    for (int i = tid; i < NT * 64; i += nthr) {
      const int tok = i >> 3, pg = i & 7;
      if (tok >= ntok) continue;
      float lo, hi;
      group_sum<NT>(rb, w.ks, tok, pg, lo, hi);
      const int e0 = 16 * sl + pg;
      if (e0 < E) {
        s_lg[tok][e0] = lo;
        a.logits[(size_t)(tok0 + tok) * E + e0] = lo;
      }
      if (e0 + 8 < E) {
        s_lg[tok][e0 + 8] = hi;
        a.logits[(size_t)(tok0 + tok) * E + e0 + 8] = hi;
      }
    }
  };
  run_stream<F16, NT>(us, w, ring, p.slot, red, bp, NT, epi);
  if (kPdlLate & PDL_ROUTER) pdl_launch_dependents();
  cluster.sync();  // every CTA's logits are in its shared memory, rank 0's masks are clear

  {  // the group's rows are ranked by all CTAs of the cluster: row r by rank r % cs
    unsigned* mask0 = cluster.map_shared_rank(&s_mask[0], 0);
    unsigned long long* jbits0 = cluster.map_shared_rank(&s_jbits[0], 0);
    const int k = a.k;
    const int qn = (E + 31) / 32;
    for (int r = rank + cs * warp; r < ntok; r += cs * kWarps) {
      RowLogits rl;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = lane + 32 * q;
        rl.v[q] = -INFINITY;
        if (e < E) {
          const float* peer = cluster.map_shared_rank(&s_lg[0][0], (e >> 4) % cs);
          rl.v[q] = peer[r * 256 + e];
        }
      }
      auto emit = [&](auto qn_tag) {
        constexpr int QN = decltype(qn_tag)::value;
        int rk[QN];
        float wt[QN];
        topk_rank<QN>(rl, E, k, lane, rk, wt);
#pragma unroll
        for (int q = 0; q < QN; ++q) {
          const int e = lane + 32 * q;
          if (e < E && rk[q] < k) {
            a.idx[(tok0 + r) * k + rk[q]] = e;
            a.wts[(tok0 + r) * k + rk[q]] = wt[q];
            atomicOr(&mask0[e], 1u << r);  // a row picks an expert at most once
            // the row's 3-bit slot, as 32-bit ORs on the two halves of the expert's word
            const unsigned long long bits = (unsigned long long)rk[q] << (3 * r);
            unsigned* jw = reinterpret_cast<unsigned*>(jbits0 + e);
            if ((unsigned)bits) atomicOr(jw, (unsigned)bits);
            if ((unsigned)(bits >> 32)) atomicOr(jw + 1, (unsigned)(bits >> 32));
          }
        }
      };
      if (qn <= 2) emit(std::integral_constant<int, 2>{});
      else if (qn <= 4) emit(std::integral_constant<int, 4>{});
      else emit(std::integral_constant<int, 8>{});
    }
  }
  // the remote ORs are complete and visible at cluster scope before the barrier
  asm volatile("fence.acq_rel.cluster;" ::: "memory");
  cluster.sync();  // every rank's choices are in rank 0's masks; no CTA reads a peer after this

  if (rank == 0) {
    const int e = threadIdx.x;
    const unsigned mk = e < E ? s_mask[e] : 0u;
    const unsigned long long jb = e < E ? s_jbits[e] : 0ull;
    int4* rec = a.rec + (size_t)g * a.n_units;
    if (a.by_slot) {  // one token group: unit i = the i-th expert that received a token
      int4 tot;
      const int4 ex = block_excl_scan4(make_int4(mk != 0u, 0, 0, 0), tot, s_scan);
      if (mk) rec[ex.x] = make_int4(e, (int)mk, (int)(uint32_t)jb, (int)(uint32_t)(jb >> 32));
      for (int i = tot.x + threadIdx.x; i < a.n_units; i += kThreads) rec[i] = make_int4(-1, 0, 0, 0);
    } else if (e < E) {
      rec[e] = make_int4(mk ? e : -1, (int)mk, (int)(uint32_t)jb, (int)(uint32_t)(jb >> 32));
    }
  }
}

// ------------------------------------------------------------------ gate/up
// One grid for every token group: a routed CTA takes its unit's rows over the
// whole step (the records of all token groups), so each expert's weights are
// streamed once per 16 of its rows, not once per token group; shared-expert
// CTAs take every row.  Rows go through in passes of 16 (NT n-tiles); a pass
// after the first streams the CTA's slabs again (from L2).
template <int FR, int FS, int NT>
__global__ void __launch_bounds__(kThreads, kMinBlocks) k_expert_gateup(const ExpertArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ RouteSmem rs;
  const StreamPlan& p = a.sp;
  __half* xs = reinterpret_cast<__half*>(smem + p.xs_off);
  float* red = reinterpret_cast<float*>(smem + p.red_off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + p.ring_off + (size_t)warp * kRingDepth * p.slot;

  if (!(kPdlLate & PDL_EXPERT)) pdl_launch_dependents();
  ExpertCta ec = expert_cta(a);
  int s0 = 0, s1 = 0;
  SlabWork w;
  UnitStream<FS> uss;
  UnitStream<FR> usr;
  bool streaming = false;
  if (ec.shared) {  // the shared experts need nothing from the router: start streaming now
    part_range(a.ws.n_slabs, groups_of(a.ws.U), ec.part, ec.parts, s0, s1);
    w = slab_work(s0, 1, s1 - s0, a.ws.U);
    uss.start(a.ws.q, a.ws.s, w);
    uss.prefetch(ring, p.slot, w, lane);
    streaming = true;
  } else if (!a.by_slot) {  // expert-id layout: the head of this expert's weights, before the routing is known
    part_range(a.wr.n_slabs, groups_of(a.wr.U), ec.part, ec.parts, s0, s1);
    w = slab_work(s0, 1, s1 - s0, a.wr.U);
    usr.start(a.wr.q + (size_t)ec.i * a.wr.q_stride, a.wr.s + (size_t)ec.i * a.wr.s_stride, w);
    usr.prefetch(ring, p.slot, w, lane);
    streaming = true;
  }
  NormW nw;
  load_norm_w(nw, a.norm_w, a.H);
  pdl_wait();

  if (blockIdx.x == 0) write_grouping(rs, a);
  // this CTA's rows
  int e = -1, ntk = a.ntok;
  if (!ec.shared) {
    if (a.by_slot) {  // one token group
      const int t = threadIdx.x;
      rs.grec[0] = record_by_slot(a, t < a.n_units ? __ldcg(a.rec + t) : make_int4(-1, 0, 0, 0), ec, rs);
    } else if ((int)threadIdx.x < a.tg) {
      rs.grec[threadIdx.x] = __ldcg(a.rec + (size_t)threadIdx.x * a.n_units + ec.i);
    }
    __syncthreads();
    e = rs.grec[0].x;
    for (int g = 1; g < a.tg; ++g) e = e >= 0 ? e : rs.grec[g].x;
    ntk = e >= 0 ? gather_unit_rows(rs, a.by_slot ? 1 : a.tg, a.k) : 0;
    if (ntk == 0) {
      if (streaming) cp_wait<0>();  // copies in flight land before the CTA leaves
      return;
    }
    if (a.by_slot) {
      part_range(a.wr.n_slabs, groups_of(a.wr.U), ec.part, ec.parts, s0, s1);
      if (s0 == s1) return;  // a part without a round (nothing in flight yet)
      w = slab_work(s0, 1, s1 - s0, a.wr.U);
      usr.start(a.wr.q + (size_t)e * a.wr.q_stride, a.wr.s + (size_t)e * a.wr.s_stride, w);
      usr.prefetch(ring, p.slot, w, lane);
    }
  } else {
    for (int t = threadIdx.x; t < ntk; t += kThreads) rs.rows[t] = t;
  }
  for (int pass = 0; pass * 16 < ntk; ++pass) {
    const int r0 = pass * 16, n = min(16, ntk - r0);
    if (pass > 0) {  // the same slabs again for the next 16 rows (L2-resident by now)
      if (ec.shared) {
        uss.start(a.ws.q, a.ws.s, w);
        uss.prefetch(ring, p.slot, w, lane);
      } else {
        usr.start(a.wr.q + (size_t)e * a.wr.q_stride, a.wr.s + (size_t)e * a.wr.s_stride, w);
        usr.prefetch(ring, p.slot, w, lane);
      }
    }
    __syncthreads();  // the previous pass's readers of xs are done
    // the pass's rows, normalised, packed into consecutive tokens
    stage_norm_gather(xs, p.ldx, a.h, a.H, rs.rows + r0, n, NT * 8, a.norm_w, nw, a.H, a.eps);
    __syncthreads();
    const int nt_used = (n + 7) >> 3;
    const BSmem bp(xs, p.ldx);
    if (ec.shared) {
      auto epi = [&](int sl, const float* rb, int tid, int nthr) {
        for (int i = tid; i < NT * 64; i += nthr) {
          const int tok = i >> 3, pg = i & 7;
          if (tok >= n) continue;
          float lo, hi;
          group_sum<NT>(rb, w.ks, tok, pg, lo, hi);
          const int r = r0 + tok;
          *reinterpret_cast<__half*>(a.act_s + bfrag_offset(r >> 3, r & 7, 8 * sl + pg, a.Ish >> 5)) =
              __float2half_rn(silu(lo) * hi);
        }
      };
      run_stream<FS, NT>(uss, w, ring, p.slot, red, bp, nt_used, epi);
    } else {
      const int tile0 = (e * a.tg + pass) * 2;  // two 8-token tiles per (expert, pass)
      auto epi = [&](int sl, const float* rb, int tid, int nthr) {
        for (int i = tid; i < NT * 64; i += nthr) {
          const int tok = i >> 3, pg = i & 7;
          if (tok >= n) continue;
          float lo, hi;
          group_sum<NT>(rb, w.ks, tok, pg, lo, hi);
          *reinterpret_cast<__half*>(a.act_r + bfrag_offset(tile0 + (tok >> 3), tok & 7, 8 * sl + pg, a.Ie >> 5)) =
              __float2half_rn(silu(lo) * hi);
        }
      };
      run_stream<FR, NT>(usr, w, ring, p.slot, red, bp, nt_used, epi);
    }
  }
  if (kPdlLate & PDL_EXPERT) pdl_launch_dependents();
}

// ------------------------------------------------------------------ down + combine
template <int FR, int FS, int NT>
__global__ void __launch_bounds__(kThreads, kMinBlocks) k_expert_down(const ExpertArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ RouteSmem rs;
  const StreamPlan& p = a.sp;
  float* red = reinterpret_cast<float*>(smem + p.red_off);
  uint8_t* btile = smem + p.extra_off;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + p.ring_off + (size_t)warp * kRingDepth * p.slot;

  if (!(kPdlLate & PDL_EXPERT)) pdl_launch_dependents();
  ExpertCta ec = expert_cta(a);
  const int H = a.H, k = a.k, rows = a.ntok;
  int s0 = 0, s1 = 0;
  SlabWork w;
  UnitStream<FS> uss;
  UnitStream<FR> usr;
  bool streaming = false;
  if (ec.shared) {
    part_range(H / 16, groups_of(a.ws.U), ec.part, ec.parts, s0, s1);
    w = slab_work(s0, 1, s1 - s0, a.ws.U);
    uss.start(a.ws.q, a.ws.s, w);
    uss.prefetch(ring, p.slot, w, lane);
    streaming = true;
  } else if (!a.by_slot) {
    part_range(H / 16, groups_of(a.wr.U), ec.part, ec.parts, s0, s1);
    w = slab_work(s0, 1, s1 - s0, a.wr.U);
    usr.start(a.wr.q + (size_t)ec.i * a.wr.q_stride, a.wr.s + (size_t)ec.i * a.wr.s_stride, w);
    usr.prefetch(ring, p.slot, w, lane);
    streaming = true;
  }
  pdl_wait();
  int4 mine = make_int4(-1, 0, 0, 0);  // active-slot units: record threadIdx.x of the (single) group
  if (a.by_slot && (int)threadIdx.x < a.n_units) mine = __ldcg(a.rec + threadIdx.x);
  int e = -1, ntk = rows;
  const int k32 = (ec.shared ? a.Ish : a.Ie) >> 5;
  if (!ec.shared) {
    if (a.by_slot) {
      rs.grec[0] = record_by_slot(a, mine, ec, rs);
    } else if ((int)threadIdx.x < a.tg) {
      rs.grec[threadIdx.x] = __ldcg(a.rec + (size_t)threadIdx.x * a.n_units + ec.i);
    }
    __syncthreads();
    e = rs.grec[0].x;
    for (int g = 1; g < a.tg; ++g) e = e >= 0 ? e : rs.grec[g].x;
    ntk = e >= 0 ? gather_unit_rows(rs, a.by_slot ? 1 : a.tg, k) : 0;
    if (ntk == 0) {
      if (streaming) cp_wait<0>();
      return;
    }
    if (a.by_slot) {
      part_range(H / 16, groups_of(a.wr.U), ec.part, ec.parts, s0, s1);
      if (s0 == s1) return;  // a part without a round (nothing in flight yet)
      w = slab_work(s0, 1, s1 - s0, a.wr.U);
      usr.start(a.wr.q + (size_t)e * a.wr.q_stride, a.wr.s + (size_t)e * a.wr.s_stride, w);
      usr.prefetch(ring, p.slot, w, lane);
    }
  }
  for (int pass = 0; pass * 16 < ntk; ++pass) {
    const int r0 = pass * 16, n = min(16, ntk - r0);
    if (pass > 0) {
      if (ec.shared) {
        uss.start(a.ws.q, a.ws.s, w);
        uss.prefetch(ring, p.slot, w, lane);
      } else {
        usr.start(a.wr.q + (size_t)e * a.wr.q_stride, a.wr.s + (size_t)e * a.wr.s_stride, w);
        usr.prefetch(ring, p.slot, w, lane);
      }
    }
    const int tiles = (n + 7) >> 3;
    const uint8_t* bsrc = ec.shared ? a.act_s + (size_t)(r0 >> 3) * k32 * 512
                                    : a.act_r + (size_t)((e * a.tg + pass) * 2) * k32 * 512;
    __syncthreads();  // the previous pass's readers of btile are done
    stage_bytes(btile, bsrc, tiles * k32 * 512);
    __syncthreads();
    const BSmemFrag bp{btile, k32};
    auto epi = [&](int sl, const float* rb, int tid, int nthr) {
      for (int i = tid; i < NT * 64; i += nthr) {
        const int tok = i >> 3, pg = i & 7;
        if (tok >= n) continue;
        float lo, hi;
        group_sum<NT>(rb, w.ks, tok, pg, lo, hi);
        float* dst = ec.shared ? a.part_s + (size_t)(r0 + tok) * H : a.part_r + (size_t)rs.ent[r0 + tok] * H;
        dst[16 * sl + pg] = lo;
        dst[16 * sl + pg + 8] = hi;
      }
    };
    if (ec.shared)
      run_stream<FS, NT>(uss, w, ring, p.slot, red, bp, tiles, epi);
    else
      run_stream<FR, NT>(usr, w, ring, p.slot, red, bp, tiles, epi);
  }
  if (kPdlLate & PDL_EXPERT) pdl_launch_dependents();

}

// ------------------------------------------------------------------ combine
// out[r][c] = h[r][c] + sum_j w[r][j] * part_r[r*k + j][c] (slot order) + part_s[r][c]:
// one thread per output, after every expert CTA of the down launch has written
// its partials (griddepcontrol.wait), in the same fixed order for every row.
__global__ void __launch_bounds__(256) k_expert_combine(const ExpertArgs a) {
  pdl_launch_dependents();
  const int H = a.H, k = a.k;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int r = i / H, c = i - r * H;
  float w[8];
  const bool ok = r < a.ntok;
  pdl_wait();
  if (!ok) return;
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = j < k ? __ldcg(a.wts + r * k + j) : 0.f;
  float pr[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) pr[j] = j < k ? __ldcg(a.part_r + (size_t)(r * k + j) * H + c) : 0.f;
  const float ps = a.ws.n_slabs > 0 ? __ldcg(a.part_s + (size_t)r * H + c) : 0.f;
  float v = a.h[(size_t)r * H + c];
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < k) v += w[j] * pr[j];
  a.out[(size_t)r * H + c] = v + ps;
}

// ------------------------------------------------------------------ launchers
int router_cluster(int n_slabs) { return n_slabs < 8 ? n_slabs : 8; }

cudaError_t launch_router(const RouterArgs& a, cudaStream_t st, bool pdl) {
  const int cs = router_cluster(a.w.n_slabs);
  const dim3 grid(cs, a.tg);
  if (a.sp.nt == 1) return launch_kernel_cluster(k_router<1>, grid, dim3(kThreads), a.sp.bytes, st, pdl, cs, a);
  return launch_kernel_cluster(k_router<2>, grid, dim3(kThreads), a.sp.bytes, st, pdl, cs, a);
}

#define UOCR_PAIRS(X, NT_) \
  X(Q8_0, Q8_0, NT_) X(Q4_0, Q8_0, NT_) X(Q4_0, Q4_0, NT_) X(Q8_0, Q4_0, NT_) X(I8ASYM, I8ASYM, NT_)

static dim3 expert_grid(const ExpertArgs& a) {
  return dim3((a.ws.n_slabs > 0 ? a.cpes : 0) + (a.by_slot ? a.n_rctas : a.n_units * a.cpe), 1);
}

cudaError_t launch_expert_gateup(int fr, int fs, const ExpertArgs& a, cudaStream_t st, bool pdl) {
  const dim3 grid = expert_grid(a);
#define X(FR_, FS_, NT_)                                                                               \
  if (fr == FR_ && fs == FS_ && a.sp.nt == NT_)                                                        \
    return launch_kernel(k_expert_gateup<FR_, FS_, NT_>, grid, dim3(kThreads), a.sp.bytes, st, pdl, a);
  UOCR_PAIRS(X, 1)
  UOCR_PAIRS(X, 2)
#undef X
  return cudaErrorInvalidValue;
}

cudaError_t launch_expert_combine(const ExpertArgs& a, cudaStream_t st, bool pdl) {
  const int n = a.ntok * a.H;
  return launch_kernel(k_expert_combine, dim3((n + 255) / 256), dim3(256), 0, st, pdl, a);
}

cudaError_t launch_expert_down(int fr, int fs, const ExpertArgs& a, cudaStream_t st, bool pdl) {
  const dim3 grid = expert_grid(a);
#define X(FR_, FS_, NT_)                                                                             \
  if (fr == FR_ && fs == FS_ && a.sp.nt == NT_)                                                      \
    return launch_kernel(k_expert_down<FR_, FS_, NT_>, grid, dim3(kThreads), a.sp.bytes, st, pdl, a);
  UOCR_PAIRS(X, 1)
  UOCR_PAIRS(X, 2)
#undef X
  return cudaErrorInvalidValue;
}

cudaError_t init_moe_attributes() {
  cudaError_t e = allow_max_dyn_smem(k_router<1>);
  if (e == cudaSuccess) e = allow_max_dyn_smem(k_router<2>);
#define X(FR_, FS_, NT_)                                                      \
  if (e == cudaSuccess) e = allow_max_dyn_smem(k_expert_gateup<FR_, FS_, NT_>); \
  if (e == cudaSuccess) e = allow_max_dyn_smem(k_expert_down<FR_, FS_, NT_>);
  UOCR_PAIRS(X, 1)
  UOCR_PAIRS(X, 2)
#undef X
  return e;
}

}  // namespace uocr
