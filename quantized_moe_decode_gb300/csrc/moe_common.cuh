// Routing state and work assignment shared by the expert kernels (the
// fragment-GEMV ones and the tensor-core ones): the token grouping written
// from the router's choices, a routed unit's rows over all token groups, and
// which CTA takes which unit and which part of its slabs.  Block-size generic.
#pragma once
#include "launch.h"

namespace uocr {

// Block-wide exclusive prefix sum of four counters (one value per thread).
__device__ __forceinline__ int4 block_excl_scan4(int4 v, int4& total, int4* s_warp) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int4 inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, inc.x, o), y = __shfl_up_sync(0xffffffffu, inc.y, o);
    const int z = __shfl_up_sync(0xffffffffu, inc.z, o), w = __shfl_up_sync(0xffffffffu, inc.w, o);
    if (lane >= o) {
      inc.x += x;
      inc.y += y;
      inc.z += z;
      inc.w += w;
    }
  }
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  int4 base = make_int4(0, 0, 0, 0);
  total = make_int4(0, 0, 0, 0);
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    const int4 t = s_warp[w];
    if (w < warp) {
      base.x += t.x;
      base.y += t.y;
      base.z += t.z;
      base.w += t.w;
    }
    total.x += t.x;
    total.y += t.y;
    total.z += t.z;
    total.w += t.w;
  }
  __syncthreads();  // s_warp may be reused by the caller's next scan
  return make_int4(base.x + inc.x - v.x, base.y + inc.y - v.y, base.z + inc.z - v.z, base.w + inc.w - v.w);
}

// Routing state of a CTA in shared memory.
struct RouteSmem {
  int idx[64 * 8];                  // [row][k] chosen experts
  unsigned long long rowmask[256];  // [E] rows that chose expert e (bit r)
  int off[256];
  int4 scan[16];                    // per-warp partials of block_excl_scan4 (<= 16 warps)
  int4 rec;                         // this CTA's routing record (active-slot units)
  int4 grec[4];                     // this CTA's unit's record of each token group
  int rows[64];                     // the unit's rows over all token groups, ascending
  int ent[64];                      // their entries row * k + slot
  int e, n;
};

// The rows of a routed unit over all token groups (ascending) and their entries
// row * k + slot, from the unit's record of each group (rs.grec[0..tg)): warp 0
// builds the list, one lane per group.  Returns the row count (all threads).
__device__ __forceinline__ int gather_unit_rows(RouteSmem& rs, int tg, int k) {
  if (threadIdx.x < 32) {
    const int g = threadIdx.x;
    const int4 r = g < tg ? rs.grec[g] : make_int4(-1, 0, 0, 0);
    const unsigned m = r.x >= 0 ? (unsigned)r.y : 0u;
    const int c = __popc(m);
    int base = c;  // inclusive scan over the (at most 4) groups
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, base, o);
      if (g >= o) base += y;
    }
    if (g == 3) rs.n = base;  // groups >= tg count zero rows
    base -= c;
    const unsigned long long jb = (unsigned long long)(uint32_t)r.z | ((unsigned long long)(uint32_t)r.w << 32);
    for (unsigned mm = m; mm; mm &= mm - 1u) {
      const int bit = __ffs(mm) - 1;
      const int row = 16 * g + bit;
      rs.rows[base] = row;
      rs.ent[base] = row * k + (int)((jb >> (3 * bit)) & 7ull);
      ++base;
    }
  }
  __syncthreads();
  return rs.n;
}

__device__ __forceinline__ void clear_rowmask(RouteSmem& rs, int E) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) rs.rowmask[e] = 0ull;
}

// The grouping of the step: count[e] (histogram), offset = exclusive scan,
// perm = entries row*k + slot grouped by expert ascending, rows ascending
// within an expert; inv = position of each entry in perm.  From the router's
// choices idx[rows][k].  All threads.
__device__ __forceinline__ void write_grouping(RouteSmem& rs, const ExpertArgs& a) {
  const int rows = a.ntok, E = a.E, k = a.k;
  clear_rowmask(rs, E);
  __syncthreads();
  for (int i = threadIdx.x; i < rows * k; i += blockDim.x) {
    const int ei = __ldcg(a.idx + i);
    rs.idx[i] = ei;
    atomicOr(&rs.rowmask[ei], 1ull << (i / k));  // a row picks an expert at most once
  }
  __syncthreads();
  const int e = threadIdx.x;
  const unsigned long long rm = e < E ? rs.rowmask[e] : 0ull;
  int4 tot;
  const int4 ex = block_excl_scan4(make_int4(__popcll(rm), 0, 0, 0), tot, rs.scan);
  if (e < E) {
    a.count[e] = __popcll(rm);
    a.offset[e] = ex.x;
    rs.off[e] = ex.x;
  }
  if (threadIdx.x == 0) a.offset[E] = tot.x;
  __syncthreads();
  for (int i = threadIdx.x; i < rows * k; i += blockDim.x) {
    const int ei = rs.idx[i], r = i / k;
    const int pos = rs.off[ei] + __popcll(rs.rowmask[ei] & ((1ull << r) - 1ull));
    a.perm[pos] = i;
    a.inv[i] = pos;
  }
}

// ------------------------------------------------------------------ expert CTAs
// blockIdx.x < ns (= cpes when there are shared experts, else 0): part x of
// the shared experts.  Then routed CTAs.  With expert-id units: unit i =
// (x - ns) / cpe, part (x - ns) % cpe of its slabs.  With active-slot units
// the n_rctas routed CTAs are dealt out over the n active slots once the
// router has counted them (slot_assign): every routed CTA has work and the
// grid is one wave whatever the number of experts that received a token.
// The grid has one row (blockIdx.y = 0): a CTA covers every token group.
struct ExpertCta {
  bool shared;
  int i, part, parts;
};
__device__ __forceinline__ ExpertCta expert_cta(const ExpertArgs& a) {
  ExpertCta c;
  const int ns = a.ws.n_slabs > 0 ? a.cpes : 0;
  const int x = blockIdx.x;
  c.shared = x < ns;
  if (c.shared) {
    c.i = -1;
    c.part = x;
    c.parts = a.cpes;
  } else if (a.by_slot) {  // known after the router: slot_assign
    c.i = -1;
    c.part = 0;
    c.parts = 1;
  } else {
    c.i = (x - ns) / a.cpe;
    c.part = (x - ns) - c.i * a.cpe;
    c.parts = a.cpe;
  }
  return c;
}

// R routed CTAs over n active slots (1 <= n <= R, which the host guarantees by
// launching at least as many routed CTAs as experts can receive a token): the
// first R % n slots get R / n + 1 CTAs, the others R / n, in slot order.
__device__ __forceinline__ void slot_assign(int xr, int R, int n, ExpertCta& c) {
  const int base = R / n, rem = R - base * n;
  const int cut = rem * (base + 1);
  if (xr < cut) {
    c.i = xr / (base + 1);
    c.part = xr - c.i * (base + 1);
    c.parts = base + 1;
  } else {
    const int y = xr - cut;
    c.i = rem + y / base;
    c.part = y - (c.i - rem) * base;
    c.parts = base;
  }
}
__device__ __forceinline__ void assign_routed(const ExpertArgs& a, int n, ExpertCta& c) {
  if (c.shared || !a.by_slot) return;
  const int ns = a.ws.n_slabs > 0 ? a.cpes : 0;
  if (n < 1 || n > a.n_rctas) {  // cannot happen (n_rctas >= most experts a group can pick)
    c.i = -1;
    return;
  }
  slot_assign((int)blockIdx.x - ns, a.n_rctas, n, c);
}
// Active-slot units (one token group, at most kThreads records): thread t
// holds record t (`mine`).  The records with rows are the active slots, in
// slot order, so their count deals the routed CTAs out (slot_assign) without a
// separate load of the count, and the thread holding this CTA's record passes
// it on through shared memory.  All threads of the CTA; two barriers.
__device__ __forceinline__ int4 record_by_slot(const ExpertArgs& a, int4 mine, ExpertCta& c, RouteSmem& rs) {
  assign_routed(a, __syncthreads_count(mine.y != 0), c);
  if (c.i >= 0 && (int)threadIdx.x == c.i) rs.rec = mine;
  __syncthreads();
  return c.i >= 0 ? rs.rec : make_int4(-1, 0, 0, 0);
}

// Slabs [lo, hi) of part `part` of `parts`: n slabs cut in runs of gran (the
// slabs of one round of a CTA) so that every group of warps gets whole rounds.
// Each part takes ceil(rounds / parts) rounds; the parts this leaves without
// a round (e.g. the 8th of 8 parts of 20 rounds) get none, which keeps the
// longest part as short as an even split would and leaves their SM to the
// CTAs that have work.
__device__ __forceinline__ void part_range(int n, int gran, int part, int parts, int& lo, int& hi) {
  const int nr = (n + gran - 1) / gran;
  const int per = (nr + parts - 1) / parts;
  lo = min(n, gran * min(nr, part * per));
  hi = min(n, gran * min(nr, (part + 1) * per));
}
__device__ __forceinline__ int groups_of(int U) { return kWarps / warps_per_slab(U); }

}  // namespace uocr
