// sv_tree.cu -- verification of drafted token trees (multi-candidate rejection
// sampling), sm_103a.
//
// Method. The DSpark Guide names tree verification ("Deep Dive into the DSpark
// Architecture", step 4: the verified prefix goes to the target "with tree / sequence
// mask"; "3. Comprehensive Technical Feature Matrix": "Static / Tree" verification) and
// the DSpark Deep Dive ("The Speculative Decoding Solution") gives the chain rule it
// extends. Reading implemented here: the walk starts at node 0; at node c the children
// are tested in index order against a residual distribution r that starts as p_c; child
// n with token x is accepted when u_n * q_c(x) < r(x), and the walk moves to n; after a
// rejection r <- normalize(max(0, r - q_c)). When every child is rejected the token is
// sampled from r by inverse CDF at u_{b,0}; at a leaf, from p_c. At T == 0 the first
// child drafting the lowest-index argmax of p_c is accepted, else that argmax is emitted.
//
// Closed form. After i rejections r = max(0, p - lam_i q) / W_i, with lam_0 = 0,
// W_0 = 1, lam_{i+1} = lam_i + W_i and W_{i+1} = sum_v max(0, p_v - lam_{i+1} q_v)
// (because max(0, max(0, a) - b) = max(0, a - b) for b >= 0). A rejection therefore
// costs one pass over the node's two rows, and no residual is ever stored.
//
// Layout. One cluster of C CTAs per request (C = 1..8, picked by the host so the batch
// is resident at once). Each row is cut into 16-byte vectors on a grid anchored at the
// row's own alignment, 32 vectors make a tile, and each CTA owns a contiguous range of
// tiles, each warp a contiguous sub-range (lanes read consecutive vectors: coalesced).
// Per visited node the cluster makes one pass for the softmax statistics of both rows
// (argmax of the target row at T == 0), one pass per rejection for W, and samples from
// the last pass's totals in three levels (CTA, warp group of tiles, element). Every
// warp leaves its partial result in shared memory; after one hardware cluster barrier
// warp 0 of every CTA reads all C x 16 partials over distributed shared memory and
// merges them in a fixed order (softmax statistics in one frame: the maximum first,
// then each partial rescaled once), so all CTAs reach bit-identical values, take the
// same branches and arrive at the same barriers. Only rows the walk reaches are read.
#include <cfloat>
#include <atomic>
#include <cooperative_groups.h>

#include "sv_cluster.cuh"
#include "sv_tree.cuh"

namespace cg = cooperative_groups;

namespace sv {
namespace {

using namespace clx;

constexpr int TW = 16;          // warps per CTA
constexpr int TT = 32 * TW;     // threads per CTA
constexpr int UNR = 4;          // tiles a lane has in flight per row (two-row passes)
constexpr int UNR_G = 8;        // the same for the one-row greedy pass
static_assert(32 % TW == 0, "a CTA's warp partials fill whole halves of a warp");
constexpr int NGRP = 32;        // group totals kept per warp for the inverse CDF
constexpr int MAXC = 8;         // largest cluster

// ---------------------------------------------------------------------------
// Shared state of one CTA.
// ---------------------------------------------------------------------------
struct Xch {  // a partial or merged result
  Soft st, sd;
  float best;
  int idx;
  int bad;
  ff tot;
};

struct __align__(16) Xw {  // one warp's partial result, read by every CTA of the cluster
  Soft st, sd;
  float best;
  int idx;
  int bad;
  int pad;
  ff tot;
  ff pad2;
};

struct Smem {
  int par[SV_MAX_TREE];
  int tok[SV_MAX_TREE];
  float u[SV_MAX_TREE];
  float czt[SV_MAX_TREE], czd[SV_MAX_TREE];  // logits of each child's token (T > 0)
  int nn;
  int ok;
  int dec;
  int sel_w, sel_g;
  ff sel_cum;
  ff gtot[TW][NGRP];
  ff ctot[MAXC];
  Xw xw[2][TW];  // per-warp partials, alternating between passes
  Soft sst[TW];  // per-warp statistics of the target row from the node's statistics pass
  ff pw[TW];     // per-warp totals of p (sample without a weight pass)
  Xch res;
  int lastbuf;   // the xw buffer of the last pass
};

// Tiles [t0, t1) of warp w in CTA `rank` of C, for a row of `ntiles` tiles.
__device__ __forceinline__ void warp_tiles(int ntiles, int C, int rank, int w, int& t0,
                                           int& t1) {
  const int tpc = (ntiles + C - 1) / C;
  const int c0 = min(ntiles, rank * tpc), c1 = min(ntiles, c0 + tpc);
  const int tpw = (c1 - c0 + TW - 1) / TW;
  t0 = min(c1, c0 + w * tpw);
  t1 = min(c1, t0 + tpw);
}

// Tiles per group: at least a round of UNR (one warp reduction per round), and few
// enough groups to fit NGRP.
__device__ __forceinline__ int group_size(int nt) { return max(UNR, (nt + NGRP - 1) / NGRP); }

// ---------------------------------------------------------------------------
// Passes over one node's rows. Each ends with the cluster-wide result in sm.res and
// every thread past a CTA barrier.
// ---------------------------------------------------------------------------
struct Geo {
  int V, off, nvec, ntiles, t0, t1;
};

template <typename T>
__device__ __forceinline__ Geo make_geo(const T* tr, int V, int C, int rank, int w) {
  constexpr int VEC = EV<T>::VEC;
  Geo g;
  g.V = V;
  g.off = row_off(tr);
  g.nvec = (V + g.off + VEC - 1) / VEC;
  g.ntiles = (g.nvec + 31) / 32;
  warp_tiles(g.ntiles, C, rank, w, g.t0, g.t1);
  return g;
}

// A round of UNR tiles from tile tb on is interior when all its tiles belong to the warp
// and every vector in them is whole (vector j covers elements j*VEC - off ..): no
// per-vector checks then. `d_off_grid`: the draft row is off the grid (never interior).
template <typename T>
__device__ __forceinline__ bool interior_round(const Geo& g, int tb, bool d_off_grid) {
  constexpr int VEC = EV<T>::VEC;
  const int jlo = g.off > 0 ? 1 : 0, jhi = (g.V + g.off) / VEC;  // whole vectors: [jlo, jhi)
  return !d_off_grid && tb + UNR <= g.t1 && tb * 32 >= jlo && (tb + UNR) * 32 <= jhi;
}

// Waits for every warp of the cluster to have stored its partial in sm.xw[buf], then
// warp 0 of each CTA merges the C x TW partials (over distributed shared memory) in a
// fixed order into sm.res, so all CTAs reach bit-identical values: the statistics in
// one frame (the maximum first, then each partial rescaled once into it), the argmax,
// or the weight totals per CTA (warps in order; into sm.ctot) and over the cluster
// (CTAs in rank order).
template <int KIND>
__device__ __forceinline__ void exchange(Smem& sm, cg::cluster_group& cl, int C, int buf,
                                         float a) {
  cl.sync();  // also a CTA barrier
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int n = C * TW;
    constexpr int PER = MAXC * TW / 32;  // entries per lane at most
    Xch r;
    r.st = soft_empty();
    r.sd = soft_empty();
    r.best = -INFINITY;
    r.idx = INT_MAX;
    r.bad = 0;
    r.tot = ff{0.f, 0.f};
    if (KIND == 0) {
      Soft et[PER], ed[PER];
      bool bad = false;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int e = lane + 32 * i;
        et[i] = ed[i] = soft_empty();
        if (e < n) {
          const Xw* x = cl.map_shared_rank(&sm.xw[buf][e % TW], e / TW);
          et[i] = x->st;
          ed[i] = x->sd;
          bad |= x->bad != 0;
        }
      }
      r.bad = __any_sync(FULLM, bad);
      r.st = soft_frame_merge<PER>(et, a);
      r.sd = soft_frame_merge<PER>(ed, a);
    } else if (KIND == 1) {
      bool bad = false;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int e = lane + 32 * i;
        if (e < n) {
          const Xw* x = cl.map_shared_rank(&sm.xw[buf][e % TW], e / TW);
          arg_merge(r.best, r.idx, x->best, x->idx);
          bad |= x->bad != 0;
        }
      }
      r.bad = __any_sync(FULLM, bad);
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float b2 = __shfl_xor_sync(FULLM, r.best, o);
        const int i2 = __shfl_xor_sync(FULLM, r.idx, o);
        arg_merge(r.best, r.idx, b2, i2);
      }
    } else {
      // Entry e = lane + 32 i is warp e % TW of CTA e / TW (all loads in flight); a
      // fixed butterfly over each TW-lane half adds a CTA's warps, and the cluster's
      // total adds the CTAs in rank order, the order the sample's search walks them.
      ff v[PER];
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < n ? cl.map_shared_rank(&sm.xw[buf][e % TW], e / TW)->tot : ff{0.f, 0.f};
      }
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        ff t = v[i];
#pragma unroll
        for (int o = TW / 2; o; o >>= 1) t = ff_add(t, ff_shfl_xor(t, o));
        const int k = (lane + 32 * i) / TW;
        if (lane % TW == 0 && k < C) sm.ctot[k] = t;
      }
      __syncwarp();
      ff c{0.f, 0.f};
      for (int k = 0; k < C; ++k) c = ff_add(c, sm.ctot[k]);
      r.tot = c;
    }
    if (lane == 0) {
      sm.res = r;
      sm.lastbuf = buf;
    }
  }
  __syncthreads();
}

// Softmax statistics of the target row (and the draft row when use_d).
template <typename T>
__device__ void stats_pass(Smem& sm, cg::cluster_group& cl, int C, int& buf, const Geo& g,
                           const T* tr, const T* dr, bool dfast, bool use_d, float a) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  Soft st = soft_empty(), sd = soft_empty();
  bool bad = false;
  const uint4* t4 = reinterpret_cast<const uint4*>(tr - g.off);  // vector 0 of the grid
  const uint4* d4 = reinterpret_cast<const uint4*>(dr - g.off);
  for (int tb = g.t0; tb < g.t1; tb += UNR) {
    uint4 vt[UNR], vd[UNR];
    if (interior_round<T>(g, tb, use_d && !dfast)) {  // whole vectors on both rows' grids
#pragma unroll
      for (int k = 0; k < UNR; ++k) {
        const int j = (tb + k) * 32 + lane;
        vt[k] = __ldg(t4 + j);
        if (use_d) vd[k] = __ldg(d4 + j);
      }
    } else {
#pragma unroll
      for (int k = 0; k < UNR; ++k) {
        const int j = (tb + k) * 32 + lane;
        vt[k] = tb + k < g.t1 ? fetch<T>(tr, true, g.V, g.off, j) : neg_inf_vec<T>();
        if (use_d) vd[k] = tb + k < g.t1 ? fetch<T>(dr, dfast, g.V, g.off, j) : neg_inf_vec<T>();
      }
    }
    soft_round<T, UNR>(st, vt, a, bad);
    if (use_d) soft_round<T, UNR>(sd, vd, a, bad);
  }
  st = soft_warp1(st, a);
  sd = use_d ? soft_warp1(sd, a) : soft_empty();
  const bool wb = __any_sync(FULLM, bad);
  if (lane == 0) {
    Xw& x = sm.xw[buf][w];
    x.st = st;
    x.sd = sd;
    x.bad = wb;
    sm.sst[w] = st;
  }
  exchange<0>(sm, cl, C, buf, a);
  buf ^= 1;
}

// Maximum and lowest-index argmax of the target row (greedy verification).
template <typename T>
__device__ void argmax_pass(Smem& sm, cg::cluster_group& cl, int C, int& buf, const Geo& g,
                            const T* tr) {
  constexpr int VEC = EV<T>::VEC;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  float best = -INFINITY;
  int idx = INT_MAX;
  bool bad = false;
  const uint4* t4 = reinterpret_cast<const uint4*>(tr - g.off);  // vector 0 of the grid
  const int jlo = g.off > 0 ? 1 : 0, jhi = (g.V + g.off) / VEC;   // whole vectors
  for (int tb = g.t0; tb < g.t1; tb += UNR_G) {
    uint4 vt[UNR_G];
    if (tb + UNR_G <= g.t1 && tb * 32 >= jlo && (tb + UNR_G) * 32 <= jhi) {
#pragma unroll
      for (int k = 0; k < UNR_G; ++k) vt[k] = __ldg(t4 + (tb + k) * 32 + lane);
    } else {
#pragma unroll
      for (int k = 0; k < UNR_G; ++k)
        vt[k] = tb + k < g.t1 ? fetch<T>(tr, true, g.V, g.off, (tb + k) * 32 + lane)
                              : neg_inf_vec<T>();
    }
    const float vm = vmax_n<T, UNR_G>(vt);
    bad |= (vm != vm) || (vm == INFINITY);
    if (vm > best) {  // rare: find the round's first element equal to its maximum
      best = vm;
      int e = -1;
#pragma unroll
      for (int k = 0; k < UNR_G; ++k) {
        float z[VEC];
        unpack<T>(vt[k], z);
#pragma unroll
        for (int i = 0; i < VEC; ++i)
          if (e < 0 && z[i] == vm) e = ((tb + k) * 32 + lane) * VEC - g.off + i;
      }
      idx = e;
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float b2 = __shfl_xor_sync(FULLM, best, o);
    const int i2 = __shfl_xor_sync(FULLM, idx, o);
    arg_merge(best, idx, b2, i2);
  }
  const bool wb = __any_sync(FULLM, bad);
  if (lane == 0) {
    Xw& x = sm.xw[buf][w];
    x.best = best;
    x.idx = idx;
    x.bad = wb;
  }
  exchange<1>(sm, cl, C, buf, 0.f);
  buf ^= 1;
}

// Sum of the weights over the row (cluster total in sm.res.tot, CTA totals in sm.ctot),
// keeping per-warp group totals (sm.gtot) and warp totals (sm.wtot) for the sample.
template <typename T>
__device__ void wsum_pass(Smem& sm, cg::cluster_group& cl, int C, int& buf, const Geo& g,
                          const T* tr, const T* dr, bool dfast, const WPar& P) {
  constexpr int VEC = EV<T>::VEC;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int nt = g.t1 - g.t0;
  const int gsz = group_size(nt);
  ff wt{0.f, 0.f};
  float ls = 0.f, lc = 0.f;
  const uint4* t4 = reinterpret_cast<const uint4*>(tr - g.off);  // vector 0 of the grid
  const uint4* d4 = reinterpret_cast<const uint4*>(dr - g.off);
  for (int tb = 0; tb < nt; tb += UNR) {
    uint4 vt[UNR], vd[UNR];
    if (interior_round<T>(g, g.t0 + tb, P.use_d && !dfast)) {  // whole vectors on both grids
#pragma unroll
      for (int k = 0; k < UNR; ++k) {
        const int j = (g.t0 + tb + k) * 32 + lane;
        vt[k] = __ldg(t4 + j);
        if (P.use_d) vd[k] = __ldg(d4 + j);
      }
    } else {
#pragma unroll
      for (int k = 0; k < UNR; ++k) {
        if (tb + k < nt) {
          const int j = (g.t0 + tb + k) * 32 + lane;
          vt[k] = fetch<T>(tr, true, g.V, g.off, j);
          if (P.use_d) vd[k] = fetch<T>(dr, dfast, g.V, g.off, j);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < UNR; ++k) {
      const int lt = tb + k;
      if (lt < nt) {
        float wv[VEC];
        acc2(ls, lc, vec_weights<T>(P, vt[k], P.use_d ? vd[k] : vt[k], wv));
        if ((lt + 1) % gsz == 0 || lt + 1 == nt) {  // the group ends (warp-uniform)
          const ff gt = ff_warp_sum(ff_two_sum(ls, lc));
          if (lane == 0) sm.gtot[w][lt / gsz] = gt;
          wt = ff_add(wt, gt);
          ls = 0.f;
          lc = 0.f;
        }
      }
    }
  }
  if (lane == 0) {
    sm.xw[buf][w].tot = wt;
    sm.xw[buf][w].bad = 0;
  }
  exchange<2>(sm, cl, C, buf, 0.f);
  buf ^= 1;
}

// Inverse CDF at target = u * total: CTA, then warp and group of tiles, then element
// (one warp). Weights of the last wsum_pass (from_s false: totals kept by that pass), or
// p itself (from_s: CTA and warp totals rescaled from the statistics pass's per-warp
// partials, group totals of the chosen warp's tiles summed by all warps of the CTA, so
// no pass over the whole row). Returns the element in lane 0 of the warp that found it
// and -1 elsewhere; only the owning CTA finds one.
template <typename T>
__device__ int locate(Smem& sm, cg::cluster_group& cl, int C, int rank, const Geo& g,
                      const T* tr, const T* dr, bool dfast, const WPar& P, float u,
                      bool from_s) {
  constexpr int VEC = EV<T>::VEC;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (from_s) {
    if (threadIdx.x < 32) {
      // Entry e = lane + 32 i is warp e % TW of CTA e / TW: its statistics rescaled to
      // p's frame (all loads in flight); a fixed butterfly over each TW-lane half adds a
      // CTA's warps; the cluster's total adds the CTAs in rank order.
      const int n = C * TW;
      constexpr int PER = MAXC * TW / 32;
      Soft v[PER];
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < n ? *cl.map_shared_rank(&sm.sst[e % TW], e / TW) : soft_empty();
      }
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int e = lane + 32 * i, k = e / TW;
        ff t = v[i].m > -INFINITY
                   ? ff_mul_f(ff_mul_f(v[i].S, ex2(__fsub_rn(v[i].F, P.Ft))), P.iSt)
                   : ff{0.f, 0.f};
        if (k == rank && e < n) sm.pw[e % TW] = t;
#pragma unroll
        for (int o = TW / 2; o; o >>= 1) t = ff_add(t, ff_shfl_xor(t, o));
        if (lane % TW == 0 && k < C) sm.ctot[k] = t;
      }
      __syncwarp();
      ff c{0.f, 0.f};
      for (int k = 0; k < C; ++k) c = ff_add(c, sm.ctot[k]);
      if (lane == 0) sm.res.tot = c;
    }
    __syncthreads();
  }
  const ff target = ff_mul_f(sm.res.tot, u);
  ff cum{0.f, 0.f};
  int cs = select_item(sm.ctot, C, target, cum);
  if (cs < 0) cs = 0;  // no mass at all cannot happen (the largest p weight is ~1)
  if (cs != rank) return -1;
  int ga, gb, scan_w;
  if (!from_s) {
    if (threadIdx.x == 0) {
      ff wtot[TW];
      for (int k = 0; k < TW; ++k) wtot[k] = sm.xw[sm.lastbuf][k].tot;
      int ws = select_item(wtot, TW, target, cum);
      if (ws < 0) ws = 0;
      int t0, t1;
      warp_tiles(g.ntiles, C, rank, ws, t0, t1);
      const int nt = t1 - t0;
      const int gsz = group_size(nt);
      int gs = select_item(sm.gtot[ws], (nt + gsz - 1) / gsz, target, cum);
      if (gs < 0) gs = 0;
      sm.sel_w = ws;
      sm.sel_g = gs;
      sm.sel_cum = cum;
    }
    __syncthreads();
    scan_w = sm.sel_w;
    int t0, t1;
    warp_tiles(g.ntiles, C, rank, scan_w, t0, t1);
    const int gsz = group_size(t1 - t0);
    ga = t0 + sm.sel_g * gsz;
    gb = min(t1, ga + gsz);
  } else {
    if (threadIdx.x == 0) {
      int ws = select_item(sm.pw, TW, target, cum);
      if (ws < 0) ws = 0;
      sm.sel_w = ws;
      sm.sel_cum = cum;
    }
    __syncthreads();
    int t0, t1;
    warp_tiles(g.ntiles, C, rank, sm.sel_w, t0, t1);
    const int nt = t1 - t0;
    const int gsz = max(1, (nt + NGRP - 1) / NGRP);
    const int ngrp = (nt + gsz - 1) / gsz;
    for (int grp = w; grp < ngrp; grp += TW) {  // group totals of p, dealt over the warps
      float ls = 0.f, lc = 0.f;
      const int te = min(t1, t0 + (grp + 1) * gsz);
      for (int t = t0 + grp * gsz; t < te; ++t) {
        const uint4 vt = fetch<T>(tr, true, g.V, g.off, t * 32 + lane);
        float wv[VEC];
        acc2(ls, lc, vec_weights<T>(P, vt, vt, wv));
      }
      const ff gt = ff_warp_sum(ff_two_sum(ls, lc));
      if (lane == 0) sm.gtot[0][grp] = gt;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      cum = sm.sel_cum;
      int gs = select_item(sm.gtot[0], ngrp, target, cum);
      if (gs < 0) gs = 0;
      sm.sel_g = gs;
      sm.sel_cum = cum;
    }
    __syncthreads();
    scan_w = 0;
    ga = t0 + sm.sel_g * gsz;
    gb = min(t1, ga + gsz);
  }
  if (w != scan_w) return -1;
  cum = sm.sel_cum;
  int found = -1, last_pos = -1;
  for (int t = ga; t < gb; ++t) {
    const int j = t * 32 + lane;
    const uint4 vt = fetch<T>(tr, true, g.V, g.off, j);
    const uint4 vd = P.use_d ? fetch<T>(dr, dfast, g.V, g.off, j) : vt;
    float wv[VEC];
    const float s = vec_weights<T>(P, vt, vd, wv);
    const ff incl = ff_warp_incl_scan(ff{s, 0.f}, lane);
    const ff excl{__shfl_up_sync(FULLM, incl.hi, 1), __shfl_up_sync(FULLM, incl.lo, 1)};
    const unsigned hit = __ballot_sync(FULLM, ff_lt(target, ff_add(cum, incl)) && s > 0.f);
    int lp = -1;  // this lane's last element of positive weight
#pragma unroll
    for (int i = 0; i < VEC; ++i)
      if (wv[i] > 0.f) lp = j * VEC - g.off + i;
    if (hit) {
      const int L = __ffs(hit) - 1;
      int e = -1;
      if (lane == L) {
        ff c = lane ? ff_add(cum, excl) : cum;
        for (int i = 0; i < VEC && e < 0; ++i) {
          if (wv[i] > 0.f) {
            const ff s2 = ff_two_sum(c.hi, wv[i]);
            c = ff_norm(s2.hi, __fadd_rn(s2.lo, c.lo));
            if (ff_lt(target, c)) e = j * VEC - g.off + i;
          }
        }
        if (e < 0) e = lp;  // rounding: the lane's last positive element
      }
      found = __shfl_sync(FULLM, e, L);
      break;
    }
    // the last positive element so far (elements grow with lane, then tile)
#pragma unroll
    for (int o = 16; o; o >>= 1) lp = max(lp, __shfl_xor_sync(FULLM, lp, o));
    if (lp >= 0) last_pos = lp;
    cum = ff_add(cum, ff{__shfl_sync(FULLM, incl.hi, 31), __shfl_sync(FULLM, incl.lo, 31)});
  }
  if (found < 0) found = last_pos;
  if (found < 0) found = max(0, ga * 32 * VEC - g.off);  // a group whose weights all rounded to 0
  return lane == 0 ? found : -1;
}

// ---------------------------------------------------------------------------
// The kernel: one cluster per request.
// ---------------------------------------------------------------------------
template <typename T, bool GREEDY>
__global__ void __launch_bounds__(TT, 1) tree_kernel(const TreeArgs A) {
  __shared__ Smem sm;
  cg::cluster_group cl = cg::this_cluster();
  const int C = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int b = blockIdx.x / C;
  const int tid = threadIdx.x, w = tid >> 5;
  const int N = A.N, V = A.V;
  const size_t base = (size_t)b * N;
  const T* tgt = static_cast<const T*>(A.tgt);
  const T* drf = static_cast<const T*>(A.drf);

  if (tid < N) {
    sm.par[tid] = A.par[base + tid];
    sm.tok[tid] = A.tok[base + tid];
    sm.u[tid] = GREEDY ? 0.f : A.uni[base + tid];
  }
  if (tid == 0) sm.nn = A.nn[b];
  __syncthreads();
  if (tid == 0) {
    const int nn = sm.nn;
    bool ok = nn >= 1 && nn <= N;
    for (int n = 1; ok && n < nn; ++n)
      ok = sm.par[n] >= 0 && sm.par[n] < n && sm.tok[n] >= 0 && sm.tok[n] < V;
    if (!GREEDY)
      for (int n = 0; ok && n < nn; ++n) ok = sm.u[n] >= 0.f && sm.u[n] < 1.f;
    sm.ok = ok;
  }
  __syncthreads();
  const int nn = sm.nn;
  bool valid = sm.ok != 0;
  int depth = 0, c = 0, buf = 0;
  int32_t* otok = A.out_tok + base;
  int32_t* opath = A.out_path ? A.out_path + base : nullptr;
  const bool writer = rank == 0 && tid == 0;

  while (valid) {
    const T* tr = tgt + (base + c) * (size_t)V;
    const Geo g = make_geo(tr, V, C, rank, w);
    int first_child = -1;
    for (int n = c + 1; n < nn; ++n)
      if (sm.par[n] == c) {
        first_child = n;
        break;
      }

    if (GREEDY) {
      argmax_pass<T>(sm, cl, C, buf, g, tr);
      if (sm.res.bad || !(sm.res.best > -INFINITY)) {
        valid = false;
        break;
      }
      const int am = sm.res.idx;
      int next = -1;
      for (int n = c + 1; n < nn && next < 0; ++n)
        if (sm.par[n] == c && sm.tok[n] == am) next = n;
      if (next < 0) {
        if (writer) otok[depth] = am;
        break;
      }
      if (writer) {
        otok[depth] = sm.tok[next];
        if (opath) opath[depth] = next;
      }
      ++depth;
      c = next;
      continue;
    }

    const bool kids = first_child >= 0;
    const T* dr = drf + (base + c) * (size_t)V;
    const bool dfast = kids && row_off(dr) == g.off;
    // Thread n fetches the logits of child n's token; they land during the pass.
    float czt = 0.f, czd = 0.f;
    const bool is_child = tid > c && tid < nn && sm.par[tid] == c;
    if (is_child) {
      czt = logit_at(tr + sm.tok[tid]);
      czd = logit_at(dr + sm.tok[tid]);
    }
    stats_pass<T>(sm, cl, C, buf, g, tr, dr, dfast, kids, A.a);
    if (sm.res.bad || !(sm.res.st.m > -INFINITY) || (kids && !(sm.res.sd.m > -INFINITY))) {
      valid = false;
      break;
    }
    // Frames and inverse sums (1/(hi + lo) to float precision).
    const Soft st = sm.res.st, sd = sm.res.sd;
    const float iSt = fmaf(-__fdiv_rn(1.f, st.S.hi), __fdiv_rn(st.S.lo, st.S.hi),
                           __fdiv_rn(1.f, st.S.hi));
    const float iSd = kids ? fmaf(-__fdiv_rn(1.f, sd.S.hi), __fdiv_rn(sd.S.lo, sd.S.hi),
                                  __fdiv_rn(1.f, sd.S.hi))
                           : 0.f;
    if (is_child) {
      sm.czt[tid] = czt;
      sm.czd[tid] = czd;
    }
    __syncthreads();
    WPar P{A.a, st.F, iSt, sd.F, 0.f, false};
    bool totals = false;  // sm.gtot/wtot/ctot hold the weights of P
    int next = -1;
    if (kids) {
      ff lam{0.f, 0.f}, W{1.f, 0.f};
      for (int n = first_child; n < nn; ++n) {
        if (sm.par[n] != c) continue;
        if (tid == 0) {
          const float px = __fmul_rn(term_precise(sm.czt[n], A.a, A.a_lo, st.F), iSt);
          const float qx = __fmul_rn(term_precise(sm.czd[n], A.a, A.a_lo, sd.F), iSd);
          // u * q(x) < r(x) with r = max(0, p - lam q) / W, division-free.
          sm.dec = __fmul_rn(__fmul_rn(sm.u[n], qx), W.hi) < fmaxf(fmaf(-lam.hi, qx, px), 0.f);
        }
        __syncthreads();
        if (sm.dec) {
          next = n;
          break;
        }
        lam = ff_add(lam, W);
        P = WPar{A.a, st.F, iSt, sd.F, __fmul_rn(lam.hi, iSd), true};
        wsum_pass<T>(sm, cl, C, buf, g, tr, dr, dfast, P);
        if (sm.res.tot.hi > 0.f) {
          W = sm.res.tot;
          totals = true;
        } else {  // no residual mass left: start again from p
          lam = ff{0.f, 0.f};
          W = ff{1.f, 0.f};
          totals = false;
        }
      }
    }
    if (next >= 0) {
      if (writer) {
        otok[depth] = sm.tok[next];
        if (opath) opath[depth] = next;
      }
      ++depth;
      c = next;
      continue;
    }
    // Terminal sample: the residual after the last rejection (its totals kept by that
    // pass), or p (leaf, or restart) from the statistics pass's partials.
    if (!totals) P = WPar{A.a, st.F, iSt, sd.F, 0.f, false};
    const int y = locate<T>(sm, cl, C, rank, g, tr, dr, dfast, P, sm.u[0], !totals);
    if (y >= 0) otok[depth] = y;
    break;
  }

  if (writer) {
    if (!valid) {
      for (int i = 0; i < N; ++i) {
        otok[i] = -1;
        if (opath) opath[i] = -1;
      }
      A.out_acc[b] = -1;
      atomicOr(&A.hdr->status, ST_DEVICE_INPUT);
    } else {
      for (int i = depth + 1; i < N; ++i) otok[i] = -1;
      if (opath)
        for (int i = depth; i < N; ++i) opath[i] = -1;
      A.out_acc[b] = depth;
    }
  }
  // No CTA leaves while another may still read its shared memory.
  cl.sync();
}

template <typename T, bool G>
cudaError_t launch_variant(const TreeArgs& A, cudaStream_t st, int* cluster_out) {
  // Largest cluster (8, 4, 2) for which every request's cluster is resident at once.
  static std::atomic<int> max_clusters[MAXC + 1];
  int C = 1;
  for (int cand = MAXC; cand >= 2; cand >>= 1) {
    int n = max_clusters[cand].load(std::memory_order_relaxed);
    if (n == 0) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = cand;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(cand);
      cfg.blockDim = dim3(TT);
      cfg.attrs = at;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, tree_kernel<T, G>, &cfg) != cudaSuccess || n < 1)
        n = -1;
      (void)cudaGetLastError();
      max_clusters[cand].store(n, std::memory_order_relaxed);
    }
    if (n >= A.B) {
      C = cand;
      break;
    }
  }
  if (cluster_out) *cluster_out = C;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(A.B * C);
  cfg.blockDim = dim3(TT);
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tree_kernel<T, G>, A);
}

}  // namespace

cudaError_t launch_tree(const TreeArgs& A, bool bf16, bool greedy, cudaStream_t st,
                        int* cluster_out) {
  if (bf16)
    return greedy ? launch_variant<uint16_t, true>(A, st, cluster_out)
                  : launch_variant<uint16_t, false>(A, st, cluster_out);
  return greedy ? launch_variant<float, true>(A, st, cluster_out)
                : launch_variant<float, false>(A, st, cluster_out);
}

}  // namespace sv
