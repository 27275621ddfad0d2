// sv_cluster.cuh -- device helpers of the cluster-per-request tree verification kernel:
// rows read as 16-byte vectors on a grid anchored at a row's own alignment, float-float
// sums, online softmax statistics, sample weights and the inverse-CDF selection over
// partial totals.
#pragma once
#include <cfloat>
#include <climits>

#include "sv_common.cuh"

namespace sv {
namespace clx {

constexpr unsigned FULLM = 0xffffffffu;

template <typename T>
struct EV;
template <>
struct EV<uint16_t> {
  static constexpr int VEC = 8;
};
template <>
struct EV<float> {
  static constexpr int VEC = 4;
};

__device__ __forceinline__ float logit_at(const float* p) { return __ldg(p); }
__device__ __forceinline__ float logit_at(const uint16_t* p) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(p)) << 16);
}

template <typename T>
__device__ __forceinline__ void unpack(const uint4 v, float* z) {
  if constexpr (EV<T>::VEC == 8) {
    z[0] = bf_lo(v.x); z[1] = bf_hi(v.x); z[2] = bf_lo(v.y); z[3] = bf_hi(v.y);
    z[4] = bf_lo(v.z); z[5] = bf_hi(v.z); z[6] = bf_lo(v.w); z[7] = bf_hi(v.w);
  } else {
    z[0] = __uint_as_float(v.x); z[1] = __uint_as_float(v.y);
    z[2] = __uint_as_float(v.z); z[3] = __uint_as_float(v.w);
  }
}

// Vector j of a row on the grid anchored at element offset `off`: elements
// [j*VEC - off, j*VEC - off + VEC), -inf outside [0, V). `fast`: this row's own
// 16-byte boundaries fall on the grid, so whole in-range vectors are one 16-byte load.
template <typename T>
__device__ __forceinline__ uint4 fetch(const T* p, bool fast, int V, int off, int j) {
  constexpr int VEC = EV<T>::VEC;
  const int e0 = j * VEC - off;
  if (fast && e0 >= 0 && e0 + VEC <= V) return __ldg(reinterpret_cast<const uint4*>(p + e0));
  uint32_t w[4];
  if constexpr (VEC == 8) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = e0 + 2 * i;
      const uint32_t lo = (e >= 0 && e < V) ? static_cast<uint32_t>(__ldg(p + e)) : 0xff80u;
      const uint32_t hi = (e + 1 >= 0 && e + 1 < V) ? static_cast<uint32_t>(__ldg(p + e + 1))
                                                    : 0xff80u;
      w[i] = lo | (hi << 16);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = e0 + i;
      w[i] = (e >= 0 && e < V) ? __float_as_uint(__ldg(p + e)) : 0xff800000u;
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T>
__device__ __forceinline__ int row_off(const T* p) {
  return static_cast<int>((reinterpret_cast<uintptr_t>(p) & 15u) / sizeof(T));
}

// ---------------------------------------------------------------------------
// Float-float values (hi + lo, about 48 significant bits) for sums and prefixes.
// ---------------------------------------------------------------------------
struct ff {
  float hi, lo;
};

__device__ __forceinline__ ff ff_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  return ff{s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp))};
}
__device__ __forceinline__ ff ff_norm(float s, float e) {
  const float h = __fadd_rn(s, e);
  return ff{h, __fsub_rn(e, __fsub_rn(h, s))};
}
// Commutative bit for bit (the TwoSum error is exact whatever the order).
__device__ __forceinline__ ff ff_add(ff a, ff b) {
  const ff s = ff_two_sum(a.hi, b.hi);
  return ff_norm(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ ff ff_mul_f(ff a, float u) {
  const float p = __fmul_rn(a.hi, u);
  return ff_norm(p, fmaf(a.lo, u, fmaf(a.hi, u, -p)));
}
__device__ __forceinline__ bool ff_lt(ff a, ff b) {
  return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}
__device__ __forceinline__ ff ff_shfl_xor(ff x, int o) {
  return ff{__shfl_xor_sync(FULLM, x.hi, o), __shfl_xor_sync(FULLM, x.lo, o)};
}
__device__ __forceinline__ ff ff_warp_sum(ff x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = ff_add(x, ff_shfl_xor(x, o));
  return x;
}
__device__ __forceinline__ ff ff_warp_incl_scan(ff x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff y{__shfl_up_sync(FULLM, x.hi, o), __shfl_up_sync(FULLM, x.lo, o)};
    if (lane >= o) x = ff_add(y, x);
  }
  return x;
}
// Compensated accumulation of a float into (s, c).
__device__ __forceinline__ void acc2(float& s, float& c, float w) {
  const float t = __fadd_rn(s, w);
  const float bp = __fsub_rn(t, s);
  c = __fadd_rn(c, __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(w, bp)));
  s = t;
}

// ---------------------------------------------------------------------------
// Softmax statistics: m = running max of the raw logits, F = fl(m*a) the frame,
// S = sum of 2^(z*a - F) (float-float; a = log2(e)/T rounded to fp32).
// ---------------------------------------------------------------------------
struct Soft {
  float m, F;
  ff S;
};

__device__ __forceinline__ Soft soft_empty() { return Soft{-INFINITY, 0.f, ff{0.f, 0.f}}; }

// 2^(z*(a + a_lo) - F) with the exponent carried in two floats (exact product error by
// fma, TwoSum error of the subtraction), for the probabilities the accept tests use.
__device__ __forceinline__ float term_precise(float z, float a, float alo, float F) {
  if (!(z > -INFINITY)) return 0.f;
  const float ph = __fmul_rn(z, a);
  const float pl = fmaf(z, a, -ph);
  const float yh = __fsub_rn(ph, F);
  const float bp = __fsub_rn(yh, ph);
  const float el = __fadd_rn(__fsub_rn(ph, __fsub_rn(yh, bp)), __fsub_rn(-F, bp));
  const float yl = fmaf(z, alo, __fadd_rn(pl, el));
  const float e = ex2(yh);
  return fmaf(e, __fmul_rn(yl, 0.6931471805599453f), e);
}

// Packed fp32x2 fused multiply-add (one instruction for two lanes of values).
__device__ __forceinline__ float2 fma2(float2 x, float2 y, float2 z) {
  float2 d;
  asm("{\n\t.reg .b64 rx, ry, rz, rd;\n\t"
      "mov.b64 rx, {%2, %3};\n\tmov.b64 ry, {%4, %5};\n\tmov.b64 rz, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, rx, ry, rz;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(x.x), "f"(x.y), "f"(y.x), "f"(y.y), "f"(z.x), "f"(z.y));
  return d;
}

__device__ __forceinline__ float2 add2(float2 x, float2 y) {
  float2 d;
  asm("{\n\t.reg .b64 rx, ry, rd;\n\t"
      "mov.b64 rx, {%2, %3};\n\tmov.b64 ry, {%4, %5};\n\t"
      "add.rn.f32x2 rd, rx, ry;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(x.x), "f"(x.y), "f"(y.x), "f"(y.y));
  return d;
}

// The VEC logits of a raw vector as VEC/2 pairs.
template <typename T>
__device__ __forceinline__ float2 pair_of(const uint4 v, int i) {
  const uint32_t w = i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
  if constexpr (EV<T>::VEC == 8) {
    return make_float2(bf_lo(w), bf_hi(w));
  } else {
    const uint32_t w2 = i == 0 ? v.y : v.w;
    return make_float2(__uint_as_float(i == 0 ? v.x : v.z), __uint_as_float(w2));
  }
}

template <typename T>
__device__ __forceinline__ uint4 neg_inf_vec() {
  if constexpr (EV<T>::VEC == 8) return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
  return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
}

// Maximum of a vector; NaN if any element is NaN.
template <typename T>
__device__ __forceinline__ float vmax(const uint4 v) {
  if constexpr (EV<T>::VEC == 8) {
    const uint32_t m = bmax2_nan(bmax2_nan(v.x, v.y), bmax2_nan(v.z, v.w));
    return fmax_nan(bf_lo(m), bf_hi(m));
  } else {
    return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                    fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
}

// Maximum of n vectors; NaN if any element is NaN. bf16 vectors are combined as packed
// pairs and unpacked once.
template <typename T, int n>
__device__ __forceinline__ float vmax_n(const uint4* v) {
  if constexpr (EV<T>::VEC == 8) {
    uint32_t m = bmax2_nan(bmax2_nan(v[0].x, v[0].y), bmax2_nan(v[0].z, v[0].w));
#pragma unroll
    for (int k = 1; k < n; ++k)
      m = bmax2_nan(m, bmax2_nan(bmax2_nan(v[k].x, v[k].y), bmax2_nan(v[k].z, v[k].w)));
    return fmax_nan(bf_lo(m), bf_hi(m));
  } else {
    float m = vmax<T>(v[0]);
#pragma unroll
    for (int k = 1; k < n; ++k) m = fmax_nan(m, vmax<T>(v[k]));
    return m;
  }
}

// Sum of 2^(z*a - F) over a vector (nF = -F): each element's unnormalised weight in
// frame F (0 for -inf). The rounding of a = log2(e)/T moves every exponent by
// (z - M)*a_lo plus a constant that the normalisation cancels: below 1e-6 relative for
// the terms that carry the mass.
template <typename T>
__device__ __forceinline__ float vexpsum(const uint4 v, float a, float nF) {
  constexpr int NP = EV<T>::VEC / 2;
  const float2 aa = make_float2(a, a), cc = make_float2(nF, nF);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const float2 y = fma2(pair_of<T>(v, i), aa, cc);
    acc = add2(acc, make_float2(ex2(y.x), ex2(y.y)));
  }
  return acc.x + acc.y;
}

// One round of UNR vectors into a softmax state: one max, at most one rescale, then
// the exponentials. `bad` collects NaN and +inf.
template <typename T, int UNR>
__device__ __forceinline__ void soft_round(Soft& s, const uint4* v, float a, bool& bad) {
  const float vm = vmax_n<T, UNR>(v);
  bad |= (vm != vm) || (vm == INFINITY);
  if (vm > s.m) {
    const float Fn = __fmul_rn(vm, a);
    const float f = (s.m == -INFINITY) ? 0.f : ex2(__fsub_rn(s.F, Fn));
    s.S = ff_mul_f(s.S, f);
    s.m = vm;
    s.F = Fn;
  }
  if (s.m == -INFINITY) return;
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < UNR; ++k) sum += vexpsum<T>(v[k], a, -s.F);
  const ff r = ff_two_sum(s.S.hi, sum);
  s.S = ff_norm(r.hi, __fadd_rn(r.lo, s.S.lo));
}

// Warp merge in one frame: the warp's maximum first, then each lane's sum rescaled once
// into it and the sums added by a butterfly (every lane ends with the same bits). Lanes
// whose statistics hold nothing (m = -inf) add nothing.
__device__ __forceinline__ Soft soft_warp1(const Soft& s, float a) {
  float m = s.m;
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULLM, m, o));
  if (!(m > -INFINITY)) return soft_empty();
  const float F = __fmul_rn(m, a);
  const ff S = s.m > -INFINITY ? ff_mul_f(s.S, ex2(__fsub_rn(s.F, F))) : ff{0.f, 0.f};
  return Soft{m, F, ff_warp_sum(S)};
}

// The same over PER statistics per lane (added in index order, then the butterfly).
template <int PER>
__device__ __forceinline__ Soft soft_frame_merge(const Soft* s, float a) {
  float m = s[0].m;
#pragma unroll
  for (int i = 1; i < PER; ++i) m = fmaxf(m, s[i].m);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULLM, m, o));
  if (!(m > -INFINITY)) return soft_empty();
  const float F = __fmul_rn(m, a);
  ff S{0.f, 0.f};
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (s[i].m > -INFINITY) S = ff_add(S, ff_mul_f(s[i].S, ex2(__fsub_rn(s[i].F, F))));
  return Soft{m, F, ff_warp_sum(S)};
}

// Argmax with ties to the lowest index.
__device__ __forceinline__ void arg_merge(float& best, int& idx, float b2, int i2) {
  if (b2 > best || (b2 == best && i2 < idx)) {
    best = b2;
    idx = i2;
  }
}

// ---------------------------------------------------------------------------
// Residual and sample weights: w = max(0, p - lam*q), or p when use_d is false.
// p = 2^(zt*a - Ft) * iSt, q likewise; lq = lam * iSd.
// ---------------------------------------------------------------------------
struct WPar {
  float a, Ft, iSt, Fd, lq;
  bool use_d;
};

// Weights of the VEC elements of one vector of t (and d); returns their sum.
template <typename T>
__device__ __forceinline__ float vec_weights(const WPar& P, uint4 vt, uint4 vd, float* w) {
  constexpr int NP = EV<T>::VEC / 2;
  const float2 aa = make_float2(P.a, P.a), ct = make_float2(-P.Ft, -P.Ft);
  const float2 st = make_float2(P.iSt, P.iSt), z0 = make_float2(0.f, 0.f);
  const float2 cd = make_float2(-P.Fd, -P.Fd), nl = make_float2(-P.lq, -P.lq);
  float2 sum = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const float2 yt = fma2(pair_of<T>(vt, i), aa, ct);
    float2 pt = fma2(make_float2(ex2(yt.x), ex2(yt.y)), st, z0);
    if (P.use_d) {
      const float2 yd = fma2(pair_of<T>(vd, i), aa, cd);
      pt = fma2(nl, make_float2(ex2(yd.x), ex2(yd.y)), pt);
      pt.x = fmaxf(pt.x, 0.f);
      pt.y = fmaxf(pt.y, 0.f);
    }
    w[2 * i] = pt.x;
    w[2 * i + 1] = pt.y;
    sum = add2(sum, pt);
  }
  return sum.x + sum.y;
}

// First item whose running total passes `target` (items of zero total never qualify);
// `cum` enters as the total before item 0 and leaves as the total before the chosen one.
// If rounding lets no item pass, the last item with a positive total; -1 if none.
__device__ inline int select_item(const ff* tot, int n, ff target, ff& cum) {
  ff c = cum, c_last = cum;
  int last = -1;
  for (int i = 0; i < n; ++i) {
    const ff nx = ff_add(c, tot[i]);
    if (tot[i].hi > 0.f) {
      last = i;
      c_last = c;
      if (ff_lt(target, nx)) {
        cum = c;
        return i;
      }
    }
    c = nx;
  }
  cum = c_last;
  return last;
}

}  // namespace clx
}  // namespace sv
