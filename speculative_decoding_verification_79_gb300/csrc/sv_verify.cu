// sv_verify.cu -- fused batched verification of drafted token blocks (sm_103a).
//
// Method: standard speculative rejection sampling, as the DSpark pages describe it
// (DSpark Deep Dive, "The Speculative Decoding Solution"; DSpark Guide, "1. The
// Mathematics of Suffix Decay"; perchy.ai Technology, "Verified by the target").
//
// One launch on the caller's stream, no CPU round trip: sv_verify_kernel, one
// persistent CTA per SM, in two phases.
//  1. Stream phase. Work list: every active logit row
//     of the batch (request b: target rows 0..L_b, and at T > 0 draft rows
//     0..L_b-1) cut into pieces of SLOT_BYTES, ordered request-major; every warp of
//     the grid takes an equal contiguous range of it. Each warp owns SLOTS_PER_WARP
//     shared-memory slots and is its own producer: lane 0 issues a 1-D bulk copy
//     (cp.async.bulk, TMA) of the next piece into the slot the warp has just
//     finished, guarded by an mbarrier, while the warp reduces the other slots.
//     Pieces are reduced whole: online softmax (running max + sum of
//     2^(z*log2e/T - max)) at T > 0, or (max, lowest argmax) at T == 0, and merged in
//     registers while consecutive pieces belong to the same row. Each row segment is
//     published with a release-ordered atomic ticket whose value the warp inspects
//     only after its next wait, so the round trip stays off the critical path. The
//     warp completing a row combines it; the warp completing a request decides it:
//     p_k(x_k), q_k(x_k),
//     the accept tests u*q < p, a ballot for the first rejection j, the outputs,
//     and (T > 0) the terminal-sample job of the request.
//  2. Terminal phase (T > 0 only), after a grid-wide barrier (the launch is
//     cooperative, so all CTAs are resident): the (request, piece) tasks of the
//     terminal rows (residual max(0, p_j - q_j), or p of the bonus row) are split
//     over all warps and copied through the same slots; each sums its piece's weights
//     with compensated fp32 arithmetic, reduced as float-float pairs; the last piece
//     of a request locates the token by inverse CDF at u_{b,K} (float-float prefix
//     over piece sums, one piece re-scanned).
//  Every wait is bounded in time; on expiry the kernel sets SV_ERR_TIMEOUT in the
//  status word, lets its copies in flight land, and returns.
#include <cfloat>
#include <climits>

#include "sv_common.cuh"

namespace sv {

enum : int { K_STREAM = 0, K_TERM = 1 };

// A contiguous run of elements of one row, split by 16-byte alignment into a head
// read directly from global memory, a body copied to shared memory, and a tail
// read directly.
struct Seg {
  const unsigned char* g;  // address of the run's first element
  int head, body, n;
};

struct __align__(16) SlotMeta {
  int kind, b, r, p;  // request, row slot (stream) or terminal row (terminal), piece
  int e0;             // first element of the piece within its row
  int direct;         // terminal piece: 1 = rows read straight from global memory
  int jkind;          // terminal piece: J_RESID or J_BONUS
  int pad;
  Seg s0, s1;         // stream piece: s0; terminal piece: target (s0) and draft (s1)
  float Mt, iSt, Md, iSd;
};

struct Shared {
  SlotMeta meta[NSLOT];
  uint64_t full[NSLOT];
  int abort_flag;
  int grid_ok;
  int last_cta;
  int total_rows;
  int scan[32];
};

template <typename T>
struct ET;
template <>
struct ET<float> {
  static constexpr int VEC = 4;
};
template <>
struct ET<uint16_t> {
  static constexpr int VEC = 8;
};

__device__ __forceinline__ float ld_logit(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ld_logit(const uint16_t* p) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(p)) << 16);
}

constexpr unsigned FULL = 0xffffffffu;

// ---------------------------------------------------------------------------
// Online softmax pieces. State (m, s): m = running max of the raw logits, s = sum of
// 2^(z*a - fl(m*a)). Merging uses the same rounded fl(m*a) on both sides.
// ---------------------------------------------------------------------------
// The frame of a partial sum is the ROUNDED product fl(m*a); every product below is
// rounded explicitly (__fmul_rn) so the compiler cannot fuse it into an FMA with the
// following subtraction, which would rescale a sum already in the right frame by
// 2^(m*a - fl(m*a)) once per merge level.
__device__ __forceinline__ void soft_merge(float& m, float& s, float m2, float s2, float a) {
  const float mn = fmax_nan(m, m2);
  if (mn == -INFINITY) return;  // both empty
  const float man = __fmul_rn(mn, a);
  const float f1 = (m == -INFINITY) ? 0.f : ex2(__fmul_rn(m, a) - man);
  const float f2 = (m2 == -INFINITY) ? 0.f : ex2(__fmul_rn(m2, a) - man);
  s = fmaf(s, f1, s2 * f2);
  m = mn;
}

__device__ __forceinline__ void soft_rescale(float& m, float& ma, float& s, float lm, float a) {
  if (lm > m || lm != lm) {
    const float mn = fmax_nan(m, lm);
    const float man = __fmul_rn(mn, a);
    s = s * ex2(ma - man);
    m = mn;
    ma = man;
  }
}

__device__ __forceinline__ void soft_add1(float& m, float& ma, float& s, float z, float a) {
  soft_rescale(m, ma, s, z, a);
  if (m != -INFINITY) s += ex2(fmaf(z, a, -ma));
}

__device__ __forceinline__ void soft_add_vec(float& m, float& ma, float& s, uint4 v, float a,
                                             uint16_t) {
  const uint32_t mx = bmax2_nan(bmax2_nan(v.x, v.y), bmax2_nan(v.z, v.w));
  soft_rescale(m, ma, s, fmax_nan(bf_lo(mx), bf_hi(mx)), a);
  if (m == -INFINITY) return;
  const float nma = -ma;
  const float e0 = ex2(fmaf(bf_lo(v.x), a, nma)), e1 = ex2(fmaf(bf_hi(v.x), a, nma));
  const float e2 = ex2(fmaf(bf_lo(v.y), a, nma)), e3 = ex2(fmaf(bf_hi(v.y), a, nma));
  const float e4 = ex2(fmaf(bf_lo(v.z), a, nma)), e5 = ex2(fmaf(bf_hi(v.z), a, nma));
  const float e6 = ex2(fmaf(bf_lo(v.w), a, nma)), e7 = ex2(fmaf(bf_hi(v.w), a, nma));
  s += ((e0 + e1) + (e2 + e3)) + ((e4 + e5) + (e6 + e7));
}

__device__ __forceinline__ void soft_add_vec(float& m, float& ma, float& s, uint4 v, float a,
                                             float) {
  const float x0 = __uint_as_float(v.x), x1 = __uint_as_float(v.y);
  const float x2 = __uint_as_float(v.z), x3 = __uint_as_float(v.w);
  soft_rescale(m, ma, s, fmax_nan(fmax_nan(x0, x1), fmax_nan(x2, x3)), a);
  if (m == -INFINITY) return;
  const float nma = -ma;
  const float e0 = ex2(fmaf(x0, a, nma)), e1 = ex2(fmaf(x1, a, nma));
  const float e2 = ex2(fmaf(x2, a, nma)), e3 = ex2(fmaf(x3, a, nma));
  s += (e0 + e1) + (e2 + e3);
}

// Warp merge in a fixed tree; every lane ends with the same (m, s).
__device__ __forceinline__ void soft_warp(float& m, float& s, float a, int lane) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float m2 = __shfl_xor_sync(FULL, m, o), s2 = __shfl_xor_sync(FULL, s, o);
    float lm = m, ls = s, hm = m2, hs = s2;
    if (lane & o) {
      lm = m2;
      ls = s2;
      hm = m;
      hs = s;
    }
    soft_merge(lm, ls, hm, hs, a);
    m = lm;
    s = ls;
  }
}

// 2^(z*(a + a_lo) - MA) with the exponent carried to about twice fp32 precision:
// y = z*a - MA split as y_hi + y_lo (exact product error by fma, TwoSum error of
// the difference), then 2^y = 2^y_hi * (1 + y_lo*ln2). Explicit roundings keep the
// compiler from fusing the pieces.
__device__ __forceinline__ float exp2_precise(float z, float a, float a_lo, float MA) {
  const float ph = __fmul_rn(z, a);
  const float pl = fmaf(z, a, -ph);  // exact error of the product
  const float yh = __fsub_rn(ph, MA);
  const float bp = __fsub_rn(yh, ph);  // TwoSum error of ph - MA
  const float el = __fadd_rn(__fsub_rn(ph, __fsub_rn(yh, bp)), __fsub_rn(-MA, bp));
  const float yl = fmaf(z, a_lo, pl + el);
  const float e = ex2(yh);
  return fmaf(e, yl * 0.6931471805599453f, e);
}

// 2^((z - M)*(a + a_lo)) for a row maximum M: z - M is exact for bf16 logits (and
// nearly so for fp32), the product is split as above; -inf logits give 0.
__device__ __forceinline__ float exp2_diff(float z, float M, float a, float a_lo) {
  const float d = __fsub_rn(z, M);
  const float yh = __fmul_rn(d, a);
  const float yl = fmaf(d, a_lo, fmaf(d, a, -yh));
  const float e = ex2(yh);
  return (d == -INFINITY) ? 0.f : fmaf(e, yl * 0.6931471805599453f, e);
}

// ---------------------------------------------------------------------------
// Greedy pieces: (best, idx) with ties to the lowest index, plus a NaN flag.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void arg_add1(float& best, int& idx, bool& bad, float z, int i) {
  if (z > best) {
    best = z;
    idx = i;
  } else if (z != z) {
    bad = true;
  }
}

__device__ __forceinline__ void arg_add_vec(float& best, int& idx, bool& bad, uint4 v, int base,
                                            uint16_t) {
  const uint32_t mx = bmax2_nan(bmax2_nan(v.x, v.y), bmax2_nan(v.z, v.w));
  const float lm = fmax_nan(bf_lo(mx), bf_hi(mx));
  if (lm > best || lm != lm) {
    if (lm != lm) {
      bad = true;
      return;
    }
    int e = 7;
    if (bf_lo(v.w) == lm) e = 6;
    if (bf_hi(v.z) == lm) e = 5;
    if (bf_lo(v.z) == lm) e = 4;
    if (bf_hi(v.y) == lm) e = 3;
    if (bf_lo(v.y) == lm) e = 2;
    if (bf_hi(v.x) == lm) e = 1;
    if (bf_lo(v.x) == lm) e = 0;
    best = lm;
    idx = base + e;
  }
}

__device__ __forceinline__ void arg_add_vec(float& best, int& idx, bool& bad, uint4 v, int base,
                                            float) {
  const float x0 = __uint_as_float(v.x), x1 = __uint_as_float(v.y);
  const float x2 = __uint_as_float(v.z), x3 = __uint_as_float(v.w);
  const float lm = fmax_nan(fmax_nan(x0, x1), fmax_nan(x2, x3));
  if (lm > best || lm != lm) {
    if (lm != lm) {
      bad = true;
      return;
    }
    int e = 3;
    if (x2 == lm) e = 2;
    if (x1 == lm) e = 1;
    if (x0 == lm) e = 0;
    best = lm;
    idx = base + e;
  }
}

__device__ __forceinline__ void arg_warp(float& best, int& idx, bool& bad) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float b2 = __shfl_xor_sync(FULL, best, o);
    const int i2 = __shfl_xor_sync(FULL, idx, o);
    if (b2 > best || (b2 == best && i2 < idx)) {
      best = b2;
      idx = i2;
    }
  }
  bad = __any_sync(FULL, bad);
}

// Compensated (TwoSum) accumulation in fp32: s + c carries the running sum with
// about twice the precision of fp32.
__device__ __forceinline__ void two_sum(float& s, float& c, float w) {
  const float t = s + w;
  const float bp = t - s;
  c += (s - (t - bp)) + (w - bp);
  s = t;
}

// ---------------------------------------------------------------------------
// Float-float ("double-fp32") values: hi + lo with |lo| <= ulp(hi)/2, about 48
// significant bits. The terminal-sample sums and prefixes use them instead of fp64,
// whose throughput on this GPU is a small fraction of fp32's.
// ---------------------------------------------------------------------------
struct ff {
  float hi, lo;
};

// Exact sum of two floats as a normalised pair (Knuth's TwoSum).
__device__ __forceinline__ ff two_sum_ff(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
  return ff{s, e};
}

// Normalise s + e when |s| >= |e| (Dekker's FastTwoSum).
__device__ __forceinline__ ff fast_two_sum_ff(float s, float e) {
  const float h = __fadd_rn(s, e);
  return ff{h, __fsub_rn(e, __fsub_rn(h, s))};
}

// a + b. Commutative bit for bit, so both lanes of a butterfly step agree.
__device__ __forceinline__ ff ff_add(ff a, ff b) {
  const ff s = two_sum_ff(a.hi, b.hi);
  return fast_two_sum_ff(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}

__device__ __forceinline__ ff ff_neg(ff a) { return ff{-a.hi, -a.lo}; }

// a * u for a float u (exact product of the high parts by fma).
__device__ __forceinline__ ff ff_mul_f(ff a, float u) {
  const float p = __fmul_rn(a.hi, u);
  const float e = fmaf(a.hi, u, -p);
  return fast_two_sum_ff(p, fmaf(a.lo, u, e));
}

// a < b for normalised pairs.
__device__ __forceinline__ bool ff_lt(ff a, ff b) {
  return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}

__device__ __forceinline__ ff shfl_xor_ff(ff x, int o) {
  return ff{__shfl_xor_sync(FULL, x.hi, o), __shfl_xor_sync(FULL, x.lo, o)};
}

__device__ __forceinline__ ff warp_sum_ff(ff x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = ff_add(x, shfl_xor_ff(x, o));
  return x;
}

__device__ __forceinline__ ff warp_incl_scan_ff(ff x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff y{__shfl_up_sync(FULL, x.hi, o), __shfl_up_sync(FULL, x.lo, o)};
    if (lane >= o) x = ff_add(y, x);
  }
  return x;
}

// ---------------------------------------------------------------------------
// Row addressing and piece splitting.
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ const T* row_ptr(const VerifyArgs& A, int b, int rslot, int L) {
  if (rslot <= L) return static_cast<const T*>(A.tgt) + ((size_t)b * (A.K + 1) + rslot) * A.V;
  return static_cast<const T*>(A.drf) + ((size_t)b * A.K + (rslot - L - 1)) * A.V;
}

__device__ __forceinline__ Seg make_seg(const unsigned char* g, int n, int eb) {
  Seg s;
  s.g = g;
  s.n = n;
  const uintptr_t A0 = reinterpret_cast<uintptr_t>(g);
  const uintptr_t a0 = (A0 + 15) & ~static_cast<uintptr_t>(15);
  int head = static_cast<int>((a0 - A0) / eb);
  if (head > n) head = n;
  s.head = head;
  s.body = (((n - head) * eb) & ~15) / eb;
  return s;
}

__device__ __forceinline__ int nrows_of(const VerifyArgs& A, int b, bool greedy) {
  const int L = A.vlen[b];
  if (L < 0 || L > A.K) return 0;
  return greedy ? L + 1 : 2 * L + 1;
}

__device__ __forceinline__ int L_of_rows(int nrows, bool greedy) {
  return greedy ? nrows - 1 : (nrows - 1) / 2;
}

__device__ void raise_status(const VerifyArgs& A, uint32_t bits) { atomicOr(&A.hdr->status, bits); }

// Bounded wait on an mbarrier phase; false on abort or timeout.
__device__ bool wait_phase(uint64_t* bar, uint32_t parity, Shared& S, const VerifyArgs& A) {
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (*reinterpret_cast<volatile int*>(&S.abort_flag)) return false;
    if (clock64() - t0 > WAIT_CYCLES) {
      S.abort_flag = 1;
      raise_status(A, ST_TIMEOUT);
      return false;
    }
  }
  return true;
}


// Acquire-ordered load (GPU scope).
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* addr) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}

// Release-ordered atomic add (GPU scope): earlier stores of this thread become
// visible to whoever observes the new count.
__device__ __forceinline__ uint32_t atom_add_release(uint32_t* addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(addr), "r"(v)
               : "memory");
  return old;
}

__device__ void emit_invalid(const VerifyArgs& A, int b, int lane) {
  int32_t* ot = A.out_tok + (size_t)b * (A.K + 1);
  for (int k = lane; k <= A.K; k += 32) ot[k] = -1;
  const float nan = __int_as_float(0x7fc00000);
  if (A.out_p)
    for (int k = lane; k < A.K; k += 32) A.out_p[(size_t)b * A.K + k] = nan;
  if (A.out_q)
    for (int k = lane; k < A.K; k += 32) A.out_q[(size_t)b * A.K + k] = nan;
  if (lane == 0) {
    A.out_acc[b] = -1;
    A.jobs[b].kind = J_NONE;
    raise_status(A, ST_DEVICE_INPUT);
  }
}

// Decision for one request at T > 0 (one warp).
template <typename T>
__device__ void decide_sample(const VerifyArgs& A, int b, int L, int lane) {
  const int K = A.K, V = A.V;
  const size_t rb = (size_t)b * A.RS;
  float p = __int_as_float(0x7fc00000), q = p, MAt = 0.f, MAd = 0.f, iSt = 0.f, iSd = 0.f;
  int x = -1;
  bool ok = true, acc = false;
  if (lane < L) {
    const float2 st = __ldcg(A.rowstat + rb + lane);
    const float2 sd = __ldcg(A.rowstat + rb + L + 1 + lane);
    x = __ldg(A.tok + (size_t)b * K + lane);
    const float u = __ldg(A.uni + (size_t)b * (K + 1) + lane);
    ok = x >= 0 && x < V && finitef(st.x) && finitef(sd.x) && st.y > 0.f && finitef(st.y) &&
         sd.y > 0.f && finitef(sd.y) && u >= 0.f && u < 1.f;
    if (ok) {
      MAt = __fmul_rn(st.x, A.a);
      MAd = __fmul_rn(sd.x, A.a);
      const T* tr = static_cast<const T*>(A.tgt) + ((size_t)b * (K + 1) + lane) * V;
      const T* dr = static_cast<const T*>(A.drf) + ((size_t)b * K + lane) * V;
      const float et = exp2_precise(ld_logit(tr + x), A.a, A.a_lo, MAt);
      const float ed = exp2_precise(ld_logit(dr + x), A.a, A.a_lo, MAd);
      p = __fdiv_rn(et, st.y);
      q = __fdiv_rn(ed, sd.y);
      iSt = __fdiv_rn(1.f, st.y);
      iSd = __fdiv_rn(1.f, sd.y);
      acc = u * q < p;
    }
  }
  const float2 sL = __ldcg(A.rowstat + rb + L);
  const float uK = __ldg(A.uni + (size_t)b * (K + 1) + K);
  const bool okL = finitef(sL.x) && sL.y > 0.f && finitef(sL.y) && uK >= 0.f && uK < 1.f;
  if (__any_sync(FULL, !ok) || !okL) {
    emit_invalid(A, b, lane);
    return;
  }
  const unsigned am = __ballot_sync(FULL, lane < L && acc);
  const unsigned lm = (L >= 32) ? FULL : ((1u << L) - 1u);
  const int j = ((am & lm) == lm) ? L : (__ffs(~am) - 1);
  int32_t* ot = A.out_tok + (size_t)b * (K + 1);
  for (int k = lane; k <= K; k += 32)
    if (k != j) ot[k] = (k < j) ? x : -1;
  if (A.out_p && lane < K) A.out_p[(size_t)b * K + lane] = p;
  if (A.out_q && lane < K) A.out_q[(size_t)b * K + lane] = q;
  if (A.acc_cnt && lane < L && lane < j) atomicAdd(A.acc_cnt + lane, 1u);
  if (A.tst_cnt && lane < L && lane <= j) atomicAdd(A.tst_cnt + lane, 1u);
  // Terminal-sample job. Weights are computed as 2^((z - M)*a) against the exact
  // maximum, so each inverse row sum absorbs the frame offset 2^(M*a - fl(M*a)).
  const float jM = (lane < L) ? __ldcg(A.rowstat + rb + lane).x : 0.f;
  const float jMd = (lane < L) ? __ldcg(A.rowstat + rb + L + 1 + lane).x : 0.f;
  const float cSt = iSt * ex2(fmaf(jM, A.a, -MAt));
  const float cSd = iSd * ex2(fmaf(jMd, A.a, -MAd));
  const float jMt = __shfl_sync(FULL, jM, j & 31), jSt = __shfl_sync(FULL, cSt, j & 31);
  const float jMdd = __shfl_sync(FULL, jMd, j & 31), jSd = __shfl_sync(FULL, cSd, j & 31);
  if (lane == 0) {
    A.out_acc[b] = j;
    TermJob J;
    J.j = j;
    if (j == L) {  // every draft accepted: bonus sample from p_L
      J.kind = J_BONUS;
      J.MAt = sL.x;
      J.invSt = J.MAd = J.invSd = 0.f;
    } else {  // first rejection at j: residual sample
      J.kind = J_RESID;
      J.MAt = jMt;
      J.invSt = jSt;
      J.MAd = jMdd;
      J.invSd = jSd;
    }
    J.pad[0] = J.pad[1] = 0;
    A.jobs[b] = J;
  }
}

// Decision for one request at T == 0 (one warp): argmax matching.
__device__ void decide_greedy(const VerifyArgs& A, int b, int L, int lane) {
  const int K = A.K, V = A.V;
  const size_t rb = (size_t)b * A.RS;
  int x = -1, am = -1;
  bool ok = true;
  if (lane < L) {
    const float2 st = __ldcg(A.rowstat + rb + lane);
    x = __ldg(A.tok + (size_t)b * K + lane);
    am = __float_as_int(st.y);
    ok = finitef(st.x) && x >= 0 && x < V;
  }
  const float2 sL = __ldcg(A.rowstat + rb + L);
  const bool okL = finitef(sL.x);
  if (__any_sync(FULL, !ok) || !okL) {
    emit_invalid(A, b, lane);
    return;
  }
  const unsigned acc = __ballot_sync(FULL, lane < L && x == am);
  const unsigned lm = (L >= 32) ? FULL : ((1u << L) - 1u);
  const int j = ((acc & lm) == lm) ? L : (__ffs(~acc) - 1);
  int y = __shfl_sync(FULL, am, j & 31);
  if (j == L) y = __float_as_int(sL.y);
  int32_t* ot = A.out_tok + (size_t)b * (K + 1);
  for (int k = lane; k <= K; k += 32) ot[k] = (k < j) ? x : (k == j ? y : -1);
  const float nan = __int_as_float(0x7fc00000);
  if (A.out_p && lane < K) A.out_p[(size_t)b * K + lane] = nan;
  if (A.out_q && lane < K) A.out_q[(size_t)b * K + lane] = nan;
  if (A.acc_cnt && lane < L && lane < j) atomicAdd(A.acc_cnt + lane, 1u);
  if (A.tst_cnt && lane < L && lane <= j) atomicAdd(A.tst_cnt + lane, 1u);
  if (lane == 0) {
    A.out_acc[b] = j;
    A.jobs[b].kind = J_NONE;
  }
}

// Per-lane running state of a row segment: (m, ma = fl(m*a), s) at T > 0, or
// (best, idx, bad) at T == 0. Lanes accumulate independently over the segment's
// pieces; the warp reduces the lanes once, when the segment is published.
struct LaneState {
  float m, ma, s;  // softmax; greedy uses m = best, s = idx bits
  bool bad;
};

__device__ __forceinline__ void lane_reset(LaneState& st) {
  st.m = -INFINITY;
  st.ma = -INFINITY;
  st.s = 0.f;
  st.bad = false;
}

__device__ __forceinline__ float vec_max(uint4 v, uint16_t) {
  const uint32_t mx = bmax2_nan(bmax2_nan(v.x, v.y), bmax2_nan(v.z, v.w));
  return fmax_nan(bf_lo(mx), bf_hi(mx));
}
__device__ __forceinline__ float vec_max(uint4 v, float) {
  return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                  fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
}
__device__ __forceinline__ uint32_t vmax_raw(uint32_t a, uint32_t b, uint16_t) {
  return bmax2_nan(a, b);
}

// Sum of 2^(z*a - ma) over one uint4 of elements.
__device__ __forceinline__ float vec_expsum(uint4 v, float a, float nma, uint16_t) {
  const float e0 = ex2(fmaf(bf_lo(v.x), a, nma)), e1 = ex2(fmaf(bf_hi(v.x), a, nma));
  const float e2 = ex2(fmaf(bf_lo(v.y), a, nma)), e3 = ex2(fmaf(bf_hi(v.y), a, nma));
  const float e4 = ex2(fmaf(bf_lo(v.z), a, nma)), e5 = ex2(fmaf(bf_hi(v.z), a, nma));
  const float e6 = ex2(fmaf(bf_lo(v.w), a, nma)), e7 = ex2(fmaf(bf_hi(v.w), a, nma));
  return ((e0 + e1) + (e2 + e3)) + ((e4 + e5) + (e6 + e7));
}
__device__ __forceinline__ float vec_expsum(uint4 v, float a, float nma, float) {
  const float e0 = ex2(fmaf(__uint_as_float(v.x), a, nma));
  const float e1 = ex2(fmaf(__uint_as_float(v.y), a, nma));
  const float e2 = ex2(fmaf(__uint_as_float(v.z), a, nma));
  const float e3 = ex2(fmaf(__uint_as_float(v.w), a, nma));
  return (e0 + e1) + (e2 + e3);
}

// Index (0..VEC-1) of the first element of v equal to lm.
__device__ __forceinline__ int vec_first(uint4 v, float lm, uint16_t) {
  int e = 7;
  if (bf_lo(v.w) == lm) e = 6;
  if (bf_hi(v.z) == lm) e = 5;
  if (bf_lo(v.z) == lm) e = 4;
  if (bf_hi(v.y) == lm) e = 3;
  if (bf_lo(v.y) == lm) e = 2;
  if (bf_hi(v.x) == lm) e = 1;
  if (bf_lo(v.x) == lm) e = 0;
  return e;
}
__device__ __forceinline__ int vec_first(uint4 v, float lm, float) {
  int e = 3;
  if (__uint_as_float(v.z) == lm) e = 2;
  if (__uint_as_float(v.y) == lm) e = 1;
  if (__uint_as_float(v.x) == lm) e = 0;
  return e;
}

// Fold one stream piece into the lane states: a max pass over the lane's vectors in
// shared memory, one rescale, then an exp-sum pass (T > 0); or a max pass and, only
// when a lane's piece maximum beats its running best, a search for its first index
// (T == 0). Head and tail elements outside the bulk copy are read from global memory.
template <typename T, bool GREEDY>
__device__ void fold_piece(LaneState& st, const VerifyArgs& A, const SlotMeta& M,
                           const unsigned char* slot, int lane) {
  constexpr int VEC = ET<T>::VEC;
  const Seg& sg = M.s0;
  const T* g = reinterpret_cast<const T*>(sg.g);
  const int tail = sg.n - sg.head - sg.body;
  const int nv = sg.body / VEC;
  const uint4* v4 = reinterpret_cast<const uint4*>(slot);
  const int base = M.e0 + sg.head;
  if (GREEDY) {
    int idx = __float_as_int(st.s);
    if (lane < sg.head) arg_add1(st.m, idx, st.bad, ld_logit(g + lane), M.e0 + lane);
    float lm = -INFINITY;
#pragma unroll 4
    for (int i = lane; i < nv; i += 32) lm = fmax_nan(lm, vec_max(v4[i], T()));
    if (lm != lm) {
      st.bad = true;
    } else if (lm > st.m) {  // new best in this piece: its first occurrence
      for (int i = lane; i < nv; i += 32) {
        const uint4 v = v4[i];
        if (vec_max(v, T()) == lm) {
          idx = base + i * VEC + vec_first(v, lm, T());
          break;
        }
      }
      st.m = lm;
    }
    if (lane < tail)
      arg_add1(st.m, idx, st.bad, ld_logit(g + sg.head + sg.body + lane), base + sg.body + lane);
    st.s = __int_as_float(idx);
    return;
  }
  const float a = A.a;
  if (lane < sg.head) soft_add1(st.m, st.ma, st.s, ld_logit(g + lane), a);
  float lm = -INFINITY;
#pragma unroll 4
  for (int i = lane; i < nv; i += 32) lm = fmax_nan(lm, vec_max(v4[i], T()));
  soft_rescale(st.m, st.ma, st.s, lm, a);
  if (st.m != -INFINITY) {
    const float nma = -st.ma;
    float acc = 0.f;
#pragma unroll 4
    for (int i = lane; i < nv; i += 32) acc += vec_expsum(v4[i], a, nma, T());
    st.s += acc;
  }
  if (lane < tail) soft_add1(st.m, st.ma, st.s, ld_logit(g + sg.head + sg.body + lane), a);
}

// Running partial of one row segment (consecutive pieces of one row handled by one
// warp).
struct Segment {
  int valid, b, r, p0, p1;  // pieces [p0, p1] of row slot r of request b
};

// A published segment whose ticket value has not been inspected yet.
struct Pending {
  int valid, b, r, count;
  uint32_t old;  // ticket value returned to lane 0
};

// Publish a segment: reduce the lane states, store the partial at slot p0 and
// neutral partials at p0+1..p1, then a release-ordered ticket increment by the number
// of pieces. Lane 0 writes everything.
template <bool GREEDY>
__device__ Pending publish(const VerifyArgs& A, const Segment& sg, LaneState st, int lane) {
  float2 v;
  if (GREEDY) {
    int idx = __float_as_int(st.s);
    bool bad = st.bad;
    arg_warp(st.m, idx, bad);
    v = make_float2(bad ? __int_as_float(0x7fc00000) : st.m, __int_as_float(idx));
  } else {
    float m = st.m, s = st.s;
    soft_warp(m, s, A.a, lane);
    v = make_float2(m, s);
  }
  Pending pd;
  pd.valid = 1;
  pd.b = sg.b;
  pd.r = sg.r;
  pd.count = sg.p1 - sg.p0 + 1;
  pd.old = 0;
  if (lane == 0) {
    const size_t rowid = (size_t)sg.b * A.RS + sg.r;
    float2* pr = A.part + rowid * A.P;
    pr[sg.p0] = v;
    const float2 neutral = GREEDY ? make_float2(-INFINITY, __int_as_float(INT_MAX))
                                  : make_float2(-INFINITY, 0.f);
    for (int q = sg.p0 + 1; q <= sg.p1; ++q) pr[q] = neutral;
    pd.old = atom_add_release(A.t_row + rowid, (uint32_t)pd.count);
  }
  return pd;
}

// Inspect a pending ticket: the warp that completed a row combines it, the warp that
// completed a request decides it.
template <typename T, bool GREEDY>
__device__ void settle(const VerifyArgs& A, const Pending& pd, const int* prefix, int lane) {
  const uint32_t old = __shfl_sync(FULL, pd.old, 0);
  const int P = A.P;
  if (old + (uint32_t)pd.count != (uint32_t)P) return;
  __threadfence();
  const int b = pd.b;
  const size_t rowid = (size_t)b * A.RS + pd.r;
  const float2* pr = A.part + rowid * P;
  float2 rs;
  if (GREEDY) {
    float best = -INFINITY;
    int idx = INT_MAX;
    bool bad = false;
    for (int p = lane; p < P; p += 32) {
      const float2 v = __ldcg(pr + p);
      const int vi = __float_as_int(v.y);
      if (v.x != v.x) {
        bad = true;
      } else if (v.x > best || (v.x == best && vi < idx)) {
        best = v.x;
        idx = vi;
      }
    }
    arg_warp(best, idx, bad);
    rs = make_float2(bad ? __int_as_float(0x7fc00000) : best, __int_as_float(idx));
  } else {
    float m = -INFINITY, s = 0.f;
    for (int p = lane; p < P; p += 32) {
      const float2 v = __ldcg(pr + p);
      soft_merge(m, s, v.x, v.y, A.a);
    }
    soft_warp(m, s, A.a, lane);
    rs = make_float2(m, s);
  }
  const int nrows = prefix[b + 1] - prefix[b];
  uint32_t o2 = 0;
  if (lane == 0) {
    A.rowstat[rowid] = rs;
    A.t_row[rowid] = 0;
    o2 = atom_add_release(A.t_req + b, 1u);
  }
  o2 = __shfl_sync(FULL, o2, 0);
  if (o2 != (uint32_t)(nrows - 1)) return;
  __threadfence();
  if (lane == 0) A.t_req[b] = 0;
  const int L = L_of_rows(nrows, GREEDY);
  if (GREEDY)
    decide_greedy(A, b, L, lane);
  else
    decide_sample<T>(A, b, L, lane);
}

// ---------------------------------------------------------------------------
// Per-warp work: a contiguous range [i0, i1) of the work list (equal shares), walked
// by a cursor in lane 0 that issues the bulk copy of each piece into the warp's
// next free slot.
// ---------------------------------------------------------------------------
struct Cursor {
  unsigned long long cur, end;
  int cb, cr, cp, cL, cn;  // request, row slot, piece, L, rows of the current item
};

template <bool GREEDY>
__device__ void cursor_init(Cursor& c, const VerifyArgs& A, const int* prefix,
                            unsigned long long i0, unsigned long long i1) {
  c.cur = i0;
  c.end = i1;
  if (i0 >= i1) return;
  const int P = A.P;
  const unsigned long long g = i0 / P;
  c.cp = static_cast<int>(i0 - g * P);
  int lo = 0, hi = A.B - 1;
  while (lo < hi) {  // last request whose prefix is <= g
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<unsigned long long>(prefix[mid]) <= g)
      lo = mid;
    else
      hi = mid - 1;
  }
  c.cb = lo;
  c.cr = static_cast<int>(g - prefix[lo]);
  c.cn = prefix[lo + 1] - prefix[lo];
  c.cL = L_of_rows(c.cn, GREEDY);
}

// Next piece of the warp's range into a slot: fills the slot's metadata and starts
// its bulk copy. Returns false at the end of the range. Lane 0 only.
template <typename T, bool GREEDY>
__device__ bool issue_next(const VerifyArgs& A, Cursor& c, const int* prefix, SlotMeta& meta,
                           uint64_t* full, unsigned char* slot) {
  constexpr int eb = sizeof(T);
  const int P = A.P, B = A.B;
  if (c.cur >= c.end) return false;
  const T* row = row_ptr<T>(A, c.cb, c.cr, c.cL);
  const int e0 = c.cp * A.E;
  const int n = min(A.E, A.V - e0);
  meta.kind = K_STREAM;
  meta.b = c.cb;
  meta.r = c.cr;
  meta.p = c.cp;
  meta.e0 = e0;
  meta.s0 = make_seg(reinterpret_cast<const unsigned char*>(row + e0), n, eb);
  ++c.cur;
  if (++c.cp == P) {
    c.cp = 0;
    if (++c.cr == c.cn) {
      c.cr = 0;
      do {
        ++c.cb;
      } while (c.cb < B && prefix[c.cb + 1] == prefix[c.cb]);
      if (c.cb < B) {
        c.cn = prefix[c.cb + 1] - prefix[c.cb];
        c.cL = L_of_rows(c.cn, GREEDY);
      }
    }
  }
  const uint32_t tx = meta.s0.body * eb;
  if (tx) {
    mbar_arrive_expect_tx(full, tx);
    bulk_g2s(slot, meta.s0.g + meta.s0.head * eb, tx, full);
  } else {
    mbar_arrive(full);
  }
  return true;
}

// One warp: its range of pieces through SLOTS_PER_WARP slots; each slot is refilled
// right after the warp has reduced it.
template <typename T, bool GREEDY>
__device__ void warp_loop(const VerifyArgs& A, Shared& S, unsigned char* slots, const int* prefix,
                          int w, int lane, uint32_t* cons) {
  const unsigned long long total =
      static_cast<unsigned long long>(S.total_rows) * static_cast<unsigned long long>(A.P);
  const unsigned long long nw = (unsigned long long)gridDim.x * NCW;
  const unsigned long long gw = (unsigned long long)blockIdx.x * NCW + w;
  const unsigned long long i0 = total * gw / nw, i1 = total * (gw + 1) / nw;
  Cursor c;
  int have[SLOTS_PER_WARP];
#pragma unroll
  for (int q = 0; q < SLOTS_PER_WARP; ++q) have[q] = 0;
  if (lane == 0) {
    cursor_init<GREEDY>(c, A, prefix, i0, i1);
#pragma unroll
    for (int q = 0; q < SLOTS_PER_WARP; ++q) {
      const int s = SLOTS_PER_WARP * w + q;
      have[q] = issue_next<T, GREEDY>(A, c, prefix, S.meta[s], &S.full[s],
                                      slots + (size_t)s * SLOT_BYTES);
    }
  }
#pragma unroll
  for (int q = 0; q < SLOTS_PER_WARP; ++q) have[q] = __shfl_sync(FULL, have[q], 0);
  Pending pd;
  pd.valid = 0;
  Segment sg;
  sg.valid = 0;
  LaneState st;
  lane_reset(st);
  if (GREEDY) st.s = __int_as_float(INT_MAX);
  unsigned long long item = i0;
  int k = 0;
  bool aborted = false;
  while (have[k]) {
    const int s = SLOTS_PER_WARP * w + k;
    const bool ok = wait_phase(&S.full[s], cons[k] & 1, S, A);
    if (!__all_sync(FULL, ok)) {
      aborted = true;
      break;
    }
    if (pd.valid) {  // the previous segment's ticket has had a whole wait to come back
      settle<T, GREEDY>(A, pd, prefix, lane);
      pd.valid = 0;
    }
    const SlotMeta M = S.meta[s];
    unsigned char* slot = slots + (size_t)s * SLOT_BYTES;
    if (!(sg.valid && sg.b == M.b && sg.r == M.r)) {  // a new row segment starts here
      sg.valid = 1;
      sg.b = M.b;
      sg.r = M.r;
      sg.p0 = M.p;
      lane_reset(st);
      if (GREEDY) st.s = __int_as_float(INT_MAX);
    }
    sg.p1 = M.p;
    fold_piece<T, GREEDY>(st, A, M, slot, lane);
    ++cons[k];
    __syncwarp();
    int h = 0;
    if (lane == 0) {
      // The slot's shared-memory reads are done; order them before the async-proxy
      // write of the next copy into the same slot.
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      h = issue_next<T, GREEDY>(A, c, prefix, S.meta[s], &S.full[s], slot);
    }
    have[k] = __shfl_sync(FULL, h, 0);
    // Publish at the row's last piece or the range's last piece.
    ++item;
    if (M.p == A.P - 1 || item == i1) {
      if (pd.valid) {
        settle<T, GREEDY>(A, pd, prefix, lane);
        pd.valid = 0;
      }
      pd = publish<GREEDY>(A, sg, st, lane);
      sg.valid = 0;
    }
    k = (k + 1 == SLOTS_PER_WARP) ? 0 : k + 1;
  }
  if (pd.valid) settle<T, GREEDY>(A, pd, prefix, lane);
  if (aborted) {
    // Let this warp's copies in flight land before the CTA may exit.
    for (int q = 0; q < SLOTS_PER_WARP; ++q) {
      if (!have[q]) continue;
      const long long t0 = clock64();
      while (!mbar_test(&S.full[SLOTS_PER_WARP * w + q], cons[q] & 1) &&
             clock64() - t0 < WAIT_CYCLES) {
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Terminal sample (T > 0): weights, piece sums, inverse-CDF location.
// ---------------------------------------------------------------------------

// Weight of one element: residual max(0, p - q), or the unnormalised target weight
// 2^((z - M)*a) of a plain sample. Mt, Md are the raw row maxima; iSt, iSd the
// inverse row sums in that frame.
struct TermW {
  float a, a_lo, Mt, iSt, Md, iSd;
  bool resid;
  __device__ __forceinline__ float operator()(float zt, float zd) const {
    const float et = exp2_diff(zt, Mt, a, a_lo);
    if (!resid) return et;
    return fmaxf(et * iSt - exp2_diff(zd, Md, a, a_lo) * iSd, 0.f);
  }
};

// Weights of the elements of one uint4 of t (and d).
template <typename T>
__device__ __forceinline__ void vec_weights(const uint4 vt, const uint4 vd, const TermW& W,
                                            float* w) {
  if (ET<T>::VEC == 8) {
    w[0] = W(bf_lo(vt.x), bf_lo(vd.x));
    w[1] = W(bf_hi(vt.x), bf_hi(vd.x));
    w[2] = W(bf_lo(vt.y), bf_lo(vd.y));
    w[3] = W(bf_hi(vt.y), bf_hi(vd.y));
    w[4] = W(bf_lo(vt.z), bf_lo(vd.z));
    w[5] = W(bf_hi(vt.z), bf_hi(vd.z));
    w[6] = W(bf_lo(vt.w), bf_lo(vd.w));
    w[7] = W(bf_hi(vt.w), bf_hi(vd.w));
  } else {
    w[0] = W(__uint_as_float(vt.x), __uint_as_float(vd.x));
    w[1] = W(__uint_as_float(vt.y), __uint_as_float(vd.y));
    w[2] = W(__uint_as_float(vt.z), __uint_as_float(vd.z));
    w[3] = W(__uint_as_float(vt.w), __uint_as_float(vd.w));
  }
}

// Compensated total of the weights of elements [0, n) of rows t (and d), n <= E2,
// read from global memory; with wbuf != nullptr the weights are also stored there
// (shared, per warp). Vector loads are issued a half-piece at a time before use.
template <typename T>
__device__ ff piece_weights(const T* t, const T* d, int n, const TermW& W, float* wbuf,
                            int lane) {
  constexpr int VEC = ET<T>::VEC;
  constexpr int HALF = SLOT_BYTES / 2 / 16 / 32 / 2;  // uint4 per lane per half-piece
  const bool vec = ((reinterpret_cast<uintptr_t>(t) | reinterpret_cast<uintptr_t>(d)) & 15) == 0;
  float hs = 0.f, hc = 0.f;
  int done = 0;
  if (vec) {
    const int nv = n / VEC;
    const uint4* t4 = reinterpret_cast<const uint4*>(t);
    const uint4* d4 = reinterpret_cast<const uint4*>(d);
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      uint4 vt[HALF], vd[HALF];
#pragma unroll
      for (int u = 0; u < HALF; ++u) {
        const int i = lane + 32 * (u + HALF * h);
        if (i < nv) {
          vt[u] = __ldg(t4 + i);
          vd[u] = W.resid ? __ldg(d4 + i) : vt[u];
        }
      }
#pragma unroll
      for (int u = 0; u < HALF; ++u) {
        const int i = lane + 32 * (u + HALF * h);
        if (i < nv) {
          float w[VEC];
          vec_weights<T>(vt[u], vd[u], W, w);
#pragma unroll
          for (int e = 0; e < VEC; ++e) two_sum(hs, hc, w[e]);
          if (wbuf) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) wbuf[i * VEC + e] = w[e];
          }
        }
      }
    }
    done = nv * VEC;
  }
  for (int e = done + lane; e < n; e += 32) {
    const float w = W(ld_logit(t + e), ld_logit(d + e));
    if (wbuf) wbuf[e] = w;
    two_sum(hs, hc, w);
  }
  __syncwarp();
  return warp_sum_ff(two_sum_ff(hs, hc));
}

// Inverse-CDF step over weights wbuf[0, n): the smallest v with target < cum(v), cum
// a float-float prefix. Lanes take contiguous ranges; falls back to the last positive
// weight when rounding leaves target past the end.
__device__ int locate_weights(const float* wbuf, int n, ff target, int lane) {
  const int c = (n + 31) / 32;
  const int v0 = min(n, lane * c), v1 = min(n, v0 + c);
  float hs = 0.f, hc = 0.f;
  int lastpos = -1;
  for (int v = v0; v < v1; ++v) {
    const float w = wbuf[v];
    two_sum(hs, hc, w);
    if (w > 0.f) lastpos = v;
  }
  const ff ls = two_sum_ff(hs, hc);
  const ff incl = warp_incl_scan_ff(ls, lane);
  const unsigned hit = __ballot_sync(FULL, ff_lt(target, incl));
  int y = -1;
  if (hit) {
    const int ln = __ffs(hit) - 1;
    if (lane == ln) {
      // Running prefix in float-float from the lane's exclusive prefix.
      ff cum = ff_add(incl, ff_neg(ls));
      for (int v = v0; v < v1; ++v) {
        cum = ff_add(cum, ff{wbuf[v], 0.f});
        if (ff_lt(target, cum)) {
          y = v;
          break;
        }
      }
      if (y < 0) y = lastpos;
    }
    y = __shfl_sync(FULL, y, ln);
  }
  if (y < 0) {
    const unsigned has = __ballot_sync(FULL, lastpos >= 0);
    y = has ? __shfl_sync(FULL, lastpos, 31 - __clz(has)) : 0;
  }
  return y;
}

// Locate the terminal token of request b from its R piece sums.
template <typename T>
__device__ int term_locate(const VerifyArgs& A, int b, const TermJob& J, const TermW& W,
                           float* wbuf, int lane) {
  const int R = A.R, K = A.K, j = J.j;
  const T* trow = static_cast<const T*>(A.tgt) + ((size_t)b * (K + 1) + j) * A.V;
  const T* drow = W.resid ? static_cast<const T*>(A.drf) + ((size_t)b * K + j) * A.V : trow;
  const float uK = __ldg(A.uni + (size_t)b * (K + 1) + K);
  const float2* rp = A.rpart + (size_t)b * A.Rmax;
  const int c = (R + 31) / 32;
  const int p0 = min(R, lane * c), p1 = min(R, p0 + c);
  ff ls{0.f, 0.f};
  int lastpos = -1;
  for (int p = p0; p < p1; ++p) {
    const float2 w = __ldcg(rp + p);
    ls = ff_add(ls, ff{w.x, w.y});
    if (w.x > 0.f) lastpos = p;
  }
  const ff incl = warp_incl_scan_ff(ls, lane);
  ff Z{__shfl_sync(FULL, incl.hi, 31), __shfl_sync(FULL, incl.lo, 31)};
  TermW Wl = W;
  bool whole_row = false;
  if (W.resid && !(Z.hi > 0.f && Z.hi <= 3.402823466e38f)) {
    // No residual mass left (p == q up to rounding): sample p_j itself instead, piece
    // by piece over the whole row.
    Wl.resid = false;
    whole_row = true;
    Z = ff{0.f, 0.f};
    for (int p = 0; p < R; ++p) {
      const int e0 = p * A.E2;
      Z = ff_add(Z, piece_weights<T>(trow + e0, trow + e0, min(A.E2, A.V - e0), Wl, nullptr, lane));
      __syncwarp();
    }
  }
  const ff target = ff_mul_f(Z, uK);
  int pstar = -1;
  ff base{0.f, 0.f};
  bool past_end = false;
  if (whole_row) {
    for (int p = 0; p < R && pstar < 0; ++p) {
      const int e0 = p * A.E2;
      const ff w = piece_weights<T>(trow + e0, trow + e0, min(A.E2, A.V - e0), Wl, nullptr, lane);
      __syncwarp();
      const ff nb = ff_add(base, w);
      if (ff_lt(target, nb)) pstar = p;
      else if (p == R - 1) {
        pstar = p;
        past_end = true;
      } else {
        base = nb;
      }
    }
  } else {
    const unsigned hit = __ballot_sync(FULL, ff_lt(target, incl));
    if (hit) {
      const int ln = __ffs(hit) - 1;
      if (lane == ln) {
        ff cum = ff_add(incl, ff_neg(ls));
        for (int p = p0; p < p1; ++p) {
          const float2 w = __ldcg(rp + p);
          const ff nc = ff_add(cum, ff{w.x, w.y});
          if (ff_lt(target, nc)) {
            pstar = p;
            break;
          }
          cum = nc;
        }
        if (pstar < 0) {
          pstar = lastpos;
          past_end = true;
        }
        base = cum;
      }
      pstar = __shfl_sync(FULL, pstar, ln);
      past_end = __shfl_sync(FULL, past_end, ln);
      base = ff{__shfl_sync(FULL, base.hi, ln), __shfl_sync(FULL, base.lo, ln)};
    }
    if (pstar < 0) {  // rounding put the target past the last piece
      const unsigned has = __ballot_sync(FULL, lastpos >= 0);
      const int ln = has ? 31 - __clz(has) : 0;
      pstar = has ? __shfl_sync(FULL, lastpos, ln) : 0;
      past_end = true;
    }
  }
  const int e0 = pstar * A.E2;
  const int ne = min(A.E2, A.V - e0);
  piece_weights<T>(trow + e0, drow + e0, ne, Wl, wbuf, lane);
  // Past the end: the last positive weight of the piece.
  const ff t2 = past_end ? ff{INFINITY, 0.f} : ff_add(target, ff_neg(base));
  return e0 + locate_weights(wbuf, ne, t2, lane);
}

// ---------------------------------------------------------------------------
// Terminal phase (T > 0), after every CTA has finished its stream work: the terminal
// piece tasks (request b, piece p) are split in equal contiguous ranges over all warps
// and fed through the same slots. Each task sums the weights of its piece (compensated
// fp32, reduced as float-float); the task completing a request locates its token.
// ---------------------------------------------------------------------------

// Next terminal task of the warp's range that has a job, into a slot (lane 0 only).
// Returns false at the end of the range.
template <typename T>
__device__ bool issue_term(const VerifyArgs& A, long long& tc, long long t1, SlotMeta& meta,
                           uint64_t* full, unsigned char* slot) {
  constexpr int eb = sizeof(T);
  const int R = A.R, K = A.K;
  while (tc < t1) {
    const int b = (int)(tc / R), p = (int)(tc - (long long)b * R);
    ++tc;
    const int kind = __ldcg(&A.jobs[b].kind), j = __ldcg(&A.jobs[b].j);
    if (!((kind == J_RESID && j >= 0 && j < K) || (kind == J_BONUS && j >= 0 && j <= K))) continue;
    const int e0 = p * A.E2;
    const int n = min(A.E2, A.V - e0);
    const T* tr = static_cast<const T*>(A.tgt) + ((size_t)b * (K + 1) + j) * A.V + e0;
    meta.kind = K_TERM;
    meta.jkind = kind;
    meta.b = b;
    meta.r = j;
    meta.p = p;
    meta.e0 = e0;
    meta.Mt = __ldcg(&A.jobs[b].MAt);
    meta.iSt = __ldcg(&A.jobs[b].invSt);
    meta.Md = __ldcg(&A.jobs[b].MAd);
    meta.iSd = __ldcg(&A.jobs[b].invSd);
    meta.s0 = make_seg(reinterpret_cast<const unsigned char*>(tr), n, eb);
    bool whole = meta.s0.head == 0 && meta.s0.body == n;
    if (kind == J_RESID) {
      const T* dr = static_cast<const T*>(A.drf) + ((size_t)b * K + j) * A.V + e0;
      meta.s1 = make_seg(reinterpret_cast<const unsigned char*>(dr), n, eb);
      whole = whole && meta.s1.head == 0 && meta.s1.body == n;
    } else {
      meta.s1 = meta.s0;
    }
    // A piece whose rows are not both 16-byte aligned and whole multiples of 16 bytes
    // is read straight from global memory.
    meta.direct = !whole;
    if (whole) {
      const uint32_t bytes = (uint32_t)(n * eb);
      mbar_arrive_expect_tx(full, (kind == J_RESID ? 2u : 1u) * bytes);
      bulk_g2s(slot, meta.s0.g, bytes, full);
      if (kind == J_RESID) bulk_g2s(slot + SLOT_BYTES / 2, meta.s1.g, bytes, full);
    } else {
      mbar_arrive(full);
    }
    return true;
  }
  return false;
}

// Weight total of one terminal piece, from its slot (or from global memory in direct
// mode): compensated fp32 per lane, reduced as float-float.
template <typename T>
__device__ ff term_piece_sum(const SlotMeta& M, const TermW& W, const unsigned char* slot,
                                 int lane) {
  constexpr int VEC = ET<T>::VEC;
  const int n = M.s0.n;
  if (M.direct)
    return piece_weights<T>(reinterpret_cast<const T*>(M.s0.g),
                            reinterpret_cast<const T*>(M.s1.g), n, W, nullptr, lane);
  const uint4* t4 = reinterpret_cast<const uint4*>(slot);
  const uint4* d4 = reinterpret_cast<const uint4*>(W.resid ? slot + SLOT_BYTES / 2 : slot);
  float hs = 0.f, hc = 0.f;
  const int nv = n / VEC;
#pragma unroll 2
  for (int i = lane; i < nv; i += 32) {
    float w[VEC];
    vec_weights<T>(t4[i], d4[i], W, w);
#pragma unroll
    for (int e = 0; e < VEC; ++e) two_sum(hs, hc, w[e]);
  }
  return warp_sum_ff(two_sum_ff(hs, hc));
}

// One warp's range of terminal tasks. cons[] carries the slots' consumed-phase counts
// from the stream phase.
template <typename T>
__device__ void term_loop(const VerifyArgs& A, Shared& S, unsigned char* slots, int w, int lane,
                          uint32_t* cons) {
  const long long N2 = (long long)A.B * A.R;
  const long long nw = (long long)gridDim.x * NCW;
  const long long gw = (long long)blockIdx.x * NCW + w;
  const long long t1 = N2 * (gw + 1) / nw;
  long long tc = N2 * gw / nw;
  int have[SLOTS_PER_WARP];
#pragma unroll
  for (int q = 0; q < SLOTS_PER_WARP; ++q) {
    int h = 0;
    if (lane == 0) {
      const int s = SLOTS_PER_WARP * w + q;
      h = issue_term<T>(A, tc, t1, S.meta[s], &S.full[s], slots + (size_t)s * SLOT_BYTES);
    }
    have[q] = __shfl_sync(FULL, h, 0);
  }
  int k = 0;
  bool aborted = false;
  while (have[k]) {
    const int s = SLOTS_PER_WARP * w + k;
    const bool ok = wait_phase(&S.full[s], cons[k] & 1, S, A);
    if (!__all_sync(FULL, ok)) {
      aborted = true;
      break;
    }
    const SlotMeta M = S.meta[s];
    unsigned char* slot = slots + (size_t)s * SLOT_BYTES;
    const TermW W{A.a, A.a_lo, M.Mt, M.iSt, M.Md, M.iSd, M.jkind == J_RESID};
    const ff acc = term_piece_sum<T>(M, W, slot, lane);
    ++cons[k];
    const int b = M.b;
    uint32_t old = 0;
    if (lane == 0) {
      A.rpart[(size_t)b * A.Rmax + M.p] = make_float2(acc.hi, acc.lo);
      old = atom_add_release(A.t_res + b, 1u);
    }
    old = __shfl_sync(FULL, old, 0);
    __syncwarp();
    if (old == (uint32_t)(A.R - 1)) {  // last piece of this request: locate its token
      __threadfence();
      if (lane == 0) A.t_res[b] = 0;
      TermJob J;
      J.kind = M.jkind;
      J.j = M.r;
      // The slot's data has been consumed: it serves as the warp's weight buffer.
      const int y = term_locate<T>(A, b, J, W, reinterpret_cast<float*>(slot), lane);
      if (lane == 0) A.out_tok[(size_t)b * (A.K + 1) + M.r] = y;
      __syncwarp();
    }
    int h = 0;
    if (lane == 0) {
      // Order this warp's generic reads and writes of the slot before the async-proxy
      // write of the next copy.
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      h = issue_term<T>(A, tc, t1, S.meta[s], &S.full[s], slot);
    }
    have[k] = __shfl_sync(FULL, h, 0);
    k = (k + 1 == SLOTS_PER_WARP) ? 0 : k + 1;
  }
  if (aborted) {
    for (int q = 0; q < SLOTS_PER_WARP; ++q) {
      if (!have[q]) continue;
      const long long c0 = clock64();
      while (!mbar_test(&S.full[SLOTS_PER_WARP * w + q], cons[q] & 1) &&
             clock64() - c0 < WAIT_CYCLES) {
      }
    }
  }
}

template <typename T, bool GREEDY>
__global__ void __launch_bounds__(NTHREADS, 1) sv_verify_kernel(const VerifyArgs A) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ Shared S;
  unsigned char* slots = dsm;
  int* prefix = reinterpret_cast<int*>(dsm + (size_t)NSLOT * SLOT_BYTES);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = A.B;

  // Exclusive prefix of active rows per request (every CTA computes the same one).
  const int per = (B + NTHREADS - 1) / NTHREADS;
  const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
  int local = 0;
  for (int b = b0; b < b1; ++b) local += nrows_of(A, b, GREEDY);
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) S.scan[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = (lane < NTHREADS / 32) ? S.scan[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL, v, o);
      if (lane >= o) v += y;
    }
    if (lane < NTHREADS / 32) S.scan[lane] = v;
  }
  __syncthreads();
  int run = incl - local + (warp ? S.scan[warp - 1] : 0);
  for (int b = b0; b < b1; ++b) {
    prefix[b] = run;
    run += nrows_of(A, b, GREEDY);
  }
  if (tid == 0) {
    S.total_rows = S.scan[NTHREADS / 32 - 1];
    prefix[B] = S.scan[NTHREADS / 32 - 1];
    S.abort_flag = 0;
    S.last_cta = 0;
    for (int s = 0; s < NSLOT; ++s) mbar_init(&S.full[s], 1);
    fence_mbar_init();
  }
  // Requests whose verify length is out of range have no rows: CTA 0 marks them.
  if (blockIdx.x == 0) {
    for (int b = warp; b < B; b += NTHREADS / 32) {
      const int L = A.vlen[b];
      if (L < 0 || L > A.K) emit_invalid(A, b, lane);
    }
  }
  __syncthreads();

  uint32_t cons[SLOTS_PER_WARP];
#pragma unroll
  for (int q = 0; q < SLOTS_PER_WARP; ++q) cons[q] = 0;
  warp_loop<T, GREEDY>(A, S, slots, prefix, warp, lane, cons);
  __syncthreads();

  if (!GREEDY) {
    // Grid-wide barrier: every request has been decided (and its terminal job
    // written) once all CTAs have arrived. The wait is bounded; after a timeout
    // anywhere the terminal phase is skipped (the status word reports it).
    if (tid == 0) {
      __threadfence();
      atomicAdd(&A.hdr->grid_sync, 1u);
      const long long c0 = clock64();
      int ok = 1;
      while (ld_acquire(&A.hdr->grid_sync) < gridDim.x) {
        if (clock64() - c0 > WAIT_CYCLES) {
          raise_status(A, ST_TIMEOUT);
          ok = 0;
          break;
        }
      }
      __threadfence();
      if (*reinterpret_cast<volatile uint32_t*>(&A.hdr->status) & ST_TIMEOUT) ok = 0;
      S.grid_ok = ok && !S.abort_flag;
    }
    __syncthreads();
    if (S.grid_ok) term_loop<T>(A, S, slots, warp, lane, cons);
    __syncthreads();
  }

  // The last CTA to finish resets the CTA counter (and, after an abort, every
  // ticket) so the workspace is ready for the next call.
  if (tid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(&A.hdr->cta_done, 1u);
    S.last_cta = (old == gridDim.x - 1);
  }
  __syncthreads();
  if (S.last_cta) {
    __threadfence();
    const bool dirty = (*reinterpret_cast<volatile uint32_t*>(&A.hdr->status) & ST_TIMEOUT) != 0;
    if (dirty) {
      for (size_t i = tid; i < TICKET_ROW_WORDS; i += NTHREADS) A.t_row[i] = 0;
      for (int i = tid; i < SV_MAX_B; i += NTHREADS) {
        A.t_req[i] = 0;
        A.t_res[i] = 0;
      }
    }
    if (tid == 0) {
      A.hdr->grid_sync = 0;
      A.hdr->cta_done = 0;
    }
  }
}

// ---------------------------------------------------------------------------
// Host launcher (called from the C-ABI layer).
// ---------------------------------------------------------------------------
template <typename T, bool GREEDY>
static cudaError_t launch_t(const VerifyArgs& A, int grid, size_t dsmem, cudaStream_t st) {
  static bool attr_set = false;  // per instantiation; idempotent if raced
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(sv_verify_kernel<T, GREEDY>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)(NSLOT * SLOT_BYTES + 4 * (SV_MAX_B + 1) + 256));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // At T > 0 the kernel holds a grid-wide barrier between its two phases: a cooperative
  // launch guarantees that all its CTAs (at most one per SM) are resident together.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = dsmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = GREEDY ? 0 : 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sv_verify_kernel<T, GREEDY>, A);
}

cudaError_t launch_verify(const VerifyArgs& A, bool bf16, bool greedy, int grid, cudaStream_t st) {
  const size_t dsmem = (size_t)NSLOT * SLOT_BYTES + align_up(4 * ((size_t)A.B + 1), 16);
  if (bf16)
    return greedy ? launch_t<uint16_t, true>(A, grid, dsmem, st)
                  : launch_t<uint16_t, false>(A, grid, dsmem, st);
  return greedy ? launch_t<float, true>(A, grid, dsmem, st)
                : launch_t<float, false>(A, grid, dsmem, st);
}

}  // namespace sv
