// sv_verify.cu -- fused batched verification of drafted token blocks (sm_103a).
//
// Method: standard speculative rejection sampling, as the DSpark pages describe it
// (DSpark Deep Dive, "The Speculative Decoding Solution"; DSpark Guide, "1. The
// Mathematics of Suffix Decay"; perchy.ai Technology, "Verified by the target").
//
// Design (one launch, one persistent CTA per SM, no CPU round trip):
//  * Work list: every active logit row of the batch (request b: target rows 0..L_b,
//    and at T > 0 draft rows 0..L_b-1) cut into fixed pieces of SLOT_BYTES. Pieces
//    are ordered request-major and claimed in batches from one atomic counter, so
//    a request's rows are streamed close together in time.
//  * Producer warp: one lane issues 1-D bulk copies (cp.async.bulk, TMA) of each
//    piece into a shared-memory slot and signals an mbarrier with the byte count.
//  * Consumer warps: each owns two slots and reduces whole pieces: online softmax
//    (running max + sum of 2^(z*log2e/T - max)) at T > 0, or (max, lowest argmax) at
//    T == 0. The piece result goes to the workspace; an atomic ticket per row and per
//    request elects the last arriving warp, which combines the row, and then the
//    request: p_k(x_k), q_k(x_k), the accept tests u*q < p, a ballot for the first
//    rejection j, the outputs.
//  * Terminal sample at T > 0: the deciding warp posts a job to its CTA's producer,
//    which streams the terminal rows again (t_j and d_j for a residual sample, or the
//    bonus row t_L; they were read microseconds earlier and are L2-resident) through
//    the same slots. Each job piece is summed with compensated fp32 arithmetic and
//    reduced in float64; the last piece locates the token by inverse CDF (float64
//    prefix over piece sums, one piece re-scanned in float64).
//  * Every wait is bounded in time; on expiry the kernel sets SV_ERR_TIMEOUT in the
//    status word, lets its copies in flight land, and returns.
#include <cfloat>
#include <climits>

#include "sv_common.cuh"

namespace sv {

enum : int { K_STREAM = 0, K_JOB = 1, K_STOP = 2 };

// Terminal-sample jobs: the residual max(0, p_j - q_j) over rows t_j and d_j, or a
// plain sample of p over one target row (the bonus row, or row j when the residual
// has no mass left).
enum : int { J_RESID = 0, J_BONUS = 1 };

// A contiguous run of elements of one row, split by 16-byte alignment into a head
// read directly from global memory, a body copied to shared memory, and a tail
// read directly.
struct Seg {
  const unsigned char* g;  // address of the run's first element
  int head, body, n;
};

struct __align__(16) SlotMeta {
  int kind, b, r, p;  // r: row slot (stream) or terminal row j / L (job piece)
  int e0;             // first element of the piece within its row
  int direct;         // job piece: 1 = rows read straight from global memory
  int jkind;          // job piece: J_RESID or J_BONUS
  int pad0;
  Seg s0, s1;
  float MAt, invSt, MAd, invSd;
};

struct Job {
  int b, j, jkind;
  float MAt, invSt, MAd, invSd;
};

struct Shared {
  SlotMeta meta[NSLOT];
  uint64_t full[NSLOT];
  uint64_t empty[NSLOT];
  Job mbox[MBOX];
  int mbox_flag[MBOX];
  int mbox_tail;
  int mbox_head;
  int abort_flag;
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
__device__ __forceinline__ void soft_merge(float& m, float& s, float m2, float s2, float a) {
  const float mn = fmax_nan(m, m2);
  if (mn == -INFINITY) return;  // both empty
  const float man = mn * a;
  const float f1 = (m == -INFINITY) ? 0.f : ex2(m * a - man);
  const float f2 = (m2 == -INFINITY) ? 0.f : ex2(m2 * a - man);
  s = fmaf(s, f1, s2 * f2);
  m = mn;
}

__device__ __forceinline__ void soft_rescale(float& m, float& ma, float& s, float lm, float a) {
  if (lm > m || lm != lm) {
    const float mn = fmax_nan(m, lm);
    const float man = mn * a;
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
// the difference), then 2^y = 2^y_hi * (1 + y_lo*ln2). Used where single values or
// terminal-sample weights must agree closely with float64.
__device__ __forceinline__ float exp2_precise(float z, float a, float a_lo, float MA) {
  const float ph = z * a;
  const float pl = fmaf(z, a, -ph);  // exact error of the product
  const float yh = ph - MA;
  const float bp = yh - ph;  // TwoSum error of ph - MA
  const float el = (ph - (yh - bp)) + (-MA - bp);
  const float yl = fmaf(z, a_lo, pl + el);
  const float e = ex2(yh);
  return fmaf(e, yl * 0.6931471805599453f, e);
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

__device__ __forceinline__ double warp_sum_d(double x, int lane) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const double y = __shfl_xor_sync(FULL, x, o);
    x = (lane & o) ? (y + x) : (x + y);
  }
  return x;
}

__device__ __forceinline__ double warp_incl_scan_d(double x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(FULL, x, o);
    if (lane >= o) x = y + x;
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

__device__ __forceinline__ void proxy_fence_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

// Copy n elements of a row (starting at src) into shared memory at dst (16-byte
// aligned). Vector loads when src is 16-byte aligned.
template <typename T>
__device__ void stage_row(unsigned char* dst, const T* src, int n, int lane) {
  constexpr int eb = sizeof(T);
  T* d = reinterpret_cast<T*>(dst);
  if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
    const int nv = n * eb / 16;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll 4
    for (int i = lane; i < nv; i += 32) d4[i] = __ldg(s4 + i);
    for (int e = nv * 16 / eb + lane; e < n; e += 32) d[e] = src[e];
  } else {
    for (int e = lane; e < n; e += 32) d[e] = src[e];
  }
}

__device__ __forceinline__ float smem_logit(const unsigned char* base, int e, float) {
  return reinterpret_cast<const float*>(base)[e];
}
__device__ __forceinline__ float smem_logit(const unsigned char* base, int e, uint16_t) {
  return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(base)[e]) << 16);
}

// Inverse-CDF step inside one staged piece of n elements: the smallest element v
// with target < cum(v), cum in float64 over fp32 weights w(v) evaluated identically
// by every lane. Falls back to the last positive-weight element when rounding leaves
// target past the end of the piece.
template <typename WF>
__device__ int locate_in_piece(WF wf, int n, double target, int lane) {
  const int c = (n + 31) / 32;
  const int v0 = lane * c, v1 = min(n, v0 + c);
  float hs = 0.f, hc = 0.f;
  int lastpos = -1;
  for (int v = v0; v < v1; ++v) {
    const float w = wf(v);
    two_sum(hs, hc, w);
    if (w > 0.f) lastpos = v;
  }
  const double ls = (double)hs + (double)hc;
  const double incl = warp_incl_scan_d(ls, lane);
  const unsigned hit = __ballot_sync(FULL, target < incl);
  int y = -1;
  if (hit) {
    const int ln = __ffs(hit) - 1;
    if (lane == ln) {
      double cum = incl - ls;
      for (int v = v0; v < v1; ++v) {
        cum += (double)wf(v);
        if (target < cum) {
          y = v;
          break;
        }
      }
      if (y < 0) y = lastpos;
    }
    y = __shfl_sync(FULL, y, ln);
  }
  if (y < 0) {  // past the end by rounding: last positive weight of the piece
    const unsigned has = __ballot_sync(FULL, lastpos >= 0);
    y = has ? __shfl_sync(FULL, lastpos, 31 - __clz(has)) : 0;
  }
  return y;
}

__device__ void emit_invalid(const VerifyArgs& A, int b, int lane) {
  int32_t* ot = A.out_tok + (size_t)b * (A.K + 1);
  for (int k = lane; k <= A.K; k += 32) ot[k] = -1;
  if (A.out_p)
    for (int k = lane; k < A.K; k += 32) A.out_p[(size_t)b * A.K + k] = __int_as_float(0x7fc00000);
  if (A.out_q)
    for (int k = lane; k < A.K; k += 32) A.out_q[(size_t)b * A.K + k] = __int_as_float(0x7fc00000);
  if (lane == 0) {
    A.out_acc[b] = -1;
    raise_status(A, ST_DEVICE_INPUT);
  }
}

// Post a terminal-sample job to this CTA's producer (one lane).
__device__ void post_job(Shared& S, const VerifyArgs& A, const Job& J) {
  const int idx = atomicAdd(&S.mbox_tail, 1);
  const long long t0 = clock64();
  while (idx - *reinterpret_cast<volatile int*>(&S.mbox_head) >= MBOX) {
    if (*reinterpret_cast<volatile int*>(&S.abort_flag)) return;
    if (clock64() - t0 > WAIT_CYCLES) {
      S.abort_flag = 1;
      raise_status(A, ST_TIMEOUT);
      return;
    }
  }
  S.mbox[idx & (MBOX - 1)] = J;
  __threadfence_block();
  *reinterpret_cast<volatile int*>(&S.mbox_flag[idx & (MBOX - 1)]) = 1;
}

// Decision for one request at T > 0 (one warp).
template <typename T>
__device__ void decide_sample(const VerifyArgs& A, Shared& S, int b, int L, int lane) {
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
      MAt = st.x * A.a;
      MAd = sd.x * A.a;
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
  if (lane == 0) A.out_acc[b] = j;
  if (A.out_p && lane < K) A.out_p[(size_t)b * K + lane] = p;
  if (A.out_q && lane < K) A.out_q[(size_t)b * K + lane] = q;
  if (A.acc_cnt && lane < L && lane < j) atomicAdd(A.acc_cnt + lane, 1u);
  if (A.tst_cnt && lane < L && lane <= j) atomicAdd(A.tst_cnt + lane, 1u);
  Job J;
  J.b = b;
  J.j = j;
  if (j == L) {  // every draft accepted: bonus sample from p_L
    J.jkind = J_BONUS;
    J.MAt = sL.x * A.a;
    J.invSt = J.MAd = J.invSd = 0.f;
  } else {  // first rejection at j: residual sample
    J.jkind = J_RESID;
    J.MAt = __shfl_sync(FULL, MAt, j & 31);
    J.invSt = __shfl_sync(FULL, iSt, j & 31);
    J.MAd = __shfl_sync(FULL, MAd, j & 31);
    J.invSd = __shfl_sync(FULL, iSd, j & 31);
  }
  if (lane == 0) post_job(S, A, J);
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
  if (lane == 0) A.out_acc[b] = j;
  const float nan = __int_as_float(0x7fc00000);
  if (A.out_p && lane < K) A.out_p[(size_t)b * K + lane] = nan;
  if (A.out_q && lane < K) A.out_q[(size_t)b * K + lane] = nan;
  if (A.acc_cnt && lane < L && lane < j) atomicAdd(A.acc_cnt + lane, 1u);
  if (A.tst_cnt && lane < L && lane <= j) atomicAdd(A.tst_cnt + lane, 1u);
}

// Process one stream piece; on completion of its row (and request) do the row
// combine (and the decision).
template <typename T, bool GREEDY>
__device__ void stream_piece(const VerifyArgs& A, Shared& S, const SlotMeta& M,
                             unsigned char* slot, const int* prefix, int lane) {
  constexpr int VEC = ET<T>::VEC;
  const Seg& sg = M.s0;
  const T* g = reinterpret_cast<const T*>(sg.g);
  const int tail = sg.n - sg.head - sg.body;
  const int nv = sg.body / VEC;
  const uint4* v4 = reinterpret_cast<const uint4*>(slot);
  float2 res;
  if (GREEDY) {
    float best = -INFINITY;
    int idx = INT_MAX;
    bool bad = false;
    if (lane < sg.head) arg_add1(best, idx, bad, ld_logit(g + lane), M.e0 + lane);
    const int base = M.e0 + sg.head;
#pragma unroll 4
    for (int i = lane; i < nv; i += 32) arg_add_vec(best, idx, bad, v4[i], base + i * VEC, T());
    if (lane < tail)
      arg_add1(best, idx, bad, ld_logit(g + sg.head + sg.body + lane), base + sg.body + lane);
    arg_warp(best, idx, bad);
    res = make_float2(bad ? __int_as_float(0x7fc00000) : best, __int_as_float(idx));
  } else {
    const float a = A.a;
    float m = -INFINITY, ma = -INFINITY, s = 0.f;
    if (lane < sg.head) soft_add1(m, ma, s, ld_logit(g + lane), a);
#pragma unroll 4
    for (int i = lane; i < nv; i += 32) soft_add_vec(m, ma, s, v4[i], a, T());
    if (lane < tail) soft_add1(m, ma, s, ld_logit(g + sg.head + sg.body + lane), a);
    soft_warp(m, s, a, lane);
    res = make_float2(m, s);
  }
  const int b = M.b, r = M.r, P = A.P;
  const size_t rowid = (size_t)b * A.RS + r;
  uint32_t old = 0;
  if (lane == 0) {
    A.part[rowid * P + M.p] = res;
    __threadfence();
    old = atomicAdd(A.t_row + rowid, 1u);
  }
  old = __shfl_sync(FULL, old, 0);
  if (old != (uint32_t)(P - 1)) return;

  // Last piece of this row: combine the row.
  __threadfence();
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
  if (lane == 0) {
    A.rowstat[rowid] = rs;
    A.t_row[rowid] = 0;
    __threadfence();
    old = atomicAdd(A.t_req + b, 1u);
  }
  old = __shfl_sync(FULL, old, 0);
  if (old != (uint32_t)(nrows - 1)) return;

  // Last row of this request: decide.
  __threadfence();
  if (lane == 0) A.t_req[b] = 0;
  const int L = L_of_rows(nrows, GREEDY);
  if (GREEDY)
    decide_greedy(A, b, L, lane);
  else
    decide_sample<T>(A, S, b, L, lane);
}

// Terminal-sample weights of one element: residual max(0, p - q), or the
// unnormalised target weight 2^(z*a - MA) of a plain sample.
struct TermW {
  float a, a_lo, MAt, iSt, MAd, iSd;
  bool resid;
  __device__ __forceinline__ float operator()(float zt, float zd) const {
    const float et = exp2_precise(zt, a, a_lo, MAt);
    if (!resid) return et;
    return fmaxf(et * iSt - exp2_precise(zd, a, a_lo, MAd) * iSd, 0.f);
  }
};

// Process one terminal-job piece: compensated sum of its weights, reduced in fp64.
// The last piece of a request locates the terminal token by inverse CDF at u_{b,K}
// (float64 prefix over the piece sums, then one piece re-scanned in float64).
template <typename T>
__device__ void job_piece(const VerifyArgs& A, Shared& S, const SlotMeta& M, unsigned char* slot,
                          int lane) {
  constexpr int VEC = ET<T>::VEC;
  const bool resid = M.jkind == J_RESID;
  const TermW W{A.a, A.a_lo, M.MAt, M.invSt, M.MAd, M.invSd, resid};
  float hs = 0.f, hc = 0.f;
  const int n = M.s0.n;
  if (!M.direct) {
    const uint4* t4 = reinterpret_cast<const uint4*>(slot);
    const uint4* d4 = reinterpret_cast<const uint4*>(slot + SLOT_BYTES / 2);
    const int nv = n / VEC;
    for (int i = lane; i < nv; i += 32) {
      const uint4 vt = t4[i];
      const uint4 vd = resid ? d4[i] : vt;
      if (VEC == 8) {
        two_sum(hs, hc, W(bf_lo(vt.x), bf_lo(vd.x)));
        two_sum(hs, hc, W(bf_hi(vt.x), bf_hi(vd.x)));
        two_sum(hs, hc, W(bf_lo(vt.y), bf_lo(vd.y)));
        two_sum(hs, hc, W(bf_hi(vt.y), bf_hi(vd.y)));
        two_sum(hs, hc, W(bf_lo(vt.z), bf_lo(vd.z)));
        two_sum(hs, hc, W(bf_hi(vt.z), bf_hi(vd.z)));
        two_sum(hs, hc, W(bf_lo(vt.w), bf_lo(vd.w)));
        two_sum(hs, hc, W(bf_hi(vt.w), bf_hi(vd.w)));
      } else {
        two_sum(hs, hc, W(__uint_as_float(vt.x), __uint_as_float(vd.x)));
        two_sum(hs, hc, W(__uint_as_float(vt.y), __uint_as_float(vd.y)));
        two_sum(hs, hc, W(__uint_as_float(vt.z), __uint_as_float(vd.z)));
        two_sum(hs, hc, W(__uint_as_float(vt.w), __uint_as_float(vd.w)));
      }
    }
  } else {
    const T* gt = reinterpret_cast<const T*>(M.s0.g);
    const T* gd = resid ? reinterpret_cast<const T*>(M.s1.g) : gt;
    for (int e = lane; e < n; e += 32) two_sum(hs, hc, W(ld_logit(gt + e), ld_logit(gd + e)));
  }
  const double acc = warp_sum_d((double)hs + (double)hc, lane);
  const int b = M.b;
  uint32_t old = 0;
  if (lane == 0) {
    A.rpart[(size_t)b * A.Rmax + M.p] = acc;
    __threadfence();
    old = atomicAdd(A.t_res + b, 1u);
  }
  old = __shfl_sync(FULL, old, 0);
  if (old != (uint32_t)(A.R - 1)) return;

  // Last piece of this job: locate the terminal token.
  __threadfence();
  if (lane == 0) A.t_res[b] = 0;
  const int R = A.R, j = M.r, K = A.K;
  const double uK = (double)__ldg(A.uni + (size_t)b * (K + 1) + K);
  const double* rp = A.rpart + (size_t)b * A.Rmax;
  const int c = (R + 31) / 32;
  const int p0 = lane * c, p1 = min(R, p0 + c);
  double ls = 0.0;
  int lastpos = -1;
  for (int p = p0; p < p1; ++p) {
    const double w = __ldcg(rp + p);
    ls += w;
    if (w > 0.0) lastpos = p;
  }
  const double incl = warp_incl_scan_d(ls, lane);
  const double Z = __shfl_sync(FULL, incl, 31);
  if (resid && (!(Z > 0.0) || !(Z < 1e300))) {
    // No residual mass left (p == q up to rounding): sample p_j itself instead.
    if (lane == 0) {
      Job J;
      J.b = b;
      J.j = j;
      J.jkind = J_BONUS;
      J.MAt = M.MAt;
      J.invSt = J.MAd = J.invSd = 0.f;
      post_job(S, A, J);
    }
    return;
  }
  const double target = uK * Z;
  const unsigned hit = __ballot_sync(FULL, target < incl);
  int pstar = -1;
  double base = 0.0;
  if (hit) {
    const int ln = __ffs(hit) - 1;
    if (lane == ln) {
      double cum = incl - ls;
      for (int p = p0; p < p1; ++p) {
        const double w = __ldcg(rp + p);
        if (target < cum + w) {
          pstar = p;
          break;
        }
        cum += w;
      }
      if (pstar < 0) pstar = lastpos;
      base = cum;
    }
    pstar = __shfl_sync(FULL, pstar, ln);
    base = __shfl_sync(FULL, base, ln);
  }
  if (pstar < 0) {  // rounding put the target past the last piece
    const unsigned has = __ballot_sync(FULL, lastpos >= 0);
    const int ln = has ? 31 - __clz(has) : 0;
    pstar = has ? __shfl_sync(FULL, lastpos, ln) : 0;
    base = target;
  }
  const int e0 = pstar * A.E2;
  const int ne = min(A.E2, A.V - e0);
  unsigned char* s1 = slot + SLOT_BYTES / 2;
  stage_row<T>(slot, static_cast<const T*>(A.tgt) + ((size_t)b * (K + 1) + j) * A.V + e0, ne, lane);
  if (resid)
    stage_row<T>(s1, static_cast<const T*>(A.drf) + ((size_t)b * K + j) * A.V + e0, ne, lane);
  __syncwarp();
  auto wf = [&](int v) {
    const float zt = smem_logit(slot, v, T());
    return W(zt, resid ? smem_logit(s1, v, T()) : zt);
  };
  const int y = e0 + locate_in_piece(wf, ne, target - base, lane);
  if (lane == 0) A.out_tok[(size_t)b * (K + 1) + j] = y;
  proxy_fence_shared();
}

// ---------------------------------------------------------------------------
// Producer: one lane. Fills slots in per-warp alternation, terminal jobs first.
// ---------------------------------------------------------------------------
template <typename T, bool GREEDY>
__device__ void producer(const VerifyArgs& A, Shared& S, unsigned char* slots, const int* prefix) {
  constexpr int eb = sizeof(T);
  const int P = A.P, B = A.B;
  const unsigned long long total =
      static_cast<unsigned long long>(S.total_rows) * static_cast<unsigned long long>(P);
  uint32_t fills[NCW];
#pragma unroll
  for (int w = 0; w < NCW; ++w) fills[w] = 0;
  int wrr = 0;

  // Work-list cursor.
  unsigned long long cur = atomicAdd(&A.hdr->q1_next, (unsigned)Q1_BATCH);
  unsigned long long nxt = (cur < total) ? atomicAdd(&A.hdr->q1_next, (unsigned)Q1_BATCH) : total;
  unsigned long long item = cur, item_end = min(cur + Q1_BATCH, total);
  int cb = -1, cr = 0, cp = 0, cL = 0, cn = 0;  // request, row slot, piece, L, rows

  // Terminal job state.
  bool job = false;
  Job J{};
  int jp = 0;
  int mh = 0;  // mailbox head

  bool aborted = false;
  long long idle_t0 = -1;

  while (true) {
    if (*reinterpret_cast<volatile int*>(&S.abort_flag)) {
      aborted = true;
      break;
    }
    SlotMeta m;
    bool have = false;
    if (!job && *reinterpret_cast<volatile int*>(&S.mbox_flag[mh & (MBOX - 1)])) {
      __threadfence_block();
      J = S.mbox[mh & (MBOX - 1)];
      *reinterpret_cast<volatile int*>(&S.mbox_flag[mh & (MBOX - 1)]) = 0;
      ++mh;
      *reinterpret_cast<volatile int*>(&S.mbox_head) = mh;
      job = true;
      jp = 0;
    }
    if (job) {
      const int e0 = jp * A.E2;
      const int n = min(A.E2, A.V - e0);
      const T* tr = static_cast<const T*>(A.tgt) + ((size_t)J.b * (A.K + 1) + J.j) * A.V + e0;
      m.kind = K_JOB;
      m.jkind = J.jkind;
      m.b = J.b;
      m.r = J.j;
      m.p = jp;
      m.e0 = e0;
      m.s0 = make_seg(reinterpret_cast<const unsigned char*>(tr), n, eb);
      bool aligned_all = m.s0.head == 0 && m.s0.body == n;
      if (J.jkind == J_RESID) {
        const T* dr = static_cast<const T*>(A.drf) + ((size_t)J.b * A.K + J.j) * A.V + e0;
        m.s1 = make_seg(reinterpret_cast<const unsigned char*>(dr), n, eb);
        aligned_all = aligned_all && m.s1.head == 0 && m.s1.body == n;
      }
      m.direct = !aligned_all;
      m.MAt = J.MAt;
      m.invSt = J.invSt;
      m.MAd = J.MAd;
      m.invSd = J.invSd;
      if (++jp == A.R) job = false;
      have = true;
    } else if (item < item_end) {
      if (cb < 0) {  // locate the item's row: binary search over the prefix
        const unsigned long long g = item / P;
        cp = static_cast<int>(item - g * P);
        int lo = 0, hi = B - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (static_cast<unsigned long long>(prefix[mid]) <= g)
            lo = mid;
          else
            hi = mid - 1;
        }
        cb = lo;
        cr = static_cast<int>(g - prefix[cb]);
        cn = prefix[cb + 1] - prefix[cb];
        cL = L_of_rows(cn, GREEDY);
      }
      const T* row = row_ptr<T>(A, cb, cr, cL);
      const int e0 = cp * A.E;
      const int n = min(A.E, A.V - e0);
      m.kind = K_STREAM;
      m.b = cb;
      m.r = cr;
      m.p = cp;
      m.e0 = e0;
      m.direct = 0;
      m.s0 = make_seg(reinterpret_cast<const unsigned char*>(row + e0), n, eb);
      have = true;
      ++item;
      if (++cp == P) {
        cp = 0;
        if (++cr == cn) {
          cr = 0;
          do {
            ++cb;
          } while (cb < B && prefix[cb + 1] == prefix[cb]);
          if (cb < B) {
            cn = prefix[cb + 1] - prefix[cb];
            cL = L_of_rows(cn, GREEDY);
          }
        }
      }
    } else if (cur < total) {
      cur = nxt;
      item = cur;
      item_end = min(cur + Q1_BATCH, total);
      cb = -1;
      if (cur < total) nxt = atomicAdd(&A.hdr->q1_next, (unsigned)Q1_BATCH);
      continue;
    }

    if (!have) {
      // Nothing to issue: finish once every slot is released and no job is pending.
      bool idle = true;
      for (int w = 0; w < NCW && idle; ++w) {
#pragma unroll
        for (int i = 0; i < SLOTS_PER_WARP; ++i) {
          const uint32_t ns = (fills[w] > (uint32_t)i) ? (fills[w] - i + 1) / 2 : 0;
          if (ns && !mbar_test(&S.empty[2 * w + i], (ns - 1) & 1)) idle = false;
        }
      }
      if (idle && !*reinterpret_cast<volatile int*>(&S.mbox_flag[mh & (MBOX - 1)])) break;
      if (idle_t0 < 0) idle_t0 = clock64();
      if (clock64() - idle_t0 > WAIT_CYCLES) {
        S.abort_flag = 1;
        raise_status(A, ST_TIMEOUT);
        aborted = true;
        break;
      }
      continue;
    }
    idle_t0 = -1;

    // Find a consumer warp whose next slot is free (polling, no sleeps).
    int w = -1;
    const long long t0 = clock64();
    while (w < 0) {
      for (int c = 0; c < NCW; ++c) {
        const int ww = (wrr + c) % NCW;
        const uint32_t f = fills[ww];
        const int s = 2 * ww + (f & 1);
        const uint32_t k = f >> 1;
        if (k == 0 || mbar_test(&S.empty[s], (k - 1) & 1)) {
          w = ww;
          break;
        }
      }
      if (w >= 0) break;
      if (*reinterpret_cast<volatile int*>(&S.abort_flag)) break;
      if (clock64() - t0 > WAIT_CYCLES) {
        S.abort_flag = 1;
        raise_status(A, ST_TIMEOUT);
        break;
      }
    }
    if (w < 0) {
      aborted = true;
      break;
    }
    wrr = (w + 1) % NCW;
    const int s = 2 * w + (fills[w] & 1);
    unsigned char* dst = slots + (size_t)s * SLOT_BYTES;
    S.meta[s] = m;
    uint32_t tx = 0;
    if (m.kind == K_STREAM) {
      tx = m.s0.body * eb;
    } else if (!m.direct) {
      tx = (m.jkind == J_RESID ? 2 : 1) * m.s0.body * eb;
    }
    if (tx) {
      mbar_arrive_expect_tx(&S.full[s], tx);
      if (m.kind == K_STREAM) {
        bulk_g2s(dst, m.s0.g + m.s0.head * eb, m.s0.body * eb, &S.full[s]);
      } else {
        bulk_g2s(dst, m.s0.g, m.s0.body * eb, &S.full[s]);
        if (m.jkind == J_RESID)
          bulk_g2s(dst + SLOT_BYTES / 2, m.s1.g, m.s1.body * eb, &S.full[s]);
      }
    } else {
      mbar_arrive(&S.full[s]);
    }
    ++fills[w];
  }

  if (aborted) {
    // Let every copy in flight land before the CTA may exit.
    for (int w = 0; w < NCW; ++w)
      for (int i = 0; i < SLOTS_PER_WARP; ++i) {
        const uint32_t ns = (fills[w] > (uint32_t)i) ? (fills[w] - i + 1) / 2 : 0;
        if (!ns) continue;
        const long long t0 = clock64();
        while (!mbar_test(&S.full[2 * w + i], (ns - 1) & 1) && clock64() - t0 < WAIT_CYCLES) {
        }
      }
    return;
  }
  // Send every consumer warp its stop slot.
  for (int w = 0; w < NCW; ++w) {
    const int s = 2 * w + (fills[w] & 1);
    S.meta[s].kind = K_STOP;
    mbar_arrive(&S.full[s]);
    ++fills[w];
  }
}

template <typename T, bool GREEDY>
__device__ void consumer(const VerifyArgs& A, Shared& S, unsigned char* slots, const int* prefix,
                         int w, int lane) {
  uint32_t it = 0;
  while (true) {
    const int s = 2 * w + (it & 1);
    const bool ok = wait_phase(&S.full[s], (it >> 1) & 1, S, A);
    if (!__all_sync(FULL, ok)) break;
    const SlotMeta M = S.meta[s];
    if (M.kind == K_STOP) break;
    unsigned char* slot = slots + (size_t)s * SLOT_BYTES;
    if (M.kind == K_STREAM)
      stream_piece<T, GREEDY>(A, S, M, slot, prefix, lane);
    else
      job_piece<T>(A, S, M, slot, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);
    ++it;
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
    S.mbox_tail = 0;
    S.mbox_head = 0;
    S.abort_flag = 0;
    S.last_cta = 0;
    for (int i = 0; i < MBOX; ++i) S.mbox_flag[i] = 0;
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
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

  if (warp == NCW) {
    if (lane == 0) producer<T, GREEDY>(A, S, slots, prefix);
  } else {
    consumer<T, GREEDY>(A, S, slots, prefix, warp, lane);
  }
  __syncthreads();

  // The last CTA to finish resets the work counter (and, after an abort, every
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
      A.hdr->q1_next = 0;
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
  sv_verify_kernel<T, GREEDY><<<grid, NTHREADS, dsmem, st>>>(A);
  return cudaGetLastError();
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
