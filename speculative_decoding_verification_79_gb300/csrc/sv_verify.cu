// sv_verify.cu -- fused batched verification of drafted token blocks (sm_103a).
//
// Method: standard speculative rejection sampling, as the DSpark pages describe it
// (DSpark Deep Dive, "The Speculative Decoding Solution"; DSpark Guide, "1. The
// Mathematics of Suffix Decay"; perchy.ai Technology, "Verified by the target").
//
// One launch on the caller's stream, no CPU round trip: sv_verify_kernel, one
// persistent CTA per SM of NCW warps.
//  - Stream work. Work list: every active logit row of the batch (request b: target
//    rows 0..L_b, and at T > 0 draft rows 0..L_b-1) cut into pieces of SLOT_BYTES,
//    ordered request-major and split into equal contiguous ranges, one per warp of
//    the grid. Each warp owns SLOTS_PER_WARP shared-memory slots and is its own
//    producer: lane 0 issues a 1-D bulk copy (cp.async.bulk, TMA) of the next piece
//    into the slot the warp has just finished, guarded by an mbarrier, while the warp
//    reduces the other slots. Pieces are reduced whole: online softmax (running max
//    + sum of 2^(z*log2e/T - max)) at T > 0, or (max, lowest argmax) at T == 0,
//    merged in registers while consecutive pieces belong to the same row. A warp's
//    run of pieces of one row is published as one self-validating 64-bit word and a
//    relaxed ticket increment, whose value the warp inspects only after its next
//    wait, so the round trip stays off the critical path (no fences on the stream
//    path). The warp completing a row combines its partials in piece order; the
//    warp completing a request decides it: p_k(x_k), q_k(x_k), the accept tests
//    u*q < p, a ballot for the first rejection j, the outputs, and (T > 0) the
//    request's terminal-sample job, announced by a release-ordered decision flag.
//  - Terminal tasks (T > 0). The terminal rows of a request (residual
//    max(0, p_j - q_j), or p of the bonus row) are cut into R pieces; the tasks
//    (b, p), request-major, are split into equal contiguous shares, one per warp.
//    Once its stream range is done, a warp feeds its terminal tasks through the same
//    slots, each as soon as its request's flag is up (no grid-wide barrier); the
//    deciding warp has already asked L2 to prefetch the request's terminal rows. Each task sums its piece's weights
//    (compensated fp32, float-float across lanes) and stores the 32 lane-range
//    totals; the task completing a request finds the token by inverse CDF at u_{b,K}
//    over piece totals, lane-range totals and at most one lane range of elements.
//  - Near-tie flags (optional output): the deciding warp marks accept tests within
//    1e-5 of their ratio and tests with p, q < 1e-30 among positions 0..j; the task
//    completing the terminal sample adds a sample within 1e-5 of a CDF bucket edge
//    and a residual of less than 1e-5 mass.
//  Every wait is bounded: waits for another warp's result by the call's wait limit,
//  waits for a copy to land by a fixed bound. The first wait to run out reports
//  SV_ERR_TIMEOUT in the status word and sets the call's abort word, which every other
//  wait checks; the warps let their copies in flight land and return, and the last
//  CTA clears the workspace (every ticket and published word) and the abort word.
#include <cfloat>
#include <climits>

#include "sv_common.cuh"

namespace sv {

enum : int { K_STREAM = 0, K_TERM = 1 };

// Near-tie flag bits of a request (the oracle's meaning): an accept test within 1e-5
// of its ratio, a terminal sample within 1e-5 (normalised) of a CDF bucket edge, p and
// q both below 1e-30 at a test, a residual with less than 1e-5 of mass, an invalid
// request.
enum : int { F_ACCEPT_TIE = 1, F_CDF_EDGE = 2, F_TINY_PROB = 4, F_SMALL_RESID = 8, F_INVALID = 16 };
constexpr float NEAR_TIE = 1e-5f;

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
  int last;           // stream piece: the warp's row segment ends here
  int xk;             // stream piece (T > 0): the drafted token of its row, or -1
  int tflags;         // terminal piece: near-tie flags of the request's decision
  Seg s0, s1;         // stream piece: s0; terminal piece: target (s0) and draft (s1)
  float Mt, iSt, Md, iSd;
};

struct Shared {
  SlotMeta meta[NSLOT];
  uint64_t full[NSLOT];
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
__device__ __forceinline__ float sm_logit(const float* p) { return *p; }
__device__ __forceinline__ float sm_logit(const uint16_t* p) {
  return __uint_as_float(static_cast<uint32_t>(*p) << 16);
}
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

__device__ __forceinline__ float ff_to_f(ff a) { return a.hi + a.lo; }

__device__ __forceinline__ ff shfl_xor_ff(ff x, int o) {
  return ff{__shfl_xor_sync(FULL, x.hi, o), __shfl_xor_sync(FULL, x.lo, o)};
}

__device__ __forceinline__ ff shfl_ff(ff x, int src) {
  return ff{__shfl_sync(FULL, x.hi, src), __shfl_sync(FULL, x.lo, src)};
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
__device__ __forceinline__ const T* tgt_row(const VerifyArgs& A, int b, int k) {
  return static_cast<const T*>(A.tgt) + ((size_t)b * (A.K + 1) + k) * A.V;
}
template <typename T>
__device__ __forceinline__ const T* drf_row(const VerifyArgs& A, int b, int k) {
  return static_cast<const T*>(A.drf) + ((size_t)b * A.K + k) * A.V;
}

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

// The call's abort word: set by the first wait that gives up, so that every other
// wait of the call returns at once; the last CTA resets it. (The status word only
// reports: a report left from an earlier call does not stop this one.)
__device__ __forceinline__ bool call_aborted(const VerifyArgs& A) {
  return *reinterpret_cast<volatile uint32_t*>(&A.hdr->abort) != 0;
}
__device__ void give_up(const VerifyArgs& A) {
  raise_status(A, ST_TIMEOUT);
  atomicExch(&A.hdr->abort, 1u);
}

// ---------------------------------------------------------------------------
// Fence-free publication. Results passed between warps (row partials, row
// statistics, drafted-token logits) are single 64-bit words written and read with
// relaxed GPU-scope accesses (single-copy atomic); a word is never 0 once written
// (its high half is stored bit-inverted and is the bits of a value >= 0 or of an
// index), so 0 means "not visible yet". The reader waits (bounded) for a non-zero
// word and resets it to 0 once consumed. Tickets are relaxed atomics. Nothing on the
// stream path then waits for a memory fence, which under full HBM load can take
// microseconds.
// ---------------------------------------------------------------------------
typedef unsigned long long u64;

__device__ __forceinline__ u64 enc_pair(float x, uint32_t y_bits) {
  return (static_cast<u64>(~y_bits) << 32) | __float_as_uint(x);
}
__device__ __forceinline__ float dec_x(u64 w) { return __uint_as_float(static_cast<uint32_t>(w)); }
__device__ __forceinline__ uint32_t dec_y(u64 w) { return ~static_cast<uint32_t>(w >> 32); }

__device__ __forceinline__ void st_word(u64* p, u64 v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ u64 ld_word(const u64* p) {
  u64 v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// A published word: waits (bounded) until it is visible, then resets the slot.
__device__ u64 take_word(const VerifyArgs& A, u64* p) {
  u64 w = ld_word(p);
  if (w == 0) {
    const long long t0 = clock64();
    while ((w = ld_word(p)) == 0) {
      if (call_aborted(A)) return 0;
      if (clock64() - t0 > A.wait_limit) {
        give_up(A);
        return 0;
      }
      __nanosleep(32);
    }
  }
  st_word(p, 0ull);
  return w;
}

// A published word that stays in place for several readers (job words): waits
// (bounded) until it is visible.
__device__ u64 wait_word(const VerifyArgs& A, const u64* p) {
  u64 w = ld_word(p);
  if (w == 0) {
    const long long t0 = clock64();
    while ((w = ld_word(p)) == 0) {
      if (call_aborted(A)) return 0;
      if (clock64() - t0 > A.wait_limit) {
        give_up(A);
        return 0;
      }
      __nanosleep(32);
    }
  }
  return w;
}

// Bounded wait on an mbarrier phase; false on abort or timeout.
__device__ bool wait_phase(uint64_t* bar, uint32_t parity, Shared& S, const VerifyArgs& A) {
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (*reinterpret_cast<volatile int*>(&S.abort_flag)) return false;
    if (clock64() - t0 > WAIT_CYCLES) {
      S.abort_flag = 1;
      give_up(A);
      return false;
    }
  }
  return true;
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
    if (A.out_flags) A.out_flags[b] = F_INVALID;
    raise_status(A, ST_DEVICE_INPUT);
    st_release(A.dec_flag + b, 2u);  // decided, no terminal sample
  }
}

// Ask L2 to fetch [p, p + bytes) ahead of its use: the 16-byte aligned interior, in
// pieces of up to 64 KB spread over the warp's lanes.
__device__ void prefetch_l2(const void* p, size_t bytes, int lane) {
  constexpr size_t CH = 65536;
  const uintptr_t a0 = (reinterpret_cast<uintptr_t>(p) + 15) & ~static_cast<uintptr_t>(15);
  const uintptr_t a1 = (reinterpret_cast<uintptr_t>(p) + bytes) & ~static_cast<uintptr_t>(15);
  if (a1 <= a0) return;
  const size_t n = a1 - a0;
  for (size_t off = (size_t)lane * CH; off < n; off += 32 * CH) {
    const uint32_t sz = static_cast<uint32_t>(n - off < CH ? n - off : CH);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a0 + off), "r"(sz) : "memory");
  }
}

// Decision for one request at T > 0 (one warp).
template <typename T>
__device__ void decide_sample(const VerifyArgs& A, int b, int L, int lane) {
  const int K = A.K, V = A.V;
  const size_t rb = (size_t)b * A.RS;
  float p = __int_as_float(0x7fc00000), q = p, MAt = 0.f, MAd = 0.f, iSt = 0.f, iSd = 0.f;
  int x = -1;
  bool ok = true, acc = false, tie = false, tiny = false;
  // Every load of the decision is issued up front. The drafted tokens' logits were
  // picked up while their rows streamed past.
  const float uK = __ldg(A.uni + (size_t)b * (K + 1) + K);
  float u = 0.f;
  if (lane < L) {
    x = __ldg(A.tok + (size_t)b * K + lane);
    u = __ldg(A.uni + (size_t)b * (K + 1) + lane);
  }
  u64* rsw = reinterpret_cast<u64*>(A.rowstat) + rb;
  u64* xzw = A.xz + rb;
  const u64 wL = take_word(A, rsw + L);
  const float2 sL = make_float2(dec_x(wL), __uint_as_float(dec_y(wL)));
  float2 st = make_float2(0.f, 0.f), sd = st;
  float zt = 0.f, zd = 0.f;
  if (lane < L) {
    const u64 w1 = take_word(A, rsw + lane), w2 = take_word(A, rsw + L + 1 + lane);
    st = make_float2(dec_x(w1), __uint_as_float(dec_y(w1)));
    sd = make_float2(dec_x(w2), __uint_as_float(dec_y(w2)));
    if (x >= 0 && x < V) {  // the stream stored these logits exactly when x is in range
      zt = dec_x(take_word(A, xzw + lane));
      zd = dec_x(take_word(A, xzw + L + 1 + lane));
    }
  }
  if (lane < L) {
    ok = x >= 0 && x < V && finitef(st.x) && finitef(sd.x) && st.y > 0.f && finitef(st.y) &&
         sd.y > 0.f && finitef(sd.y) && u >= 0.f && u < 1.f;
    if (ok) {
      MAt = __fmul_rn(st.x, A.a);
      MAd = __fmul_rn(sd.x, A.a);
      const float et = exp2_precise(zt, A.a, A.a_lo, MAt);
      const float ed = exp2_precise(zd, A.a, A.a_lo, MAd);
      p = __fdiv_rn(et, st.y);
      q = __fdiv_rn(ed, sd.y);
      iSt = __fdiv_rn(1.f, st.y);
      iSd = __fdiv_rn(1.f, sd.y);
      acc = u * q < p;
      const float ratio = q > 0.f ? fminf(__fdiv_rn(p, q), 1.f) : (p > 0.f ? 1.f : 0.f);
      tie = fabsf(u - ratio) < NEAR_TIE;
      tiny = p < 1e-30f && q < 1e-30f;
    }
  }
  const bool okL = finitef(sL.x) && sL.y > 0.f && finitef(sL.y) && uK >= 0.f && uK < 1.f;
  if (__any_sync(FULL, !ok) || !okL) {
    emit_invalid(A, b, lane);
    return;
  }
  const unsigned am = __ballot_sync(FULL, lane < L && acc);
  const unsigned lm = (L >= 32) ? FULL : ((1u << L) - 1u);
  const int j = ((am & lm) == lm) ? L : (__ffs(~am) - 1);
  // Near ties among the tests that were decisive (positions 0..j).
  const bool tested = lane < L && lane <= j;
  const int dflags = (__any_sync(FULL, tested && tie) ? F_ACCEPT_TIE : 0) |
                     (__any_sync(FULL, tested && tiny) ? F_TINY_PROB : 0);
  int32_t* ot = A.out_tok + (size_t)b * (K + 1);
  for (int k = lane; k <= K; k += 32)
    if (k != j) ot[k] = (k < j) ? x : -1;
  if (A.out_p && lane < K) A.out_p[(size_t)b * K + lane] = p;
  if (A.out_q && lane < K) A.out_q[(size_t)b * K + lane] = q;
  if (A.acc_cnt && lane < L && lane < j) atomicAdd(A.acc_cnt + lane, 1u);
  if (A.tst_cnt && lane < L && lane <= j) atomicAdd(A.tst_cnt + lane, 1u);
  // Terminal-sample job: a row's weights are taken in the frame its sum was formed
  // in, 2^(fl(z*a - fl(M*a))), so that weight * (1/S) is p (or q) directly.
  const float jMt = __shfl_sync(FULL, MAt, j & 31), jSt = __shfl_sync(FULL, iSt, j & 31);
  const float jMdd = __shfl_sync(FULL, MAd, j & 31), jSd = __shfl_sync(FULL, iSd, j & 31);
  if (lane == 0) {
    A.out_acc[b] = j;
    TermJob J;
    J.j = j;
    if (j == L) {  // every draft accepted: bonus sample from p_L
      J.kind = J_BONUS;
      J.MAt = __fmul_rn(sL.x, A.a);
      J.invSt = J.MAd = J.invSd = 0.f;
    } else {  // first rejection at j: residual sample
      J.kind = J_RESID;
      J.MAt = jMt;
      J.invSt = jSt;
      J.MAd = jMdd;
      J.invSd = jSd;
    }
    // The job's frames travel as two published words and its kind, row and near-tie
    // flags in the flag itself (1 | bonus << 2 | flags << 4 | (row + 1) << 8), so
    // neither side needs a fence.
    u64* jw = reinterpret_cast<u64*>(A.jobs + b);
    st_word(jw, enc_pair(J.MAt, __float_as_uint(J.invSt)));
    st_word(jw + 1, enc_pair(J.MAd, __float_as_uint(J.invSd)));
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(A.dec_flag + b),
                 "r"(1u | (J.kind == J_BONUS ? 4u : 0u) | (static_cast<uint32_t>(dflags) << 4) |
                     (static_cast<uint32_t>(j + 1) << 8))
                 : "memory");
  }
  // The terminal rows are read again shortly by the terminal tasks: start fetching
  // them into L2 now.
  prefetch_l2(static_cast<const T*>(A.tgt) + ((size_t)b * (K + 1) + j) * V, (size_t)V * sizeof(T),
              lane);
  if (j < L)
    prefetch_l2(static_cast<const T*>(A.drf) + ((size_t)b * K + j) * V, (size_t)V * sizeof(T), lane);
}

// Decision for one request at T == 0 (one warp): argmax matching.
__device__ void decide_greedy(const VerifyArgs& A, int b, int L, int lane) {
  const int K = A.K, V = A.V;
  const size_t rb = (size_t)b * A.RS;
  int x = -1, am = -1;
  bool ok = true;
  u64* rsw = reinterpret_cast<u64*>(A.rowstat) + rb;
  if (lane < L) {
    const u64 w = take_word(A, rsw + lane);
    x = __ldg(A.tok + (size_t)b * K + lane);
    am = static_cast<int>(dec_y(w));
    ok = finitef(dec_x(w)) && x >= 0 && x < V;
  }
  const u64 wL = take_word(A, rsw + L);
  const float2 sL = make_float2(dec_x(wL), __int_as_float(static_cast<int>(dec_y(wL))));
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
    if (A.out_flags) A.out_flags[b] = 0;
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

// Packed fp32x2 arithmetic: one instruction for a pair of values.
__device__ __forceinline__ float2 ffma2(float2 x, float2 y, float2 z) {
  float2 d;
  asm("{\n\t.reg .b64 rx, ry, rz, rd;\n\t"
      "mov.b64 rx, {%2, %3};\n\tmov.b64 ry, {%4, %5};\n\tmov.b64 rz, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, rx, ry, rz;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(x.x), "f"(x.y), "f"(y.x), "f"(y.y), "f"(z.x), "f"(z.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 x, float2 y) {
  float2 d;
  asm("{\n\t.reg .b64 rx, ry, rd;\n\t"
      "mov.b64 rx, {%2, %3};\n\tmov.b64 ry, {%4, %5};\n\t"
      "add.rn.f32x2 rd, rx, ry;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(x.x), "f"(x.y), "f"(y.x), "f"(y.y));
  return d;
}

// Sum of 2^(z*a - ma) over one uint4 of elements (8 bf16 / 4 fp32).
__device__ __forceinline__ float vec_expsum(uint4 v, float a, float nma, uint16_t) {
  const float2 aa = make_float2(a, a), cc = make_float2(nma, nma);
  const float2 y0 = ffma2(make_float2(bf_lo(v.x), bf_hi(v.x)), aa, cc);
  const float2 y1 = ffma2(make_float2(bf_lo(v.y), bf_hi(v.y)), aa, cc);
  const float2 y2 = ffma2(make_float2(bf_lo(v.z), bf_hi(v.z)), aa, cc);
  const float2 y3 = ffma2(make_float2(bf_lo(v.w), bf_hi(v.w)), aa, cc);
  const float2 e0 = make_float2(ex2(y0.x), ex2(y0.y)), e1 = make_float2(ex2(y1.x), ex2(y1.y));
  const float2 e2 = make_float2(ex2(y2.x), ex2(y2.y)), e3 = make_float2(ex2(y3.x), ex2(y3.y));
  const float2 s = fadd2(fadd2(e0, e1), fadd2(e2, e3));
  return s.x + s.y;
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
// neutral partials at p0+1..p1, then a ticket increment by the number of pieces.
// Lane 0 writes everything (fence-free: see take_word).
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
    u64* pr = reinterpret_cast<u64*>(A.part) + rowid * A.P;
    st_word(pr + sg.p0, enc_pair(v.x, __float_as_uint(v.y)));
    const u64 neutral = GREEDY ? enc_pair(-INFINITY, static_cast<uint32_t>(INT_MAX))
                               : enc_pair(-INFINITY, 0u);
    for (int q = sg.p0 + 1; q <= sg.p1; ++q) st_word(pr + q, neutral);
    pd.old = atomicAdd(A.t_row + rowid, (uint32_t)pd.count);
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
  const int b = pd.b;
  const size_t rowid = (size_t)b * A.RS + pd.r;
  u64* pr = reinterpret_cast<u64*>(A.part) + rowid * P;
  float2 rs;
  if (GREEDY) {
    float best = -INFINITY;
    int idx = INT_MAX;
    bool bad = false;
    for (int p = lane; p < P; p += 32) {
      const u64 w = take_word(A, pr + p);
      const float2 v = make_float2(dec_x(w), 0.f);
      const int vi = static_cast<int>(dec_y(w));
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
      const u64 w = take_word(A, pr + p);
      soft_merge(m, s, dec_x(w), __uint_as_float(dec_y(w)), A.a);
    }
    soft_warp(m, s, A.a, lane);
    rs = make_float2(m, s);
  }
  const int nrows = prefix[b + 1] - prefix[b];
  uint32_t o2 = 0;
  if (lane == 0) {
    st_word(reinterpret_cast<u64*>(A.rowstat) + rowid, enc_pair(rs.x, __float_as_uint(rs.y)));
    A.t_row[rowid] = 0;
    o2 = atomicAdd(A.t_req + b, 1u);
  }
  o2 = __shfl_sync(FULL, o2, 0);
  if (o2 != (uint32_t)(nrows - 1)) return;
  if (lane == 0) A.t_req[b] = 0;
  const int L = L_of_rows(nrows, GREEDY);
  if (GREEDY)
    decide_greedy(A, b, L, lane);
  else
    decide_sample<T>(A, b, L, lane);
}

// ---------------------------------------------------------------------------
// Terminal-sample weights.
// ---------------------------------------------------------------------------
// Weight of one element: residual max(0, p - q), or the unnormalised target weight
// 2^(z*a - MA) of a plain sample. MAt, MAd are the frames fl(M*a) the row sums were
// formed in, iSt, iSd the inverse row sums, so 2^(z*a - MA) * iS is the probability.
// A -inf logit (a masked token) gives 2^-inf = 0.
struct TermW {
  float a, MAt, iSt, MAd, iSd;
  bool resid;
  __device__ __forceinline__ float operator()(float zt, float zd) const {
    const float et = ex2(fmaf(zt, a, -MAt));
    if (!resid) return et;
    return fmaxf(fmaf(et, iSt, -(ex2(fmaf(zd, a, -MAd)) * iSd)), 0.f);
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


// ---------------------------------------------------------------------------
// Terminal sample (T > 0): residual max(0, p_j - q_j) at the first rejection j, or
// p_L when every draft was accepted, sampled by inverse CDF at u_{b,K}.
//
// A request's terminal rows are cut into R pieces of E2 elements (one task each);
// inside a piece, lane l covers one contiguous range of whole vectors. A task stores
// the piece's total (float-float) and its 32 lane-range totals; the task completing
// the request then finds the token in three levels (piece, lane range, element), so
// only one lane range (at most 64 elements) is evaluated again.
// ---------------------------------------------------------------------------

// Length of each lane's contiguous range in a terminal piece of n elements: a whole
// number of vectors, ceil(n / 32) rounded up to a vector.
template <typename T>
__device__ __forceinline__ int range_len(int n) {
  constexpr int VEC = ET<T>::VEC;
  return VEC * ((n + 32 * VEC - 1) / (32 * VEC));
}

// Sum of the weights of one vector as a balanced fp32 tree.
template <typename T>
__device__ __forceinline__ float vec_wsum(const uint4 vt, const uint4 vd, const TermW& W) {
  float w[ET<T>::VEC];
  vec_weights<T>(vt, vd, W, w);
  if constexpr (ET<T>::VEC == 8) {
    return ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
  } else {
    return (w[0] + w[1]) + (w[2] + w[3]);
  }
}

// Weight total of this lane's range of a terminal piece held in a slot (target row
// in the first half, draft row in the second), or read from global memory in direct
// mode. Compensated fp32.
template <typename T>
__device__ ff lane_range_sum(const SlotMeta& M, const TermW& W, const unsigned char* slot,
                             int lane) {
  constexpr int VEC = ET<T>::VEC;
  const int n = M.s0.n;
  const int ce = range_len<T>(n);
  const int lo = min(n, lane * ce), hi = min(n, lo + ce);
  float hs = 0.f, hc = 0.f;
  if (M.direct) {
    const T* t = reinterpret_cast<const T*>(M.s0.g);
    const T* d = reinterpret_cast<const T*>(M.s1.g);
    for (int e = lo; e < hi; ++e) two_sum(hs, hc, W(ld_logit(t + e), ld_logit(d + e)));
  } else {
    const uint4* t4 = reinterpret_cast<const uint4*>(slot);
    const uint4* d4 = reinterpret_cast<const uint4*>(W.resid ? slot + SLOT_BYTES / 2 : slot);
    const int v0 = lo / VEC, nvl = (hi - lo) / VEC;
    // Each lane starts at a different vector of its range, so that the lanes of one
    // shared-memory wavefront read distinct banks.
    if (nvl == 8) {  // every full piece of 8 KB slots
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int q = v0 + ((lane + i) & 7);
        two_sum(hs, hc, vec_wsum<T>(t4[q], d4[q], W));
      }
    } else {
      int q = nvl ? lane % nvl : 0;
      for (int i = 0; i < nvl; ++i) {
        two_sum(hs, hc, vec_wsum<T>(t4[v0 + q], d4[v0 + q], W));
        q = (q + 1 == nvl) ? 0 : q + 1;
      }
    }
  }
  return two_sum_ff(hs, hc);
}

// The same lane-range total read from global memory (whole-row fallback only).
template <typename T>
__device__ ff range_sum_global(const T* t, const T* d, int n, const TermW& W, int lane) {
  const int ce = range_len<T>(n);
  const int lo = min(n, lane * ce), hi = min(n, lo + ce);
  float hs = 0.f, hc = 0.f;
  for (int e = lo; e < hi; ++e) two_sum(hs, hc, W(ld_logit(t + e), ld_logit(d + e)));
  return two_sum_ff(hs, hc);
}

// A terminal task whose ticket value has not been inspected yet.
struct TermPend {
  int valid, b, j, jkind, tflags;
  float Mt, iSt, Md, iSd;
  uint32_t old;  // ticket value returned to lane 0
};

// Sum one terminal piece: lane-range totals staged in the (consumed) slot and
// written by lane 0 with the piece total. The ticket increment follows one slot later
// (term_ticket), when these stores have long completed and the release costs little.
template <typename T>
__device__ TermPend term_consume(const VerifyArgs& A, const SlotMeta& M, unsigned char* slot,
                                 int lane) {
  const TermW W{A.a, M.Mt, M.iSt, M.Md, M.iSd, M.jkind == J_RESID};
  const ff mine = lane_range_sum<T>(M, W, slot, lane);
  const ff tot = warp_sum_ff(mine);
  float* stage = reinterpret_cast<float*>(slot);
  __syncwarp();  // every lane has finished reading the slot
  stage[lane] = mine.hi;
  // Order the staging write before the async-proxy write of the slot's next copy.
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
  TermPend pt;
  pt.valid = 1;
  pt.b = M.b;
  pt.j = M.r;
  pt.jkind = M.jkind;
  pt.tflags = M.tflags;
  pt.Mt = M.Mt;
  pt.iSt = M.iSt;
  pt.Md = M.Md;
  pt.iSd = M.iSd;
  pt.old = 0;
  if (lane == 0) {
    const size_t pid = (size_t)M.b * A.Rmax + M.p;
    float4* dst = reinterpret_cast<float4*>(A.lsum + pid * 32);
    const float4* src = reinterpret_cast<const float4*>(stage);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = src[i];
    A.rpart[pid] = make_float2(tot.hi, tot.lo);
  }
  return pt;
}

// Release-ordered ticket increment for a summed terminal piece (lane 0); its value is
// inspected by term_settle a slot later.
__device__ __forceinline__ void term_ticket(const VerifyArgs& A, TermPend& pt, int lane) {
  if (lane == 0) pt.old = atom_add_release(A.t_res + pt.b, 1u);
}

// ---------------------------------------------------------------------------
// Locating the terminal token (inverse CDF at u_{b,K}).
// ---------------------------------------------------------------------------
struct Located {
  int y;
  float gap;  // distance of the target to the nearest edge of y's bucket, over Z
};

// Element level: the first element e in [r0, r1) of rows t, d with t3 < cumulative
// weight from r0 (or the last positive element when `past`, or when rounding leaves
// t3 beyond the range's total). Each lane takes up to EPL consecutive elements and
// keeps their weights in registers.
template <typename T>
__device__ Located locate_elems(const T* t, const T* d, int r0, int r1, ff t3, bool past, ff Z,
                                const TermW& W, int lane) {
  constexpr int VEC = ET<T>::VEC;
  constexpr int E2 = SLOT_BYTES / 2 / (int)sizeof(T);
  constexpr int EPL = (VEC * ((E2 + 32 * VEC - 1) / (32 * VEC)) + 31) / 32;
  static_assert(EPL >= 1 && EPL <= 4, "lane ranges of at most 128 elements");
  const int e0 = min(r1, r0 + lane * EPL);
  float w[EPL];
  float hs = 0.f, hc = 0.f;
  int lastpos = -1;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    w[i] = (e0 + i < r1) ? W(ld_logit(t + e0 + i), ld_logit(d + e0 + i)) : 0.f;
    two_sum(hs, hc, w[i]);
    if (w[i] > 0.f) lastpos = e0 + i;
  }
  const ff ls = two_sum_ff(hs, hc);
  const ff incl = warp_incl_scan_ff(ls, lane);
  Located r{-1, 0.f};
  const unsigned hit = past ? 0u : __ballot_sync(FULL, ff_lt(t3, incl));
  if (hit) {
    const int ln = __ffs(hit) - 1;
    float gap = 0.f;
    if (lane == ln) {
      ff cum = ff_add(incl, ff_neg(ls));
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const ff nc = ff_add(cum, ff{w[i], 0.f});
        if (r.y < 0 && e0 + i < r1 && ff_lt(t3, nc)) {
          r.y = e0 + i;
          const float glo = ff_to_f(ff_add(t3, ff_neg(cum)));
          const float ghi = ff_to_f(ff_add(nc, ff_neg(t3)));
          gap = fminf(glo, ghi) / ff_to_f(Z);
        }
        cum = nc;
      }
      if (r.y < 0) r.y = lastpos;
    }
    r.y = __shfl_sync(FULL, r.y, ln);
    r.gap = __shfl_sync(FULL, gap, ln);
  }
  if (r.y < 0) {
    const unsigned has = __ballot_sync(FULL, lastpos >= 0);
    r.y = has ? __shfl_sync(FULL, lastpos, 31 - __clz(has)) : r0;
    r.gap = 0.f;
  }
  return r;
}

// Lane-range and element levels inside piece `pstar` of rows trow, drow, given each
// lane's range total `lsv` and the target t2 relative to the piece start.
template <typename T>
__device__ Located locate_in_piece(const VerifyArgs& A, const T* trow, const T* drow, int pstar,
                                   float lsv, ff t2, bool past, ff Z, const TermW& W, int lane) {
  const ff mine{lsv, 0.f};
  const ff incl = warp_incl_scan_ff(mine, lane);
  int lstar;
  ff t3{0.f, 0.f};
  const unsigned hit = past ? 0u : __ballot_sync(FULL, ff_lt(t2, incl));
  if (hit) {
    lstar = __ffs(hit) - 1;
    const ff ex = ff_add(incl, ff_neg(mine));
    t3 = ff_add(t2, ff_neg(shfl_ff(ex, lstar)));
  } else {
    const unsigned has = __ballot_sync(FULL, lsv > 0.f);
    lstar = has ? 31 - __clz(has) : 0;
    past = true;
  }
  const int e0 = pstar * A.E2;
  const int n = min(A.E2, A.V - e0);
  const int ce = range_len<T>(n);
  const int r0 = min(n, lstar * ce), r1 = min(n, r0 + ce);
  Located r = locate_elems<T>(trow + e0, drow + e0, r0, r1, t3, past, Z, W, lane);
  r.y += e0;
  return r;
}

// No residual mass left (p == q up to rounding): sample p_j itself instead, its piece
// totals computed here, piece by piece.
template <typename T>
__device__ Located locate_whole_row(const VerifyArgs& A, const T* trow, float uK, TermW W,
                                    int lane) {
  W.resid = false;
  const int R = A.R;
  ff Z{0.f, 0.f};
  for (int p = 0; p < R; ++p) {
    const int e0 = p * A.E2;
    Z = ff_add(Z, warp_sum_ff(range_sum_global<T>(trow + e0, trow + e0, min(A.E2, A.V - e0), W,
                                                  lane)));
  }
  const ff target = ff_mul_f(Z, uK);
  ff base{0.f, 0.f};
  int pstar = R - 1;
  bool past = true;
  float lsv = 0.f;
  for (int p = 0; p < R; ++p) {
    const int e0 = p * A.E2;
    const ff mine = range_sum_global<T>(trow + e0, trow + e0, min(A.E2, A.V - e0), W, lane);
    const ff nb = ff_add(base, warp_sum_ff(mine));
    lsv = mine.hi;
    if (ff_lt(target, nb)) {
      pstar = p;
      past = false;
      break;
    }
    base = nb;
  }
  return locate_in_piece<T>(A, trow, trow, pstar, lsv, ff_add(target, ff_neg(base)), past, Z, W,
                            lane);
}

// Locate the terminal token of request b (row j) from its piece and lane-range totals
// (whole warp). Also reports the residual's mass through `Zout` (residual jobs).
template <typename T>
__device__ Located term_locate(const VerifyArgs& A, int b, int j, const TermW& W, float& Zout,
                               int lane) {
  const int R = A.R, K = A.K;
  const T* trow = tgt_row<T>(A, b, j);
  const T* drow = W.resid ? drf_row<T>(A, b, j) : trow;
  const float uK = __ldg(A.uni + (size_t)b * (K + 1) + K);
  const float2* rp = A.rpart + (size_t)b * A.Rmax;
  const int c = (R + 31) / 32;
  const int p0 = min(R, lane * c), p1 = min(R, p0 + c);
  constexpr int CREG = 4;  // piece totals a lane keeps in registers (R <= 128)
  float2 wr[CREG];
  ff ls{0.f, 0.f};
  int lastpos = -1;
  if (c <= CREG) {
#pragma unroll
    for (int i = 0; i < CREG; ++i)
      wr[i] = (p0 + i < p1) ? __ldcg(rp + p0 + i) : make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < CREG; ++i) {
      ls = ff_add(ls, ff{wr[i].x, wr[i].y});
      if (wr[i].x > 0.f) lastpos = p0 + i;
    }
  } else {
    for (int p = p0; p < p1; ++p) {
      const float2 w = __ldcg(rp + p);
      ls = ff_add(ls, ff{w.x, w.y});
      if (w.x > 0.f) lastpos = p;
    }
  }
  const ff incl = warp_incl_scan_ff(ls, lane);
  const ff Z = shfl_ff(incl, 31);
  Zout = ff_to_f(Z);
  if (W.resid && !(Z.hi > 0.f && Z.hi <= 3.402823466e38f))
    return locate_whole_row<T>(A, trow, uK, W, lane);
  const ff target = ff_mul_f(Z, uK);
  // Piece level.
  int pstar = -1;
  bool past = false;
  ff base{0.f, 0.f};
  const unsigned hit = __ballot_sync(FULL, ff_lt(target, incl));
  if (hit) {
    const int ln = __ffs(hit) - 1;
    if (lane == ln) {
      ff cum = ff_add(incl, ff_neg(ls));
      if (c <= CREG) {
#pragma unroll
        for (int i = 0; i < CREG; ++i) {
          if (pstar < 0 && p0 + i < p1) {
            const ff nc = ff_add(cum, ff{wr[i].x, wr[i].y});
            if (ff_lt(target, nc))
              pstar = p0 + i;
            else
              cum = nc;
          }
        }
      } else {
        for (int p = p0; p < p1; ++p) {
          const float2 w = __ldcg(rp + p);
          const ff nc = ff_add(cum, ff{w.x, w.y});
          if (ff_lt(target, nc)) {
            pstar = p;
            break;
          }
          cum = nc;
        }
      }
      if (pstar < 0) {
        pstar = lastpos;
        past = true;
      }
      base = cum;
    }
    pstar = __shfl_sync(FULL, pstar, ln);
    past = __shfl_sync(FULL, (int)past, ln) != 0;
    base = shfl_ff(base, ln);
  }
  if (pstar < 0) {  // rounding put the target past the last piece
    const unsigned has = __ballot_sync(FULL, lastpos >= 0);
    pstar = has ? __shfl_sync(FULL, lastpos, 31 - __clz(has)) : 0;
    past = true;
  }
  const float lsv = __ldcg(A.lsum + ((size_t)b * A.Rmax + pstar) * 32 + lane);
  const ff t2 = past ? ff{0.f, 0.f} : ff_add(target, ff_neg(base));
  return locate_in_piece<T>(A, trow, drow, pstar, lsv, t2, past, Z, W, lane);
}

// Inspect a terminal ticket: the task completing its request locates the token.
template <typename T>
__device__ void term_settle(const VerifyArgs& A, const TermPend& pt, int lane) {
  const uint32_t old = __shfl_sync(FULL, pt.old, 0);
  if (old != (uint32_t)(A.R - 1)) return;
  fence_acq_rel();
  if (lane == 0) A.t_res[pt.b] = 0;
  const TermW W{A.a, pt.Mt, pt.iSt, pt.Md, pt.iSd, pt.jkind == J_RESID};
  float Z = 0.f;
  const Located r = term_locate<T>(A, pt.b, pt.j, W, Z, lane);
  if (lane == 0) {
    A.out_tok[(size_t)pt.b * (A.K + 1) + pt.j] = r.y;
    if (A.out_flags) {
      int f = pt.tflags;
      if (r.gap < NEAR_TIE) f |= F_CDF_EDGE;
      if (W.resid && Z < NEAR_TIE) f |= F_SMALL_RESID;
      A.out_flags[pt.b] = f;
    }
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Per-warp work. Stream: the work list (every active row of the batch, request-major,
// cut into pieces) is split into equal contiguous ranges, one per warp of the grid.
// Terminal tasks (T > 0), request-major, likewise; a warp takes them up once its
// stream range is done, each as soon as its request is decided.
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
  while (lo < hi) {  // last request whose first row is <= g
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

// Next stream piece of the warp's range into a slot (lane 0 only); false at the end.
template <typename T, bool GREEDY>
__device__ bool issue_stream(const VerifyArgs& A, Cursor& c, const int* prefix, SlotMeta& meta,
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
  const int kpos0 = (c.cr <= c.cL) ? c.cr : c.cr - c.cL - 1;
  meta.xk = -1;
  if (!GREEDY) {
    const int k = (c.cr <= c.cL) ? c.cr : c.cr - c.cL - 1;  // target row k or draft row k
    if (k < c.cL) meta.xk = __ldg(A.tok + (size_t)c.cb * A.K + k);
  }
  ++c.cur;
  // The warp's segment of this row ends at the row's last piece or the range's end.
  meta.last = (c.cp == P - 1 || c.cur == c.end) ? 1 : 0;
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
    // Rows of the first two positions of a request are the likeliest terminal rows
    // (read again after the decision): ask L2 to keep them; the rest is read once.
    const uint64_t pol = (!GREEDY && kpos0 <= 1) ? policy_evict_last() : policy_evict_first();
    bulk_g2s_hint(slot, meta.s0.g + meta.s0.head * eb, tx, full, pol);
  } else {
    mbar_arrive(full);
  }
  return true;
}

// Terminal task (request b, piece p) into a slot (lane 0 only; the request's job is
// published).
template <typename T>
__device__ void issue_term(const VerifyArgs& A, int b, int p, const TermJob& J, SlotMeta& meta,
                           uint64_t* full, unsigned char* slot) {
  constexpr int eb = sizeof(T);
  const int K = A.K;
  const int kind = J.kind, j = J.j;
  const int e0 = p * A.E2;
  const int n = min(A.E2, A.V - e0);
  const T* tr = static_cast<const T*>(A.tgt) + ((size_t)b * (K + 1) + j) * A.V + e0;
  meta.kind = K_TERM;
  meta.jkind = kind;
  meta.b = b;
  meta.r = j;
  meta.p = p;
  meta.e0 = e0;
  meta.Mt = J.MAt;
  meta.iSt = J.invSt;
  meta.Md = J.MAd;
  meta.iSd = J.invSd;
  meta.tflags = J.flags;
  meta.s0 = make_seg(reinterpret_cast<const unsigned char*>(tr), n, eb);
  bool whole = meta.s0.head == 0 && meta.s0.body == n;
  if (kind == J_RESID) {
    const T* dr = static_cast<const T*>(A.drf) + ((size_t)b * K + j) * A.V + e0;
    meta.s1 = make_seg(reinterpret_cast<const unsigned char*>(dr), n, eb);
    whole = whole && meta.s1.head == 0 && meta.s1.body == n;
  } else {
    meta.s1 = meta.s0;
  }
  // Rows that are not 16-byte aligned whole multiples of 16 bytes are read straight
  // from global memory.
  meta.direct = !whole;
  if (whole) {
    const uint32_t bytes = (uint32_t)(n * eb);
    mbar_arrive_expect_tx(full, (kind == J_RESID ? 2u : 1u) * bytes);
    const uint64_t pol = policy_evict_first();
    bulk_g2s_hint(slot, meta.s0.g, bytes, full, pol);
    if (kind == J_RESID) bulk_g2s_hint(slot + SLOT_BYTES / 2, meta.s1.g, bytes, full, pol);
  } else {
    mbar_arrive(full);
  }
}

enum : int { SLOT_EMPTY = 0, SLOT_FULL = 1, SLOT_DEFERRED = 2 };

// Per-warp issue state (meaningful in lane 0).
struct Issuer {
  Cursor c;
  long long nw;      // warps in the grid
  long long tt, te;  // this warp's terminal tasks still to issue: [tt, te)
  uint32_t pf;       // decision flag of task tt's request, loaded earlier
  int pacq;          // pf came from an acquire load (no fence needed before the job)
  int jb;            // request whose job record J holds (-1: none)
  TermJob J;
};

// Refill a slot (lane 0): the next stream piece while the warp's range lasts, then
// its terminal tasks, each once its request is decided. Returns SLOT_FULL, SLOT_EMPTY
// (nothing left at all), or SLOT_DEFERRED (only terminal tasks of undecided requests
// are left). `fresh`: read the decision flag now instead of using the prefetched one.
template <typename T, bool GREEDY>
__device__ int refill(const VerifyArgs& A, Issuer& I, const int* prefix, bool fresh,
                      SlotMeta& meta, uint64_t* full, unsigned char* slot) {
  if (issue_stream<T, GREEDY>(A, I.c, prefix, meta, full, slot)) return SLOT_FULL;
  if (!GREEDY) {
    bool acq = I.pacq;  // I.pf was read with acquire semantics
    I.pacq = 0;
    while (I.tt < I.te) {
      const int b = static_cast<int>(I.tt / A.R);
      if (b != I.jb) {  // first task of this request: its flag, then its job record
        uint32_t f = I.pf;
        if (fresh) {
          f = ld_relaxed(A.dec_flag + b);
          acq = false;
        }
        if (f == 0) break;
        fresh = true;  // a later request's flag has not been read yet
        if ((f & 3u) != 1u) {  // the request has no terminal sample: skip its tasks
          I.tt = min(I.te, (long long)(b + 1) * A.R);
          continue;
        }
        (void)acq;
        const u64* jw = reinterpret_cast<const u64*>(A.jobs + b);
        const u64 w1 = wait_word(A, jw), w2 = wait_word(A, jw + 1);
        I.J.kind = (f & 4u) ? J_BONUS : J_RESID;
        I.J.flags = static_cast<int>((f >> 4) & 15u);
        I.J.j = static_cast<int>(f >> 8) - 1;
        I.J.MAt = dec_x(w1);
        I.J.invSt = __uint_as_float(dec_y(w1));
        I.J.MAd = dec_x(w2);
        I.J.invSd = __uint_as_float(dec_y(w2));
        I.jb = b;
      }
      issue_term<T>(A, b, static_cast<int>(I.tt - (long long)b * A.R), I.J, meta, full, slot);
      ++I.tt;
      I.pf = 0;
      return SLOT_FULL;
    }
  }
  return (!GREEDY && I.tt < I.te) ? SLOT_DEFERRED : SLOT_EMPTY;
}

// A refill that found nothing at all left: slots waiting for a terminal task have
// nothing to wait for either.
__device__ __forceinline__ void drop_deferred(int* st, int h) {
  if (h != SLOT_EMPTY) return;
#pragma unroll
  for (int q = 0; q < SLOTS_PER_WARP; ++q)
    if (st[q] == SLOT_DEFERRED) st[q] = SLOT_EMPTY;
}

// Bounded wait until the request of terminal task tt is decided (lane 0).
// On success I.pf holds the flag, read with acquire semantics.
__device__ bool wait_decided(const VerifyArgs& A, Shared& S, Issuer& I) {
  if (I.tt >= I.te) return true;
  const int b = static_cast<int>(I.tt / A.R);
  const long long t0 = clock64();
  // Every idle warp of the grid may be polling: back off between polls so that the
  // flags' and the status word's cache lines stay free for the warps still working.
  uint32_t f;
  for (unsigned it = 1; (f = ld_relaxed(A.dec_flag + b)) == 0; ++it) {
    __nanosleep(256);
    if ((it & 15) != 0) continue;
    if (*reinterpret_cast<volatile int*>(&S.abort_flag)) return false;
    if (call_aborted(A)) {
      S.abort_flag = 1;
      return false;
    }
    if (clock64() - t0 > A.wait_limit) {
      S.abort_flag = 1;
      give_up(A);
      return false;
    }
  }
  I.pf = f;
  I.pacq = 1;
  return true;
}

// One warp: its stream range and then its terminal tasks through SLOTS_PER_WARP
// slots; each slot is refilled right after the warp has consumed it.
template <typename T, bool GREEDY>
__device__ void warp_loop(const VerifyArgs& A, Shared& S, unsigned char* slots, const int* prefix,
                          int w, int lane) {
  Issuer I;
  I.nw = (long long)gridDim.x * NCW;
  const long long gw = (long long)blockIdx.x * NCW + w;
  {
    // Terminal tasks (b, p) in request-major order, an equal contiguous share per
    // warp: a warp's tasks mostly belong to one request, whose job it reads once.
    const long long NT = GREEDY ? 0 : (long long)A.B * A.R;
    I.tt = NT * gw / I.nw;
    I.te = NT * (gw + 1) / I.nw;
  }
  I.pf = 0;
  I.pacq = 0;
  I.jb = -1;
  {
    const unsigned long long total =
        static_cast<unsigned long long>(S.total_rows) * static_cast<unsigned long long>(A.P);
    const unsigned long long nw = I.nw, g = gw;
    if (lane == 0) cursor_init<GREEDY>(I.c, A, prefix, total * g / nw, total * (g + 1) / nw);
  }
  int st[SLOTS_PER_WARP];
  uint32_t cons[SLOTS_PER_WARP];
#pragma unroll
  for (int q = 0; q < SLOTS_PER_WARP; ++q) {
    const int s = SLOTS_PER_WARP * w + q;
    int h = 0;
    if (lane == 0)
      h = refill<T, GREEDY>(A, I, prefix, true, S.meta[s], &S.full[s],
                            slots + (size_t)s * SLOT_BYTES);
    st[q] = __shfl_sync(FULL, h, 0);
    cons[q] = 0;
  }
  Pending pd;
  pd.valid = 0;
  TermPend pti, pts;  // terminal pieces summed (ticket not taken yet) / ticket taken
  pti.valid = 0;
  pts.valid = 0;
  Segment sg;
  sg.valid = 0;
  LaneState ls;
  lane_reset(ls);
  if (GREEDY) ls.s = __int_as_float(INT_MAX);
  int k = 0;
  bool aborted = false;
  while (true) {
    const int s = SLOTS_PER_WARP * w + k;
    unsigned char* slot = slots + (size_t)s * SLOT_BYTES;
    if (!GREEDY && st[k] == SLOT_DEFERRED) {  // retry a refill that had to wait
      int h = 0;
      if (lane == 0)
        h = refill<T, GREEDY>(A, I, prefix, !I.pacq, S.meta[s], &S.full[s], slot);
      st[k] = __shfl_sync(FULL, h, 0);
      drop_deferred(st, st[k]);
    }
    if (st[k] == SLOT_FULL) {
      const bool ok = wait_phase(&S.full[s], cons[k] & 1, S, A);
      if (!__all_sync(FULL, ok)) {
        aborted = true;
        break;
      }
      ++cons[k];
      st[k] = SLOT_EMPTY;
      if (pd.valid) {  // the previous segment's ticket has had a whole wait to come back
        settle<T, GREEDY>(A, pd, prefix, lane);
        pd.valid = 0;
      }
      if (!GREEDY && pts.valid) {
        term_settle<T>(A, pts, lane);
        pts.valid = 0;
      }
      if (!GREEDY && pti.valid) {
        pts = pti;
        term_ticket(A, pts, lane);
        pti.valid = 0;
      }
      // Once the stream range is done, prefetch the decision flag the next refill
      // will look at.
      if (!GREEDY && lane == 0 && I.c.cur >= I.c.end && I.tt < I.te &&
          I.tt / A.R != I.jb) {
        I.pf = ld_relaxed(A.dec_flag + I.tt / A.R);
        I.pacq = 0;
      }
      const SlotMeta M = S.meta[s];
      if (GREEDY || M.kind == K_STREAM) {
        if (!(sg.valid && sg.b == M.b && sg.r == M.r)) {  // a new row segment starts here
          sg.valid = 1;
          sg.b = M.b;
          sg.r = M.r;
          sg.p0 = M.p;
          lane_reset(ls);
          if (GREEDY) ls.s = __int_as_float(INT_MAX);
        }
        sg.p1 = M.p;
        fold_piece<T, GREEDY>(ls, A, M, slot, lane);
        if (!GREEDY && lane == 0 && M.xk >= M.e0 && M.xk < M.e0 + M.s0.n) {
          // This piece holds the row's drafted token: keep its logit for the decision.
          const int off = M.xk - M.e0;
          const T* g = reinterpret_cast<const T*>(M.s0.g);
          const float z = (off >= M.s0.head && off < M.s0.head + M.s0.body)
                              ? sm_logit(reinterpret_cast<const T*>(slot) + (off - M.s0.head))
                              : ld_logit(g + off);
          st_word(A.xz + (size_t)M.b * A.RS + M.r, enc_pair(z, 0u));
        }
      } else {
        pti = term_consume<T>(A, M, slot, lane);
      }
      __syncwarp();
      int h = 0;
      if (lane == 0) {
        // The slot's shared-memory accesses are done; order them before the
        // async-proxy write of the next copy into the same slot.
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        h = refill<T, GREEDY>(A, I, prefix, false, S.meta[s], &S.full[s], slot);
      }
      st[k] = __shfl_sync(FULL, h, 0);
      drop_deferred(st, st[k]);
      if ((GREEDY || M.kind == K_STREAM) && M.last) {
        if (pd.valid) {
          settle<T, GREEDY>(A, pd, prefix, lane);
          pd.valid = 0;
        }
        pd = publish<GREEDY>(A, sg, ls, lane);
        sg.valid = 0;
      }
      k = (k + 1 == SLOTS_PER_WARP) ? 0 : k + 1;
      continue;
    }
    // Slot k has nothing to consume: move on to a slot that has.
    bool any_full = false, any_def = false;
#pragma unroll
    for (int q = 0; q < SLOTS_PER_WARP; ++q) {
      any_full |= st[q] == SLOT_FULL;
      any_def |= st[q] == SLOT_DEFERRED;
    }
    if (any_full) {
      k = (k + 1 == SLOTS_PER_WARP) ? 0 : k + 1;
      continue;
    }
    if (GREEDY || !any_def) break;
    // Only terminal tasks of undecided requests are left. Settle the pending tickets
    // first (the awaited decision may be one this warp owes), then wait for it.
    if (pd.valid) {
      settle<T, GREEDY>(A, pd, prefix, lane);
      pd.valid = 0;
    }
    if (pts.valid) {
      term_settle<T>(A, pts, lane);
      pts.valid = 0;
    }
    if (pti.valid) {
      term_ticket(A, pti, lane);
      term_settle<T>(A, pti, lane);
      pti.valid = 0;
    }
    int ok = 1;
    if (lane == 0) ok = wait_decided(A, S, I);
    if (!__shfl_sync(FULL, ok, 0)) {
      aborted = true;
      break;
    }
    while (st[k] != SLOT_DEFERRED) k = (k + 1 == SLOTS_PER_WARP) ? 0 : k + 1;
  }
  if (pd.valid) settle<T, GREEDY>(A, pd, prefix, lane);
  if (!GREEDY && pts.valid) term_settle<T>(A, pts, lane);
  if (!GREEDY && pti.valid) {
    term_ticket(A, pti, lane);
    term_settle<T>(A, pti, lane);
  }
  if (aborted) {
    // Let this warp's copies in flight land before the CTA may exit.
    for (int q = 0; q < SLOTS_PER_WARP; ++q) {
      if (st[q] != SLOT_FULL) continue;
      const long long t0 = clock64();
      while (!mbar_test(&S.full[SLOTS_PER_WARP * w + q], cons[q] & 1) &&
             clock64() - t0 < WAIT_CYCLES) {
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

  warp_loop<T, GREEDY>(A, S, slots, prefix, warp, lane);
  __syncthreads();

  // The last CTA to finish resets the CTA counter and the decision flags (and, after
  // an abort, every ticket) so the workspace is ready for the next call.
  if (tid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(&A.hdr->cta_done, 1u);
    S.last_cta = (old == gridDim.x - 1);
  }
  __syncthreads();
  if (S.last_cta) {
    __threadfence();
    const bool dirty = call_aborted(A);
    if (dirty) {
      // An aborted call can leave published words behind: clear them all.
      const size_t nrow = (size_t)B * A.RS;
      u64* pw = reinterpret_cast<u64*>(A.part);
      for (size_t i = tid; i < nrow * A.P; i += NTHREADS) pw[i] = 0ull;
      for (size_t i = tid; i < nrow; i += NTHREADS) {
        reinterpret_cast<u64*>(A.rowstat)[i] = 0ull;
        A.xz[i] = 0ull;
      }
      for (size_t i = tid; i < TICKET_ROW_WORDS; i += NTHREADS) A.t_row[i] = 0;
      for (int i = tid; i < SV_MAX_B; i += NTHREADS) {
        A.t_req[i] = 0;
        A.t_res[i] = 0;
      }
    }
    for (int i = tid; i < B; i += NTHREADS) {
      A.dec_flag[i] = 0;
      reinterpret_cast<u64*>(A.jobs + i)[0] = 0ull;
      reinterpret_cast<u64*>(A.jobs + i)[1] = 0ull;
    }
    __syncthreads();
    if (tid == 0) {
      A.hdr->abort = 0;
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
  // At T > 0 warps wait for decisions made in other CTAs: a cooperative launch
  // guarantees that all the CTAs (at most one per SM) are resident together.
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
