// sv_schedule.cu -- GPU-resident confidence schedule (sm_103a).
//
// Computes per-request verify lengths from per-position draft confidences, on the
// device, in one small launch (DSpark Deep Dive, "GPU-Resident Scheduling": the
// scheduling decision is a CUDA kernel that reads the confidence scores and writes a
// verification length per request, with no CPU round trip).
//
//  1. S_{b,k} = c_{b,0} * ... * c_{b,k} in float64, left to right (DSpark Guide,
//     "2. Confidence-Scheduled Dynamic Verification": prefix survival C_k).
//  2. L0_b = max(1, #{k : S_{b,k} >= tau}) (truncate at the first C_k < tau, keep at
//     least one token; DSpark Guide sketch, DSpark Deep Dive "Variable-Length Drafts").
//  3. If sum L0 > budget: keep the budget best positions (floor positions first when
//     budget >= B; then S descending, k ascending, b ascending), found by an MSB-first
//     radix select on the 64-bit patterns of S (order-preserving for S >= 0) and a
//     k-major prefix count that ranks positions tied with the threshold
//     (DSpark Deep Dive, "The Optimization Logic").
//  0. Optional prologue: sequential temperature scaling of each confidence,
//     c' = sigmoid(logit(c) / T_k) with one temperature per draft position (DSpark
//     Deep Dive, "Sequential Temperature Scaling"), in fp32; and the load-aware
//     threshold tau = tau_min + (tau_max - tau_min) * LF^2, LF = 0.6 Q/Q_max +
//     0.4 M/M_max clamped to 1 (DSpark Guide, "Dynamic Verification Scheduling
//     Algorithm"), in fp64 from the device-resident load state.
// One CTA of 1024 threads; everything lives in shared memory.
#include "sv_common.cuh"
#include "sv_launch.cuh"

namespace sv {

constexpr int SCHED_THREADS = 1024;

struct ScheduleArgs {
  const float* conf;
  const float* temps;  // [K] or nullptr: no calibration
  const float* load;   // [4] {Q, Q_max, M_gpu, M_max} or nullptr: tau as given
  const float* curve;  // [2 * n_pts] tokens then tokens/s, or nullptr: budget as given
  int n_pts;
  int32_t* n_out;      // [1] or nullptr: the budget the curve chose
  double* g_out;       // [1] or nullptr: its goodput
  int B, K;
  float tau, tau_min, tau_max;
  int budget;
  int32_t* out_len;
  float* conf_cal;     // [B,K] or nullptr
  double* tau_out;     // [1] or nullptr
  WsHeader* hdr;
};

// sigmoid(logit(c) / T) in fp32; the end points stay fixed. logit(c) is taken as the
// log of one rounded ratio c / (1 - c): near c = 1/2 this avoids the cancellation of
// log(c) - log(1 - c), and elsewhere the error is that of logf itself (an absolute
// error of a few ulps of |logit c|, scaled by (1 - c') / T in c').
__device__ __forceinline__ float calibrate(float c, float T) {
  if (c <= 0.f) return 0.f;
  if (c >= 1.f) return 1.f;
  const float z = __fdiv_rn(logf(__fdiv_rn(c, __fsub_rn(1.f, c))), T);
  return __fdiv_rn(1.f, __fadd_rn(1.f, expf(-z)));
}

// The throughput curve at x tokens (fp64, each step rounded once): linear between its
// points, flat beyond the first and the last.
// x is a whole number of tokens below 2^24, exact in fp32, so the segment is found
// with fp32 compares; only the interpolation runs on the (slow) fp64 pipe.
__device__ double curve_at(const float* cx, const float* cy, int n, double x) {
  const float xf = static_cast<float>(x);
  if (xf <= cx[0]) return cy[0];
  for (int i = 1; i < n; ++i) {
    if (xf <= cx[i]) {
      const double x0 = cx[i - 1], x1 = cx[i], y0 = cy[i - 1], y1 = cy[i];
      return __dadd_rn(y0, __dmul_rn(__dsub_rn(y1, y0), __ddiv_rn(__dsub_rn(x, x0), __dsub_rn(x1, x0))));
    }
  }
  return cy[n - 1];
}

// Load-aware threshold in fp64 (no contraction: each step rounds once). Returns a
// negative value for an invalid load state.
__device__ double load_tau(const float* load, double tau_min, double tau_max) {
  const double Q = load[0], Qm = load[1], M = load[2], Mm = load[3];
  if (!(isfinite(Q) && isfinite(Qm) && isfinite(M) && isfinite(Mm))) return -1.0;
  if (Q < 0.0 || M < 0.0 || !(Qm > 0.0) || !(Mm > 0.0)) return -1.0;
  double lf = __dadd_rn(__dmul_rn(0.6, __ddiv_rn(Q, Qm)), __dmul_rn(0.4, __ddiv_rn(M, Mm)));
  if (lf > 1.0) lf = 1.0;
  return __dadd_rn(tau_min, __dmul_rn(__dsub_rn(tau_max, tau_min), __dmul_rn(lf, lf)));
}

__device__ __forceinline__ unsigned long long surv_key(double s) {
  return static_cast<unsigned long long>(__double_as_longlong(s == 0.0 ? 0.0 : s));
}

// Throughput-curve budget (DSpark Deep Dive, "The Throughput Curve", "The Optimization
// Logic"): the smallest N in [N_lo, N_hi] maximising the goodput
// G(N) = (B + A(N)) T(B + N) / (B + N), A(N) the sum of the N best survivals in the trim
// order (the floor positions first when the budget allows one per request), T the curve.
// The competing survivals are sorted (bitonic, descending) in C, prefix-summed in
// float64, and every N is evaluated by some thread; the block keeps the best (G, N).
__device__ long long curve_budget(const ScheduleArgs& A, const double* S, const int* L0,
                                  double* C, long long total, const float* cx, const float* cy) {
  __shared__ unsigned int s_nc;
  __shared__ double s_red[SCHED_THREADS / 32];
  __shared__ double s_floor;
  __shared__ long long s_n;
  __shared__ unsigned long long s_bestn[SCHED_THREADS / 32];
  __shared__ double s_bestg[SCHED_THREADS / 32];
  const int B = A.B, K = A.K, N = B * K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool floors = A.budget >= B;
  const long long n_hi = total < A.budget ? total : A.budget;
  const long long n_lo = floors ? B : 0;
  // Competing survivals into C (any order: they are sorted next), the floors' sum.
  if (tid == 0) s_nc = 0;
  __syncthreads();
  double fsum = 0.0;
  for (int i = tid; i < N; i += SCHED_THREADS) {
    const int b = i / K, k = i - b * K;
    if (k >= L0[b]) continue;
    if (floors && k == 0)
      fsum += S[i];
    else
      C[atomicAdd(&s_nc, 1u)] = S[i];
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) fsum += __shfl_xor_sync(0xffffffffu, fsum, o);
  if (lane == 0) s_red[warp] = fsum;
  __syncthreads();
  const int nc = static_cast<int>(s_nc);
  int P = 1;
  while (P < nc) P <<= 1;
  for (int i = nc + tid; i < P; i += SCHED_THREADS) C[i] = 0.0;  // padding sorts last
  if (tid == 0) {  // the floors' sum, once (fp64 work is scarce on this GPU)
    double a = 0.0;
    for (int w = 0; w < SCHED_THREADS / 32; ++w) a += s_red[w];
    s_floor = a;
  }
  __syncthreads();
  const double a_floor = s_floor;
  // Bitonic sort, descending, on the bit patterns (S >= 0 orders like its bits).
  unsigned long long* Ck = reinterpret_cast<unsigned long long*>(C);
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < P; i += SCHED_THREADS) {
        const int l = i ^ j;
        if (l > i) {
          const unsigned long long x = Ck[i], y = Ck[l];
          const bool desc = (i & k) == 0;
          if (desc ? (x < y) : (x > y)) {
            Ck[i] = y;
            Ck[l] = x;
          }
        }
      }
      __syncthreads();
    }
  }
  // Inclusive prefix sums of the first nc values: a chunk per thread, then the chunks.
  const int per = (nc + SCHED_THREADS - 1) / SCHED_THREADS;
  const int i0 = min(nc, tid * per), i1 = min(nc, i0 + per);
  double run = 0.0;
  for (int i = i0; i < i1; ++i) {
    run += C[i];
    C[i] = run;
  }
  double incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  __syncthreads();
  if (lane == 31) s_red[warp] = incl;
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the warps' totals, once
    const double v = s_red[lane];
    double e = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, e, o);
      if (lane >= o) e += y;
    }
    __syncwarp();
    s_red[lane] = e - v;
  }
  __syncthreads();
  const double off = (incl - run) + s_red[warp];
  for (int i = i0; i < i1; ++i) C[i] += off;
  __syncthreads();
  // Goodput of every N; the best (largest G, then smallest N) over the block.
  double bg = -1.0;
  long long bn = n_lo;
  for (long long n = n_lo + tid; n <= n_hi; n += SCHED_THREADS) {
    const double a = (n > n_lo) ? __dadd_rn(a_floor, C[n - n_lo - 1]) : a_floor;
    const double x = static_cast<double>(B) + static_cast<double>(n);
    const double g = __ddiv_rn(__dmul_rn(__dadd_rn(static_cast<double>(B), a),
                                         curve_at(cx, cy, A.n_pts, x)), x);
    if (g > bg) {
      bg = g;
      bn = n;
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const double g2 = __shfl_xor_sync(0xffffffffu, bg, o);
    const long long n2 = __shfl_xor_sync(0xffffffffu, bn, o);
    if (g2 > bg || (g2 == bg && n2 < bn)) {
      bg = g2;
      bn = n2;
    }
  }
  if (lane == 0) {
    s_bestg[warp] = bg;
    s_bestn[warp] = static_cast<unsigned long long>(bn);
  }
  __syncthreads();
  if (warp == 0) {  // the best over the warps, once
    double g = s_bestg[lane];
    long long n = static_cast<long long>(s_bestn[lane]);
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const double g2 = __shfl_xor_sync(0xffffffffu, g, o);
      const long long n2 = __shfl_xor_sync(0xffffffffu, n, o);
      if (g2 > g || (g2 == g && n2 < n)) {
        g = g2;
        n = n2;
      }
    }
    if (lane == 0) {
      s_n = n;
      if (A.n_out) *A.n_out = static_cast<int32_t>(n);
      if (A.g_out) *A.g_out = g;
    }
  }
  __syncthreads();
  return s_n;
}

__global__ void __launch_bounds__(SCHED_THREADS, 1) sv_schedule_kernel(const ScheduleArgs A) {
  extern __shared__ __align__(16) unsigned char dsm[];
  const int B = A.B, K = A.K, N = B * K;
  double* S = reinterpret_cast<double*>(dsm);  // [B*K], request-major
  int* L0 = reinterpret_cast<int*>(S + N);     // [B]
  int* cnt = L0 + B;                           // [B] kept competing positions
  __shared__ unsigned int hist[256];
  __shared__ unsigned long long s_prefix;
  __shared__ unsigned int s_rem;
  __shared__ int s_scan[32];
  __shared__ unsigned long long s_total;
  __shared__ float s_temps[SV_MAX_K];
  __shared__ double s_tau;
  __shared__ float s_cx[SV_MAX_CURVE], s_cy[SV_MAX_CURVE];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // 0. Threshold (as given, or from the load state by thread 0) and the position
  // temperatures; barriers only when either is in use.
  const bool cal = A.temps != nullptr;
  double th = static_cast<double>(A.tau);
  bool bad = false;
  if (A.load || cal || A.curve) {
    int mine = 0;
    if (A.curve && tid == 0) {  // the curve: finite, tokens/s > 0, tokens ascending
      for (int i = 0; i < A.n_pts; ++i) {
        const float x = __ldg(A.curve + i), y = __ldg(A.curve + A.n_pts + i);
        s_cx[i] = x;
        s_cy[i] = y;
        if (!(isfinite(x) && isfinite(y) && y > 0.f) || (i > 0 && !(x > s_cx[i - 1]))) mine = 1;
      }
    }
    if (A.load && tid == 0) {
      const double t = load_tau(A.load, static_cast<double>(A.tau_min),
                                static_cast<double>(A.tau_max));
      s_tau = t;
      mine = t < 0.0;
    }
    if (cal && tid < K) {
      const float t = __ldg(A.temps + tid);
      s_temps[tid] = t;
      mine |= !(isfinite(t) && t > 0.f);
    }
    bad = __syncthreads_or(mine) != 0;
    if (A.load) th = s_tau;
    if (cal) {
      // 0b. Calibrated confidences into S, one element per thread.
      for (int i = tid; i < N; i += SCHED_THREADS) {
        const float c0 = __ldg(A.conf + i);
        if (!(c0 >= 0.f && c0 <= 1.f)) bad = true;
        const float c = calibrate(c0, s_temps[i % K]);
        if (A.conf_cal) A.conf_cal[i] = c;
        S[i] = static_cast<double>(c);
      }
      __syncthreads();
    }
  }
  if (tid == 0 && A.tau_out) *A.tau_out = th;

  // 1-2. survival products and tau-lengths, one thread per request; the row of
  // confidences is loaded up front (independent loads), and S >= 0 compares with tau
  // as 64-bit patterns, keeping the slow fp64 pipe to the products alone.
  const unsigned long long tau_key = surv_key(th < 0.0 ? 0.0 : th);
  unsigned long long my_total = 0;
  for (int b = tid; b < B; b += SCHED_THREADS) {
    double run = 1.0;
    int n = 0;
    if (cal) {  // calibrated confidences are in S already
#pragma unroll
      for (int k = 0; k < SV_MAX_K; ++k) {
        if (k < K) {
          run = run * S[(size_t)b * K + k];
          S[(size_t)b * K + k] = run;
          if (surv_key(run) >= tau_key) n = k + 1;
        }
      }
    } else {
      float cv[SV_MAX_K];
#pragma unroll
      for (int k = 0; k < SV_MAX_K; ++k) cv[k] = (k < K) ? __ldg(A.conf + (size_t)b * K + k) : 0.f;
#pragma unroll
      for (int k = 0; k < SV_MAX_K; ++k) {
        if (k < K) {
          const float c = cv[k];
          if (!(c >= 0.f && c <= 1.f)) bad = true;
          if (A.conf_cal) A.conf_cal[(size_t)b * K + k] = c;
          run = run * static_cast<double>(c);
          S[(size_t)b * K + k] = run;
          if (surv_key(run) >= tau_key) n = k + 1;
        }
      }
    }
    if (n < 1) n = 1;
    L0[b] = n;
    cnt[b] = 0;
    my_total += n;
  }
  if (tid == 0) s_total = 0;
  if (__syncthreads_or(bad)) {
    for (int b = tid; b < B; b += SCHED_THREADS) A.out_len[b] = 0;
    if (tid == 0) atomicOr(&A.hdr->status, ST_DEVICE_INPUT);
    return;
  }
  // Sum of the tau-lengths: a warp reduction, then one shared atomic per warp.
#pragma unroll
  for (int o = 16; o; o >>= 1) my_total += __shfl_xor_sync(0xffffffffu, my_total, o);
  if (lane == 0 && my_total) atomicAdd(&s_total, my_total);
  __syncthreads();
  const long long total = static_cast<long long>(s_total);
  long long budget = A.budget;
  if (A.curve) budget = curve_budget(A, S, L0, reinterpret_cast<double*>(cnt + B), total, s_cx, s_cy);
  if (total <= budget) {
    for (int b = tid; b < B; b += SCHED_THREADS) A.out_len[b] = L0[b];
    return;
  }
  const bool floor_first = budget >= B;
  const int lo = floor_first ? 1 : 0;
  const unsigned int bud = static_cast<unsigned int>(floor_first ? budget - B : budget);
  if (bud == 0) {
    for (int b = tid; b < B; b += SCHED_THREADS) A.out_len[b] = lo;
    return;
  }

  // 3a. Radix select: the bud-th largest key among competing positions
  // (lo <= k < L0_b). Their count exceeds bud because total > budget.
  if (tid == 0) {
    s_prefix = 0ull;
    s_rem = bud;
  }
  unsigned long long mask = 0ull;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += SCHED_THREADS) hist[i] = 0u;
    __syncthreads();
    const unsigned long long pre = s_prefix;
    for (int i = tid; i < N; i += SCHED_THREADS) {
      const int b = i / K, k = i - b * K;
      if (k < lo || k >= L0[b]) continue;
      const unsigned long long key = surv_key(S[i]);
      if ((key & mask) != pre) continue;
      atomicAdd(&hist[(key >> shift) & 255ull], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // The digit d holding the rem-th largest key: lane l owns digits
      // 255-8l .. 248-8l; counts above each lane's block come from a suffix scan.
      const unsigned int rem = s_rem;
      unsigned int own = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) own += hist[255 - 8 * lane - q];
      unsigned int above = own;  // inclusive prefix from the top digit down
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned int y = __shfl_up_sync(0xffffffffu, above, o);
        if (lane >= o) above += y;
      }
      const unsigned int hit = __ballot_sync(0xffffffffu, above >= rem);
      const int ln = hit ? __ffs(hit) - 1 : 31;
      if (lane == ln) {
        unsigned int acc = above - own;
        int d = 255 - 8 * lane;
        for (int q = 0; q < 7; ++q, --d) {
          if (acc + hist[d] >= rem) break;
          acc += hist[d];
        }
        s_rem = rem - acc;
        s_prefix = pre | (static_cast<unsigned long long>(d) << shift);
      }
    }
    mask |= 255ull << shift;
    __syncthreads();
  }
  const unsigned long long thr = s_prefix;
  const unsigned int need = s_rem;  // how many keys equal to thr are kept

  // 3b. Keys above the threshold are kept; ties with it are ranked in k-major order
  // (k ascending, then b ascending) by a block-wide prefix count.
  const int per = (N + SCHED_THREADS - 1) / SCHED_THREADS;
  const int i0 = min(N, tid * per), i1 = min(N, i0 + per);  // k-major index range
  int my_ties = 0;
  for (int i = i0; i < i1; ++i) {
    const int k = i / B, b = i - k * B;
    if (k < lo || k >= L0[b]) continue;
    const unsigned long long key = surv_key(S[(size_t)b * K + k]);
    if (key > thr)
      atomicAdd(&cnt[b], 1);
    else if (key == thr)
      ++my_ties;
  }
  int incl = my_ties;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = s_scan[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    s_scan[lane] = v;
  }
  __syncthreads();
  int rank = incl - my_ties + (warp ? s_scan[warp - 1] : 0);
  for (int i = i0; i < i1; ++i) {
    const int k = i / B, b = i - k * B;
    if (k < lo || k >= L0[b]) continue;
    if (surv_key(S[(size_t)b * K + k]) == thr) {
      if (static_cast<unsigned int>(rank) < need) atomicAdd(&cnt[b], 1);
      ++rank;
    }
  }
  __syncthreads();
  for (int b = tid; b < B; b += SCHED_THREADS) A.out_len[b] = lo + cnt[b];
}

static size_t schedule_smem_bytes(int B, int K, bool curve) {
  size_t sort = 0;
  if (curve) {
    size_t p = 1;
    while (p < (size_t)B * K) p <<= 1;
    sort = p * sizeof(double);
  }
  return (size_t)B * K * sizeof(double) + 2 * (size_t)B * sizeof(int) + sort;
}

cudaError_t launch_schedule(const float* conf, const float* temps, const float* load,
                            const float* curve, int n_pts, int B, int K, float tau, float tau_min,
                            float tau_max, int budget, int32_t* out_len, float* conf_cal,
                            double* tau_out, int32_t* n_out, double* g_out, WsHeader* hdr,
                            cudaStream_t st) {
  const size_t smem = schedule_smem_bytes(B, K, curve != nullptr);
  static bool attr_set = false;  // idempotent if two threads race here
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(
        sv_schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        (int)schedule_smem_bytes(SV_MAX_SCHED_B, SV_MAX_SCHED_BK / SV_MAX_SCHED_B, false));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  ScheduleArgs A{conf, temps, load, curve, n_pts, n_out, g_out, B, K, tau, tau_min, tau_max,
                 budget, out_len, conf_cal, tau_out, hdr};
  sv_schedule_kernel<<<1, SCHED_THREADS, smem, st>>>(A);
  return cudaGetLastError();
}

}  // namespace sv
