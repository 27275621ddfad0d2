// sv_calib.cu -- the online calibration loop around the schedule (sm_103a).
//
// DSpark Deep Dive, "The Calibration Loop in Practice": over a window of
// verification rounds the system compares, per draft position, the mean calibrated
// confidence with the fraction of tokens at that position the verifier accepted, and
// moves the position's temperature by a small step toward agreement; the expected
// calibration error (ECE, "The Raw Confidence Problem") measures the remaining gap.
//
//  sv_calib_observe_kernel: adds one round to the window statistics. A position
//    counts when the verifier tested it (k < L_b and k <= j_b, j_b the accepted
//    count; later positions were never tested) and was accepted when k < j_b. Per
//    position: sum of c', tested, accepted; per confidence bin (SV_CALIB_BINS equal
//    bins of [0, 1]): tested, sum of c', accepted. One CTA; each thread keeps the
//    counts of one position in registers and adds them to shared counters once;
//    sums of c' are exact fixed-point integers (see below), so the statistics do not
//    depend on the order of the additions.
//  sv_calib_update_kernel: T_k <- max(T_k + lr * (mean c'_k - acceptance_k), floor)
//    for each position with a tested token (float64, then rounded to float32), ECE =
//    sum_bins |accepted - sum c'| / tested, and the window restarts.
#include "sv_common.cuh"
#include "sv_launch.cuh"

namespace sv {

constexpr int OBS_THREADS = 512;
constexpr int NB = SV_CALIB_BINS;
constexpr float FIX_SCALE = 281474976710656.0f;  // 2^48
constexpr double FIX_UNIT = 1.0 / 281474976710656.0;

// Sums of c' are kept as integers in units of 2^-48. A float32 c' >= 2^-25 converts
// exactly, integer addition is exact and order-free, and the float64 value of the
// total is exact whenever the float64 sum of the same values is (every c' >= 2^-14
// and the total below 2^15): the window then matches a sequential float64 sum bit for
// bit, and repeated runs agree. Smaller c' round to the nearest 2^-48.
// Sum of v over the lanes in `mask`, exact: three chunks of at most 22 bits, each
// summed by the hardware reduction (32 lanes cannot overflow a chunk's 32 bits).
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned mask, unsigned long long v) {
  const unsigned a = __reduce_add_sync(mask, static_cast<unsigned>(v & 0x3fffffull));
  const unsigned b = __reduce_add_sync(mask, static_cast<unsigned>((v >> 22) & 0x3fffffull));
  const unsigned c = __reduce_add_sync(mask, static_cast<unsigned>(v >> 44));
  return static_cast<unsigned long long>(a) + (static_cast<unsigned long long>(b) << 22) +
         (static_cast<unsigned long long>(c) << 44);
}

__global__ void __launch_bounds__(OBS_THREADS, 1)
    sv_calib_observe_kernel(const float* __restrict__ conf_cal, const int32_t* __restrict__ vlen,
                            const int32_t* __restrict__ acc, int B, int K, double* stats) {
  __shared__ unsigned long long psum[SV_MAX_K], bsum[NB];
  __shared__ unsigned int pcnt[SV_MAX_K][2], bcnt[NB][2];  // tested, accepted
  const int tid = threadIdx.x;
  if (tid < SV_MAX_K) {
    psum[tid] = 0ull;
    pcnt[tid][0] = pcnt[tid][1] = 0u;
  }
  if (tid < NB) {
    bsum[tid] = 0ull;
    bcnt[tid][0] = bcnt[tid][1] = 0u;
  }
  __syncthreads();
  // Thread t takes the elements e = t, t + G, t + 2G, ... with G a multiple of K, so
  // its position k = t mod K is fixed: its counts stay in registers and meet the
  // shared counters once at the end.
  const int G = (OBS_THREADS / K) * K;
  const long long n = (long long)B * K;
  unsigned long long ps = 0ull, bs[NB];
  unsigned pt = 0u, pa = 0u, bt[NB], ba[NB];
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    bs[i] = 0ull;
    bt[i] = ba[i] = 0u;
  }
  if (tid < G) {
    const int k = tid % K;
    constexpr int U = 4;  // elements whose loads are in flight together
    for (long long e0 = tid; e0 < n; e0 += (long long)U * G) {
      int Lu[U], ju[U];
      float cu[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const long long e = e0 + (long long)u * G;
        Lu[u] = -1;
        ju[u] = -1;
        cu[u] = 0.f;
        if (e < n) {
          const int b = static_cast<int>(e / K);
          Lu[u] = __ldg(vlen + b);
          ju[u] = __ldg(acc + b);
          cu[u] = __ldg(conf_cal + e);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
      const int L = Lu[u], j = ju[u];
      if (j < 0 || L < 0 || L > K || k >= L || k > j) continue;
      const float c = cu[u];
      const unsigned a = k < j ? 1u : 0u;
      const unsigned long long f = __float2ull_rn(c * FIX_SCALE);
      // Bin floor(NB * c), taken exactly: the product rounds in fp32, so the candidate
      // is checked against its edges with one-rounding fmas, whose sign is exact.
      int bin = static_cast<int>(floorf(c * static_cast<float>(NB)));
      if (__fmaf_rn(c, static_cast<float>(NB), -static_cast<float>(bin)) < 0.f)
        --bin;
      else if (__fmaf_rn(c, static_cast<float>(NB), -static_cast<float>(bin + 1)) >= 0.f)
        ++bin;
      bin = bin < 0 ? 0 : (bin > NB - 1 ? NB - 1 : bin);
      ps += f;
      ++pt;
      pa += a;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        if (i == bin) {
          bs[i] += f;
          ++bt[i];
          ba[i] += a;
        }
      }
      }
    }
  }
  // Warp-level sums first (lanes of one position, then every lane for each bin), so
  // each shared counter sees at most one atomic per warp.
  if (tid < ((G + 31) & ~31)) {
    const unsigned act = __ballot_sync(0xffffffffu, tid < G);
    if (tid < G) {
      const int k = tid % K;
      const unsigned same = __match_any_sync(act, k);
      const unsigned long long s1 = warp_sum_u64(same, ps);
      const unsigned t1 = __reduce_add_sync(same, pt), a1 = __reduce_add_sync(same, pa);
      if ((threadIdx.x & 31) == __ffs(same) - 1 && t1) {
        atomicAdd(&psum[k], s1);
        atomicAdd(&pcnt[k][0], t1);
        atomicAdd(&pcnt[k][1], a1);
      }
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const unsigned long long s2 = warp_sum_u64(act, bs[i]);
        const unsigned t2 = __reduce_add_sync(act, bt[i]), a2 = __reduce_add_sync(act, ba[i]);
        if ((threadIdx.x & 31) == __ffs(act) - 1 && t2) {
          atomicAdd(&bsum[i], s2);
          atomicAdd(&bcnt[i][0], t2);
          atomicAdd(&bcnt[i][1], a2);
        }
      }
    }
  }
  __syncthreads();
  if (tid < K) {
    stats[3 * tid + 0] += static_cast<double>(psum[tid]) * FIX_UNIT;
    stats[3 * tid + 1] += static_cast<double>(pcnt[tid][0]);
    stats[3 * tid + 2] += static_cast<double>(pcnt[tid][1]);
  } else if (tid >= 32 && tid < 32 + NB) {
    const int i = tid - 32;
    double* bins = stats + 3 * K;
    bins[3 * i + 0] += static_cast<double>(bcnt[i][0]);
    bins[3 * i + 1] += static_cast<double>(bsum[i]) * FIX_UNIT;
    bins[3 * i + 2] += static_cast<double>(bcnt[i][1]);
  }
}

__global__ void __launch_bounds__(32, 1)
    sv_calib_update_kernel(double* stats, float* temps, int K, double lr, double temp_floor,
                           double* ece) {
  const int lane = threadIdx.x;
  if (lane < K) {
    const double n = stats[3 * lane + 1];
    if (n > 0.0) {
      const double err = __dsub_rn(__ddiv_rn(stats[3 * lane + 0], n), __ddiv_rn(stats[3 * lane + 2], n));
      float tf = __double2float_rn(__dadd_rn(static_cast<double>(temps[lane]), __dmul_rn(lr, err)));
      if (static_cast<double>(tf) < temp_floor) tf = __double2float_rn(temp_floor);
      temps[lane] = tf;
    }
  }
  __syncwarp();
  if (lane == 0) {
    const double* bins = stats + 3 * K;
    double N = 0.0, gap = 0.0;
    for (int i = 0; i < NB; ++i) {  // in bin order
      N = __dadd_rn(N, bins[3 * i + 0]);
      gap = __dadd_rn(gap, fabs(__dsub_rn(bins[3 * i + 2], bins[3 * i + 1])));
    }
    if (ece) *ece = N > 0.0 ? __ddiv_rn(gap, N) : 0.0;
  }
  __syncwarp();
  for (int i = lane; i < 3 * K + 3 * NB; i += 32) stats[i] = 0.0;
}

cudaError_t launch_calib_observe(const float* conf_cal, const int32_t* vlen, const int32_t* acc,
                                 int B, int K, double* stats, cudaStream_t st) {
  sv_calib_observe_kernel<<<1, OBS_THREADS, 0, st>>>(conf_cal, vlen, acc, B, K, stats);
  return cudaGetLastError();
}

cudaError_t launch_calib_update(double* stats, float* temps, int K, float lr, float temp_floor,
                                double* ece, cudaStream_t st) {
  sv_calib_update_kernel<<<1, 32, 0, st>>>(stats, temps, K, static_cast<double>(lr),
                                           static_cast<double>(temp_floor), ece);
  return cudaGetLastError();
}

}  // namespace sv
