// sv_api.cu -- the C-ABI boundary of libspecverify: argument checks, workspace
// layout, launches. Declarations and contracts are in include/specverify.h.
#include <atomic>
#include <cmath>

#include "sv_common.cuh"
#include "sv_launch.cuh"
#include "sv_tree.cuh"

namespace sv {

static int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace sv

using namespace sv;

extern "C" {

size_t sv_workspace_bytes(int B, int K, int V) {
  if (B < 0 || K < 1 || K > SV_MAX_K || V < 1 || V > SV_MAX_V) return 0;
  return ws_layout(B > SV_MAX_B ? SV_MAX_B : B, K, V).total;
}

sv_status sv_workspace_init(void* ws_d, size_t ws_bytes, void* stream) {
  if (!ws_d || ws_bytes < sizeof(WsHeader) || !aligned(ws_d, 256)) return SV_ERR_WORKSPACE;
  if (cudaMemsetAsync(ws_d, 0, ws_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

static sv_status schedule_any(const float* conf_d, const float* temps_d, const float* load_d,
                              float tau, float tau_min, float tau_max, const float* curve_d,
                              int n_pts, int B, int K, int token_budget, int32_t* out_len_d,
                              float* conf_cal_d, double* tau_out_d, int32_t* n_out_d,
                              double* g_out_d, void* ws_d, size_t ws_bytes, void* stream) {
  if (B < 0 || B > SV_MAX_SCHED_B || K < 1 || K > SV_MAX_K || (long long)B * K > SV_MAX_SCHED_BK)
    return SV_ERR_SHAPE;
  if (curve_d && (n_pts < 1 || n_pts > SV_MAX_CURVE || (long long)B * K > SV_MAX_CURVE_BK))
    return SV_ERR_SHAPE;
  if (!(tau >= 0.f && tau <= 1.f) || token_budget < 0) return SV_ERR_ARG;
  if (load_d && !(tau_min >= 0.f && tau_min <= 1.f && tau_max >= 0.f && tau_max <= 1.f))
    return SV_ERR_ARG;
  if (!ws_d || ws_bytes < sizeof(WsHeader) || !aligned(ws_d, 256)) return SV_ERR_WORKSPACE;
  if (B == 0) return SV_OK;
  if (!conf_d || !out_len_d || !aligned(conf_d, 4) || !aligned(out_len_d, 4)) return SV_ERR_ARG;
  if ((temps_d && !aligned(temps_d, 4)) || (load_d && !aligned(load_d, 4)) ||
      (conf_cal_d && !aligned(conf_cal_d, 4)) || (tau_out_d && !aligned(tau_out_d, 8)) ||
      (curve_d && !aligned(curve_d, 4)) || (n_out_d && !aligned(n_out_d, 4)) ||
      (g_out_d && !aligned(g_out_d, 8)))
    return SV_ERR_ARG;
  const cudaError_t e = launch_schedule(conf_d, temps_d, load_d, curve_d, n_pts, B, K, tau,
                                        tau_min, tau_max, token_budget, out_len_d, conf_cal_d,
                                        tau_out_d, n_out_d, g_out_d,
                                        static_cast<WsHeader*>(ws_d),
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status sv_schedule_cal(const float* conf_d, const float* temps_d, const float* load_d,
                          float tau, float tau_min, float tau_max, int B, int K,
                          int token_budget, int32_t* out_len_d, float* conf_cal_d,
                          double* tau_out_d, void* ws_d, size_t ws_bytes, void* stream) {
  return schedule_any(conf_d, temps_d, load_d, tau, tau_min, tau_max, nullptr, 0, B, K,
                      token_budget, out_len_d, conf_cal_d, tau_out_d, nullptr, nullptr, ws_d,
                      ws_bytes, stream);
}

sv_status sv_schedule_curve(const float* conf_d, const float* temps_d, const float* load_d,
                            float tau, float tau_min, float tau_max, const float* curve_d,
                            int n_pts, int B, int K, int token_budget, int32_t* out_len_d,
                            float* conf_cal_d, double* tau_out_d, int32_t* n_out_d,
                            double* g_out_d, void* ws_d, size_t ws_bytes, void* stream) {
  if (!curve_d) return SV_ERR_ARG;
  return schedule_any(conf_d, temps_d, load_d, tau, tau_min, tau_max, curve_d, n_pts, B, K,
                      token_budget, out_len_d, conf_cal_d, tau_out_d, n_out_d, g_out_d, ws_d,
                      ws_bytes, stream);
}

sv_status sv_schedule(const float* conf_d, int B, int K, float tau, int token_budget,
                      int32_t* out_len_d, void* ws_d, size_t ws_bytes, void* stream) {
  return sv_schedule_cal(conf_d, nullptr, nullptr, tau, 0.f, 0.f, B, K, token_budget, out_len_d,
                         nullptr, nullptr, ws_d, ws_bytes, stream);
}

size_t sv_markov_keys_len(int B, int K) {
  if (B < 0 || B > SV_MAX_B || K < 1 || K > SV_MAX_K) return 0;
  return (size_t)B * K;
}

sv_status sv_markov_draft(const void* logits_d, const void* U_d, const void* Vm_d,
                          const int32_t* prev_tok_d, int B, int K, int V, int r,
                          void* corrected_d, int32_t* draft_tok_d, unsigned long long* keys_d,
                          void* ws_d, size_t ws_bytes, void* stream) {
  if (B < 0 || B > SV_MAX_B || K < 1 || K > SV_MAX_K || V < 1 || V > SV_MAX_V) return SV_ERR_SHAPE;
  if (r < 16 || r > SV_MAX_MARKOV_R || r % 16 != 0) return SV_ERR_SHAPE;
  if (!ws_d || ws_bytes < sizeof(WsHeader) || !aligned(ws_d, 256)) return SV_ERR_WORKSPACE;
  if (B == 0) return SV_OK;
  if (!logits_d || !U_d || !Vm_d || !prev_tok_d || !corrected_d || !draft_tok_d || !keys_d)
    return SV_ERR_ARG;
  if (!aligned(logits_d, 16) || !aligned(U_d, 16) || !aligned(Vm_d, 16) ||
      !aligned(corrected_d, 16) || !aligned(prev_tok_d, 4) || !aligned(draft_tok_d, 4) ||
      !aligned(keys_d, 8))
    return SV_ERR_ARG;
  const cudaError_t e = launch_markov(
      static_cast<const uint16_t*>(logits_d), static_cast<const uint16_t*>(U_d),
      static_cast<const uint16_t*>(Vm_d), prev_tok_d, B, K, V, r,
      static_cast<uint16_t*>(corrected_d), draft_tok_d, keys_d, static_cast<WsHeader*>(ws_d),
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

size_t sv_calib_stats_len(int K) {
  if (K < 1 || K > SV_MAX_K) return 0;
  return 3 * (size_t)K + 3 * (size_t)SV_CALIB_BINS;
}

sv_status sv_calib_observe(const float* conf_cal_d, const int32_t* verify_len_d,
                           const int32_t* accepted_d, int B, int K, double* stats_d,
                           void* stream) {
  if (B < 0 || B > SV_MAX_B || K < 1 || K > SV_MAX_K) return SV_ERR_SHAPE;
  if (B == 0) return SV_OK;
  if (!conf_cal_d || !verify_len_d || !accepted_d || !stats_d || !aligned(conf_cal_d, 4) ||
      !aligned(verify_len_d, 4) || !aligned(accepted_d, 4) || !aligned(stats_d, 8))
    return SV_ERR_ARG;
  const cudaError_t e = launch_calib_observe(conf_cal_d, verify_len_d, accepted_d, B, K, stats_d,
                                             static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status sv_calib_update(double* stats_d, float* temps_d, int K, float lr, float temp_floor,
                          double* ece_d, void* stream) {
  if (K < 1 || K > SV_MAX_K) return SV_ERR_SHAPE;
  if (!std::isfinite(lr) || !std::isfinite(temp_floor) || !(temp_floor > 0.f)) return SV_ERR_ARG;
  if (!stats_d || !temps_d || !aligned(stats_d, 8) || !aligned(temps_d, 4) ||
      (ece_d && !aligned(ece_d, 8)))
    return SV_ERR_ARG;
  const cudaError_t e = launch_calib_update(stats_d, temps_d, K, lr, temp_floor, ece_d,
                                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // extern "C"

namespace sv {

// Bound on a verify call's waits for other warps' results (clock cycles); a testing
// aid can shorten it (sv_set_wait_limit).
static std::atomic<long long> g_wait_limit{WAIT_CYCLES};

// Every host-side check of a verify call, then the kernel arguments (nothing is
// enqueued here).
sv_status verify_prepare(const void* target_d, const void* draft_d, sv_dtype dtype,
                         const int32_t* draft_tok_d, const int32_t* verify_len_d,
                         const float* uniforms_d, int B, int K, int V, float temperature,
                         int32_t* out_tok_d, int32_t* out_accepted_d, float* out_p_d,
                         float* out_q_d, uint32_t* accept_count_d, uint32_t* tested_count_d,
                         int32_t* near_tie_flags_d, void* ws_d, size_t ws_bytes,
                         VerifyArgs* out, int* grid_out) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (B < 0 || B > SV_MAX_B || K < 1 || K > SV_MAX_K || V < 1 || V > SV_MAX_V)
    return SV_ERR_SHAPE;
  const bool greedy = temperature == 0.f;
  if (!std::isfinite(temperature) || temperature < 0.f ||
      (!greedy && (temperature < 1e-6f || temperature > 1e6f)))
    return SV_ERR_ARG;
  const WsLayout L = ws_layout(B, K, V);
  if (!ws_d || !aligned(ws_d, 256) || ws_bytes < L.total) return SV_ERR_WORKSPACE;
  *grid_out = 0;
  if (B == 0) return SV_OK;
  const size_t eb = dtype == SV_BF16 ? 2 : 4;
  if (!target_d || !draft_tok_d || !verify_len_d || !out_tok_d || !out_accepted_d)
    return SV_ERR_ARG;
  if (!greedy && (!draft_d || !uniforms_d)) return SV_ERR_ARG;
  if (!aligned(target_d, eb) || (draft_d && !aligned(draft_d, eb)) || !aligned(draft_tok_d, 4) ||
      !aligned(verify_len_d, 4) || (uniforms_d && !aligned(uniforms_d, 4)) ||
      !aligned(out_tok_d, 4) || !aligned(out_accepted_d, 4) || (out_p_d && !aligned(out_p_d, 4)) ||
      (out_q_d && !aligned(out_q_d, 4)) || (accept_count_d && !aligned(accept_count_d, 4)) ||
      (tested_count_d && !aligned(tested_count_d, 4)) ||
      (near_tie_flags_d && !aligned(near_tie_flags_d, 4)))
    return SV_ERR_ARG;
  const int sms = sm_count();
  if (sms <= 0) return SV_ERR_CUDA;

  unsigned char* ws = static_cast<unsigned char*>(ws_d);
  VerifyArgs& A = *out;
  A.tgt = target_d;
  A.drf = greedy ? nullptr : draft_d;
  A.tok = draft_tok_d;
  A.vlen = verify_len_d;
  A.uni = greedy ? nullptr : uniforms_d;
  A.B = B;
  A.K = K;
  A.V = V;
  {
    const double ad = greedy ? 0.0 : 1.4426950408889634 / (double)temperature;
    A.a = (float)ad;
    A.a_lo = (float)(ad - (double)A.a);
  }
  A.P = pieces_per_row(V, (int)eb);
  A.E = SLOT_BYTES / (int)eb;
  A.R = resid_pieces(V, (int)eb);
  A.E2 = SLOT_BYTES / 2 / (int)eb;
  A.RS = L.RS;
  A.Rmax = L.Rmax;
  A.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  A.out_tok = out_tok_d;
  A.out_acc = out_accepted_d;
  A.out_p = out_p_d;
  A.out_q = out_q_d;
  A.acc_cnt = accept_count_d;
  A.tst_cnt = tested_count_d;
  A.out_flags = near_tie_flags_d;
  A.hdr = reinterpret_cast<WsHeader*>(ws);
  A.t_row = reinterpret_cast<uint32_t*>(ws + L.t_row);
  A.t_req = reinterpret_cast<uint32_t*>(ws + L.t_req);
  A.t_res = reinterpret_cast<uint32_t*>(ws + L.t_res);
  A.rowstat = reinterpret_cast<float2*>(ws + L.rowstat);
  A.xz = reinterpret_cast<unsigned long long*>(ws + L.xz);
  A.part = reinterpret_cast<float2*>(ws + L.part);
  A.rpart = reinterpret_cast<float2*>(ws + L.rpart);
  A.jobs = reinterpret_cast<TermJob*>(ws + L.jobs);
  A.dec_flag = reinterpret_cast<uint32_t*>(ws + L.dec);
  A.lsum = reinterpret_cast<float*>(ws + L.lsum);
  // One persistent CTA per SM, fewer when the batch cannot give every warp a piece.
  const long long max_pieces = (long long)B * (greedy ? K + 1 : 2 * K + 1) * A.P;
  const long long want = (max_pieces + NCW - 1) / NCW;
  *grid_out = (int)(want < sms ? want : sms);
  return SV_OK;
}

sv_status verify_launch(const VerifyArgs& A, sv_dtype dtype, float temperature, int grid,
                        void* stream) {
  if (grid <= 0) return SV_OK;
  const cudaError_t e = launch_verify(A, dtype == SV_BF16, temperature == 0.f, grid,
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace sv

extern "C" {

sv_status sv_verify_diag(const void* target_d, const void* draft_d, sv_dtype dtype,
                         const int32_t* draft_tok_d, const int32_t* verify_len_d,
                         const float* uniforms_d, int B, int K, int V, float temperature,
                         int32_t* out_tok_d, int32_t* out_accepted_d, float* out_p_d,
                         float* out_q_d, uint32_t* accept_count_d, uint32_t* tested_count_d,
                         int32_t* near_tie_flags_d, void* ws_d, size_t ws_bytes, void* stream) {
  VerifyArgs A;
  int grid = 0;
  const sv_status st = verify_prepare(target_d, draft_d, dtype, draft_tok_d, verify_len_d,
                                      uniforms_d, B, K, V, temperature, out_tok_d,
                                      out_accepted_d, out_p_d, out_q_d, accept_count_d,
                                      tested_count_d, near_tie_flags_d, ws_d, ws_bytes, &A, &grid);
  if (st != SV_OK) return st;
  return verify_launch(A, dtype, temperature, grid, stream);
}

sv_status sv_verify(const void* target_d, const void* draft_d, sv_dtype dtype,
                    const int32_t* draft_tok_d, const int32_t* verify_len_d,
                    const float* uniforms_d, int B, int K, int V, float temperature,
                    int32_t* out_tok_d, int32_t* out_accepted_d, void* ws_d, size_t ws_bytes,
                    void* stream) {
  return sv_verify_diag(target_d, draft_d, dtype, draft_tok_d, verify_len_d, uniforms_d, B, K, V,
                        temperature, out_tok_d, out_accepted_d, nullptr, nullptr, nullptr,
                        nullptr, nullptr, ws_d, ws_bytes, stream);
}

long long sv_set_wait_limit(long long cycles) {
  const long long prev = g_wait_limit.load(std::memory_order_relaxed);
  g_wait_limit.store(cycles > 0 ? cycles : WAIT_CYCLES, std::memory_order_relaxed);
  return prev;
}

sv_status sv_verify_tree(const void* target_d, const void* draft_d, sv_dtype dtype,
                         const int32_t* parent_d, const int32_t* draft_tok_d,
                         const int32_t* n_nodes_d, const float* uniforms_d, int B, int N, int V,
                         float temperature, int32_t* out_tok_d, int32_t* out_accepted_d,
                         int32_t* out_path_d, void* ws_d, size_t ws_bytes, void* stream) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (B < 0 || B > SV_MAX_B || N < 1 || N > SV_MAX_TREE || V < 1 || V > SV_MAX_V)
    return SV_ERR_SHAPE;
  const bool greedy = temperature == 0.f;
  if (!std::isfinite(temperature) || temperature < 0.f ||
      (!greedy && (temperature < 1e-6f || temperature > 1e6f)))
    return SV_ERR_ARG;
  if (!ws_d || !aligned(ws_d, 256) || ws_bytes < sizeof(WsHeader)) return SV_ERR_WORKSPACE;
  if (B == 0) return SV_OK;
  const size_t eb = dtype == SV_BF16 ? 2 : 4;
  if (!target_d || !parent_d || !draft_tok_d || !n_nodes_d || !out_tok_d || !out_accepted_d)
    return SV_ERR_ARG;
  if (!greedy && (!draft_d || !uniforms_d)) return SV_ERR_ARG;
  if (!aligned(target_d, eb) || (draft_d && !aligned(draft_d, eb)) || !aligned(parent_d, 4) ||
      !aligned(draft_tok_d, 4) || !aligned(n_nodes_d, 4) ||
      (uniforms_d && !aligned(uniforms_d, 4)) || !aligned(out_tok_d, 4) ||
      !aligned(out_accepted_d, 4) || (out_path_d && !aligned(out_path_d, 4)))
    return SV_ERR_ARG;
  TreeArgs A;
  A.tgt = target_d;
  A.drf = greedy ? nullptr : draft_d;
  A.par = parent_d;
  A.tok = draft_tok_d;
  A.nn = n_nodes_d;
  A.uni = greedy ? nullptr : uniforms_d;
  A.B = B;
  A.N = N;
  A.V = V;
  {
    const double ad = greedy ? 0.0 : 1.4426950408889634 / (double)temperature;
    A.a = (float)ad;
    A.a_lo = (float)(ad - (double)A.a);
  }
  A.out_tok = out_tok_d;
  A.out_acc = out_accepted_d;
  A.out_path = out_path_d;
  A.hdr = static_cast<WsHeader*>(ws_d);
  const cudaError_t e = launch_tree(A, dtype == SV_BF16, greedy,
                                    static_cast<cudaStream_t>(stream), nullptr);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status sv_get_status(void* ws_d, void* stream, int clear, int32_t* status_out) {
  if (!ws_d || !status_out) return SV_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t bits = 0;
  if (cudaMemcpyAsync(&bits, ws_d, sizeof(bits), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SV_ERR_CUDA;
  *status_out = (bits & ST_TIMEOUT) ? SV_ERR_TIMEOUT
                : (bits & ST_DEVICE_INPUT) ? SV_ERR_DEVICE_INPUT
                                           : SV_OK;
  if (clear) {
    if (cudaMemsetAsync(ws_d, 0, sizeof(bits), st) != cudaSuccess) return SV_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SV_ERR_CUDA;
  }
  return SV_OK;
}

const char* sv_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "ok";
    case SV_ERR_ARG: return "invalid argument";
    case SV_ERR_SHAPE: return "unsupported shape";
    case SV_ERR_DTYPE: return "unsupported dtype";
    case SV_ERR_CUDA: return "CUDA runtime error";
    case SV_ERR_DEVICE_INPUT: return "invalid device-resident input";
    case SV_ERR_TIMEOUT: return "device wait timed out";
    case SV_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
  }
  return "unknown status";
}

int sv_version(void) { return 100; }

}  // extern "C"
