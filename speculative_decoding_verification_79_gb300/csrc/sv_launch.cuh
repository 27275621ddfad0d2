// sv_launch.cuh -- launch entry points of the schedule, calibration and Markov kernels
// (the verify kernel's is in sv_common.cuh, the tree kernel's in sv_tree.cuh).
#pragma once
#include "sv_common.cuh"

namespace sv {

cudaError_t launch_schedule(const float* conf, const float* temps, const float* load,
                            const float* curve, int n_pts, int B, int K, float tau, float tau_min,
                            float tau_max, int budget, int32_t* out_len, float* conf_cal,
                            double* tau_out, int32_t* n_out, double* g_out, WsHeader* hdr,
                            cudaStream_t st);
cudaError_t launch_markov(const uint16_t* L, const uint16_t* U, const uint16_t* Vm,
                          const int32_t* prev, int B, int K, int V, int r, uint16_t* out,
                          int32_t* tok, unsigned long long* keys, WsHeader* hdr, cudaStream_t st);
cudaError_t launch_calib_observe(const float* conf_cal, const int32_t* vlen, const int32_t* acc,
                                 int B, int K, double* stats, cudaStream_t st);
cudaError_t launch_calib_update(double* stats, float* temps, int K, float lr, float temp_floor,
                                double* ece, cudaStream_t st);

}  // namespace sv
