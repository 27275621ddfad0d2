// sv_static.cu -- sv_verify_static: verification with no allocation at all.
//
// Some callers cannot call cudaMalloc: plugins whose host application owns every
// device allocation, runtimes that plan all their memory up front and allow no
// allocation afterwards, and allocator-less embedded deployments. This entry point lets
// them verify without providing a workspace: the scratch lives in one file-scope
// device array that the library image carries, sized SV_STATIC_SCRATCH_BYTES, which
// every GPU that loads the library keeps until the process exits.
#include <atomic>
#include <mutex>

#include "sv_common.cuh"

namespace sv {

static __device__ __align__(256) unsigned char g_static_scratch[SV_STATIC_SCRATCH_BYTES];

// Device address of the array, looked up once per device with that device current.
// In host code `g_static_scratch` names a host-side stand-in, never the device memory.
static std::atomic<void*> g_scratch_addr[64];
static std::mutex g_scratch_mu;

static sv_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SV_ERR_CUDA;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    p = g_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!p) {
      if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return SV_ERR_CUDA;
      g_scratch_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return SV_OK;
}

}  // namespace sv

using namespace sv;

extern "C" sv_status sv_verify_static(const void* target_d, const void* draft_d, sv_dtype dtype,
                                      const int32_t* draft_tok_d, const int32_t* verify_len_d,
                                      const float* uniforms_d, int B, int K, int V,
                                      float temperature, int32_t* out_tok_d,
                                      int32_t* out_accepted_d, void* stream) {
  if (B < 0 || B > SV_MAX_B || K < 1 || K > SV_MAX_K || V < 1 || V > SV_MAX_V)
    return SV_ERR_SHAPE;
  const size_t need = ws_layout(B, K, V).total;
  if (need > (size_t)SV_STATIC_SCRATCH_BYTES) return SV_ERR_WORKSPACE;  // too big for the array
  // No device work (and no address lookup) for an empty batch: its arguments are
  // still checked.
  void* ws = reinterpret_cast<void*>(static_cast<uintptr_t>(256));
  if (B > 0) {
    const sv_status sa = scratch_address(&ws);
    if (sa != SV_OK) return sa;
  }
  // Every argument check runs before anything is enqueued.
  VerifyArgs A;
  int grid = 0;
  const sv_status st = verify_prepare(target_d, draft_d, dtype, draft_tok_d, verify_len_d,
                                      uniforms_d, B, K, V, temperature, out_tok_d,
                                      out_accepted_d, nullptr, nullptr, nullptr, nullptr, nullptr,
                                      ws, need, &A, &grid);
  if (st != SV_OK || grid == 0) return st;
  // The array keeps the previous call's contents. Every call leaves its counters and
  // published words at zero (and the array starts at zero when the library loads), so
  // only the 256-byte header, whose status word collects reports, is cleared here.
  if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SV_ERR_CUDA;
  return verify_launch(A, dtype, temperature, grid, stream);
}
