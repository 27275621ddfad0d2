// sv_common.cuh -- device helpers, kernel arguments and the workspace layout shared
// by the libspecverify kernels (sm_103a only).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "specverify.h"

namespace sv {

// ---------------------------------------------------------------------------
// Tuning constants of the fused verify kernel.
// One persistent CTA per SM of NCW warps; each warp owns SLOTS_PER_WARP shared-memory
// slots, issues its own 1-D bulk copies (TMA) of row pieces into them and reduces
// whole pieces on its own.
// ---------------------------------------------------------------------------
#ifndef SV_SLOT_BYTES
#define SV_SLOT_BYTES 8192
#endif
#ifndef SV_NCW
#define SV_NCW 12
#endif
#ifndef SV_SLOTS_PER_WARP
#define SV_SLOTS_PER_WARP 2
#endif
constexpr int SLOT_BYTES = SV_SLOT_BYTES;
constexpr int NCW = SV_NCW;
constexpr int SLOTS_PER_WARP = SV_SLOTS_PER_WARP;
static_assert(SLOT_BYTES % 32 == 0 && NCW * SLOTS_PER_WARP * SLOT_BYTES <= 200 * 1024,
              "slots must fit in shared memory next to the request prefix");
constexpr int NSLOT = NCW * SLOTS_PER_WARP;
constexpr int NTHREADS = 32 * NCW;
constexpr long long WAIT_CYCLES = 4000000000LL;  // ~2 s at 2 GHz: bound on any wait

// Status word bits (sticky reports, in the workspace header; cleared only by the
// caller).
constexpr uint32_t ST_DEVICE_INPUT = 1u;
constexpr uint32_t ST_TIMEOUT = 2u;

// ---------------------------------------------------------------------------
// Workspace layout (computed identically on host and device from B, K, V).
// ---------------------------------------------------------------------------
struct WsHeader {
  uint32_t status;    // ST_* bits: sticky report
  uint32_t abort;     // verify: set when a wait of this call gave up; reset at its end
  uint32_t cta_done;  // verify: CTAs that have finished
  uint32_t mk_pos;    // Markov: CTAs through the position barriers (reset after each call)
  uint32_t pad[60];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// Terminal-sample job of one request, written by the deciding warp and read by the
// warps running its terminal tasks: the residual max(0, p_j - q_j) over rows
// t_j and d_j, a plain sample of p over target row j (the bonus row L), or nothing
// (an invalid request, or greedy verification).
enum : int { J_NONE = -1, J_RESID = 0, J_BONUS = 1 };
struct __align__(32) TermJob {
  int kind, j;
  // Target and draft rows j: raw maximum M and 2^(M*a - fl(M*a)) / S, the inverse
  // row sum in the frame of the exact maximum.
  float MAt, invSt, MAd, invSd;
  int flags;  // near-tie flags of the decision (accept-test ties, tiny probabilities)
  int pad;
};

struct WsLayout {
  size_t t_row, t_req, t_res;  // uint32 tickets: [B*RS], [B], [B]
  size_t dec;                  // uint32 decision flags [B]
  size_t rowstat;              // float2 [B*RS]
  size_t xz;                   // u64 [B*RS]: logit of the drafted token in each row
  size_t part;                 // float2 [B*RS*Pmax]
  size_t rpart;                // float2 [B*Rmax] (float-float piece sums)
  size_t jobs;                 // TermJob [B]
  size_t lsum;                 // float [B*Rmax*32] lane-range totals of terminal pieces
  size_t total;
  int RS, Pmax, Rmax;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Pieces per row for element size `eb`: SLOT_BYTES per stream piece; terminal-sample
// pieces are half as long (a residual piece covers the same range of two rows).
__host__ __device__ inline int pieces_per_row(int V, int eb) {
  const int E = SLOT_BYTES / eb;
  return (V + E - 1) / E;
}
__host__ __device__ inline int resid_pieces(int V, int eb) {
  const int E2 = SLOT_BYTES / 2 / eb;
  return (V + E2 - 1) / E2;
}

// The ticket counters and decision flags sit at fixed offsets sized for the library
// maxima, so that calls of different shapes sharing one workspace never find another
// call's data where they expect a counter. Every one is back to zero when a call ends.
constexpr size_t TICKET_ROW_WORDS = (size_t)SV_MAX_B * (2 * SV_MAX_K + 1);
constexpr size_t TICKET_BYTES = 4 * (TICKET_ROW_WORDS + 3 * (size_t)SV_MAX_B);

__host__ __device__ inline WsLayout ws_layout(int B, int K, int V) {
  WsLayout L;
  L.RS = 2 * K + 1;
  L.Pmax = pieces_per_row(V, 4);  // fp32 needs the most pieces
  L.Rmax = resid_pieces(V, 4);
  const size_t nb = (size_t)(B > 0 ? B : 1);
  L.t_row = sizeof(WsHeader);
  L.t_req = L.t_row + 4 * TICKET_ROW_WORDS;
  L.t_res = L.t_req + 4 * (size_t)SV_MAX_B;
  L.dec = L.t_res + 4 * (size_t)SV_MAX_B;
  size_t off = align_up(sizeof(WsHeader) + TICKET_BYTES, 256);
  L.rowstat = off; off = align_up(off + 8 * nb * L.RS, 256);
  L.xz = off;      off = align_up(off + 8 * nb * L.RS, 256);
  L.part = off;    off = align_up(off + 8 * nb * L.RS * (size_t)L.Pmax, 256);
  L.rpart = off;   off = align_up(off + 8 * nb * (size_t)L.Rmax, 256);
  L.jobs = off;    off = align_up(off + sizeof(TermJob) * nb, 256);
  L.lsum = off;    off = align_up(off + 4 * 32 * nb * (size_t)L.Rmax, 256);
  L.total = off;
  return L;
}

// Arguments of the fused verify kernel (built by the C-ABI layer).
struct VerifyArgs {
  const void* tgt;
  const void* drf;
  const int32_t* tok;
  const int32_t* vlen;
  const float* uni;
  int B, K, V;
  float a;     // log2(e) / T rounded to fp32, T > 0
  float a_lo;  // log2(e) / T - a (the rounding error of a)
  int P;       // stream pieces per row
  int E;       // elements per stream piece
  int R;       // terminal-job pieces per request
  int E2;      // elements per terminal-job piece (per row)
  int RS;      // row slots per request, 2K+1
  int Rmax;    // stride of the terminal-partial array
  long long wait_limit;  // bound, in clock cycles, on waits for other warps' results
  int32_t* out_tok;
  int32_t* out_acc;
  float* out_p;
  float* out_q;
  uint32_t* acc_cnt;
  uint32_t* tst_cnt;
  int32_t* out_flags;
  WsHeader* hdr;
  uint32_t* t_row;
  uint32_t* t_req;
  uint32_t* t_res;
  uint32_t* dec_flag;  // per request: 0 undecided, 1 terminal job published, 2 no job
  float2* rowstat;
  unsigned long long* xz;
  float2* part;
  float2* rpart;
  TermJob* jobs;
  float* lsum;
};

cudaError_t launch_verify(const VerifyArgs& A, bool bf16, bool greedy, int grid, cudaStream_t st);

// Host side of a verify call (sv_api.cu): every argument check, then the kernel
// arguments and grid (grid 0: nothing to launch); and the launch itself.
sv_status verify_prepare(const void* target_d, const void* draft_d, sv_dtype dtype,
                         const int32_t* draft_tok_d, const int32_t* verify_len_d,
                         const float* uniforms_d, int B, int K, int V, float temperature,
                         int32_t* out_tok_d, int32_t* out_accepted_d, float* out_p_d,
                         float* out_q_d, uint32_t* accept_count_d, uint32_t* tested_count_d,
                         int32_t* near_tie_flags_d, void* ws_d, size_t ws_bytes,
                         VerifyArgs* out, int* grid_out);
sv_status verify_launch(const VerifyArgs& A, sv_dtype dtype, float temperature, int grid,
                        void* stream);

// ---------------------------------------------------------------------------
// PTX wrappers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

// Non-blocking probe: has the phase with this parity completed?
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Potentially blocking probe (the hardware may suspend the thread for a short,
// system-defined time before returning false).
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Acquire-ordered load (GPU scope).
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* addr) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}

// Relaxed load (GPU scope): a poll that orders nothing.
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* addr) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}

// Release-ordered store (GPU scope): earlier writes of this thread become visible to
// whoever observes the value (after an acquire fence).
__device__ __forceinline__ void st_release(uint32_t* addr, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

// Acquire-release fence (GPU scope): after a relaxed load that saw a released value,
// later reads see what was written before the release.
__device__ __forceinline__ void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// 1-D bulk copy global -> shared with an L2 eviction-priority hint (a policy made by
// createpolicy): evict_first for data read once, evict_last for data read again soon.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2^x on the special-function unit (hardware approximation).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max that returns NaN when either input is NaN.
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// Lane-wise max of two packed bf16 pairs, NaN-propagating.
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ bool finitef(float x) { return fabsf(x) <= 3.402823466e38f; }

}  // namespace sv
