// sv_markov.cu -- the Markov logit-bias head of the drafter (sm_103a).
//
// DSpark Guide, "1. The Markov Logit-Bias Head": the parallel backbone's raw logits of
// draft position k are corrected by a low-rank bigram term of the token drafted at
// position k-1,
//     L'_k = L_k + U (Vm[y_{k-1}, :])^T,   U, Vm in R^{V x r},
// and the next token is drafted from L'_k (greedy here: the lowest-index argmax, as
// in the page's sketch), so the positions run one after another.
//
// For a group of up to 128 requests the correction is the product D = X U^T, X [128, r]
// the gathered rows Vm[y_b, :] (zero past the batch), U [V, r]: a dense contraction on
// the fifth-generation tensor cores. A persistent CTA per SM (and request group) gathers
// X into shared memory in the canonical K-major 128-byte-swizzled layout, then walks its
// vocabulary tiles of 128 rows with four roles coupled only by mbarriers:
//  - one thread streams U tiles by 2-D tensor-map TMA (cp.async.bulk.tensor, 128-byte
//    swizzle, one box of 128 rows x 64 columns per 64 of r; rows past V and columns past
//    r are filled with zeros) into a ring of four buffers (two at r > 128);
//  - one thread copies the raw logits of each tile (the group's rows x 128 columns) by
//    3-D tensor-map TMA into a second ring of stages, so that each SM keeps 32-64 KB of
//    them in flight (loads held in registers one tile ahead kept only ~16 KB in flight
//    and left the epilogue waiting on HBM latency); a stage is released only after its
//    values have been used;
//  - one thread issues the tile's tcgen05.mma (kind::f16, bf16 inputs, M = 128 requests,
//    N = 128 vocabulary rows, K = 16 each) into one of four TMEM accumulators of 128 fp32
//    columns (all 512) and commits them to mbarriers;
//  - while the next tile multiplies, eight epilogue warps read the accumulator with
//    tcgen05.ld (a thread holds 32 consecutive values of one request), add the raw
//    logits, round once to bf16, store, and keep the request's running maximum and its
//    first index. A group of at most 64 requests fills X twice (rows 64..127 repeat rows
//    0..63), so that all four TMEM lane groups hold its products: lane groups 0-1 take
//    the tile's columns 0..63 and 2-3 columns 64..127, 32 per warp.
// At B <= 128 one cooperative launch runs all K positions, with a grid barrier between
// positions (see the kernel); otherwise one launch per position.
// key = (order-preserving bits of the bf16 value) << 32 | (0xffffffff - v): the largest
// value wins and, among equal values, the lowest index. Each CTA ends with one
// atomicMax per request; max is order-free, so results do not depend on scheduling.
// The next position reads y from those keys; a last small launch writes the tokens.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "sv_common.cuh"
#include "sv_launch.cuh"

namespace sv {

constexpr int MK_M = 128;        // requests per group (UMMA M; rows past the batch are zero)
constexpr int MK_N = 128;        // vocabulary rows per tile (UMMA N)
constexpr int MK_KB = 64;        // K elements per 128-byte swizzle block
constexpr int MK_EPI_WARPS = 8;  // epilogue warps: two per TMEM lane group, half a tile each
// and a U TMA warp, an MMA warp and a raw-logit TMA warp
constexpr int MK_THREADS = 32 * (3 + MK_EPI_WARPS);
constexpr int MK_XBLK = MK_M * 128;      // one block of X: 128 rows x 128 bytes
constexpr int MK_UBLK = MK_N * 128;      // one block of a U tile: 128 rows x 128 bytes
constexpr int MK_RING = 4;               // most U tiles in flight
constexpr int MK_ACC = 4;                    // accumulator stages in TMEM
constexpr uint32_t MK_TMEM_COLS = MK_ACC * MK_N;
constexpr int MK_RAWBOX = 64 * 128;  // raw logits of 64 requests x 64 columns (bf16)
constexpr int MK_RSTAGES = 8;        // most raw-logit stages
// U buffers: four at r <= 128, two above (shared memory).
__host__ __device__ constexpr int mk_uring(int nkb) { return nkb <= 2 ? 4 : 2; }
// Bytes of the raw-logit ring: 64 KB, or at r > 192 the 32 KB that the 227 KB of
// shared memory leave next to X, the U ring, alignment and static variables.
__host__ __device__ constexpr int mk_raw_bytes(int nkb) { return nkb <= 3 ? 65536 : 32768; }

struct MarkovArgs {
  const uint16_t* L;     // [B, K, V] raw logits (bf16 bits)
  const uint16_t* U;     // [V, r]
  const uint16_t* Vm;    // [V, r]
  const int32_t* prev;   // [B]
  uint16_t* out;         // [B, K, V] corrected logits
  unsigned long long* keys;  // [K, B]
  int32_t* tok;          // [B, K]
  WsHeader* hdr;
  int B, K, V, r;
  int k, kend;  // positions k .. kend - 1 in this launch
};

__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// Order-preserving 16-bit code of a bf16 value (-0 counts as +0).
__device__ __forceinline__ uint32_t bf_order(uint16_t h) {
  if (h == 0x8000u) h = 0;
  return (h & 0x8000u) ? static_cast<uint32_t>(~h & 0xffffu) : static_cast<uint32_t>(h | 0x8000u);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)),
               "l"(src), "l"(pol)
               : "memory");
}
// Box (x = column, y = position, z = request) of a 3-D tensor map into shared memory.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Tensor-core (tcgen05) and tensor-map TMA wrappers.
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor of a K-major operand in the canonical 128-byte
// swizzled layout: 8-row groups 1024 bytes apart (stride byte offset), rows of 128
// bytes, the leading byte offset unused; descriptor version 1, swizzle mode 128 B.
// The buffer must be 1024-byte aligned.
__device__ __forceinline__ uint64_t sw128_desc(const void* smem) {
  const uint32_t a = smem_addr(smem);
  return static_cast<uint64_t>((a >> 4) & 0x3fffu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both K-major,
// N = MK_N, M = MK_M.
constexpr uint32_t MK_IDESC = (1u << 4) | (1u << 7) | (1u << 10) |
                              (static_cast<uint32_t>(MK_N >> 3) << 17) |
                              (static_cast<uint32_t>(MK_M >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(MK_IDESC), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// Tile (x = column, y = row) of a 2-D tensor map into shared memory, with an L2 cache
// policy.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Probe of an mbarrier phase that may suspend the thread for up to `ns` nanoseconds
// (or until the phase completes), so waiting lanes do not spin through issue slots.
__device__ __forceinline__ bool mbar_try_ns(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Barrier `id` among the first `n` threads that reach it (whole warps).
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Bounded wait for an mbarrier phase; false (and a status report) when it runs out.
__device__ bool mk_wait(uint64_t* bar, uint32_t parity, const MarkovArgs& A) {
  const long long t0 = clock64();
  while (!mbar_try_ns(bar, parity, 2000u)) {
    if (clock64() - t0 > WAIT_CYCLES) {
      atomicOr(&A.hdr->status, ST_TIMEOUT);
      return false;
    }
  }
  return true;
}

// The token drafted at position kk-1 of request b (kk > 0), or prev[b]; -1 if invalid.
// The keys are read from L2: other CTAs of the same launch may have written them.
__device__ __forceinline__ int prev_token(const MarkovArgs& A, int kk, int b) {
  if (kk == 0) {
    const int y = __ldg(A.prev + b);
    return (y >= 0 && y < A.V) ? y : -1;
  }
  const unsigned long long key = __ldcg(A.keys + (size_t)(kk - 1) * A.B + b);
  if (key == 0ull) return -1;
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(key));
}

// Shared memory of the step kernel: X (nkb blocks of 128 rows x 128 bytes), the ring
// of U tiles (nkb blocks of 64 rows x 128 bytes each), then the raw-logit ring,
// 1024-byte aligned; at least 116 KB, so that one CTA is resident per SM.
size_t markov_smem_bytes(int r) {
  const int nkb = (r + MK_KB - 1) / MK_KB;
  const size_t need =
      1024 + (size_t)nkb * (MK_XBLK + mk_uring(nkb) * MK_UBLK) + (size_t)mk_raw_bytes(nkb);
  return need > (size_t)116 * 1024 ? need : (size_t)116 * 1024;
}

// RING: the raw logits reach the epilogue through the shared-memory ring, filled by TMA
// from tmL (rows 16-byte aligned); otherwise by plain loads.
// Positions A.k .. A.kend - 1 run in this launch. With more than one, the launch is
// cooperative (one CTA per SM, gridDim.y == 1): between positions the epilogue warps of
// every CTA meet at a grid barrier (a counter in the workspace header) before they read
// the previous position's argmax and gather the next X, while U and the raw logits of
// the next position keep streaming into their rings. Every (position, tile) pair of the
// CTA has one running index g, which the rings and accumulator stages follow.
template <bool RING, int NUR>
__global__ void __launch_bounds__(MK_THREADS, 1)
    sv_markov_step_kernel(const MarkovArgs A, const __grid_constant__ CUtensorMap tmU,
                          const __grid_constant__ CUtensorMap tmL) {
  extern __shared__ __align__(1024) unsigned char dsm_raw[];
  unsigned char* dsm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // ufull: U tile landed; uempty: its product is done (the buffer may be refilled);
  // afull: accumulator ready; aempty: the epilogue warps have read it;
  // rfull / rempty: a raw-logit stage landed / was used by its epilogue warps;
  // xfull: X of the next position gathered.
  __shared__ uint64_t ufull[MK_RING], uempty[MK_RING], afull[MK_ACC], aempty[MK_ACC];
  __shared__ uint64_t rfull[MK_RSTAGES], rempty[MK_RSTAGES], xfull;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;     // a grid barrier gave up: skip the remaining ones
  __shared__ int yrow[MK_M];  // the previous token of each row of X (-1: a zero row)
  const int r = A.r, V = A.V, B = A.B;
  const int nkb = (r + MK_KB - 1) / MK_KB;
  unsigned char* Xs = dsm;
  auto ubuf = [&](int q) { return dsm + (size_t)nkb * (MK_XBLK + q * MK_UBLK); };
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g0 = blockIdx.y * MK_M;                 // first request of the group
  const int nb = min(MK_M, B - g0);                 // requests in the group
  const int ntiles = (V + MK_N - 1) / MK_N;
  const uint32_t tile_bytes = static_cast<uint32_t>(nkb) * MK_UBLK;
  // A group of at most 64 requests is multiplied twice (rows 64..127 of X repeat rows
  // 0..63), so that the epilogue warps of all four TMEM lane quadrants hold its products
  // and the two halves take the two column halves of every tile.
  const bool dup = nb <= MK_M / 2;
  int nmine = 0;  // tiles of this CTA per position: blockIdx.x, blockIdx.x + gridDim.x, ...
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x) ++nmine;
  const int npos = A.kend - A.k;
  const int total = npos * nmine;  // (position, tile) pairs, position-major
  // Raw-logit stages: per 64 requests two boxes of 64 rows x 128 bytes (the tile's two
  // 64-column halves), twice that for a group of more; the 128-byte swizzle puts row j's
  // 16-byte chunk c at chunk c ^ (j & 7), so that the epilogue's reads of 32 rows spread
  // over all banks. The number of stages is a power of two (1, 2 or 4).
  constexpr bool rt = RING;
  constexpr int LGU = NUR == 4 ? 2 : 1;  // log2 of the U buffers
  static_assert(NUR == 2 || NUR == 4, "U ring");
  const int nbox = dup ? 1 : 2;          // 64-request blocks of a raw stage
  const int rsb = nbox * 2 * MK_RAWBOX;  // and two 64-column halves
  const int nrs = min(MK_RSTAGES, mk_raw_bytes(nkb) / rsb);
  const int lgr = 31 - __clz(nrs);
  unsigned char* rawq = dsm + (size_t)nkb * (MK_XBLK + NUR * MK_UBLK);
  constexpr int RAW_W = 2 + MK_EPI_WARPS;  // the raw-logit copy warp
  constexpr int EPI0 = 64;                 // first thread of the epilogue warps
  // Pair g (position kk, tile i)'s raw logits into stage g % nrs (one thread): boxes of
  // 64 requests x 1 position x 64 columns, box (hb, ch) at (2 hb + ch) x 8 KB for request
  // block hb and column half ch.
  auto issue_raw = [&](int g, int kk, int i) {
    const int q = g & (nrs - 1);
    const int v0 = (blockIdx.x + i * gridDim.x) * MK_N;
    const uint64_t once = policy_evict_first();
    mbar_arrive_expect_tx(&rfull[q], static_cast<uint32_t>(rsb));
    for (int hb = 0; hb < nbox; ++hb)
      for (int ch = 0; ch < 2; ++ch)
        tma_load_3d(rawq + (size_t)q * rsb + (size_t)(2 * hb + ch) * MK_RAWBOX, &tmL,
                    v0 + 64 * ch, kk, g0 + 64 * hb, &rfull[q], once);
  };
  auto issue_u = [&](int g, int i) {  // U tile i into buffer g % NUR (one thread)
    const int q = g & (NUR - 1);
    const uint64_t keep = policy_evict_last();  // U is read again at every position
    mbar_arrive_expect_tx(&ufull[q], tile_bytes);
    const int t = blockIdx.x + i * gridDim.x;
    for (int kb = 0; kb < nkb; ++kb)
      tma_load_2d(ubuf(q) + (size_t)kb * MK_UBLK, &tmU, kb * MK_KB, t * MK_N, &ufull[q], keep);
  };
  // X of position kk by threads t0 .. t0 + nthr - 1 (yrow holds its previous tokens): row
  // m = request g0 + m, the gathered Vm row, zero past the group, past r, or for an
  // invalid previous token; 16-byte chunks placed in the swizzled layout.
  auto gather_x = [&](int t0, int nthr) {
    const uint64_t keep = policy_evict_last();
    const int cpr = nkb * (MK_KB / 8);  // 16-byte chunks per padded row
    for (int i = tid - t0; i < MK_M * cpr; i += nthr) {
      const int m = i / cpr, c = i - m * cpr;
      const int kb = c >> 3, cc = c & 7;
      unsigned char* dst = Xs + (size_t)kb * MK_XBLK + m * 128 + ((cc ^ (m & 7)) << 4);
      const int y = c * 8 < r ? yrow[m] : -1;
      if (y >= 0)
        cp_async16(dst, A.Vm + (size_t)y * r + c * 8, keep);
      else
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    cp_async_wait_all();
    // The tensor cores read X through the async proxy.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  };
  auto set_yrow = [&](int kk, int j) {  // thread j < MK_M: row j's previous token
    const int mr = dup ? (j & (MK_M / 2 - 1)) : j;
    yrow[j] = mr < nb ? prev_token(A, kk, g0 + mr) : -1;
  };

  if (tid == 0) {
    for (int q = 0; q < NUR; ++q) {
      mbar_init(&ufull[q], 1);
      mbar_init(&uempty[q], 1);
    }
    for (int q = 0; q < MK_ACC; ++q) {
      mbar_init(&afull[q], 1);
      mbar_init(&aempty[q], MK_EPI_WARPS);
    }
    for (int q = 0; q < nrs; ++q) {
      mbar_init(&rfull[q], 1);
      mbar_init(&rempty[q], MK_EPI_WARPS);
    }
    mbar_init(&xfull, 1);
    s_abort = 0;
    fence_mbar_init();
    // U does not depend on X: the first tiles of the ring start landing while X is
    // gathered (this thread is the TMA producer).
    for (int g = 0; g < NUR && g < total; ++g) issue_u(g, g % nmine);
  }
  if (tid < MK_M) set_yrow(A.k, tid);  // one read of each request's previous token
  if (w == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_base)),
                 "r"(MK_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  __syncthreads();  // yrow and the barriers
  if (w == RAW_W) {
    // The copy thread starts the raw-logit ring while the others gather X.
    if (rt && lane == 0)
      for (int g = 0; g < nrs && g < total; ++g) issue_raw(g, A.k + g / nmine, g % nmine);
  } else {
    gather_x(0, 32 * RAW_W);
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = tmem_base;

  if (w == 0) {
    // U producer (lane 0): pair g's tile once its buffer's previous product is done.
    if (lane == 0) {
      int g = NUR, i = NUR % max(nmine, 1);
      for (; g < total; ++g) {
        if (!mk_wait(&uempty[g & (NUR - 1)], static_cast<uint32_t>(((g >> LGU) - 1) & 1), A))
          break;
        issue_u(g, i);
        if (++i == nmine) i = 0;
      }
      // After a timeout, let the copies already issued land before the CTA exits.
      for (int j = max(0, min(g, total) - NUR); j < min(g, total); ++j)
        mk_wait(&ufull[j & (NUR - 1)], static_cast<uint32_t>((j >> LGU) & 1), A);
    }
  } else if (w == 1) {
    // MMA issuer (lane 0): pair g's product into accumulator g % MK_ACC once its U tile
    // has landed, the epilogue warps have read that accumulator's previous tile, and (at
    // the first tile of a later position) that position's X is gathered.
    if (lane == 0) {
      const uint64_t ad = sw128_desc(Xs);
      const int nk = r / 16;
      int i = 0, pos = 0;
      for (int g = 0; g < total; ++g) {
        const int q = g & (NUR - 1), a = g & (MK_ACC - 1);
        if (i == 0 && pos > 0 && !mk_wait(&xfull, static_cast<uint32_t>((pos - 1) & 1), A)) break;
        if (!mk_wait(&ufull[q], static_cast<uint32_t>((g >> LGU) & 1), A)) break;
        if (g >= MK_ACC && !mk_wait(&aempty[a], static_cast<uint32_t>(((g >> 2) - 1) & 1), A))
          break;
        tmem_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(a * MK_N);
        const uint64_t bd = sw128_desc(ubuf(q));
        for (int kk = 0; kk < nk; ++kk) {
          // 16 elements = 32 bytes along K inside a 128-byte block; X's blocks and the U
          // tile's are 16 KB apart.
          const uint64_t sub = static_cast<uint64_t>((kk & 3) * 2);
          umma_bf16(d, ad + static_cast<uint64_t>((kk >> 2) * (MK_XBLK >> 4)) + sub,
                    bd + static_cast<uint64_t>((kk >> 2) * (MK_UBLK >> 4)) + sub, kk > 0 ? 1u : 0u);
        }
        umma_commit(&uempty[q]);  // the U buffer is free when these products are done
        umma_commit(&afull[a]);   // and the accumulator is ready
        if (++i == nmine) {
          i = 0;
          ++pos;
        }
      }
    }
  } else if (w < 2 + MK_EPI_WARPS) {
    // Epilogue warps: warp w reads TMEM lanes 32 (w % 4) .. + 31, i.e. request g0 + m,
    // m = 32 (w % 4) + lane, of every tile, in chunks of 32 columns: with the group
    // doubled (rows 64..127 repeat 0..63) quadrants 0-1 take columns 0..63 and 2-3
    // columns 64..127, 32 per warp; otherwise each warp takes 64 columns, as two chunks.
    const int m = 32 * (w & 3) + lane;        // TMEM lane (row of the product)
    const int mreq = dup ? (m & (MK_M / 2 - 1)) : m;
    const int h = (w - 2) >> 2;               // which of the two warps of its lane group
    const int nsub = dup ? 1 : 2;
    const int cbase = dup ? 64 * ((w & 3) >> 1) + 32 * h : 64 * h;
    const int rr = mreq & 63;                 // row of the request in its raw box
    const int hb = dup ? 0 : (mreq >> 6);     // its request block
    const size_t KV = (size_t)A.K * V;
    const int b = g0 + mreq;
    const bool live = mreq < nb;
    bool dead = false;  // a wait gave up: skip the work, keep meeting the other warps
    int g = 0;
    for (int kk = A.k; kk < A.kend; ++kk) {
      const uint16_t* Lrow = A.L + (size_t)(live ? b : 0) * KV + (size_t)kk * V;
      uint16_t* Orow = A.out + (size_t)(live ? b : 0) * KV + (size_t)kk * V;
      uint32_t best = 0;   // order-preserving code (+1) of the request's largest value so far
      int best_v = -1;     // its first index (values are visited in increasing v)
      auto see = [&](uint16_t hv, int v) {
        const uint32_t c = bf_order(hv) + 1u;
        if (c > best) {
          best = c;
          best_v = v;
        }
      };
      for (int i = 0; i < nmine; ++i, ++g) {
        if (dead) continue;
        const int a = g & (MK_ACC - 1), q = g & (nrs - 1);
        bool ok = true;
        if (lane == 0) ok = mk_wait(&afull[a], static_cast<uint32_t>((g >> 2) & 1), A);
        // Every lane reads the stage, so every lane observes its phase: the copy's
        // writes are visible to a thread through its own wait on the barrier.
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) ||
            (rt && !__all_sync(0xffffffffu,
                               mk_wait(&rfull[q], static_cast<uint32_t>((g >> lgr) & 1), A)))) {
          dead = true;
          continue;
        }
        tmem_fence_after();
        for (int sb = 0; sb < nsub; ++sb) {
        const int c0 = cbase + 32 * sb;  // the chunk's first column in the tile
        const int vq = (blockIdx.x + i * gridDim.x) * MK_N + c0;
        const bool full = rt && live && vq + 32 <= V;
        // The chunk's 32 columns of the request's row in the stage: 16-byte chunks
        // 4 ((c0 / 32) % 2) .. + 3 of row rr of box (hb, c0 / 64), placed by the 128-byte
        // swizzle.
        uint4 raw[4];
        if (rt) {
          const unsigned char* rp =
              rawq + (size_t)q * rsb + (size_t)(2 * hb + (c0 >> 6)) * MK_RAWBOX + rr * 128;
          const int c4 = 4 * ((c0 >> 5) & 1);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            raw[j] = *reinterpret_cast<const uint4*>(rp + (((c4 + j) ^ (rr & 7)) << 4));
        }
        const uint32_t tcol = tmem + ((static_cast<uint32_t>(32 * (w & 3))) << 16) +
                              static_cast<uint32_t>(a * MK_N + c0);
        float acc[32];
        tmem_ld32(tcol, acc);
        if (sb == nsub - 1) {
          // The accumulator is in registers (tcgen05.wait::ld): release it to the MMA
          // issuer.
          tmem_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&aempty[a]);
        }
        if (full) {
          // Pairs of values: one packed fp32x2 add, one rounding to bf16x2 (round to
          // nearest even, as the per-value path), then the tile's maximum by packed
          // NaN-propagating max. Only a tile whose maximum beats the running best looks
          // for its first index; a tile with a NaN takes the per-value rule.
          uint32_t hp[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t wv[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const int e = j * 8 + e2 * 2;  // elements e (low half) and e + 1 (high half)
              float2 z;
              asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
                  "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
                  "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
                  : "=f"(z.x), "=f"(z.y)
                  : "f"(bf_lo(wv[e2])), "f"(bf_hi(wv[e2])), "f"(acc[e]), "f"(acc[e + 1]));
              const __nv_bfloat162 o = __floats2bfloat162_rn(z.x, z.y);
              hp[j * 4 + e2] = *reinterpret_cast<const uint32_t*>(&o);
            }
            __stcs(reinterpret_cast<uint4*>(Orow + vq) + j,
                   make_uint4(hp[j * 4], hp[j * 4 + 1], hp[j * 4 + 2], hp[j * 4 + 3]));
          }
          // A tree of depth four over the 16 packed pairs (a chain would be 15 deep).
          __nv_bfloat162 mt[8];
#pragma unroll
          for (int t = 0; t < 8; ++t)
            mt[t] = __hmax2_nan(*reinterpret_cast<const __nv_bfloat162*>(&hp[2 * t]),
                                *reinterpret_cast<const __nv_bfloat162*>(&hp[2 * t + 1]));
#pragma unroll
          for (int t = 0; t < 4; ++t) mt[t] = __hmax2_nan(mt[2 * t], mt[2 * t + 1]);
          mt[0] = __hmax2_nan(__hmax2_nan(mt[0], mt[1]), __hmax2_nan(mt[2], mt[3]));
          const __nv_bfloat16 m = __hmax_nan(mt[0].x, mt[0].y);
          if (__hisnan(m)) {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              see(static_cast<uint16_t>(hp[t] & 0xffffu), vq + 2 * t);
              see(static_cast<uint16_t>(hp[t] >> 16), vq + 2 * t + 1);
            }
          } else {
            const uint32_t c = bf_order(__bfloat16_as_ushort(m)) + 1u;
            if (c > best) {  // the first column holding the maximum (-0 counts as +0)
              int e = 31;
#pragma unroll
              for (int t = 15; t >= 0; --t) {
                if (bf_order(static_cast<uint16_t>(hp[t] >> 16)) + 1u == c) e = 2 * t + 1;
                if (bf_order(static_cast<uint16_t>(hp[t] & 0xffffu)) + 1u == c) e = 2 * t;
              }
              best = c;
              best_v = vq + e;
            }
          }
        } else if (live) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            if (vq + e >= V) continue;
            const uint16_t hv = __bfloat16_as_ushort(
                __float2bfloat16_rn(__fadd_rn(bf2f(__ldcs(Lrow + vq + e)), acc[e])));
            __stcs(Orow + vq + e, hv);
            see(hv, vq + e);
          }
        }
        }  // chunk
        // The raw-logit stage is released only once every lane has used its values: a
        // load whose result is still pending does not hold the stage, and a refill
        // issued on an earlier release could overwrite it before it is read.
        if (rt) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&rempty[q]);
        }
      }
      if (live && best_v >= 0)
        atomicMax(A.keys + (size_t)kk * B + b,
                  (static_cast<unsigned long long>(best - 1u) << 32) |
                      (0xffffffffull - static_cast<unsigned>(best_v)));
      if (kk + 1 == A.kend) break;
      // Next position: every CTA's argmax of this one must be in before its previous
      // tokens are read. The epilogue warps of this CTA meet (named barrier 1); one
      // thread counts the CTA in and waits for all.
      named_bar_sync(1, 32 * MK_EPI_WARPS);
      if (tid == EPI0) {
        // One release-ordered add: the CTA's maxima (ordered before it by the named
        // barrier) are visible to whoever reads the count with acquire.
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&A.hdr->mk_pos) : "memory");
        const uint32_t want = gridDim.x * static_cast<uint32_t>(kk + 1 - A.k);
        const long long t0 = clock64();
        while (!s_abort && ld_acquire(&A.hdr->mk_pos) < want) {
          if (clock64() - t0 > WAIT_CYCLES) {
            atomicOr(&A.hdr->status, ST_TIMEOUT);
            s_abort = 1;
          }
        }
      }
      named_bar_sync(1, 32 * MK_EPI_WARPS);
      if (tid - EPI0 < MK_M) set_yrow(kk + 1, tid - EPI0);
      named_bar_sync(1, 32 * MK_EPI_WARPS);
      // The products of this position are done (every accumulator was waited for), so
      // X may be overwritten.
      gather_x(EPI0, 32 * MK_EPI_WARPS);
      named_bar_sync(1, 32 * MK_EPI_WARPS);
      if (tid == EPI0) mbar_arrive(&xfull);
    }
  } else if (rt && lane == 0) {
    // Raw-logit copy thread: pair g once its stage's previous pair has been used (the
    // first stages are already on their way).
    int g = nrs, kk = A.k + nrs / nmine, i = nrs % nmine;
    for (; g < total; ++g) {
      if (!mk_wait(&rempty[g & (nrs - 1)], static_cast<uint32_t>(((g >> lgr) - 1) & 1), A))
        break;
      issue_raw(g, kk, i);
      if (++i == nmine) {
        i = 0;
        ++kk;
      }
    }
    // After a timeout, let the copies already issued land before the CTA exits (at
    // once otherwise: each of these phases has been consumed).
    for (int j = max(0, min(g, total) - nrs); j < min(g, total); ++j)
      mk_wait(&rfull[j & (nrs - 1)], static_cast<uint32_t>((j >> lgr) & 1), A);
  }

  tmem_fence_before();
  __syncthreads();
  if (w == 0) {
    tmem_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(MK_TMEM_COLS)
                 : "memory");
  }
}

// Drafted tokens from the keys; requests with an invalid previous token get -1.
__global__ void sv_markov_finish_kernel(const MarkovArgs A) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= A.B) return;
  if (b == 0) A.hdr->mk_pos = 0;  // the position barrier's counter, for the next call
  const int y0 = __ldg(A.prev + b);
  const bool ok = y0 >= 0 && y0 < A.V;
  if (!ok) atomicOr(&A.hdr->status, ST_DEVICE_INPUT);
  for (int k = 0; k < A.K; ++k) {
    const unsigned long long key = A.keys[(size_t)k * A.B + b];
    A.tok[(size_t)b * A.K + k] =
        (ok && key) ? static_cast<int>(0xffffffffu - static_cast<uint32_t>(key)) : -1;
  }
}

// The driver's tensor-map encoder, looked up once through the runtime.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    (void)cudaGetLastError();
  });
  return fn;
}

cudaError_t launch_markov(const uint16_t* L, const uint16_t* U, const uint16_t* Vm,
                          const int32_t* prev, int B, int K, int V, int r, uint16_t* out,
                          int32_t* tok, unsigned long long* keys, WsHeader* hdr, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    const int smax = (int)markov_smem_bytes(SV_MAX_MARKOV_R);
    const void* ks[4] = {reinterpret_cast<const void*>(sv_markov_step_kernel<false, 2>),
                         reinterpret_cast<const void*>(sv_markov_step_kernel<false, 4>),
                         reinterpret_cast<const void*>(sv_markov_step_kernel<true, 2>),
                         reinterpret_cast<const void*>(sv_markov_step_kernel<true, 4>)};
    cudaError_t e = cudaSuccess;
    for (int j = 0; j < 4 && e == cudaSuccess; ++j)
      e = cudaFuncSetAttribute(ks[j], cudaFuncAttributeMaxDynamicSharedMemorySize, smax);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // U as a 2-D tensor [V rows, r columns] of bf16: boxes of 64 rows x 64 columns (128
  // bytes, 128-byte swizzle), zeros outside the tensor.
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tm;
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(r), static_cast<cuuint64_t>(V)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(r) * 2};
  const cuuint32_t box[2] = {MK_KB, MK_N};  // 64 columns (128 bytes) x 128 rows
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(U), gdim, gstride, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // The raw logits go through the shared-memory ring when their rows are 16-byte
  // aligned (otherwise the kernel reads them with plain loads): by TMA, as a 3-D tensor
  // [B][K][V] of bf16 in boxes of 64 columns (128 bytes, 128-byte swizzle) x 1 position
  // x 64 requests, zeros past V and B.
  const bool ring = V % 8 == 0 && reinterpret_cast<uintptr_t>(L) % 16 == 0;
  CUtensorMap tl = tm;  // a valid map, unused without the ring
  if (ring) {
    const cuuint64_t ldim[3] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(K),
                                static_cast<cuuint64_t>(B)};
    const cuuint64_t lstride[2] = {static_cast<cuuint64_t>(V) * 2,
                                   static_cast<cuuint64_t>(K) * static_cast<cuuint64_t>(V) * 2};
    const cuuint32_t lbox[3] = {64, 1, 64};
    const cuuint32_t lestr[3] = {1, 1, 1};
    if (enc(&tl, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(L), ldim, lstride,
            lbox, lestr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaMemsetAsync(keys, 0, sizeof(unsigned long long) * (size_t)K * B, st);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  MarkovArgs A{L, U, Vm, prev, out, keys, tok, hdr, B, K, V, r, 0, K};
  const int ntiles = (V + MK_N - 1) / MK_N;
  const dim3 grid(static_cast<unsigned>(ntiles < sms ? ntiles : sms),
                  static_cast<unsigned>((B + MK_M - 1) / MK_M));
  const size_t smem = markov_smem_bytes(r);
  // One group of requests (B <= 128): all K positions in one cooperative launch (its
  // CTAs, one per SM, meet at a grid barrier between positions). Otherwise one launch
  // per position.
  int coop = 0;
  if ((e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess)
    return e;
  const bool loop = grid.y == 1 && coop != 0;
  for (int k = 0; k < K; k = A.kend) {
    A.k = k;
    A.kend = loop ? K : k + 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(MK_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = loop ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool u4 = mk_uring((r + MK_KB - 1) / MK_KB) == 4;
    e = ring ? (u4 ? cudaLaunchKernelEx(&cfg, sv_markov_step_kernel<true, 4>, A, tm, tl)
                   : cudaLaunchKernelEx(&cfg, sv_markov_step_kernel<true, 2>, A, tm, tl))
             : (u4 ? cudaLaunchKernelEx(&cfg, sv_markov_step_kernel<false, 4>, A, tm, tl)
                   : cudaLaunchKernelEx(&cfg, sv_markov_step_kernel<false, 2>, A, tm, tl));
    if (e != cudaSuccess) return e;
  }
  sv_markov_finish_kernel<<<(B + 127) / 128, 128, 0, st>>>(A);
  return cudaGetLastError();
}

}  // namespace sv
