// sv_markov.cu -- the Markov logit-bias head of the drafter (sm_103a).
//
// DSpark Guide, "1. The Markov Logit-Bias Head": the parallel backbone's raw logits of
// draft position k are corrected by a low-rank bigram term of the token drafted at
// position k-1,
//     L'_k = L_k + U (Vm[y_{k-1}, :])^T,   U, Vm in R^{V x r},
// and the next token is drafted from L'_k (greedy here: the lowest-index argmax, as
// in the page's sketch), so the positions run one after another.
//
// One launch per position. For a batch of B requests the correction is a product of
// U [V, r] with X [r, B], X's columns the gathered rows Vm[y_b, :]: a dense
// contraction, done on the tensor cores (bf16 inputs, fp32 accumulation) by
// mma.sync.m16n8k16. A CTA owns 128 vocabulary rows and up to 64 requests: it copies
// its U tile (kept in L2 across positions: evict_last) and the 64 gathered rows of Vm
// into shared memory with cp.async while each thread loads the raw logits of its own
// accumulator elements into registers, multiplies (8 warps x 16 rows x 64 columns),
// adds, rounds once to bf16 and stores from the registers, and folds the tile's
// argmax of each request into a 64-bit key per (position, request) with atomicMax:
// key = (order-preserving bits of the bf16 value) << 32 | (0xffffffff - v), so the
// largest value wins and, among equal values, the lowest index; max is order-free,
// so results do not depend on CTA scheduling. The next position reads y from those
// keys; a last small launch writes the drafted tokens.
#include <cuda_bf16.h>

#include "sv_common.cuh"
#include "sv_launch.cuh"

namespace sv {

constexpr int MK_ROWS = 128;   // vocabulary rows per CTA
constexpr int MK_COLS = 64;    // requests per CTA
constexpr int MK_WARPS = 8;    // 16 rows each
constexpr int MK_THREADS = MK_WARPS * 32;
constexpr int MK_PAD = 8;      // bf16 elements of padding per shared-memory row

struct MarkovArgs {
  const uint16_t* L;     // [B, K, V] raw logits (bf16 bits)
  const uint16_t* U;     // [V, r]
  const uint16_t* Vm;    // [V, r]
  const int32_t* prev;   // [B]
  uint16_t* out;         // [B, K, V] corrected logits
  unsigned long long* keys;  // [K, B]
  int32_t* tok;          // [B, K]
  WsHeader* hdr;
  int B, K, V, r, k;
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
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3,
                                        const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
               : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t& b0, uint32_t& b1, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(b0), "=r"(b1)
               : "r"(smem_addr(p)));
}
__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The token drafted at position k-1 of request b (k > 0), or prev[b]; -1 if invalid.
__device__ __forceinline__ int prev_token(const MarkovArgs& A, int b) {
  if (A.k == 0) {
    const int y = __ldg(A.prev + b);
    return (y >= 0 && y < A.V) ? y : -1;
  }
  const unsigned long long key = A.keys[(size_t)(A.k - 1) * A.B + b];
  if (key == 0ull) return -1;
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(key));
}

__global__ void __launch_bounds__(MK_THREADS, 2) sv_markov_step_kernel(const MarkovArgs A) {
  extern __shared__ __align__(128) unsigned char dsm[];
  const int r = A.r, rs = r + MK_PAD;  // shared row stride (bf16 elements)
  uint16_t* Us = reinterpret_cast<uint16_t*>(dsm);                 // [MK_ROWS][rs]
  uint16_t* Xs = Us + (size_t)MK_ROWS * rs;                         // [MK_COLS][rs]
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int v0 = blockIdx.x * MK_ROWS, b0 = blockIdx.y * MK_COLS;
  const int nrows = min(MK_ROWS, A.V - v0), ncols = min(MK_COLS, A.B - b0);
  const uint64_t keep = policy_evict_last();
  const int cpr = r / 8;  // 16-byte chunks per row of U / Vm

  // Copies: the U tile and the gathered rows of Vm (zero rows past the ends).
  for (int i = tid; i < MK_ROWS * cpr; i += MK_THREADS) {
    const int row = i / cpr, c = i - row * cpr;
    uint16_t* dst = Us + (size_t)row * rs + c * 8;
    if (row < nrows)
      cp_async16(dst, A.U + (size_t)(v0 + row) * r + c * 8, keep);
    else
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
  }
  for (int i = tid; i < MK_COLS * cpr; i += MK_THREADS) {
    const int col = i / cpr, c = i - col * cpr;
    uint16_t* dst = Xs + (size_t)col * rs + c * 8;
    const int y = (col < ncols) ? prev_token(A, b0 + col) : -1;
    if (y >= 0)
      cp_async16(dst, A.Vm + (size_t)y * r + c * 8, keep);
    else
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
  }
  // The raw logits of this thread's accumulator elements, straight into registers
  // (their latency overlaps the copies above and the product below): element (n, e)
  // is row 16w + g (+8 for e >= 2), column 8n + 2t (+1 for odd e).
  const int g = lane >> 2, tq = lane & 3;
  const size_t KV = (size_t)A.K * A.V;
  uint16_t lraw[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int row = 16 * w + g + ((e & 2) ? 8 : 0), col = 8 * n + 2 * tq + (e & 1);
      lraw[n][e] = (row < nrows && col < ncols)
                       ? __ldcs(A.L + (size_t)(b0 + col) * KV + (size_t)A.k * A.V + v0 + row)
                       : static_cast<uint16_t>(0);
    }
  }
  cp_async_wait_all();
  __syncthreads();

  // Correction tile: warp w takes rows 16w..16w+15 and all 64 columns.
  float acc[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  const uint16_t* arow = Us + (size_t)(16 * w + (lane & 15)) * rs + (lane >> 4) * 8;
  const uint16_t* brow = Xs + (size_t)(lane & 7) * rs + ((lane >> 3) & 1) * 8;
  for (int k0 = 0; k0 < r; k0 += 16) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4(a0, a1, a2, a3, arow + k0);
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      uint32_t b0r, b1r;
      ldsm_x2(b0r, b1r, brow + (size_t)(8 * n) * rs + k0);
      mma_bf16(acc[n], a0, a1, a2, a3, b0r, b1r);
    }
  }

  // Raw logits + correction, rounded once to bf16, stored from the registers; each
  // column's best key over the warp's 16 rows, then over the 8 warps in shared memory.
  __shared__ unsigned long long red[MK_WARPS][MK_COLS];
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    unsigned long long kb[2] = {0ull, 0ull};  // columns 8n + 2t and 8n + 2t + 1
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int row = 16 * w + g + ((e & 2) ? 8 : 0), col = 8 * n + 2 * tq + (e & 1);
      const uint16_t h = __bfloat16_as_ushort(__float2bfloat16_rn(__fadd_rn(bf2f(lraw[n][e]), acc[n][e])));
      if (row < nrows && col < ncols) {
        __stcs(A.out + (size_t)(b0 + col) * KV + (size_t)A.k * A.V + v0 + row, h);
        const unsigned long long key = (static_cast<unsigned long long>(bf_order(h)) << 32) |
                                       static_cast<unsigned long long>(0xffffffffu - (uint32_t)(v0 + row));
        kb[e & 1] = key > kb[e & 1] ? key : kb[e & 1];
      }
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      unsigned long long m = kb[c];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {  // over g: lanes with the same t hold the same column
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, m, o);
        m = y > m ? y : m;
      }
      if (g == 0) red[w][8 * n + 2 * tq + c] = m;
    }
  }
  __syncthreads();
  if (tid < MK_COLS && tid < ncols) {
    unsigned long long m = 0ull;
#pragma unroll
    for (int q = 0; q < MK_WARPS; ++q) m = red[q][tid] > m ? red[q][tid] : m;
    if (m) atomicMax(A.keys + (size_t)A.k * A.B + b0 + tid, m);
  }
}

// Drafted tokens from the keys; requests with an invalid previous token get -1.
__global__ void sv_markov_finish_kernel(const MarkovArgs A) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= A.B) return;
  const int y0 = __ldg(A.prev + b);
  const bool ok = y0 >= 0 && y0 < A.V;
  if (!ok) atomicOr(&A.hdr->status, ST_DEVICE_INPUT);
  for (int k = 0; k < A.K; ++k) {
    const unsigned long long key = A.keys[(size_t)k * A.B + b];
    A.tok[(size_t)b * A.K + k] =
        (ok && key) ? static_cast<int>(0xffffffffu - static_cast<uint32_t>(key)) : -1;
  }
}

// The U tile and the gathered Vm rows.
size_t markov_smem_bytes(int r) { return (size_t)(MK_ROWS + MK_COLS) * (r + MK_PAD) * 2; }

cudaError_t launch_markov(const uint16_t* L, const uint16_t* U, const uint16_t* Vm,
                          const int32_t* prev, int B, int K, int V, int r, uint16_t* out,
                          int32_t* tok, unsigned long long* keys, WsHeader* hdr, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(sv_markov_step_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)markov_smem_bytes(SV_MAX_MARKOV_R));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaError_t e = cudaMemsetAsync(keys, 0, sizeof(unsigned long long) * (size_t)K * B, st);
  if (e != cudaSuccess) return e;
  MarkovArgs A{L, U, Vm, prev, out, keys, tok, hdr, B, K, V, r, 0};
  const dim3 grid((V + MK_ROWS - 1) / MK_ROWS, (B + MK_COLS - 1) / MK_COLS);
  for (int k = 0; k < K; ++k) {
    A.k = k;
    sv_markov_step_kernel<<<grid, MK_THREADS, markov_smem_bytes(r), st>>>(A);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  sv_markov_finish_kernel<<<(B + 127) / 128, 128, 0, st>>>(A);
  return cudaGetLastError();
}

}  // namespace sv
