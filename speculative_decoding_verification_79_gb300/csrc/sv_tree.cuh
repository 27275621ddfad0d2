// sv_tree.cuh -- arguments and launch of the tree verification kernel.
#pragma once
#include "sv_common.cuh"

namespace sv {

// Arguments of tree verification (built by the C-ABI layer). Every array is [B, N] or
// [B, N, V], row-major; see sv_verify_tree in specverify.h for their meaning.
struct TreeArgs {
  const void* tgt;       // [B, N, V] target logits
  const void* drf;       // [B, N, V] draft logits (unused at T == 0)
  const int32_t* par;    // [B, N] parent links
  const int32_t* tok;    // [B, N] drafted tokens
  const int32_t* nn;     // [B] nodes in use
  const float* uni;      // [B, N] uniforms (unused at T == 0)
  int B, N, V;
  float a;     // log2(e) / T rounded to fp32 (T > 0)
  float a_lo;  // log2(e) / T - a
  int32_t* out_tok;      // [B, N]
  int32_t* out_acc;      // [B]
  int32_t* out_path;     // [B, N] or null
  WsHeader* hdr;         // status word
};

// Launches one cluster of CTAs per request; the cluster size (1..8) is chosen so that
// the batch is resident at once when it can be. *cluster_out (if not null) receives it.
cudaError_t launch_tree(const TreeArgs& A, bool bf16, bool greedy, cudaStream_t st,
                        int* cluster_out);

}  // namespace sv
