// Batched (masked) expert layout: the routing step of fused_experts_batched.
//
// Page "fused_moe.py 分析", activation formats: after dispatch the activations
// are either Standard [M, K] or BatchedExperts [E, max_tokens, K] -- one
// buffer of max_tokens rows per local expert, filled up to that expert's token
// count; page "Blackwell 上的 DeepGEMM FusedMoE（vLLM）", §2.5 (DeepEP low-latency
// dispatch): the experts then run a masked grouped GEMM and the per-expert
// counts come with the dispatch, so no counting pass is needed.
//
// Here the layout's rows are the GEMMs' rows directly: with T = max_tokens a
// multiple of the 128-row tile, expert e owns row blocks [e T/128, (e+1) T/128)
// and a block takes part when it holds at least one of the expert's first
// count[e] rows; the other blocks get expert id -1 and every GEMM skips them.
// Counts are clamped to [0, T].  For the quantising permute, row r of expert e
// maps to itself (r < count) or to the padding id E*T (zero row, zero scale).
#include <algorithm>

#include "moe_internal.h"

namespace moe {
namespace {

__global__ void k_batched_blocks(const int32_t* __restrict__ counts, int E, int T,
                                 int32_t* __restrict__ block_expert_ids,
                                 int32_t* __restrict__ num_post_padded,
                                 int32_t* __restrict__ sorted_ids) {
  const int blocks_per_expert = T / 128;
  const int nblocks = E * blocks_per_expert;
  const int rows = E * T;
  const int stride = gridDim.x * blockDim.x;
  const int i0 = blockIdx.x * blockDim.x + threadIdx.x;
  if (i0 == 0) *num_post_padded = rows;
  for (int b = i0; b < nblocks; b += stride) {
    const int e = b / blocks_per_expert, j = b - e * blocks_per_expert;
    const int c = min(max(counts[e], 0), T);
    block_expert_ids[b] = j * 128 < c ? e : -1;
  }
  if (sorted_ids != nullptr) {
    for (int r = i0; r < rows; r += stride) {
      const int e = r / T;
      const int c = min(max(counts[e], 0), T);
      sorted_ids[r] = r - e * T < c ? r : rows;
    }
  }
}

}  // namespace

cudaError_t launch_batched_blocks(const int32_t* counts, int E, int T, int32_t* block_expert_ids,
                                  int32_t* num_post_padded, int32_t* sorted_ids,
                                  cudaStream_t stream) {
  const int rows = E * T;
  const int work = sorted_ids != nullptr ? rows : E * (T / 128);
  const int threads = 256;
  const int grid = std::max(1, std::min((work + threads - 1) / threads, 4 * num_sms()));
  k_batched_blocks<<<grid, threads, 0, stream>>>(counts, E, T, block_expert_ids, num_post_padded,
                                                 sorted_ids);
  return cudaGetLastError();
}

}  // namespace moe
