// Router: scores -> top-k experts per token (the step before the path).
//
// Page "fused_moe.py 分析", section "topk_ids, topk_weights 的由来以及内容"
// (fused_topk): per token, softmax over the E router logits or an element-wise
// sigmoid, keep the k best experts, optionally renormalise their weights;
// expert_map (same page) turns global expert ids into this shard's ids.
//
// One warp per token.  Lane l holds logits l, l + 32, ... in registers (VPL
// of them, E <= 32 VPL), so the row is read from HBM once, coalesced.
//  * selection: k rounds of a warp arg-max over the logits still in play,
//    (larger logit, then smaller index) wins; both scores increase with the
//    logit, so this is the top-k of the scores with no rounding deciding it.
//    A round is two redux.sync reductions (max of order-preserving keys, min
//    of the expert ids holding it) and a rescan in the winning lane only --
//    a shuffle arg-max with a full rescan per round took 3x longer at k = 8;
//  * softmax: m = row max, Z = sum exp(l - m) (warp sums); weight exp(l - m)/Z,
//    or exp(l - m) / sum over the k kept when renormalising (Z cancels);
//  * sigmoid: 1 / (1 + exp(-l)), renormalised over the k kept if asked.
// Lane i writes slot i of the token's outputs.
#include "../../include/moe_ffn.h"
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int ROUTER_WARPS = 8;

__device__ __forceinline__ float load_logit(const void* p, size_t i, bool bf16) {
  return bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i])
              : reinterpret_cast<const float*>(p)[i];
}

template <int VPL>
__global__ void __launch_bounds__(ROUTER_WARPS * 32)
    k_topk_router(const void* __restrict__ logits, bool bf16, int M, int E, int k, bool sigmoid,
                  bool renorm, const int32_t* __restrict__ expert_map, float* __restrict__ w_out,
                  int32_t* __restrict__ id_out, int32_t* __restrict__ tei_out) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * ROUTER_WARPS + (threadIdx.x >> 5);
  if (t >= M) return;
  const size_t row = (size_t)t * E;
  float v[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = j * 32 + lane;
    v[j] = e < E ? load_logit(logits, row + e, bf16) : -INFINITY;
  }
  // row maximum and softmax denominator
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < VPL; ++j) m = fmaxf(m, v[j]);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float z = 0.0f;
  if (!sigmoid) {
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      if (j * 32 + lane < E) z += expf(v[j] - m);
#pragma unroll
    for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  }
  // k rounds of arg-max; slot i's winner ends up in lane i.  Each lane keeps
  // the position of its best logit still in play (ties: the lower position,
  // i.e. the lower expert); a round is one warp max over order-preserving
  // keys of those logits and one warp min over the expert ids holding the
  // maximum, then only the winning lane looks for its next best.
  uint32_t taken = 0;          // bit j: logit j*32 + lane already selected
  auto best_pos = [&](float& val) {   // position and value of the lane's best in play
    int b = -1;
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      if (j * 32 + lane < E && !(taken >> j & 1u) && (b < 0 || v[j] > val)) {
        b = j;
        val = v[j];
      }
    return b;
  };
  float bv = 0.0f;
  int bj = best_pos(bv);
  int my_id = -1;
  float my_logit = 0.0f;
  for (int i = 0; i < k; ++i) {
    // order-preserving key of the float (larger float -> larger key; -0 is
    // keyed as +0, which compares equal); lanes with nothing left offer
    // key 0 and no expert
    const uint32_t u = __float_as_uint(bv) == 0x80000000u ? 0u : __float_as_uint(bv);
    const uint32_t key = bj < 0 ? 0u : ((u & 0x80000000u) ? ~u : (u | 0x80000000u));
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
    const uint32_t cand = (bj >= 0 && key == kmax) ? (uint32_t)(bj * 32 + lane) : 0xffffffffu;
    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    // with k <= E some lane always offers an expert (win < E)
    const int bi = win < (uint32_t)E ? (int)win : -1;
    const float wv = __shfl_sync(0xffffffffu, bv, bi >= 0 ? (bi & 31) : 0);
    if (bi >= 0 && (bi & 31) == lane) {
      taken |= 1u << (bi >> 5);
      bj = best_pos(bv);
    }
    if (lane == i) {
      my_id = bi;
      my_logit = wv;
    }
  }
  float w = 0.0f;
  if (lane < k) w = sigmoid ? 1.0f / (1.0f + expf(-my_logit)) : expf(my_logit - m);
  if (renorm || !sigmoid) {
    float d = z;                        // softmax, not renormalised: the full sum
    if (renorm) {
      d = w;                            // the k kept scores
#pragma unroll
      for (int o = 16; o; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    }
    w = w / d;
  }
  if (lane < k) {
    const size_t o = (size_t)t * k + lane;
    w_out[o] = w;
    id_out[o] = (expert_map != nullptr && my_id >= 0) ? expert_map[my_id] : my_id;
    if (tei_out != nullptr) tei_out[o] = (int32_t)o;
  }
}

}  // namespace

cudaError_t launch_topk_router(const void* logits, bool bf16, int M, int E, int k, bool sigmoid,
                               bool renorm, const int32_t* expert_map, float* w, int32_t* ids,
                               int32_t* tei, cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  const dim3 grid((M + ROUTER_WARPS - 1) / ROUTER_WARPS), block(ROUTER_WARPS * 32);
  const int vpl = (E + 31) / 32;
#define MOE_ROUTER_CASE(N)                                                                    \
  if (vpl <= N) {                                                                             \
    k_topk_router<N><<<grid, block, 0, stream>>>(logits, bf16, M, E, k, sigmoid, renorm,      \
                                                 expert_map, w, ids, tei);                    \
    return cudaGetLastError();                                                                \
  }
  MOE_ROUTER_CASE(1)
  MOE_ROUTER_CASE(2)
  MOE_ROUTER_CASE(4)
  MOE_ROUTER_CASE(8)
  MOE_ROUTER_CASE(16)
  MOE_ROUTER_CASE(32)
#undef MOE_ROUTER_CASE
  return cudaErrorInvalidValue;
}

}  // namespace moe
