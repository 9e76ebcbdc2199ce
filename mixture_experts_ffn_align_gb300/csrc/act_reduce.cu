// SiLU-and-mul (+ dynamic FP8 quantisation) and the weighted top-k
// unpermute-reduce (stages 3 and 5).
//
// Stage 3 follows the page "Blackwell 上的 DeepGEMM FusedMoE（vLLM）", §2.6.4
// (SwiGLU on the bf16 GEMM1 output, optionally quantised per 1x128 group) and
// the page "fused_moe.py 分析" (_silu_and_mul_kernel).  Stage 5 follows §2.6.5
// of the first page (ep_gather: per token and top-k slot, fetch row
// inv_perm[t,i], accumulate w * v in fp32, cast to bf16; slots with id -1 are
// skipped) -- the same result as weighting then moe_sum on page 1 (§4,
// TopKWeightAndReduceContiguous).
//
// Both are HBM-bound elementwise/gather kernels: 16-byte vector loads and
// stores, one CTA per row (token), grid-stride over rows, no shared memory.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

// z[row, :] = bf16(SiLU(bf16 g) * bf16 u) for rows below num_post_padded.
__global__ void __launch_bounds__(128)
    k_act_mul_bf16(const __nv_bfloat16* __restrict__ h1, int I, const int32_t* __restrict__ npp,
                   __nv_bfloat16* __restrict__ z) {
  const int rows = *npp;
  const int nv = I / 8;
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const uint4* g4 = reinterpret_cast<const uint4*>(h1 + (size_t)row * 2 * I);
    const uint4* u4 = reinterpret_cast<const uint4*>(h1 + (size_t)row * 2 * I + I);
    uint4* z4 = reinterpret_cast<uint4*>(z + (size_t)row * I);
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
      uint4 gv = __ldg(g4 + v), uv = __ldg(u4 + v), out;
      const __nv_bfloat16* gb = reinterpret_cast<const __nv_bfloat16*>(&gv);
      const __nv_bfloat16* ub = reinterpret_cast<const __nv_bfloat16*>(&uv);
      __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(&out);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        ob[j] = __float2bfloat16_rn(silu_f32(__bfloat162float(gb[j])) * __bfloat162float(ub[j]));
      z4[v] = out;
    }
  }
}

// Quantised variant: z in fp32, then per 1x128 group amax -> scale -> e4m3.
__global__ void __launch_bounds__(128)
    k_act_mul_fp8(const __nv_bfloat16* __restrict__ h1, int I, const int32_t* __restrict__ npp,
                  uint8_t* __restrict__ zq, float* __restrict__ zs, int ue8m0) {
  const int rows = *npp;
  const int nv = I / 8;   // multiple of 16: a 16-lane group is one 1x128 group
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const uint4* g4 = reinterpret_cast<const uint4*>(h1 + (size_t)row * 2 * I);
    const uint4* u4 = reinterpret_cast<const uint4*>(h1 + (size_t)row * 2 * I + I);
    uint2* q2 = reinterpret_cast<uint2*>(zq + (size_t)row * I);
    float* srow = zs + (size_t)row * (I / 128);
    for (int base = 0; base < nv; base += blockDim.x) {
      const int v = base + threadIdx.x;
      const bool act = v < nv;
      float f[8];
      float amax = 0.0f;
      if (act) {
        uint4 gv = __ldg(g4 + v), uv = __ldg(u4 + v);
        const __nv_bfloat16* gb = reinterpret_cast<const __nv_bfloat16*>(&gv);
        const __nv_bfloat16* ub = reinterpret_cast<const __nv_bfloat16*>(&uv);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          f[j] = silu_f32(__bfloat162float(gb[j])) * __bfloat162float(ub[j]);
          amax = fmaxf(amax, fabsf(f[j]));
        }
      }
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (act) {
        const float s = act_scale(amax, ue8m0 != 0);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) lo |= (uint32_t)f32_to_e4m3(__fdiv_rn(f[j], s)) << (8 * j);
#pragma unroll
        for (int j = 0; j < 4; ++j) hi |= (uint32_t)f32_to_e4m3(__fdiv_rn(f[4 + j], s)) << (8 * j);
        q2[v] = make_uint2(lo, hi);
        if ((v & 15) == 0) srow[v >> 4] = s;
      }
    }
  }
}

cudaError_t launch_act_mul(const void* h1, int I, const int32_t* num_post_padded, void* z,
                           float* z_scale, bool ue8m0, int cap, cudaStream_t stream) {
  if (cap <= 0) return cudaSuccess;
  const int grid = min(cap, num_sms() * 8);
  if (z_scale == nullptr) {
    k_act_mul_bf16<<<grid, 128, 0, stream>>>(static_cast<const __nv_bfloat16*>(h1), I,
                                             num_post_padded, static_cast<__nv_bfloat16*>(z));
  } else {
    k_act_mul_fp8<<<grid, 128, 0, stream>>>(static_cast<const __nv_bfloat16*>(h1), I,
                                            num_post_padded, static_cast<uint8_t*>(z), z_scale,
                                            ue8m0);
  }
  return cudaGetLastError();
}

// y[t, :] = bf16( sum_i w[t,i] * y2[inv_perm[t,i], :] ), fp32, slot order.
__global__ void __launch_bounds__(128)
    k_unpermute_reduce(const __nv_bfloat16* __restrict__ y2, int H, int M, int topk,
                       const int32_t* __restrict__ inv_perm, const float* __restrict__ w,
                       int unit_weights, __nv_bfloat16* __restrict__ y) {
  const int nv = H / 8;
  for (int t = blockIdx.x; t < M; t += gridDim.x) {
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
      for (int i = 0; i < topk; ++i) {
        const int p = __ldg(inv_perm + (size_t)t * topk + i);
        if (p < 0) continue;
        const float wi = unit_weights ? 1.0f : __ldg(w + (size_t)t * topk + i);
        uint4 u = __ldg(reinterpret_cast<const uint4*>(y2 + (size_t)p * H) + v);
        const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = fmaf(wi, __bfloat162float(b[j]), acc[j]);
      }
      uint4 out;
      __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(&out);
#pragma unroll
      for (int j = 0; j < 8; ++j) ob[j] = __float2bfloat16_rn(acc[j]);
      reinterpret_cast<uint4*>(y + (size_t)t * H)[v] = out;
    }
  }
}

cudaError_t launch_unpermute_reduce(const void* y2, int H, int M, int topk,
                                    const int32_t* inv_perm, const float* topk_weights,
                                    bool unit_weights, void* y, cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  const int grid = min(M, num_sms() * 8);
  k_unpermute_reduce<<<grid, 128, 0, stream>>>(static_cast<const __nv_bfloat16*>(y2), H, M, topk,
                                               inv_perm, topk_weights, unit_weights ? 1 : 0,
                                               static_cast<__nv_bfloat16*>(y));
  return cudaGetLastError();
}

}  // namespace moe
