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
// Both are HBM-bound: one warp per row (token), grid-stride, 16-byte vector
// loads issued in batches ahead of the arithmetic so each warp keeps several
// KB in flight; the reduce issues all k gathers of a vector pair before it
// accumulates.
#include "e4m3_pack.cuh"
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int ACT_U = 2;             // 16-byte vectors of g (and of u) per lane in flight
                                     // (2: 167 us on the DeepSeek-class FP8 act, 4: 171, 8: 188)
constexpr int ACT_THREADS = 256;

// z[row, :] = bf16(act(bf16 g, bf16 u)) for rows below num_post_padded;
// act = SiLU(g) * u, or the gemm1 alpha / beta / clamp recipe.
__global__ void __launch_bounds__(ACT_THREADS)
    k_act_mul_bf16(const __nv_bfloat16* __restrict__ h1, int I, const int32_t* __restrict__ npp,
                   __nv_bfloat16* __restrict__ z, const Epilogue act) {
  const int lane = threadIdx.x & 31;
  const int wpc = blockDim.x >> 5;
  const int rows = *npp;
  const int nv = I / 8;
  for (int row = blockIdx.x * wpc + (threadIdx.x >> 5); row < rows; row += gridDim.x * wpc) {
    const uint4* g4 = reinterpret_cast<const uint4*>(h1 + (size_t)row * 2 * I);
    const uint4* u4 = reinterpret_cast<const uint4*>(h1 + (size_t)row * 2 * I + I);
    uint4* z4 = reinterpret_cast<uint4*>(z + (size_t)row * I);
    for (int base = 0; base < nv; base += 32 * ACT_U) {
      uint4 gv[ACT_U], uv[ACT_U];
#pragma unroll
      for (int k = 0; k < ACT_U; ++k) {
        const int v = base + 32 * k + lane;
        if (v < nv) {
          gv[k] = __ldg(g4 + v);
          uv[k] = __ldg(u4 + v);
        }
      }
#pragma unroll
      for (int k = 0; k < ACT_U; ++k) {
        const int v = base + 32 * k + lane;
        if (v >= nv) continue;
        const __nv_bfloat16* gb = reinterpret_cast<const __nv_bfloat16*>(&gv[k]);
        const __nv_bfloat16* ub = reinterpret_cast<const __nv_bfloat16*>(&uv[k]);
        uint4 out;
        __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(&out);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          ob[j] = __float2bfloat16_rn(
              act_glu(act, __bfloat162float(gb[j]), __bfloat162float(ub[j])));
        z4[v] = out;
      }
    }
  }
}

// Quantised variant: z in fp32, then per group of LPG lanes x 8 values
// (16 lanes: 1x128; 4 lanes: the 1x32 groups of MXFP8) amax -> scale -> e4m3
// with one reciprocal per group.  With power-of-two scales (UE8M0) the
// reciprocal is exact and v * r is the correctly rounded quotient, so the
// correction step is skipped.
template <int LPG, bool UE8M0>
__global__ void __launch_bounds__(ACT_THREADS)
    k_act_mul_fp8(const __nv_bfloat16* __restrict__ h1, int I, const int32_t* __restrict__ npp,
                  uint8_t* __restrict__ zq, float* __restrict__ zs, const Epilogue recipe) {
  const int lane = threadIdx.x & 31;
  const int wpc = blockDim.x >> 5;
  const int rows = *npp;
  const int nv = I / 8;   // a multiple of LPG: groups never straddle rows
  for (int row = blockIdx.x * wpc + (threadIdx.x >> 5); row < rows; row += gridDim.x * wpc) {
    const uint4* g4 = reinterpret_cast<const uint4*>(h1 + (size_t)row * 2 * I);
    const uint4* u4 = reinterpret_cast<const uint4*>(h1 + (size_t)row * 2 * I + I);
    uint2* q2 = reinterpret_cast<uint2*>(zq + (size_t)row * I);
    float* srow = zs + (size_t)row * (nv / LPG);
    for (int base = 0; base < nv; base += 32 * ACT_U) {
      uint4 gv[ACT_U], uv[ACT_U];
#pragma unroll
      for (int k = 0; k < ACT_U; ++k) {
        const int v = base + 32 * k + lane;
        if (v < nv) {
          gv[k] = __ldg(g4 + v);
          uv[k] = __ldg(u4 + v);
        }
      }
#pragma unroll
      for (int k = 0; k < ACT_U; ++k) {
        const int v = base + 32 * k + lane;
        const bool act = v < nv;
        float f[8];
        float amax = 0.0f;
        if (act) {
          const __nv_bfloat16* gb = reinterpret_cast<const __nv_bfloat16*>(&gv[k]);
          const __nv_bfloat16* ub = reinterpret_cast<const __nv_bfloat16*>(&uv[k]);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            f[j] = act_glu(recipe, __bfloat162float(gb[j]), __bfloat162float(ub[j]));
            amax = fmaxf(amax, fabsf(f[j]));
          }
        }
#pragma unroll
        for (int o = LPG / 2; o >= 1; o >>= 1)
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (act) {
          const float s = act_scale(amax, UE8M0);
          const float r = __frcp_rn(s);
#pragma unroll
          for (int j = 0; j < 8; ++j) f[j] = UE8M0 ? f[j] * r : quot_rn(f[j], s, r);
          q2[v] = make_uint2(e4m3x4(f[0], f[1], f[2], f[3]), e4m3x4(f[4], f[5], f[6], f[7]));
          if (v % LPG == 0) srow[v / LPG] = s;
        }
      }
    }
  }
}

cudaError_t launch_act_mul(const void* h1, int I, const int32_t* num_post_padded, void* z,
                           float* z_scale, bool ue8m0, int group, int cap,
                           const Epilogue& act, cudaStream_t stream) {
  if (cap <= 0) return cudaSuccess;
  const int wpc = ACT_THREADS / 32;
  const int grid = min((cap + wpc - 1) / wpc, num_sms() * 8);
  if (z_scale == nullptr) {
    k_act_mul_bf16<<<grid, ACT_THREADS, 0, stream>>>(static_cast<const __nv_bfloat16*>(h1), I,
                                                     num_post_padded,
                                                     static_cast<__nv_bfloat16*>(z), act);
  } else {
    const auto* hp = static_cast<const __nv_bfloat16*>(h1);
    auto* zp = static_cast<uint8_t*>(z);
    if (group == 32 && ue8m0)
      k_act_mul_fp8<4, true><<<grid, ACT_THREADS, 0, stream>>>(hp, I, num_post_padded, zp,
                                                                z_scale, act);
    else if (group == 32)
      k_act_mul_fp8<4, false><<<grid, ACT_THREADS, 0, stream>>>(hp, I, num_post_padded, zp,
                                                                 z_scale, act);
    else if (ue8m0)
      k_act_mul_fp8<16, true><<<grid, ACT_THREADS, 0, stream>>>(hp, I, num_post_padded, zp,
                                                                 z_scale, act);
    else
      k_act_mul_fp8<16, false><<<grid, ACT_THREADS, 0, stream>>>(hp, I, num_post_padded, zp,
                                                                  z_scale, act);
  }
  return cudaGetLastError();
}

// y[t, :] = bf16( sum_i w[t,i] * y2[inv_perm[t,i], :] ), fp32, slot order.
// One warp per token; its k row indices and weights are held by lanes 0..k-1
// and broadcast by shuffles.  Per lane, two vectors x k gathers are issued
// before any accumulation (KMAX slots unrolled, the rest in a loop).
constexpr int REDUCE_THREADS = 256;

template <int KMAX>
__global__ void __launch_bounds__(REDUCE_THREADS)
    k_unpermute_reduce(const __nv_bfloat16* __restrict__ y2, int H, int M, int topk,
                       const int32_t* __restrict__ inv_perm, const float* __restrict__ w,
                       int unit_weights, __nv_bfloat16* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int wpc = blockDim.x >> 5;
  const int nv = H / 8;
  for (int t = blockIdx.x * wpc + (threadIdx.x >> 5); t < M; t += gridDim.x * wpc) {
    int my_p = -1;
    float my_w = 0.0f;
    if (lane < topk) {
      my_p = __ldg(inv_perm + (size_t)t * topk + lane);
      my_w = unit_weights ? 1.0f : __ldg(w + (size_t)t * topk + lane);
    }
    int p[KMAX];
    float wi[KMAX];
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
      p[i] = __shfl_sync(0xffffffffu, my_p, i);
      wi[i] = __shfl_sync(0xffffffffu, my_w, i);
    }
    uint4* yt = reinterpret_cast<uint4*>(y + (size_t)t * H);
    for (int v0 = lane; v0 < nv; v0 += 64) {
      const int v1 = v0 + 32;
      const bool has1 = v1 < nv;
      uint4 a[KMAX], b[KMAX];
#pragma unroll
      for (int i = 0; i < KMAX; ++i) {
        if (i < topk && p[i] >= 0) {
          const uint4* row = reinterpret_cast<const uint4*>(y2 + (size_t)p[i] * H);
          a[i] = __ldg(row + v0);
          if (has1) b[i] = __ldg(row + v1);
        }
      }
      float acc0[8], acc1[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc0[j] = acc1[j] = 0.0f;
#pragma unroll
      for (int i = 0; i < KMAX; ++i) {
        if (i < topk && p[i] >= 0) {
          const __nv_bfloat16* ab = reinterpret_cast<const __nv_bfloat16*>(&a[i]);
          const __nv_bfloat16* bb = reinterpret_cast<const __nv_bfloat16*>(&b[i]);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            acc0[j] = fmaf(wi[i], __bfloat162float(ab[j]), acc0[j]);
            if (has1) acc1[j] = fmaf(wi[i], __bfloat162float(bb[j]), acc1[j]);
          }
        }
      }
      // slots beyond KMAX (top-k up to 16): one at a time, same slot order;
      // lanes may have left the vector loop, so no shuffles here
      for (int i = KMAX; i < topk; ++i) {
        const int pi = __ldg(inv_perm + (size_t)t * topk + i);
        const float wv = unit_weights ? 1.0f : __ldg(w + (size_t)t * topk + i);
        if (pi < 0) continue;
        const uint4* row = reinterpret_cast<const uint4*>(y2 + (size_t)pi * H);
        uint4 ua = __ldg(row + v0), ub = has1 ? __ldg(row + v1) : make_uint4(0, 0, 0, 0);
        const __nv_bfloat16* ab = reinterpret_cast<const __nv_bfloat16*>(&ua);
        const __nv_bfloat16* bb = reinterpret_cast<const __nv_bfloat16*>(&ub);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          acc0[j] = fmaf(wv, __bfloat162float(ab[j]), acc0[j]);
          acc1[j] = fmaf(wv, __bfloat162float(bb[j]), acc1[j]);
        }
      }
      uint4 o0, o1;
      __nv_bfloat16* ob0 = reinterpret_cast<__nv_bfloat16*>(&o0);
      __nv_bfloat16* ob1 = reinterpret_cast<__nv_bfloat16*>(&o1);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        ob0[j] = __float2bfloat16_rn(acc0[j]);
        ob1[j] = __float2bfloat16_rn(acc1[j]);
      }
      yt[v0] = o0;
      if (has1) yt[v1] = o1;
    }
  }
}

// Split-K form: GEMM2 left one fp32 partial per K slice for every routed
// item r = t * k + i (part[(s * R + r) * H + col]).  Each (token, 256-column
// segment) is one warp's work item, lane l owning 8 columns: the slices are
// summed in order, rounded to bf16 where Y2 would have been stored, and the
// weighted sum over the slots runs in fp32 as in k_unpermute_reduce.
constexpr int kMaxSlices = 8;

// The slices of 8 columns of one routed item, summed in slice order; all
// loads are issued before the first add.
__device__ __forceinline__ void sum_slices(const float* __restrict__ part, int S, size_t stride,
                                           size_t off, float (&v)[8]) {
  float4 a[kMaxSlices], b[kMaxSlices];
#pragma unroll
  for (int sl = 0; sl < kMaxSlices; ++sl) {
    if (sl < S) {
      const float4* src = reinterpret_cast<const float4*>(part + sl * stride + off);
      a[sl] = __ldg(src);
      b[sl] = __ldg(src + 1);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = 0.0f;
#pragma unroll
  for (int sl = 0; sl < kMaxSlices; ++sl) {
    if (sl < S) {
      v[0] += a[sl].x; v[1] += a[sl].y; v[2] += a[sl].z; v[3] += a[sl].w;
      v[4] += b[sl].x; v[5] += b[sl].y; v[6] += b[sl].z; v[7] += b[sl].w;
    }
  }
}

__global__ void __launch_bounds__(REDUCE_THREADS)
    k_unpermute_reduce_split(const float* __restrict__ part, int S, int H, int M, int topk,
                             const int32_t* __restrict__ inv_perm, const float* __restrict__ w,
                             __nv_bfloat16* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nw = gridDim.x * (blockDim.x >> 5);
  const int segs = H / 256;
  const size_t R = (size_t)M * topk;
  for (int item = gw; item < M * segs; item += nw) {
    const int t = item / segs, col = (item - t * segs) * 256 + lane * 8;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int i = 0; i < topk; ++i) {
      const size_t r = (size_t)t * topk + i;
      if (__ldg(inv_perm + r) < 0) continue;       // skipped slot (same for the whole warp)
      const float wi = __ldg(w + r);
      float v[8];
      sum_slices(part, S, R * H, r * H + col, v);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = fmaf(wi, bf16_round(v[j]), acc[j]);
    }
    uint4 o;
    __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(&o);
#pragma unroll
    for (int j = 0; j < 8; ++j) ob[j] = __float2bfloat16_rn(acc[j]);
    *reinterpret_cast<uint4*>(y + (size_t)t * H + col) = o;
  }
}

cudaError_t launch_unpermute_reduce_split(const float* part, int splits, int H, int M, int topk,
                                          const int32_t* inv_perm, const float* topk_weights,
                                          void* y, cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  if (H % 256 != 0 || splits < 1 || splits > kMaxSlices) return cudaErrorInvalidValue;
  const int wpc = REDUCE_THREADS / 32;
  const int items = M * (H / 256);
  const int grid = min((items + wpc - 1) / wpc, num_sms() * 8);
  k_unpermute_reduce_split<<<grid, REDUCE_THREADS, 0, stream>>>(
      part, splits, H, M, topk, inv_perm, topk_weights, static_cast<__nv_bfloat16*>(y));
  return cudaGetLastError();
}

cudaError_t launch_unpermute_reduce(const void* y2, int H, int M, int topk,
                                    const int32_t* inv_perm, const float* topk_weights,
                                    bool unit_weights, void* y, cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  const int wpc = REDUCE_THREADS / 32;
  const int grid = min((M + wpc - 1) / wpc, num_sms() * 8);
  const auto* yy = static_cast<const __nv_bfloat16*>(y2);
  auto* out = static_cast<__nv_bfloat16*>(y);
  const int uw = unit_weights ? 1 : 0;
  if (topk <= 2)
    k_unpermute_reduce<2><<<grid, REDUCE_THREADS, 0, stream>>>(yy, H, M, topk, inv_perm,
                                                               topk_weights, uw, out);
  else if (topk <= 4)
    k_unpermute_reduce<4><<<grid, REDUCE_THREADS, 0, stream>>>(yy, H, M, topk, inv_perm,
                                                               topk_weights, uw, out);
  else
    k_unpermute_reduce<8><<<grid, REDUCE_THREADS, 0, stream>>>(yy, H, M, topk, inv_perm,
                                                               topk_weights, uw, out);
  return cudaGetLastError();
}

}  // namespace moe
