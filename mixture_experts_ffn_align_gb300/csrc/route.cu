// Block-aligned routing and permute (stage 1).
//
// Page "fused_moe.py 分析", "moe_align_block_size 的作用": routed items
// (token, slot) are sorted by expert and each expert's count is padded to the
// block size, giving sorted_token_ids, one expert id per block and
// num_tokens_post_padded.  Page "Blackwell 上的 DeepGEMM FusedMoE（vLLM）",
// §2.6.2: per-expert rounded prefix sum (ep_scatter_1), each item's
// destination row into inv_perm (ep_scatter_2), ids < 0 skipped, padding
// rows of the activation scale are zero.
//
// GB300 design: the pages' scatter claims rows with atomics, which makes the
// order inside an expert depend on timing.  Here the order is ascending item
// index, so indices are reproducible bit for bit:
//   k_route_hist    one warp per 512-item segment: per-segment histogram
//   k_route_scan    one CTA: per-expert scan over segments + padded prefix
//                   sum over experts, block ids, padding entries
//   k_route_scatter one warp per segment: __match_any_sync ranks items of the
//                   same expert within 32-item chunks; a per-warp running
//                   count in shared memory carries the rank across chunks.
//   k_route_small   small batches (decode, and the Mixtral-shaped prefill):
//                   the same three phases in one CTA, histograms in shared
//                   memory (one launch, not three).
// The data gather (k_permute_*) runs one warp per destination row with
// 16-byte vector loads batched ahead of the stores; the FP8 variant fuses the
// dynamic 1x128 quantisation.
#include "../../include/moe_ffn.h"
#include "e4m3_pack.cuh"
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

__global__ void __launch_bounds__(kRouteWarps * 32)
    k_route_hist(const int32_t* __restrict__ ids, int R, int E, int G, int32_t* __restrict__ hist,
                 int* err) {
  extern __shared__ int32_t sh_hist[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x * kRouteWarps + warp;
  int32_t* h = sh_hist + warp * E;
  for (int e = lane; e < E; e += 32) h[e] = 0;
  __syncwarp();
  if (g < G) {
    const int end = min(R, (g + 1) * kRouteSeg);
    for (int r = g * kRouteSeg + lane; r < end; r += 32) {
      const int e = __ldg(ids + r);
      if (e >= E) {
        set_dev_error(err, kDevErrBadIndex);
      } else if (e >= 0) {
        atomicAdd(h + e, 1);
      }
    }
  }
  __syncwarp();
  if (g < G)
    for (int e = lane; e < E; e += 32) hist[(size_t)g * E + e] = h[e];
}

// One CTA of 1024 threads.  Thread t works on expert e = t % E and on part
// t / E of the segments (P = 1024 / E parts, rounded down to a power of two),
// so each thread walks G / P segments instead of all G: (1) per-part sums,
// (2) per-expert counts, padded exclusive scan over experts, (3) each part
// rewrites its segments' counts as the running start row of the segment.
__global__ void __launch_bounds__(1024)
    k_route_scan(int32_t* __restrict__ hist, int G, int E, int A, int R, int cap,
                 int32_t* __restrict__ expert_offsets, int32_t* __restrict__ num_post_padded,
                 int32_t* __restrict__ block_ids, int32_t* __restrict__ sorted_ids) {
  __shared__ int32_t part_sum[1024];
  __shared__ int32_t s_off[1025];
  __shared__ int32_t s_cnt[1024];
  __shared__ int32_t warp_sums[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int P = 1;
  while (P * 2 * E <= 1024) P *= 2;
  const int e = tid % E, part = tid / E;
  const bool worker = part < P;
  const int per = (G + P - 1) / P;
  const int g0 = min(G, part * per), g1 = min(G, g0 + per);
  // (1) sum of this part's segments
  if (worker) {
    int sum = 0, g = g0;
    for (; g + 4 <= g1; g += 4)
      sum += hist[(size_t)g * E + e] + hist[(size_t)(g + 1) * E + e] +
             hist[(size_t)(g + 2) * E + e] + hist[(size_t)(g + 3) * E + e];
    for (; g < g1; ++g) sum += hist[(size_t)g * E + e];
    part_sum[part * E + e] = sum;
  }
  __syncthreads();
  // (2) expert counts and the padded exclusive scan over experts
  int count = 0;
  if (tid < E)
    for (int q = 0; q < P; ++q) count += part_sum[q * E + tid];
  const int padded = (count + A - 1) / A * A;
  int incl = padded;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = warp_sums[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    warp_sums[lane] = wi - w;   // exclusive prefix of warp totals
    if (lane == 31) s_off[1024] = wi;
  }
  __syncthreads();
  if (tid < E) {
    s_off[tid] = incl - padded + warp_sums[warp];
    s_cnt[tid] = count;
  }
  __syncthreads();
  const int total = s_off[1024];
  // (3) start row of each segment's first item of expert e
  if (worker) {
    int run = s_off[e];
    for (int q = 0; q < part; ++q) run += part_sum[q * E + e];
    int g = g0;
    for (; g + 4 <= g1; g += 4) {
      const int v0 = hist[(size_t)g * E + e], v1 = hist[(size_t)(g + 1) * E + e];
      const int v2 = hist[(size_t)(g + 2) * E + e], v3 = hist[(size_t)(g + 3) * E + e];
      hist[(size_t)g * E + e] = run; run += v0;
      hist[(size_t)(g + 1) * E + e] = run; run += v1;
      hist[(size_t)(g + 2) * E + e] = run; run += v2;
      hist[(size_t)(g + 3) * E + e] = run; run += v3;
    }
    for (; g < g1; ++g) {
      const int v = hist[(size_t)g * E + e];
      hist[(size_t)g * E + e] = run;
      run += v;
    }
    // padding entries at the end of expert e's segment
    for (int j = s_off[e] + s_cnt[e] + part; j < s_off[e] + (s_cnt[e] + A - 1) / A * A; j += P)
      sorted_ids[j] = R;
  }
  if (tid < E) expert_offsets[tid] = s_off[tid];
  if (tid == 0) {
    expert_offsets[E] = total;
    num_post_padded[0] = total;
  }
  // block expert ids: the expert whose padded range holds the block (binary
  // search over the offsets), -1 past the used blocks
  for (int b = tid; b < cap / A; b += blockDim.x) {
    int id = -1;
    if (b * A < total) {
      int lo = 0, hi = E - 1;   // last expert with s_off <= b * A and a non-empty range
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= b * A) lo = mid; else hi = mid - 1;
      }
      id = lo;
    }
    block_ids[b] = id;
  }
  for (int j = total + tid; j < cap; j += blockDim.x) sorted_ids[j] = R;
}

__global__ void __launch_bounds__(kRouteWarps * 32)
    k_route_scatter(const int32_t* __restrict__ ids, int R, int E, int G,
                    const int32_t* __restrict__ hist, int32_t* __restrict__ sorted_ids,
                    int32_t* __restrict__ inv_perm) {
  extern __shared__ int32_t sh_cnt[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x * kRouteWarps + warp;
  if (g >= G) return;
  int32_t* cnt = sh_cnt + warp * E;
  for (int e = lane; e < E; e += 32) cnt[e] = hist[(size_t)g * E + e];
  __syncwarp();
  const unsigned lt_mask = (1u << lane) - 1u;
  const int end = min(R, (g + 1) * kRouteSeg);
  for (int base = g * kRouteSeg; base < end; base += 32) {
    const int r = base + lane;
    const bool in = r < end;
    const int e = in ? __ldg(ids + r) : -1;
    const bool valid = in && e >= 0 && e < E;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
    int pos = -1;
    if (valid) pos = cnt[e] + __popc(peers & lt_mask);
    __syncwarp();
    if (valid) {
      sorted_ids[pos] = r;
      if (lane == __ffs(peers) - 1) cnt[e] += __popc(peers);
    }
    if (in) inv_perm[r] = pos;
    __syncwarp();
  }
}

// Small batches (decode): the three routing phases in one CTA of 1024
// threads, the per-segment histograms in shared memory.  Warp g < G handles
// items [g S, (g + 1) S) (S a multiple of 32, G <= 32); the outputs are the
// same as the three-kernel form's, bit for bit (same segments' order, same
// ranks inside a segment).
constexpr int kSmallThreads = 1024;
// One CTA routes up to 2048 items, or up to 8192 with at most 64 experts
// (measured on GB300, routing alone: Mixtral-shaped 8192 items over 8
// experts 10.9 vs 20.9 us for the three kernels; 16384 items over 256 experts
// 34.6 vs 31.0 us and 65536 over 256 experts 91.5 vs 37.2 us favour them).
bool route_in_one_cta(int R, int E) { return R <= 2048 || (R <= 8192 && E <= 64); }

__global__ void __launch_bounds__(kSmallThreads)
    k_route_small(const int32_t* __restrict__ ids, int R, int E, int A, int cap, int S, int G,
                  int32_t* __restrict__ expert_offsets, int32_t* __restrict__ num_post_padded,
                  int32_t* __restrict__ block_ids, int32_t* __restrict__ sorted_ids,
                  int32_t* __restrict__ inv_perm, int* err) {
  extern __shared__ int32_t hist[];     // [G][E]
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t s_total;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // (1) per-segment histograms
  if (warp < G) {
    int32_t* h = hist + warp * E;
    for (int e = lane; e < E; e += 32) h[e] = 0;
    __syncwarp();
    const int end = min(R, (warp + 1) * S);
    for (int r = warp * S + lane; r < end; r += 32) {
      const int e = __ldg(ids + r);
      if (e >= E) {
        set_dev_error(err, kDevErrBadIndex);
      } else if (e >= 0) {
        atomicAdd(h + e, 1);
      }
    }
  }
  __syncthreads();
  // (2) per-expert counts, padded exclusive scan over experts, segment starts
  int count = 0;
  if (tid < E)
    for (int g = 0; g < G; ++g) {
      const int v = hist[g * E + tid];
      hist[g * E + tid] = count;
      count += v;
    }
  const int padded = (count + A - 1) / A * A;
  int incl = padded;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = warp_sums[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    warp_sums[lane] = wi - w;
    if (lane == 31) s_total = wi;
  }
  __syncthreads();
  const int total = s_total;
  if (tid < E) {
    const int off = incl - padded + warp_sums[warp];
    expert_offsets[tid] = off;
    for (int g = 0; g < G; ++g) hist[g * E + tid] += off;
    for (int b = off / A; b < (off + padded) / A; ++b) block_ids[b] = tid;
    for (int j = off + count; j < off + padded; ++j) sorted_ids[j] = R;
  }
  if (tid == 0) {
    expert_offsets[E] = total;
    num_post_padded[0] = total;
  }
  for (int b = total / A + tid; b < cap / A; b += kSmallThreads) block_ids[b] = -1;
  for (int j = total + tid; j < cap; j += kSmallThreads) sorted_ids[j] = R;
  __syncthreads();
  // (3) stable scatter, ascending item index inside each expert
  if (warp < G) {
    int32_t* cnt = hist + warp * E;
    const unsigned lt_mask = (1u << lane) - 1u;
    const int end = min(R, (warp + 1) * S);
    for (int base = warp * S; base < end; base += 32) {
      const int r = base + lane;
      const bool in = r < end;
      const int e = in ? __ldg(ids + r) : -1;
      const bool valid = in && e >= 0 && e < E;
      const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
      int pos = -1;
      if (valid) pos = cnt[e] + __popc(peers & lt_mask);
      __syncwarp();
      if (valid) {
        sorted_ids[pos] = r;
        if (lane == __ffs(peers) - 1) cnt[e] += __popc(peers);
      }
      if (in) inv_perm[r] = pos;
      __syncwarp();
    }
  }
}

cudaError_t launch_route(const int32_t* topk_ids, int R, int E, int block_size, int cap,
                         int32_t* hist, int32_t* sorted_ids, int32_t* block_expert_ids,
                         int32_t* expert_offsets, int32_t* num_post_padded, int32_t* inv_perm,
                         cudaStream_t stream) {
  int* err = dev_error_word();
  if (err == nullptr) return cudaErrorInvalidDevice;   // no usable current device
  // small batches: one CTA, histograms in shared memory
  const int S = 32 * ((R + 32 * 32 - 1) / (32 * 32));   // items per warp, a multiple of 32
  const int Gs = R > 0 ? (R + S - 1) / S : 0;
  if (route_in_one_cta(R, E)) {
    const size_t sh_small = (size_t)Gs * E * sizeof(int32_t);   // <= 32 x 1024 x 4 B
    static DeviceOnce attr;
    const cudaError_t ea = attr.call([] {
      return cudaFuncSetAttribute(k_route_small, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  32 * MOE_MAX_EXPERTS * (int)sizeof(int32_t));
    });
    if (ea != cudaSuccess) return ea;
    k_route_small<<<1, kSmallThreads, sh_small, stream>>>(
        topk_ids, R, E, block_size, cap, S, Gs, expert_offsets, num_post_padded,
        block_expert_ids, sorted_ids, inv_perm, err);
    return cudaGetLastError();
  }
  const int G = route_segments(R);
  const int ctas = (G + kRouteWarps - 1) / kRouteWarps;
  const size_t sh = (size_t)kRouteWarps * E * sizeof(int32_t);
  if (G > 0) {
    k_route_hist<<<ctas, kRouteWarps * 32, sh, stream>>>(topk_ids, R, E, G, hist, err);
  }
  k_route_scan<<<1, 1024, 0, stream>>>(hist, G, E, block_size, R, cap, expert_offsets,
                                       num_post_padded, block_expert_ids, sorted_ids);
  if (G > 0) {
    k_route_scatter<<<ctas, kRouteWarps * 32, sh, stream>>>(topk_ids, R, E, G, hist,
                                                            sorted_ids, inv_perm);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------ data permute
// One warp per destination row (grid-stride over the used rows); each lane
// issues PERMUTE_U 16-byte loads before it stores any, so a warp keeps
// PERMUTE_U * 512 B of the row in flight.
constexpr int PERMUTE_U = 8;
constexpr int PERMUTE_THREADS = 256;

__global__ void __launch_bounds__(PERMUTE_THREADS)
    k_permute_bf16(const __nv_bfloat16* __restrict__ x, int H, int topk, int R,
                   const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ npp,
                   const float* __restrict__ row_weights, __nv_bfloat16* __restrict__ xp) {
  const int lane = threadIdx.x & 31;
  const int wpc = blockDim.x >> 5;
  const int rows = *npp;
  const int nv = H / 8;
  for (int row = blockIdx.x * wpc + (threadIdx.x >> 5); row < rows; row += gridDim.x * wpc) {
    const int sid = sorted_ids[row];
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)row * H);
    if (sid >= R) {
      for (int v = lane; v < nv; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(sid / topk) * H);
    const float w = row_weights ? row_weights[sid] : 1.0f;
    for (int base = 0; base < nv; base += 32 * PERMUTE_U) {
      uint4 buf[PERMUTE_U];
#pragma unroll
      for (int u = 0; u < PERMUTE_U; ++u) {
        const int v = base + 32 * u + lane;
        if (v < nv) buf[u] = __ldg(src + v);
      }
#pragma unroll
      for (int u = 0; u < PERMUTE_U; ++u) {
        const int v = base + 32 * u + lane;
        if (v >= nv) continue;
        if (row_weights) {
          __nv_bfloat16* b = reinterpret_cast<__nv_bfloat16*>(&buf[u]);
#pragma unroll
          for (int j = 0; j < 8; ++j) b[j] = __float2bfloat16_rn(__bfloat162float(b[j]) * w);
        }
        dst[v] = buf[u];
      }
    }
  }
}

// FP8 variant: LPG lanes x 8 values form one quantisation group (16 lanes:
// a 1x128 group; 4 lanes: the 1x32 groups of MXFP8); the lanes of a group
// share one scale, so the quotient uses one reciprocal and a correction step
// instead of a division per value.
template <int LPG>
__global__ void __launch_bounds__(PERMUTE_THREADS)
    k_permute_fp8(const __nv_bfloat16* __restrict__ x, int H, int topk, int R,
                  const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ npp,
                  const float* __restrict__ row_weights, uint8_t* __restrict__ xq,
                  float* __restrict__ xs, int ue8m0) {
  const int lane = threadIdx.x & 31;
  const int wpc = blockDim.x >> 5;
  const int rows = *npp;
  const int nv = H / 8;          // 8-element vectors per row; a multiple of LPG
  for (int row = blockIdx.x * wpc + (threadIdx.x >> 5); row < rows; row += gridDim.x * wpc) {
    const int sid = sorted_ids[row];
    uint2* dst = reinterpret_cast<uint2*>(xq + (size_t)row * H);
    float* srow = xs + (size_t)row * (nv / LPG);
    if (sid >= R) {
      for (int v = lane; v < nv; v += 32) {
        dst[v] = make_uint2(0, 0);
        if (v % LPG == 0) srow[v / LPG] = 0.0f;
      }
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(sid / topk) * H);
    const float w = row_weights ? row_weights[sid] : 1.0f;
    for (int base = 0; base < nv; base += 32 * PERMUTE_U) {
      uint4 buf[PERMUTE_U];
#pragma unroll
      for (int u = 0; u < PERMUTE_U; ++u) {
        const int v = base + 32 * u + lane;
        if (v < nv) buf[u] = __ldg(src + v);
      }
#pragma unroll
      for (int u = 0; u < PERMUTE_U; ++u) {
        const int v = base + 32 * u + lane;
        // a group is wholly inside or outside the row (nv % LPG == 0), but
        // every lane takes part in the shuffles
        const bool act = v < nv;
        float f[8];
        float amax = 0.0f;
        if (act) {
          const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&buf[u]);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            f[j] = __bfloat162float(b[j]);
            if (row_weights) f[j] = bf16_round(f[j] * w);
            amax = fmaxf(amax, fabsf(f[j]));
          }
        }
#pragma unroll
        for (int o = LPG / 2; o >= 1; o >>= 1)
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (act) {
          const float s = act_scale(amax, ue8m0 != 0);
          const float r = __frcp_rn(s);
          uint32_t lo = 0, hi = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            lo |= (uint32_t)f32_to_e4m3(quot_rn(f[j], s, r)) << (8 * j);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            hi |= (uint32_t)f32_to_e4m3(quot_rn(f[4 + j], s, r)) << (8 * j);
          dst[v] = make_uint2(lo, hi);
          if (v % LPG == 0) srow[v / LPG] = s;
        }
      }
    }
  }
}

// Token-major FP8 variant for the routed layout: one warp per token reads
// the row of x once, quantises it once and stores the codes and scales into
// each of the token's k destination rows (inv_perm); the gather form above
// reads and quantises each routed copy again (k = 8 on the DeepSeek-class
// shapes).  Each lane holds 16 consecutive values (two 16-byte loads, one
// 16-byte store of codes); LPG lanes form one quantisation group (8 lanes:
// 1x128, 2 lanes: 1x32).  Padding rows (sorted id >= R) below the used row
// count are zeroed by the same warps afterwards, one warp per row.  With
// power-of-two scales (UE8M0) v * (1/s) is already the correctly rounded
// quotient.
template <int LPG, bool UE8M0>
__global__ void __launch_bounds__(PERMUTE_THREADS)
    k_permute_fp8_tok(const __nv_bfloat16* __restrict__ x, int H, int M, int topk, int R,
                      const int32_t* __restrict__ inv_perm,
                      const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ npp,
                      uint8_t* __restrict__ xq, float* __restrict__ xs) {
  constexpr int U = 2;           // 16-value chunks per lane in flight
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nw = gridDim.x * (blockDim.x >> 5);
  const int nv = H / 16;         // 16-value chunks per row; a multiple of LPG
  const int gpr = nv / LPG;      // scale groups per row
  for (int t = gw; t < M; t += nw) {
    // lane i < topk holds the destination row of routed item (t, i)
    const int my_dst = lane < topk ? inv_perm[(size_t)t * topk + lane] : -1;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    for (int base = 0; base < nv; base += 32 * U) {
      uint4 buf[2 * U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = base + 32 * u + lane;
        if (v < nv) {
          buf[2 * u] = __ldg(src + 2 * v);
          buf[2 * u + 1] = __ldg(src + 2 * v + 1);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = base + 32 * u + lane;
        const bool act = v < nv;   // groups lie wholly inside or outside the row
        float f[16];
        float amax = 0.0f;
        if (act) {
          const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&buf[2 * u]);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            f[j] = __bfloat162float(b[j]);
            amax = fmaxf(amax, fabsf(f[j]));
          }
        }
#pragma unroll
        for (int o = LPG / 2; o >= 1; o >>= 1)
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = act_scale(amax, UE8M0);
        uint4 code = make_uint4(0, 0, 0, 0);
        if (act) {
          const float r = __frcp_rn(s);
#pragma unroll
          for (int j = 0; j < 16; ++j) f[j] = UE8M0 ? f[j] * r : quot_rn(f[j], s, r);
          code = make_uint4(e4m3x4(f[0], f[1], f[2], f[3]), e4m3x4(f[4], f[5], f[6], f[7]),
                            e4m3x4(f[8], f[9], f[10], f[11]), e4m3x4(f[12], f[13], f[14], f[15]));
        }
        for (int i = 0; i < topk; ++i) {
          const int row = __shfl_sync(0xffffffffu, my_dst, i);
          if (row < 0 || !act) continue;
          reinterpret_cast<uint4*>(xq + (size_t)row * H)[v] = code;
          if (lane % LPG == 0) xs[(size_t)row * gpr + v / LPG] = s;
        }
      }
    }
  }
  // padding rows of the used blocks (one warp per row): codes and scales zero
  const int rows = *npp;
  for (int row = gw; row < rows; row += nw) {
    if (sorted_ids[row] < R) continue;
    uint4* dst = reinterpret_cast<uint4*>(xq + (size_t)row * H);
    for (int v = lane; v < nv; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
    for (int g = lane; g < gpr; g += 32) xs[(size_t)row * gpr + g] = 0.0f;
  }
}

// Token-major bf16 form: one warp per token reads its row once (16-byte
// loads, PERMUTE_U per lane in flight) and stores it to each of its k
// destination rows; padding rows below the used count are zeroed as in the
// FP8 form.  The row is read exactly once, also when x lives in host memory
// that the kernel reads in place (fused_experts_from_host).
__global__ void __launch_bounds__(PERMUTE_THREADS)
    k_permute_bf16_tok(const __nv_bfloat16* __restrict__ x, int H, int M, int topk, int R,
                       const int32_t* __restrict__ inv_perm,
                       const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ npp,
                       __nv_bfloat16* __restrict__ xp) {
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nw = gridDim.x * (blockDim.x >> 5);
  const int nv = H / 8;          // 16-byte vectors per row
  for (int t = gw; t < M; t += nw) {
    const int my_dst = lane < topk ? inv_perm[(size_t)t * topk + lane] : -1;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    for (int base = 0; base < nv; base += 32 * PERMUTE_U) {
      uint4 buf[PERMUTE_U];
#pragma unroll
      for (int u = 0; u < PERMUTE_U; ++u) {
        const int v = base + 32 * u + lane;
        if (v < nv) buf[u] = __ldg(src + v);
      }
      for (int i = 0; i < topk; ++i) {
        const int row = __shfl_sync(0xffffffffu, my_dst, i);
        if (row < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)row * H);
#pragma unroll
        for (int u = 0; u < PERMUTE_U; ++u) {
          const int v = base + 32 * u + lane;
          if (v < nv) dst[v] = buf[u];
        }
      }
    }
  }
  const int rows = *npp;
  for (int row = gw; row < rows; row += nw) {   // padding rows, one warp per row
    if (sorted_ids[row] < R) continue;
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)row * H);
    for (int v = lane; v < nv; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
  }
}

cudaError_t launch_permute_bf16_tokens(const void* x, int H, int M, int topk, int R,
                                       const int32_t* inv_perm, const int32_t* sorted_ids,
                                       const int32_t* num_post_padded, void* x_perm, int cap,
                                       cudaStream_t stream) {
  const int wpc = PERMUTE_THREADS / 32;
  const int work = max(M, cap);
  if (work <= 0) return cudaSuccess;
  const int grid = min((work + wpc - 1) / wpc, num_sms() * 8);
  k_permute_bf16_tok<<<grid, PERMUTE_THREADS, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(x), H, M, topk, R, inv_perm, sorted_ids,
      num_post_padded, static_cast<__nv_bfloat16*>(x_perm));
  return cudaGetLastError();
}

cudaError_t launch_permute_tokens(const void* x, int H, int M, int topk, int R,
                                  const int32_t* inv_perm, const int32_t* sorted_ids,
                                  const int32_t* num_post_padded, void* x_perm, float* x_scale,
                                  bool ue8m0, int group, int cap, cudaStream_t stream) {
  const int wpc = PERMUTE_THREADS / 32;
  const int work = max(M, cap);
  if (work <= 0) return cudaSuccess;
  const int grid = min((work + wpc - 1) / wpc, num_sms() * 8);
  const auto* xp = static_cast<const __nv_bfloat16*>(x);
  auto* q = static_cast<uint8_t*>(x_perm);
  if (group == 32 && ue8m0)
    k_permute_fp8_tok<2, true><<<grid, PERMUTE_THREADS, 0, stream>>>(
        xp, H, M, topk, R, inv_perm, sorted_ids, num_post_padded, q, x_scale);
  else if (group == 32)
    k_permute_fp8_tok<2, false><<<grid, PERMUTE_THREADS, 0, stream>>>(
        xp, H, M, topk, R, inv_perm, sorted_ids, num_post_padded, q, x_scale);
  else if (ue8m0)
    k_permute_fp8_tok<8, true><<<grid, PERMUTE_THREADS, 0, stream>>>(
        xp, H, M, topk, R, inv_perm, sorted_ids, num_post_padded, q, x_scale);
  else
    k_permute_fp8_tok<8, false><<<grid, PERMUTE_THREADS, 0, stream>>>(
        xp, H, M, topk, R, inv_perm, sorted_ids, num_post_padded, q, x_scale);
  return cudaGetLastError();
}

cudaError_t launch_permute_rows(const void* x, int H, int topk, int R, const int32_t* sorted_ids,
                                const int32_t* num_post_padded, const float* row_weights,
                                void* x_perm, float* x_scale, bool ue8m0, int group, int cap,
                                cudaStream_t stream) {
  if (cap <= 0) return cudaSuccess;
  const int wpc = PERMUTE_THREADS / 32;
  const int grid = min((cap + wpc - 1) / wpc, num_sms() * 8);
  if (x_scale == nullptr) {
    k_permute_bf16<<<grid, PERMUTE_THREADS, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(x), H, topk, R, sorted_ids, num_post_padded,
        row_weights, static_cast<__nv_bfloat16*>(x_perm));
  } else {
    if (group == 32)
      k_permute_fp8<4><<<grid, PERMUTE_THREADS, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(x), H, topk, R, sorted_ids, num_post_padded,
          row_weights, static_cast<uint8_t*>(x_perm), x_scale, ue8m0);
    else
      k_permute_fp8<16><<<grid, PERMUTE_THREADS, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(x), H, topk, R, sorted_ids, num_post_padded,
          row_weights, static_cast<uint8_t*>(x_perm), x_scale, ue8m0);
  }
  return cudaGetLastError();
}

}  // namespace moe
