// The C ABI (include/moe_ffn.h): argument validation, workspace layout and
// the stage orchestration of fused_experts.
//
// Validation mirrors the checks listed on the page "fused_moe.py 分析",
// "fused_experts_impl 的执行流程" step 1 (shape agreement, activation fixed to
// SiLU), the chunk bound CHUNK_SIZE = 16 * 1024 ("分 chunk 执行"), the page
// "Blackwell 上的 DeepGEMM FusedMoE（vLLM）" §2.6.3 warning that a GEMM block
// taller than the padding granularity reads another expert's id (so the
// GEMMs cut 128-row tiles inside each expert's segment and never store rows
// past it when block_size < 128), and M == 0 returning early (page 1,
// FusedMoEKernelModularImpl._fused_experts, "M_full == 0").
#include <cmath>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "../../include/moe_ffn.h"
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

__device__ int g_dev_error_word = 0;

namespace {
std::atomic<int> g_sms[kMaxDevices];   // SM count per device, 0 until queried
int* g_err_ptr[kMaxDevices];
std::mutex g_dev_mu;
int64_t g_watchdog_ns = 0;
int g_never_arrive = 0;
int g_bf16_form = 0;   // 0: by size, 1: single SM, 2: SM pairs

// The current device, or -1 when it cannot be read or lies beyond the
// per-device caches (kMaxDevices); callers then fail instead of borrowing
// another device's cached values.
int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}
}  // namespace

int device_index() { return current_device(); }

int num_sms() {
  const int d = current_device();
  if (d < 0) return 0;            // a zero grid: the launch fails with a CUDA error
  int n = g_sms[d].load(std::memory_order_relaxed);
  if (n == 0) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    if (n <= 0) n = 1;
    g_sms[d].store(n, std::memory_order_relaxed);
  }
  return n;
}

int* dev_error_word() {
  const int d = current_device();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_err_ptr[d] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_error_word) == cudaSuccess) g_err_ptr[d] = (int*)p;
  }
  return g_err_ptr[d];
}

void watchdog_params(uint64_t* limit_ns, int* never_arrive) {
  *limit_ns = g_watchdog_ns > 0 ? (uint64_t)g_watchdog_ns : 2000000000ull;
  *never_arrive = g_never_arrive;
}

}  // namespace moe

using namespace moe;

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool valid_problem(const moe_problem* p) {
  if (p == nullptr) return false;
  if (p->M < 0 || p->M > MOE_MAX_TOKENS) return false;
  if (p->H <= 0 || p->H % 128 || p->I <= 0 || p->I % 128) return false;
  if (p->E < 1 || p->E > MOE_MAX_EXPERTS) return false;
  if (p->topk < 1 || p->topk > MOE_MAX_TOPK) return false;
  if (p->block_size != 16 && p->block_size != 32 && p->block_size != 64 &&
      p->block_size != 128)
    return false;
  if (p->quant < MOE_Q_BF16 || p->quant > MOE_Q_MXFP8_1X32) return false;
  if (p->act_scale_fmt != MOE_SCALE_FP32 && p->act_scale_fmt != MOE_SCALE_UE8M0) return false;
  if (p->apply_router_weight_on_input && p->topk != 1) return false;
  if (p->router_weight_in_gemm2 != 0 && p->router_weight_in_gemm2 != 1) return false;
  if (p->router_weight_in_gemm2 && p->apply_router_weight_on_input) return false;
  if (p->act_recipe != 0 && p->act_recipe != 1) return false;
  if (p->act_recipe &&
      !(std::isfinite(p->gemm1_alpha) && std::isfinite(p->gemm1_beta) &&
        std::isfinite(p->gemm1_clamp_limit)))
    return false;
  if (p->weight_scales_prepacked != 0 && p->weight_scales_prepacked != 1) return false;
  if (p->weight_scales_prepacked && p->quant != MOE_Q_MXFP4_W4A8 &&
      p->quant != MOE_Q_MXFP8_1X32)
    return false;
  return true;
}

// Epilogue work of one GEMM of problem p: the activation recipe, a bias and
// (GEMM2 with router_weight_in_gemm2) the router weight per row.
Epilogue make_epilogue(const moe_problem* p, const void* bias, int n_bias,
                       const int32_t* sorted_ids, const float* item_weights) {
  Epilogue ep{};
  ep.bias = static_cast<const __nv_bfloat16*>(bias);
  ep.n_bias = n_bias;
  ep.sorted_ids = item_weights != nullptr ? sorted_ids : nullptr;
  ep.item_weights = sorted_ids != nullptr ? item_weights : nullptr;
  ep.R = p->M * p->topk;
  ep.recipe = p->act_recipe;
  ep.alpha = p->act_recipe ? p->gemm1_alpha : 1.0f;
  ep.beta = p->act_recipe ? p->gemm1_beta : 0.0f;
  ep.limit = p->act_recipe ? p->gemm1_clamp_limit : 0.0f;
  return ep;
}

bool quantised(const moe_problem* p) { return p->quant != MOE_Q_BF16; }
// Activation quantisation group along K: 32 for MXFP8 (1x32), else 128.
int act_group(const moe_problem* p) { return p->quant == MOE_Q_MXFP8_1X32 ? 32 : 128; }
// The block-scaled (E8M0 per 32) GEMM serves MXFP4 and MXFP8 weights.
bool block_scaled(const moe_problem* p) {
  return p->quant == MOE_Q_MXFP4_W4A8 || p->quant == MOE_Q_MXFP8_1X32;
}

size_t cap_rows(const moe_problem* p) {
  const size_t R = (size_t)p->M * p->topk;
  const size_t A = (size_t)p->block_size;
  const size_t raw = R + std::min(R, (size_t)p->E) * (A - 1);
  return (raw + A - 1) / A * A;
}

// K slices of the bf16 GEMM2 in fused_experts.  With few routed rows per
// expert (decode) its 128 x 256 tiles -- the used blocks x H / 256 -- number
// fewer than the SMs, and each SM streams weights at a bounded rate, so SMs
// would sit idle; cutting K s ways makes s x tiles work units.  s in [1, 8]
// minimises the rounds per unit of work, ceil(tiles s / SMs) / s, on the
// expected block count (every expert that receives rows fills its blocks
// evenly).  1 for the SM-pair form, the quantised modes and H % 256 != 0.
int splits_for_tiles(const moe_problem* p, int64_t tiles);

bool use_pairs_for(const moe_problem* p, int64_t rows_per_expert);

int gemm2_splits(const moe_problem* p) {
  if (p->quant != MOE_Q_BF16 || p->H % 256 != 0 || g_bf16_form == 2) return 1;
  const int64_t R = (int64_t)p->M * p->topk;
  if (R <= 0 || use_pairs_for(p, R / p->E)) return 1;
  const int64_t experts = std::min<int64_t>(p->E, R);
  const int64_t blocks = experts * ((R / experts + 127) / 128);
  return splits_for_tiles(p, blocks * (p->H / 256));
}

// The slice count for a GEMM2 of `tiles` 128 x 256 output tiles (see above).
int splits_for_tiles(const moe_problem* p, int64_t tiles) {
  const int64_t sms = num_sms();
  if (tiles >= sms) return 1;
  int best = 1;
  double best_cost = 1.0;
  for (int sp = 2; sp <= 8; ++sp) {
    const double cost = (double)((tiles * sp + sms - 1) / sms) / sp;
    if (cost < best_cost - 1e-9) {
      best = sp;
      best_cost = cost;
    }
  }
  // slices of whole 64-deep K steps, none empty: the count the GEMM runs
  const int num_kb = p->I / 64;
  const int per = (num_kb + best - 1) / best;
  return (num_kb + per - 1) / per;
}

struct Layout {
  size_t hist, sorted, blocks, offsets, npp, inv, ctr, xperm, xscale, h1, z, zscale, y2, part,
      total;
};

// Tile counters of the SM-pair bf16 GEMMs of one call (GEMM1's, then GEMM2's:
// two ints each), zeroed on the call's stream before them.
constexpr size_t kTileCtrBytes = 4 * sizeof(int32_t);

Layout layout(const moe_problem* p) {
  Layout L{};
  const size_t cap = cap_rows(p), R = (size_t)p->M * p->topk;
  const size_t H = p->H, I = p->I;
  const size_t G = (size_t)route_segments((int)R);
  const size_t xb = quantised(p) ? 1 : 2;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  L.hist = take(std::max<size_t>(G, 1) * p->E * 4);
  L.sorted = take(cap * 4);
  L.blocks = take(cap / p->block_size * 4 + 4);
  L.offsets = take(((size_t)p->E + 1) * 4);
  L.npp = take(4);
  L.inv = take(R * 4);
  L.ctr = take(kTileCtrBytes);
  // x_perm is dead once GEMM1 has run, so GEMM2's output reuses its storage
  L.xperm = take(std::max(cap * H * xb, cap * H * 2));
  L.y2 = L.xperm;
  L.xscale = quantised(p) ? take(cap * (H / act_group(p)) * 4) : 0;
  // bf16 and block-scaled GEMM1s write z (activation, and its quantisation,
  // fused); FP8 block scales keep H1
  L.h1 = p->quant == MOE_Q_FP8_BLOCK128 ? take(cap * 2 * I * 2) : 0;
  L.z = take(cap * I * (quantised(p) ? 1 : 2));
  L.zscale = quantised(p) ? take(cap * (I / act_group(p)) * 4) : 0;
  // split-K GEMM2 partials: fp32 per K slice and routed item
  const int sp = gemm2_splits(p);
  L.part = sp > 1 ? take((size_t)sp * R * H * 4) : 0;
  L.total = o;
  return L;
}

// The batched layout [E, T, H] (T = max_tokens): T a positive multiple of the
// 128-row tile and E*T within the rows the GEMM schedules hold.
bool valid_batched(const moe_problem* p, int max_tokens) {
  if (p == nullptr || p->E < 1 || p->E > MOE_MAX_EXPERTS || p->H <= 0 || p->I <= 0 ||
      p->block_size != 128 || max_tokens <= 0 || max_tokens % 128 != 0)
    return false;
  if (p->quant < MOE_Q_BF16 || p->quant > MOE_Q_MXFP8_1X32) return false;
  if (p->act_scale_fmt != MOE_SCALE_FP32 && p->act_scale_fmt != MOE_SCALE_UE8M0) return false;
  if (p->H % 128 != 0 || p->I % 128 != 0) return false;
  return (int64_t)p->E * max_tokens <= (int64_t)MOE_MAX_TOKENS * MOE_MAX_TOPK;
}

struct BatchedLayout {
  size_t blocks, npp, ctr, sorted, xq, xscale, h1, z, zscale, total;
};

BatchedLayout batched_layout(const moe_problem* p, int max_tokens) {
  BatchedLayout L{};
  const size_t rows = (size_t)p->E * max_tokens, H = p->H, I = p->I;
  const bool q = quantised(p);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  L.blocks = take(rows / 128 * 4);
  L.npp = take(4);
  L.ctr = take(kTileCtrBytes);
  L.sorted = q ? take(rows * 4) : 0;
  L.xq = q ? take(rows * H) : 0;
  L.xscale = q ? take(rows * (H / act_group(p)) * 4) : 0;
  L.h1 = p->quant == MOE_Q_FP8_BLOCK128 ? take(rows * 2 * I * 2) : 0;
  L.z = take(rows * I * (q ? 1 : 2));
  L.zscale = q ? take(rows * (I / act_group(p)) * 4) : 0;
  L.total = o;
  return L;
}

// Device address through which kernels on the current device may read and
// write a host buffer in place: page-locked (pinned or registered) host
// memory mapped into the device's address space, 16-byte aligned for the
// kernels' vector accesses.  nullptr for any other memory.
void* device_view(const void* host) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();   // clear the (non-sticky) error an unregistered pointer may leave
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return nullptr;
  if (reinterpret_cast<uintptr_t>(a.devicePointer) & 15u) return nullptr;
  return a.devicePointer;
}

thread_local char g_last_error[256] = "";

// Records the CUDA error of a failed call for moe_last_error_string.
moe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e),
           cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

// The GEMMs cut each expert's segment into 128-row m-tiles whatever the block
// size (16, 32, 64 or 128; a partial last m-tile's rows past the segment are
// not stored), so every valid block size is served; bf16 GEMM2 tiles are 256
// columns wide.  The MXFP4 kernel applies scales in the tensor core, which
// takes powers of two only: activations need UE8M0.
bool gemm_supported(const moe_problem* p) {
  if (p->quant == MOE_Q_BF16) return p->H % 256 == 0;
  if (block_scaled(p)) return p->act_scale_fmt == MOE_SCALE_UE8M0;
  return p->quant == MOE_Q_FP8_BLOCK128;
}

}  // namespace

extern "C" {

size_t moe_m_sum_bound(const moe_problem* p) { return valid_problem(p) ? cap_rows(p) : 0; }

size_t moe_prepacked_scale_bytes(const moe_problem* p, int which) {
  if (!valid_problem(p) || !block_scaled(p) || (which != 0 && which != 1)) return 0;
  const size_t N = which == 0 ? 2 * (size_t)p->I : (size_t)p->H;
  const size_t K = which == 0 ? (size_t)p->H : (size_t)p->I;
  return (size_t)p->E * N * (K / 32);
}

moe_status moe_prepack_weights(const moe_problem* p, const void* w13_scale, const void* w2_scale,
                               void* w13_scale_packed, void* w2_scale_packed, void* stream) {
  if (!valid_problem(p)) return MOE_ERR_INVALID_ARG;
  if (!block_scaled(p)) return MOE_ERR_UNSUPPORTED;
  if (!w13_scale || !w2_scale || !w13_scale_packed || !w2_scale_packed)
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w13_scale) | reinterpret_cast<uintptr_t>(w2_scale)) & 3u ||
      (reinterpret_cast<uintptr_t>(w13_scale_packed) |
       reinterpret_cast<uintptr_t>(w2_scale_packed)) & 15u)
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_prepack_mx_scales(static_cast<const uint8_t*>(w13_scale), p->E,
                                           2 * p->I, p->H, w13_scale_packed, s);
  if (e == cudaSuccess)
    e = launch_prepack_mx_scales(static_cast<const uint8_t*>(w2_scale), p->E, p->H, p->I,
                                 w2_scale_packed, s);
  return cuda_status(e);
}

size_t moe_align_workspace_bytes(const moe_problem* p) {
  if (!valid_problem(p)) return 0;
  const size_t G = (size_t)route_segments(p->M * p->topk);
  return align_up(std::max<size_t>(G, 1) * p->E * 4);
}

size_t moe_workspace_bytes(const moe_problem* p) {
  return valid_problem(p) ? layout(p).total : 0;
}

size_t moe_host_workspace_bytes(const moe_problem* p) {
  if (!valid_problem(p)) return 0;
  const size_t MH = (size_t)p->M * p->H * 2, Mk = (size_t)p->M * p->topk * 4;
  return layout(p).total + align_up(MH) + 2 * align_up(Mk) + align_up(MH);
}

moe_status moe_align_permute(const moe_problem* p, const void* x, const int32_t* topk_ids,
                             const float* topk_weights, int32_t* sorted_ids,
                             int32_t* block_expert_ids, int32_t* expert_offsets,
                             int32_t* num_post_padded, int32_t* inv_perm, void* x_perm,
                             float* x_perm_scale, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (!valid_problem(p)) return MOE_ERR_INVALID_ARG;
  if (p->M == 0) return MOE_OK;
  if (!topk_ids || !sorted_ids || !block_expert_ids || !expert_offsets || !num_post_padded ||
      !inv_perm || !workspace)
    return MOE_ERR_INVALID_ARG;
  if ((x == nullptr) != (x_perm == nullptr)) return MOE_ERR_INVALID_ARG;
  if (x && quantised(p) && !x_perm_scale) return MOE_ERR_INVALID_ARG;
  if (x && p->apply_router_weight_on_input && !topk_weights) return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < moe_align_workspace_bytes(p)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int R = p->M * p->topk, cap = (int)cap_rows(p);
  cudaError_t e = launch_route(topk_ids, R, p->E, p->block_size, cap,
                               static_cast<int32_t*>(workspace), sorted_ids, block_expert_ids,
                               expert_offsets, num_post_padded, inv_perm, s);
  if (e != cudaSuccess) return cuda_status(e);
  if (x && quantised(p) && !p->apply_router_weight_on_input) {
    e = launch_permute_tokens(x, p->H, p->M, p->topk, R, inv_perm, sorted_ids, num_post_padded,
                              x_perm, x_perm_scale, p->act_scale_fmt == MOE_SCALE_UE8M0,
                              act_group(p), cap, s);
  } else if (x && !p->apply_router_weight_on_input) {
    e = launch_permute_bf16_tokens(x, p->H, p->M, p->topk, R, inv_perm, sorted_ids,
                                   num_post_padded, x_perm, cap, s);
  } else if (x) {
    e = launch_permute_rows(x, p->H, p->topk, R, sorted_ids, num_post_padded,
                            p->apply_router_weight_on_input ? topk_weights : nullptr, x_perm,
                            quantised(p) ? x_perm_scale : nullptr,
                            p->act_scale_fmt == MOE_SCALE_UE8M0, act_group(p), cap, s);
  }
  return cuda_status(e);
}

}  // extern "C"

namespace {
// bf16 grouped GEMM form.  SM-pair tiles halve the weight bytes each SM
// stages per MMA, which pays once the experts average two or more 128-row
// blocks; below that most pairs would carry a lone block whose second half
// repeats the first.
// rows_per_expert: the expected routed rows per expert.
// SM-pair tiles for the bf16 GEMMs once the experts average two 128-row
// blocks (the debug hook can force either form); the pair forms pair whole
// 128-row blocks, so they take block size 128 only.
bool use_pairs(int64_t rows_per_expert, int block_size) {
  if (block_size != 128) return false;
  return g_bf16_form == 2 || (g_bf16_form == 0 && rows_per_expert >= 2 * 128);
}
// The FP8-block GEMMs run on one SM unless the debug hook forces the pair
// form: with fp32 block scales each 128-deep K block's partial is read out of
// tensor memory and promoted on the CUDA cores, and that readout, not the
// shared-memory staging the pair form halves, bounds both forms (the pair form
// measured 2.64 / 1.70 ms against 2.54 / 1.54 ms for the DeepSeek-class
// GEMM1 / GEMM2).
bool use_fp8_pairs(int block_size) { return block_size == 128 && g_bf16_form == 2; }
// The block-scaled GEMMs run on one SM unless the debug hook forces the pair
// form (prepacked weight scales and 128-row blocks only): on the DeepSeek-class
// MXFP8 layer the pair form with no scale synchronisation at all (a timing
// variant) was 2.20 against 2.35 ms for GEMM1, and delivering each K block's
// scale operands to both CTAs costs more than that (3.64 ms).
bool use_mx_pairs(const moe_problem* p) {
  return p->weight_scales_prepacked && p->block_size == 128 && g_bf16_form == 2;
}
bool use_pairs_for(const moe_problem* p, int64_t rows_per_expert) {
  return use_pairs(rows_per_expert, p->block_size);
}

cudaError_t launch_bf16_gemm(int64_t rows_per_expert, const void* A, int cap, int K,
                             const void* B, int b_rows_total, int b_rows_per_expert, int n_out,
                             const int32_t* block_expert_ids, const int32_t* num_post_padded,
                             void* out, bool fuse_act, const Epilogue& ep, cudaStream_t s,
                             int* tile_ctr = nullptr, int block_size = 128) {
  if (use_pairs(rows_per_expert, block_size))
    return launch_ggemm_bf16_2sm(A, cap, K, B, b_rows_total, b_rows_per_expert, n_out,
                                 block_expert_ids, num_post_padded, out, fuse_act, ep, s,
                                 tile_ctr);
  return launch_ggemm_bf16(A, cap, K, B, b_rows_total, b_rows_per_expert, n_out,
                           block_expert_ids, num_post_padded, out, fuse_act, ep, s, 1, nullptr,
                           nullptr, 0, block_size);
}
}  // namespace

extern "C" {

}  // extern "C"

namespace {
// Stage 2 with the tile counter of the SM-pair bf16 form given (nullptr: the
// library ring), shared by the entry point and fused_experts.
moe_status gemm_w13(const moe_problem* p, const void* x_perm, const float* x_scale,
                    const void* w13, const void* w13_scale, const void* w13_bias,
                    const int32_t* block_expert_ids, const int32_t* num_post_padded, void* out,
                    float* out_scale, int fuse_act, void* stream, int* tile_ctr) {
  if (!valid_problem(p)) return MOE_ERR_INVALID_ARG;
  if (p->M == 0) return MOE_OK;
  if (!x_perm || !w13 || !block_expert_ids || !num_post_padded || !out) return MOE_ERR_INVALID_ARG;
  if (!gemm_supported(p)) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int cap = (int)cap_rows(p);
  const Epilogue ep = make_epilogue(p, w13_bias, 2 * p->I, nullptr, nullptr);
  if (p->quant == MOE_Q_BF16) {
    return cuda_status(launch_bf16_gemm((int64_t)p->M * p->topk / p->E, x_perm, cap, p->H, w13,
                                        p->E * 2 * p->I, 2 * p->I, 2 * p->I, block_expert_ids,
                                        num_post_padded, out, fuse_act != 0, ep, s, tile_ctr,
                                        p->block_size));
  }
  if (!x_scale || !w13_scale) return MOE_ERR_INVALID_ARG;
  if (fuse_act && !out_scale) return MOE_ERR_INVALID_ARG;
  if (block_scaled(p) && use_mx_pairs(p))
    return cuda_status(launch_ggemm_mx_2sm(
        x_perm, x_scale, cap, p->H, w13, static_cast<const uint8_t*>(w13_scale), p->E * 2 * p->I,
        2 * p->I, 2 * p->I, block_expert_ids, num_post_padded, out,
        p->quant == MOE_Q_MXFP8_1X32, ep, s, out_scale, fuse_act != 0,
        p->act_scale_fmt == MOE_SCALE_UE8M0, tile_ctr));
  if (block_scaled(p))
    return cuda_status(launch_ggemm_mxfp4(
        x_perm, x_scale, cap, p->H, w13, static_cast<const uint8_t*>(w13_scale), p->E * 2 * p->I,
        2 * p->I, 2 * p->I, block_expert_ids, num_post_padded, out,
        p->quant == MOE_Q_MXFP8_1X32, ep, s, out_scale, fuse_act != 0,
        p->act_scale_fmt == MOE_SCALE_UE8M0, p->weight_scales_prepacked != 0, p->block_size));
  if (!fuse_act && use_fp8_pairs(p->block_size))
    return cuda_status(launch_ggemm_fp8_2sm(x_perm, x_scale, cap, p->H, w13,
                                            static_cast<const float*>(w13_scale),
                                            p->E * 2 * p->I, 2 * p->I, 2 * p->I,
                                            block_expert_ids, num_post_padded, out, ep, s,
                                            tile_ctr));
  return cuda_status(launch_ggemm_fp8(x_perm, x_scale, cap, p->H, w13,
                                      static_cast<const float*>(w13_scale), p->E * 2 * p->I,
                                      2 * p->I, 2 * p->I, block_expert_ids, num_post_padded, out,
                                      ep, s, out_scale, fuse_act != 0,
                                      p->act_scale_fmt == MOE_SCALE_UE8M0, p->block_size));
}
}  // namespace

extern "C" {

moe_status grouped_gemm_w13_ex(const moe_problem* p, const void* x_perm, const float* x_scale,
                               const void* w13, const void* w13_scale, const void* w13_bias,
                               const int32_t* block_expert_ids,
                               const int32_t* num_post_padded, void* out, float* out_scale,
                               int fuse_act, void* stream) {
  return gemm_w13(p, x_perm, x_scale, w13, w13_scale, w13_bias, block_expert_ids,
                  num_post_padded, out, out_scale, fuse_act, stream, nullptr);
}

moe_status grouped_gemm_w13(const moe_problem* p, const void* x_perm, const float* x_scale,
                            const void* w13, const void* w13_scale,
                            const int32_t* block_expert_ids, const int32_t* num_post_padded,
                            void* out, float* out_scale, int fuse_act, void* stream) {
  return grouped_gemm_w13_ex(p, x_perm, x_scale, w13, w13_scale, nullptr, block_expert_ids,
                             num_post_padded, out, out_scale, fuse_act, stream);
}

moe_status act_mul_quant(const moe_problem* p, const void* h1, const int32_t* num_post_padded,
                         void* z, float* z_scale, void* stream) {
  if (!valid_problem(p)) return MOE_ERR_INVALID_ARG;
  if (p->M == 0) return MOE_OK;
  if (!h1 || !num_post_padded || !z) return MOE_ERR_INVALID_ARG;
  if (quantised(p) && !z_scale) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_act_mul(h1, p->I, num_post_padded, z,
                                    quantised(p) ? z_scale : nullptr,
                                    p->act_scale_fmt == MOE_SCALE_UE8M0, act_group(p),
                                    (int)cap_rows(p),
                                    make_epilogue(p, nullptr, 0, nullptr, nullptr),
                                    static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {
// Stage 4 with the SM-pair tile counter given (see gemm_w13).
moe_status gemm_w2(const moe_problem* p, const void* z, const float* z_scale, const void* w2,
                   const void* w2_scale, const void* w2_bias, const int32_t* block_expert_ids,
                   const int32_t* num_post_padded, const int32_t* sorted_ids,
                   const float* topk_weights, void* y2, void* stream, int* tile_ctr) {
  if (!valid_problem(p)) return MOE_ERR_INVALID_ARG;
  if (p->M == 0) return MOE_OK;
  if (!z || !w2 || !block_expert_ids || !num_post_padded || !y2) return MOE_ERR_INVALID_ARG;
  if (p->router_weight_in_gemm2 && (!sorted_ids || !topk_weights)) return MOE_ERR_INVALID_ARG;
  if (!gemm_supported(p)) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int cap = (int)cap_rows(p);
  const Epilogue ep =
      p->router_weight_in_gemm2 ? make_epilogue(p, w2_bias, p->H, sorted_ids, topk_weights)
                                : make_epilogue(p, w2_bias, p->H, nullptr, nullptr);
  if (p->quant == MOE_Q_BF16) {
    return cuda_status(launch_bf16_gemm((int64_t)p->M * p->topk / p->E, z, cap, p->I, w2,
                                        p->E * p->H, p->H, p->H, block_expert_ids,
                                        num_post_padded, y2, false, ep, s, tile_ctr,
                                        p->block_size));
  }
  if (!z_scale || !w2_scale) return MOE_ERR_INVALID_ARG;
  if (block_scaled(p) && use_mx_pairs(p))
    return cuda_status(launch_ggemm_mx_2sm(z, z_scale, cap, p->I, w2,
                                           static_cast<const uint8_t*>(w2_scale), p->E * p->H,
                                           p->H, p->H, block_expert_ids, num_post_padded, y2,
                                           p->quant == MOE_Q_MXFP8_1X32, ep, s, nullptr, false,
                                           true, tile_ctr));
  if (block_scaled(p))
    return cuda_status(launch_ggemm_mxfp4(z, z_scale, cap, p->I, w2,
                                          static_cast<const uint8_t*>(w2_scale), p->E * p->H,
                                          p->H, p->H, block_expert_ids, num_post_padded, y2,
                                          p->quant == MOE_Q_MXFP8_1X32, ep, s, nullptr, false,
                                          true, p->weight_scales_prepacked != 0,
                                          p->block_size));
  if (use_fp8_pairs(p->block_size))
    return cuda_status(launch_ggemm_fp8_2sm(z, z_scale, cap, p->I, w2,
                                            static_cast<const float*>(w2_scale), p->E * p->H,
                                            p->H, p->H, block_expert_ids, num_post_padded, y2,
                                            ep, s, tile_ctr));
  return cuda_status(launch_ggemm_fp8(z, z_scale, cap, p->I, w2,
                                      static_cast<const float*>(w2_scale), p->E * p->H, p->H,
                                      p->H, block_expert_ids, num_post_padded, y2, ep, s,
                                      nullptr, false, false, p->block_size));
}
}  // namespace

extern "C" {

moe_status grouped_gemm_w2_ex(const moe_problem* p, const void* z, const float* z_scale,
                              const void* w2, const void* w2_scale, const void* w2_bias,
                              const int32_t* block_expert_ids, const int32_t* num_post_padded,
                              const int32_t* sorted_ids, const float* topk_weights, void* y2,
                              void* stream) {
  return gemm_w2(p, z, z_scale, w2, w2_scale, w2_bias, block_expert_ids, num_post_padded,
                 sorted_ids, topk_weights, y2, stream, nullptr);
}

moe_status grouped_gemm_w2(const moe_problem* p, const void* z, const float* z_scale,
                           const void* w2, const void* w2_scale,
                           const int32_t* block_expert_ids, const int32_t* num_post_padded,
                           void* y2, void* stream) {
  if (p != nullptr && p->router_weight_in_gemm2) return MOE_ERR_INVALID_ARG;   // needs _ex
  return grouped_gemm_w2_ex(p, z, z_scale, w2, w2_scale, nullptr, block_expert_ids,
                            num_post_padded, nullptr, nullptr, y2, stream);
}

moe_status unpermute_reduce(const moe_problem* p, const void* y2, const int32_t* inv_perm,
                            const float* topk_weights, void* y, void* stream) {
  if (!valid_problem(p)) return MOE_ERR_INVALID_ARG;
  if (p->M == 0) return MOE_OK;
  if (!y2 || !inv_perm || !y) return MOE_ERR_INVALID_ARG;
  const bool unit = p->apply_router_weight_on_input || p->router_weight_in_gemm2;
  if (!unit && !topk_weights) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_unpermute_reduce(y2, p->H, p->M, p->topk, inv_perm, topk_weights,
                                             unit, y, static_cast<cudaStream_t>(stream)));
}

int moe_gemm2_splits(const moe_problem* p) { return valid_problem(p) ? gemm2_splits(p) : 0; }

int moe_align_permute_launches(const moe_problem* p) {
  if (!valid_problem(p) || p->M == 0) return 0;
  return (route_in_one_cta(p->M * p->topk, p->E) ? 1 : 3) + 1;
}

size_t moe_gemm2_partial_bytes(const moe_problem* p, int splits) {
  if (!valid_problem(p) || splits < 1) return 0;
  return (size_t)splits * p->M * p->topk * p->H * 4;
}

moe_status grouped_gemm_w2_split(const moe_problem* p, const void* z, const void* w2,
                                 const int32_t* block_expert_ids,
                                 const int32_t* num_post_padded, const int32_t* sorted_ids,
                                 int splits, float* partial, void* stream) {
  if (!valid_problem(p) || p->quant != MOE_Q_BF16 || p->H % 256 != 0) return MOE_ERR_INVALID_ARG;
  if (p->M == 0) return MOE_OK;
  if (!z || !w2 || !block_expert_ids || !num_post_padded || !sorted_ids || !partial ||
      splits < 1 || splits > 8 || splits > p->I / 64)
    return MOE_ERR_INVALID_ARG;
  if (!gemm_supported(p)) return MOE_ERR_UNSUPPORTED;
  const Epilogue ep = make_epilogue(p, nullptr, p->H, nullptr, nullptr);
  const cudaError_t e = launch_ggemm_bf16(z, (int)cap_rows(p), p->I, w2, p->E * p->H, p->H, p->H,
                                          block_expert_ids, num_post_padded, nullptr, false, ep,
                                          static_cast<cudaStream_t>(stream), splits, partial,
                                          sorted_ids, p->M * p->topk, p->block_size);
  return e == cudaErrorInvalidValue ? MOE_ERR_INVALID_ARG : cuda_status(e);
}

moe_status unpermute_reduce_split(const moe_problem* p, const float* partial, int splits,
                                  const int32_t* inv_perm, const float* topk_weights, void* y,
                                  void* stream) {
  if (!valid_problem(p) || p->H % 256 != 0 || p->apply_router_weight_on_input ||
      p->router_weight_in_gemm2)
    return MOE_ERR_INVALID_ARG;
  if (p->M == 0) return MOE_OK;
  if (!partial || !inv_perm || !topk_weights || !y || splits < 1 || splits > 8)
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_unpermute_reduce_split(partial, splits, p->H, p->M, p->topk, inv_perm,
                                                   topk_weights, y,
                                                   static_cast<cudaStream_t>(stream)));
}

moe_status fused_experts_ex(const moe_problem* p, const void* x, const void* w13,
                            const void* w13_scale, const void* w13_bias, const void* w2,
                            const void* w2_scale, const void* w2_bias,
                            const float* topk_weights, const int32_t* topk_ids, void* y,
                            void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_problem(p)) return MOE_ERR_INVALID_ARG;
  if (p->M == 0) return MOE_OK;
  if (!x || !w13 || !w2 || !topk_ids || !y || !workspace || !topk_weights)
    return MOE_ERR_INVALID_ARG;
  if (quantised(p) && (!w13_scale || !w2_scale)) return MOE_ERR_INVALID_ARG;
  if (!gemm_supported(p)) return MOE_ERR_UNSUPPORTED;
  const Layout L = layout(p);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto i32 = [&](size_t off) { return reinterpret_cast<int32_t*>(ws + off); };
  auto f32 = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  int32_t *sorted = i32(L.sorted), *blocks = i32(L.blocks), *offs = i32(L.offsets),
          *npp = i32(L.npp), *inv = i32(L.inv), *ctr = i32(L.ctr);
  if (cudaMemsetAsync(ctr, 0, kTileCtrBytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_status(cudaGetLastError());
  moe_status st = moe_align_permute(p, x, topk_ids, topk_weights, sorted, blocks, offs, npp, inv,
                                    ws + L.xperm, quantised(p) ? f32(L.xscale) : nullptr,
                                    ws + L.hist, L.sorted - L.hist, stream);
  if (st != MOE_OK) return st;
  const int splits = gemm2_splits(p);
  if (!quantised(p) && splits > 1 && !w2_bias && !p->router_weight_in_gemm2 &&
      !p->apply_router_weight_on_input) {
    // decode-sized: GEMM2 in K slices over all SMs, the reduce sums them
    st = gemm_w13(p, ws + L.xperm, nullptr, w13, nullptr, w13_bias, blocks, npp, ws + L.z,
                  nullptr, 1, stream, ctr);
    if (st != MOE_OK) return st;
    st = grouped_gemm_w2_split(p, ws + L.z, w2, blocks, npp, sorted, splits, f32(L.part),
                               stream);
    if (st != MOE_OK) return st;
    return unpermute_reduce_split(p, f32(L.part), splits, inv, topk_weights, y, stream);
  }
  if (!quantised(p)) {
    st = gemm_w13(p, ws + L.xperm, nullptr, w13, nullptr, w13_bias, blocks, npp, ws + L.z,
                  nullptr, 1, stream, ctr);
    if (st != MOE_OK) return st;
    st = gemm_w2(p, ws + L.z, nullptr, w2, nullptr, w2_bias, blocks, npp, sorted, topk_weights,
                 ws + L.y2, stream, ctr + 2);
  } else if (block_scaled(p)) {
    // GEMM1 writes the quantised activation directly (act_mul_quant fused)
    st = gemm_w13(p, ws + L.xperm, f32(L.xscale), w13, w13_scale, w13_bias, blocks, npp,
                  ws + L.z, f32(L.zscale), 1, stream, ctr);
    if (st != MOE_OK) return st;
    st = gemm_w2(p, ws + L.z, f32(L.zscale), w2, w2_scale, w2_bias, blocks, npp, sorted,
                 topk_weights, ws + L.y2, stream, ctr + 2);
  } else {
    // FP8 block scales: the promotion epilogue bounds this GEMM, and the
    // activation at the end of each tile lengthened it by more than the
    // separate pass costs, so H1 goes through HBM
    st = gemm_w13(p, ws + L.xperm, f32(L.xscale), w13, w13_scale, w13_bias, blocks, npp,
                  ws + L.h1, nullptr, 0, stream, ctr);
    if (st != MOE_OK) return st;
    st = act_mul_quant(p, ws + L.h1, npp, ws + L.z, f32(L.zscale), stream);
    if (st != MOE_OK) return st;
    st = gemm_w2(p, ws + L.z, f32(L.zscale), w2, w2_scale, w2_bias, blocks, npp, sorted,
                 topk_weights, ws + L.y2, stream, ctr + 2);
  }
  if (st != MOE_OK) return st;
  return unpermute_reduce(p, ws + L.y2, inv, topk_weights, y, stream);
}

moe_status fused_experts(const moe_problem* p, const void* x, const void* w13,
                         const void* w13_scale, const void* w2, const void* w2_scale,
                         const float* topk_weights, const int32_t* topk_ids, void* y,
                         void* workspace, size_t workspace_bytes, void* stream) {
  return fused_experts_ex(p, x, w13, w13_scale, nullptr, w2, w2_scale, nullptr, topk_weights,
                          topk_ids, y, workspace, workspace_bytes, stream);
}

moe_status fused_experts_from_host(const moe_problem* p, const void* host_x,
                                   const int32_t* host_topk_ids,
                                   const float* host_topk_weights, void* host_y,
                                   const void* w13, const void* w13_scale, const void* w2,
                                   const void* w2_scale, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  if (!valid_problem(p)) return MOE_ERR_INVALID_ARG;
  if (p->M == 0) return MOE_OK;
  if (!host_x || !host_topk_ids || !host_topk_weights || !host_y || !workspace)
    return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < moe_host_workspace_bytes(p)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const size_t base = layout(p).total;
  const size_t MH = (size_t)p->M * p->H * 2, Mk = (size_t)p->M * p->topk * 4;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* d_ids = reinterpret_cast<int32_t*>(ws + base + align_up(MH));
  float* d_w = reinterpret_cast<float*>(ws + base + align_up(MH) + align_up(Mk));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // x and y in page-locked host memory are read and written in place by the
  // permute and reduce kernels (each x row is read once, each y row written
  // once, over the host link); other host memory is staged with copies.
  const void* x_in = device_view(host_x);
  void* y_out = device_view(host_y);
  void* d_x = ws + base;
  void* d_y = ws + base + align_up(MH) + 2 * align_up(Mk);
  if (x_in == nullptr) {
    if (cudaMemcpyAsync(d_x, host_x, MH, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return cuda_status(cudaGetLastError());
    x_in = d_x;
  }
  if (cudaMemcpyAsync(d_ids, host_topk_ids, Mk, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(d_w, host_topk_weights, Mk, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return cuda_status(cudaGetLastError());
  moe_status st = fused_experts(p, x_in, w13, w13_scale, w2, w2_scale, d_w, d_ids,
                                y_out ? y_out : d_y, workspace, base, stream);
  if (st != MOE_OK || y_out != nullptr) return st;
  return cuda_status(cudaMemcpyAsync(host_y, d_y, MH, cudaMemcpyDeviceToHost, s));
}

moe_status moe_sync_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  int* err = dev_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (v & kDevErrTimeout) return MOE_ERR_DEVICE_TIMEOUT;
  if (v & kDevErrBadIndex) return MOE_ERR_DEVICE_BAD_INDEX;
  return MOE_OK;
}

const char* moe_last_error_string(void) { return g_last_error; }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_DEVICE_BAD_INDEX: return "MOE_ERR_DEVICE_BAD_INDEX";
  }
  return "MOE_ERR_UNKNOWN";
}

size_t moe_batched_workspace_bytes(const moe_problem* p, int max_tokens) {
  if (!valid_batched(p, max_tokens)) return 0;
  return batched_layout(p, max_tokens).total;
}

moe_status fused_experts_batched(const moe_problem* p, const void* x,
                                 const int32_t* expert_num_tokens, int max_tokens,
                                 int expected_m, const void* w13, const void* w13_scale,
                                 const void* w2, const void* w2_scale, void* y, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (!valid_batched(p, max_tokens) || expected_m < 0) return MOE_ERR_INVALID_ARG;
  if (p->router_weight_in_gemm2 || p->act_recipe < 0 || p->act_recipe > 1)
    return MOE_ERR_INVALID_ARG;   // the layout carries no router weights
  if (!x || !expert_num_tokens || !w13 || !w2 || !y || !workspace) return MOE_ERR_INVALID_ARG;
  if (quantised(p) && (!w13_scale || !w2_scale)) return MOE_ERR_INVALID_ARG;
  if (!gemm_supported(p)) return MOE_ERR_UNSUPPORTED;
  const BatchedLayout L = batched_layout(p, max_tokens);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* blocks = reinterpret_cast<int32_t*>(ws + L.blocks);
  int32_t* npp = reinterpret_cast<int32_t*>(ws + L.npp);
  int32_t* ctr = reinterpret_cast<int32_t*>(ws + L.ctr);
  int32_t* sorted = quantised(p) ? reinterpret_cast<int32_t*>(ws + L.sorted) : nullptr;
  float* xscale = reinterpret_cast<float*>(ws + L.xscale);
  float* zscale = reinterpret_cast<float*>(ws + L.zscale);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int rows = p->E * max_tokens, H = p->H, I = p->I, E = p->E;
  const bool ue8m0 = p->act_scale_fmt == MOE_SCALE_UE8M0;
  const Epilogue ep = make_epilogue(p, nullptr, 0, nullptr, nullptr);
  cudaError_t e = launch_batched_blocks(expert_num_tokens, E, max_tokens, blocks, npp, sorted, s);
  if (e != cudaSuccess) return cuda_status(e);
  if (!quantised(p)) {
    // the layout's rows are GEMM1's rows as they are: no permute
    e = cudaMemsetAsync(ctr, 0, kTileCtrBytes, s);
    if (e == cudaSuccess)
      e = launch_bf16_gemm(expected_m, x, rows, H, w13, E * 2 * I, 2 * I, 2 * I, blocks, npp,
                           ws + L.z, true, ep, s, ctr);
    if (e != cudaSuccess) return cuda_status(e);
    e = launch_bf16_gemm(expected_m, ws + L.z, rows, I, w2, E * H, H, H, blocks, npp, y, false,
                         ep, s, ctr + 2);
    return cuda_status(e);
  }
  // quantised: per-row dynamic quantisation of the layout, then the same stages
  e = launch_permute_rows(x, H, 1, rows, sorted, npp, nullptr, ws + L.xq, xscale, ue8m0,
                          act_group(p), rows, s);
  if (e != cudaSuccess) return cuda_status(e);
  if (block_scaled(p)) {
    // GEMM1 with the activation and its quantisation in the epilogue
    e = launch_ggemm_mxfp4(ws + L.xq, xscale, rows, H, w13, static_cast<const uint8_t*>(w13_scale),
                           E * 2 * I, 2 * I, 2 * I, blocks, npp, ws + L.z,
                           p->quant == MOE_Q_MXFP8_1X32, ep, s, zscale, true, ue8m0,
                           p->weight_scales_prepacked != 0);
  } else {   // FP8 block scales: two steps (see fused_experts_ex)
    e = launch_ggemm_fp8(ws + L.xq, xscale, rows, H, w13, static_cast<const float*>(w13_scale),
                         E * 2 * I, 2 * I, 2 * I, blocks, npp, ws + L.h1, ep, s);
    if (e == cudaSuccess)
      e = launch_act_mul(ws + L.h1, I, npp, ws + L.z, zscale, ue8m0, act_group(p), rows, ep, s);
  }
  if (e != cudaSuccess) return cuda_status(e);
  if (block_scaled(p))
    e = launch_ggemm_mxfp4(ws + L.z, zscale, rows, I, w2, static_cast<const uint8_t*>(w2_scale),
                           E * H, H, H, blocks, npp, y, p->quant == MOE_Q_MXFP8_1X32, ep, s,
                           nullptr, false, true, p->weight_scales_prepacked != 0);
  else
    e = launch_ggemm_fp8(ws + L.z, zscale, rows, I, w2, static_cast<const float*>(w2_scale),
                         E * H, H, H, blocks, npp, y, ep, s);
  return cuda_status(e);
}

moe_status moe_topk_router(int M, int E, int topk, const void* logits, int logits_bf16,
                           int scoring, int renormalize, const int32_t* expert_map,
                           float* topk_weights, int32_t* topk_ids,
                           int32_t* token_expert_indices, void* stream) {
  if (M < 0 || M > MOE_MAX_TOKENS || E < 1 || E > MOE_MAX_EXPERTS || topk < 1 ||
      topk > MOE_MAX_TOPK || topk > E ||
      (scoring != MOE_SCORE_SOFTMAX && scoring != MOE_SCORE_SIGMOID))
    return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  if (!logits || !topk_weights || !topk_ids) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_topk_router(logits, logits_bf16 != 0, M, E, topk,
                                        scoring == MOE_SCORE_SIGMOID, renormalize != 0,
                                        expert_map, topk_weights, topk_ids,
                                        token_expert_indices, static_cast<cudaStream_t>(stream)));
}

void moe_debug_set_watchdog(int64_t limit_ns, int never_arrive) {
  g_watchdog_ns = limit_ns > 0 ? limit_ns : 0;
  g_never_arrive = never_arrive != 0;
}

void moe_debug_set_bf16_gemm_form(int mode) { g_bf16_form = (mode == 1 || mode == 2) ? mode : 0; }

}  // extern "C"
