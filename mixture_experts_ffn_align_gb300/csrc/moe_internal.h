// Host-side launchers shared between the translation units of the library.
// Every launcher enqueues work on `stream` and returns a cudaError_t from the
// launch (argument validation happens in capi.cu before these are called).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

namespace moe {

struct Epilogue;   // optional GEMM epilogue work (moe_common.cuh)

constexpr int kRouteSeg = 512;        // routed items handled by one warp
constexpr int kRouteWarps = 8;        // warps per routing CTA

inline int route_segments(int R) { return (R + kRouteSeg - 1) / kRouteSeg; }

constexpr int kMaxDevices = 64;               // devices the per-device caches cover
// Current device in [0, kMaxDevices), or -1 when cudaGetDevice fails or the
// index is beyond the caches (the library then reports an error).
int device_index();
int num_sms();                                // SMs of the current device (0 if -1)
int* dev_error_word();                        // device address of the error word (or null)
void watchdog_params(uint64_t* limit_ns, int* never_arrive);

// One-time setup per device: kernel attributes (the dynamic shared-memory
// opt-in) belong to the device they were set on.  call(f) runs f() on the
// current device until it has succeeded there once; later calls return
// cudaSuccess without running it.  Thread-safe.
class DeviceOnce {
 public:
  template <class F>
  cudaError_t call(F&& f) {
    const int d = device_index();
    if (d < 0) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu_);
    if ((done_ >> d) & 1u) return cudaSuccess;
    const cudaError_t e = f();
    if (e == cudaSuccess) done_ |= 1ull << d;
    return e;
  }

 private:
  std::mutex mu_;
  uint64_t done_ = 0;
};

// Stage 1 routes R items over E experts in one CTA (k_route_small) rather than
// three kernels (histograms, scan, scatter).
bool route_in_one_cta(int R, int E);
// Routing half of moe_align_permute (one or three launches).
cudaError_t launch_route(const int32_t* topk_ids, int R, int E, int block_size, int cap,
                         int32_t* hist, int32_t* sorted_ids, int32_t* block_expert_ids,
                         int32_t* expert_offsets, int32_t* num_post_padded, int32_t* inv_perm,
                         cudaStream_t stream);

// Data half: gather x rows into the padded layout (bf16 copy, or fused
// dynamic 1x128 e4m3 quantisation when x_scale != nullptr).
// group: the quantisation group along H (128, or 32 for MXFP8).
cudaError_t launch_permute_rows(const void* x, int H, int topk, int R, const int32_t* sorted_ids,
                                const int32_t* num_post_padded, const float* row_weights,
                                void* x_perm, float* x_scale, bool ue8m0, int group, int cap,
                                cudaStream_t stream);

// Token-major form of the quantising permute: each token's row is read and
// quantised once and stored to its destination rows (inv_perm); padding rows
// below num_post_padded are zeroed.  No router weight on the input.
cudaError_t launch_permute_tokens(const void* x, int H, int M, int topk, int R,
                                  const int32_t* inv_perm, const int32_t* sorted_ids,
                                  const int32_t* num_post_padded, void* x_perm, float* x_scale,
                                  bool ue8m0, int group, int cap, cudaStream_t stream);

// Token-major bf16 permute (a copy of each token's row into its k rows, read
// once); padding rows below num_post_padded are zeroed.
cudaError_t launch_permute_bf16_tokens(const void* x, int H, int M, int topk, int R,
                                       const int32_t* inv_perm, const int32_t* sorted_ids,
                                       const int32_t* num_post_padded, void* x_perm, int cap,
                                       cudaStream_t stream);

// SiLU-and-mul over h1 [rows, 2I] bf16 -> z bf16, or e4m3 + scales.
// act: the gated activation recipe (recipe / alpha / beta / limit fields).
cudaError_t launch_act_mul(const void* h1, int I, const int32_t* num_post_padded, void* z,
                           float* z_scale, bool ue8m0, int group, int cap, const Epilogue& act,
                           cudaStream_t stream);

// Weighted top-k gather-reduce into y [M, H] bf16.
cudaError_t launch_unpermute_reduce(const void* y2, int H, int M, int topk,
                                    const int32_t* inv_perm, const float* topk_weights,
                                    bool unit_weights, void* y, cudaStream_t stream);

// Batched layout [E, T, H] (T % 128 == 0): per-expert counts -> block expert
// ids of the E*T/128 row blocks (-1 past a count), num_post_padded = E*T, and
// (if sorted_ids != nullptr) the identity row map with padding id E*T.
cudaError_t launch_batched_blocks(const int32_t* counts, int E, int T, int32_t* block_expert_ids,
                                  int32_t* num_post_padded, int32_t* sorted_ids,
                                  cudaStream_t stream);

// Router: softmax / sigmoid top-k per token, one warp per token.
cudaError_t launch_topk_router(const void* logits, bool bf16, int M, int E, int k, bool sigmoid,
                               bool renorm, const int32_t* expert_map, float* w, int32_t* ids,
                               int32_t* tei, cudaStream_t stream);

// The grouped GEMMs below walk each expert's segment of the padded layout in
// 128-row m-tiles (tile_sched.cuh); blk_rows is the layout's block size (16,
// 32, 64 or 128: the block ids' granularity).  The SM-pair forms take 128 only.
//
// bf16 grouped GEMM on tcgen05: out[row, n] = sum_k A[row, k] * B[e*b_rows + n, k].
//   fuse_act: B tile = 128 gate rows + 128 up rows; writes SiLU(g)*u (bf16).
//   part != nullptr (not with fuse_act): K is cut into `splits` slices (a
//   count that would leave a slice empty is an error) and each live row's
//   fp32 slice sums go to part[(slice * part_R + part_ids[row]) * n_out + n]
//   instead of out.
cudaError_t launch_ggemm_bf16(const void* A, int cap, int K, const void* B, int b_rows_total,
                              int b_rows_per_expert, int n_out, const int32_t* block_expert_ids,
                              const int32_t* num_post_padded, void* out, bool fuse_act,
                              const Epilogue& ep, cudaStream_t stream, int splits = 1,
                              float* part = nullptr, const int32_t* part_ids = nullptr,
                              int part_R = 0, int blk_rows = 128);

// Weighted top-k reduce of split-K GEMM2 partials: y[t, :] = bf16( sum_i w[t,i] *
// bf16( sum_s part[s, t*k + i, :] ) ), fp32, slots and slices in order; slots
// with inv_perm < 0 are skipped.  H % 256 == 0.
cudaError_t launch_unpermute_reduce_split(const float* part, int splits, int H, int M, int topk,
                                          const int32_t* inv_perm, const float* topk_weights,
                                          void* y, cudaStream_t stream);
// The same GEMM issued on SM pairs (cta_group::2, 256 x 256 tiles).  Tiles
// are handed out by a device counter of two ints: tile_ctr (zero when the
// launch starts; the launch leaves it zero), or with nullptr one slot of a
// library-owned ring (launches that overlap on the GPU must be fewer than its
// 64 slots, and a launch captured in a graph keeps its slot).
cudaError_t launch_ggemm_bf16_2sm(const void* A, int cap, int K, const void* B,
                                  int b_rows_total, int b_rows_per_expert, int n_out,
                                  const int32_t* block_expert_ids,
                                  const int32_t* num_post_padded, void* out, bool fuse_act,
                                  const Epilogue& ep, cudaStream_t stream,
                                  int* tile_ctr = nullptr);

// A tile counter (two ints, zero between launches) from the library-owned
// ring of the SM-pair GEMMs, for launches that bring none of their own;
// nullptr when the current device is unusable.
int* next_tile_counter();

// FP8 (e4m3) grouped GEMM with fp32 1x128 activation scales and 128x128
// weight block scales: out = sum_kb sa*sb*partial_kb (bf16 output).
// fuse_act (GEMM1 only, n_out = b_rows_per_expert = 2I): the gated
// activation quantised to e4m3 codes in out [cap, I], 1x128 scales in z_scale.
cudaError_t launch_ggemm_fp8(const void* A, const float* a_scale, int cap, int K, const void* B,
                             const float* b_scale, int b_rows_total, int b_rows_per_expert,
                             int n_out, const int32_t* block_expert_ids,
                             const int32_t* num_post_padded, void* out, const Epilogue& ep,
                             cudaStream_t stream, float* z_scale = nullptr,
                             bool fuse_act = false, bool ue8m0 = false, int blk_rows = 128);

// The same FP8 GEMM (no fused activation) issued on SM pairs (cta_group::2,
// 256 x 256 tiles); n_out == b_rows_per_expert, a multiple of 128.  Tile
// counter as for launch_ggemm_bf16_2sm.
cudaError_t launch_ggemm_fp8_2sm(const void* A, const float* a_scale, int cap, int K,
                                 const void* B, const float* b_scale, int b_rows_total,
                                 int b_rows_per_expert, int n_out,
                                 const int32_t* block_expert_ids,
                                 const int32_t* num_post_padded, void* out, const Epilogue& ep,
                                 cudaStream_t stream, int* tile_ctr = nullptr);

// MXFP4 (E2M1 + E8M0 per 32) weights x e4m3 activations with power-of-two
// 1x128 scales (or MXFP8: e4m3 weights, b_e4m3, with 1x32 scales),
// block-scaled tensor-core MMA (bf16 output).  fuse_act (GEMM1 only, n_out =
// b_rows_per_expert = 2I): the gated activation quantised to e4m3 codes in
// out [cap, I] with scales in z_scale (1x128 groups, 1x32 for MXFP8).
cudaError_t launch_ggemm_mxfp4(const void* A, const float* a_scale, int cap, int K, const void* B,
                               const uint8_t* b_scale, int b_rows_total, int b_rows_per_expert,
                               int n_out, const int32_t* block_expert_ids,
                               const int32_t* num_post_padded, void* out, bool b_e4m3,
                               const Epilogue& ep, cudaStream_t stream,
                               float* z_scale = nullptr, bool fuse_act = false,
                               bool ue8m0 = true, bool scales_prepacked = false,
                               int blk_rows = 128);

// The block-scaled GEMM on SM pairs (cta_group::2, 256 x 256 tiles) for
// prepacked weight scales (b_scale_packed, the layout below) and 128-row
// blocks; otherwise as launch_ggemm_mxfp4.  Tile counter as for
// launch_ggemm_bf16_2sm.
cudaError_t launch_ggemm_mx_2sm(const void* A, const float* a_scale, int cap, int K, const void* B,
                                const uint8_t* b_scale_packed, int b_rows_total,
                                int b_rows_per_expert, int n_out,
                                const int32_t* block_expert_ids, const int32_t* num_post_padded,
                                void* out, bool b_e4m3, const Epilogue& ep, cudaStream_t stream,
                                float* z_scale = nullptr, bool fuse_act = false,
                                bool ue8m0 = true, int* tile_ctr = nullptr);

// E8M0 weight scales [E, N, K/32] -> the operand layout the block-scaled MMA
// copies into tensor memory: [E][K/128][N/128] blocks of 512 bytes, block
// byte 16 l + 4 c + j = scale of row 32 c + l of the group, K chunk 4 kb + j.
// N and K multiples of 128, scale 4-byte and packed 16-byte aligned.
cudaError_t launch_prepack_mx_scales(const uint8_t* scale, int E, int N, int K, void* packed,
                                     cudaStream_t stream);

}  // namespace moe
