/*
 * moe_ffn.h -- C ABI of the GB300 (sm_103a) fused MoE expert forward.
 *
 * The library computes, for hidden states x[M,H], router outputs
 * topk_ids[M,k] / topk_weights[M,k] and expert weights w13[E,2I,H] (gate rows
 * [0,I), up rows [I,2I)) and w2[E,H,I]:
 *
 *   y_t = sum_{i: id[t,i] >= 0} w[t,i] * W2_e( SiLU(W1gate_e x_t) * (W1up_e x_t) )
 *
 * in the five stages described on the page "Blackwell 上的 DeepGEMM FusedMoE
 * （vLLM）" (§1.1 six-step table, §2.6) and on the page "fused_moe.py 分析"
 * (§1.2-1.3, "moe_align_block_size 的作用", "fused_moe_kernel 的核心原理"):
 *   1. block-aligned routing + permute  (moe_align_permute)
 *   2. grouped GEMM1 over w13           (grouped_gemm_w13)
 *   3. SiLU-and-mul (+ dynamic FP8)     (act_mul_quant, or fused into 2)
 *   4. grouped GEMM2 over w2            (grouped_gemm_w2, or in K slices:
 *                                        grouped_gemm_w2_split)
 *   5. weighted unpermute + reduce      (unpermute_reduce, or
 *                                        unpermute_reduce_split)
 * and fused_experts runs all five (fused_experts_ex with expert biases and
 * epilogue options, fused_experts_from_host from host buffers,
 * fused_experts_batched on the batched [E, T, H] layout).  moe_topk_router
 * is the step before: logits -> topk_ids / topk_weights.
 *
 * Conventions for every entry point:
 *  - Pointers named as device pointers must point to device memory of the
 *    current CUDA device; the caller owns every buffer (inputs, outputs and
 *    workspaces) and keeps it alive until the work on `stream` completes.
 *  - All tensors are dense, row-major, with the last dimension contiguous.
 *    Base addresses must be 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *    asynchronous on that stream; a call never synchronises the host.
 *  - Argument errors are detected on the host before any launch and return
 *    MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_WORKSPACE_TOO_SMALL
 *    with nothing enqueued.  Errors found by kernels (an expert id >= E, a
 *    bounded device wait that ran out) are recorded in a device error word
 *    and reported by moe_sync_status().
 *  - M == 0 is valid: nothing is launched and MOE_OK is returned.
 */
#ifndef MOE_FFN_H_
#define MOE_FFN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,          /* bad shape, null pointer, bad enum */
  MOE_ERR_UNSUPPORTED = 2,          /* valid problem the kernels do not cover */
  MOE_ERR_CUDA = 3,                 /* a CUDA runtime call failed */
  MOE_ERR_DEVICE_TIMEOUT = 4,       /* a bounded device wait ran out */
  MOE_ERR_WORKSPACE_TOO_SMALL = 5,  /* workspace_bytes below the requirement */
  MOE_ERR_DEVICE_BAD_INDEX = 6      /* a kernel saw an expert id >= E */
} moe_status;

/* Weight / activation formats (page "Blackwell 上的 DeepGEMM FusedMoE（vLLM）",
 * TL;DR table).
 *  MOE_Q_BF16:          bf16 x, w13, w2; bf16 intermediates.
 *  MOE_Q_FP8_BLOCK128:  w13/w2 e4m3fn codes (uint8) with fp32 scales per
 *                       128x128 block, scale arrays [E, ceil(N/128), ceil(K/128)];
 *                       activations quantised on the fly to e4m3fn per 1x128
 *                       group (dynamic scale amax/448).
 *  MOE_Q_MXFP4_W4A8:    w13/w2 E2M1 codes packed two per byte ([E, N, K/2],
 *                       low nibble = even k) with E8M0 scales per 32 along K
 *                       ([E, N, K/32] uint8); activations e4m3fn per 1x128.
 *  MOE_Q_MXFP8_1X32:    w13/w2 e4m3fn codes ([E, N, K] uint8) with E8M0
 *                       scales per 1x32 along K ([E, N, K/32] uint8);
 *                       activations e4m3fn per 1x32 group with UE8M0 scales
 *                       (act_scale_fmt must be MOE_SCALE_UE8M0), stored as
 *                       fp32 powers of two [S, K/32] (MXFP8 1x32 row of the
 *                       same table).
 */
typedef enum {
  MOE_Q_BF16 = 0,
  MOE_Q_FP8_BLOCK128 = 1,
  MOE_Q_MXFP4_W4A8 = 2,
  MOE_Q_MXFP8_1X32 = 3
} moe_quant;

/* Activation scale format of the quantised modes: fp32 amax/448, or that
 * value rounded up to a power of two (UE8M0; page "Blackwell 上的 DeepGEMM
 * FusedMoE（vLLM）", §2.8(f), FLOAT32_CEIL_UE8M0).  Scales are always stored as
 * fp32 values. */
typedef enum { MOE_SCALE_FP32 = 0, MOE_SCALE_UE8M0 = 1 } moe_scale_fmt;

/* The problem statement (page 1, "FusedMoEExpertsModular.apply" and
 * "moe_problem_size": E, M, N = 2I, K = H, topk).
 *  block_size: padding granularity of each expert's rows (BLOCK_SIZE_M);
 *              one of 16, 32, 64, 128.  The grouped GEMMs compute 128-row
 *              tiles inside each expert's padded segment (a smaller block
 *              size pads less and leaves a partial last tile per expert,
 *              whose rows past the segment are not written); the SM-pair
 *              GEMM forms and fused_experts_batched take 128 only (the
 *              others are then used).
 *  apply_router_weight_on_input: multiply x_t by its router weight before
 *              GEMM1 and reduce with weight 1 (top-k must be 1).
 *  router_weight_in_gemm2: GEMM2's epilogue multiplies each output row by its
 *              routed item's weight (fp32, after the bias, before the bf16
 *              cast) and the reduce only sums (page "fused_moe.py 分析",
 *              fused_moe_kernel post-processing "optional router weight";
 *              TopKWeightAndReduce when the experts already applied it).
 *              Not together with apply_router_weight_on_input.
 *  weight_scales_prepacked: (MOE_Q_MXFP4_W4A8, MOE_Q_MXFP8_1X32) w13_scale and
 *              w2_scale passed to the GEMM entry points are the buffers
 *              moe_prepack_weights wrote, not the [E, N, K/32] E8M0 arrays.
 *  act_recipe: 0: z = SiLU(gate) * up.  1: the recipe of gemm1_alpha,
 *              gemm1_beta and gemm1_clamp_limit (page "Blackwell 上的 DeepGEMM
 *              FusedMoE（vLLM）", §2.6.4): with L = gemm1_clamp_limit,
 *              g' = min(gate, L), u' = clamp(up, -L, L) (no clamp if L <= 0),
 *              z = (u' + beta) * g' * sigmoid(alpha * g'); alpha = 1, beta = 0
 *              and no clamp give SiLU-and-mul back.
 * Zero-initialised trailing fields select the plain path.
 */
typedef struct {
  int32_t M, H, I, E, topk, block_size;
  int32_t quant;          /* moe_quant */
  int32_t act_scale_fmt;  /* moe_scale_fmt */
  int32_t apply_router_weight_on_input;
  int32_t router_weight_in_gemm2;
  int32_t act_recipe;
  float gemm1_alpha, gemm1_beta, gemm1_clamp_limit;
  int32_t weight_scales_prepacked;
} moe_problem;

/* Limits checked by every entry point: 0 <= M <= MOE_MAX_TOKENS (the pages'
 * CHUNK_SIZE, page "fused_moe.py 分析", "分 chunk 执行"), 1 <= topk <= 16,
 * 1 <= E <= 1024, H and I positive multiples of 128. */
#define MOE_MAX_TOKENS 16384
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOPK 16

/* Rows of the padded (permuted) layout: the worst case over all routings,
 * round_up(M*k + min(M*k, E)*(block_size-1), block_size) (page "Blackwell 上的
 * DeepGEMM FusedMoE（vLLM）", §2.6.1, compute_aligned_M_and_alignment).
 * Returns 0 for an invalid problem. */
size_t moe_m_sum_bound(const moe_problem* p);

/* Bytes of scratch that moe_align_permute needs in `workspace` (per-segment
 * expert histograms).  0 for an invalid problem. */
size_t moe_align_workspace_bytes(const moe_problem* p);

/* Number of kernels moe_align_permute launches for p when it is given x and
 * x_perm (for launch accounting): the routing kernels -- 1 when the problem
 * routes in one CTA (M*topk <= 2048, or <= 8192 with E <= 64), else 3
 * (histograms, scan, scatter) -- plus the permute.  0 when M == 0 and for an
 * invalid problem.  Host-only; launches nothing. */
int moe_align_permute_launches(const moe_problem* p);

/* Bytes of workspace fused_experts needs (routing scratch, indices and every
 * intermediate, sized for moe_m_sum_bound rows, with the permuted input and
 * the GEMM2 output sharing storage as the page's workspace13 does, §2.8(a)).
 * 0 for an invalid problem. */
size_t moe_workspace_bytes(const moe_problem* p);

/* Load-time rewrite of the block-scaled weights' scales (page "Blackwell 上的
 * DeepGEMM FusedMoE（vLLM）", §2.8: the weight scale factors are transformed
 * once, when the weights are loaded, into the layout the GEMM kernel reads --
 * transform_sf_into_required_layout).  For MOE_Q_MXFP4_W4A8 and
 * MOE_Q_MXFP8_1X32 only (other modes: MOE_ERR_UNSUPPORTED).
 *  in : w13_scale [E, 2I, H/32] and w2_scale [E, H, I/32] E8M0 bytes (device).
 *  out: w13_scale_packed and w2_scale_packed (device, 16-byte aligned, each
 *       moe_prepacked_scale_bytes(p, 0 / 1) bytes, the same size as the
 *       input): for every expert e, K block kb (128 deep) and group g of 128
 *       weight rows, in that order ([E][K/128][N/128]), one 512-byte block
 *       whose byte 16 l + 4 c + j is the scale of row 128 g + 32 c + l, K
 *       chunk 4 kb + j -- the 32 x 16-byte operand the block-scaled MMA copies
 *       into tensor memory, so the GEMM loads it as it is.
 * The weights themselves keep their layout.  Set p->weight_scales_prepacked
 * and pass the packed buffers as w13_scale / w2_scale to the GEMM entry points
 * and fused_experts; results are identical to the unpacked call.  Asynchronous
 * on `stream`; the inputs must not be written until it completes. */
size_t moe_prepacked_scale_bytes(const moe_problem* p, int which /* 0: w13, 1: w2 */);
moe_status moe_prepack_weights(const moe_problem* p, const void* w13_scale, const void* w2_scale,
                               void* w13_scale_packed, void* w2_scale_packed, void* stream);

/* Stage 1: block-aligned routing and permute (page "fused_moe.py 分析",
 * "moe_align_block_size 的作用"; page "Blackwell 上的 DeepGEMM FusedMoE（vLLM）",
 * §2.6.2 ep_scatter).  Routed item r = t*k + i (token r / k).
 *  in : topk_ids [M*k] int32 device (-1 = skip the slot; >= E is an error),
 *       x [M,H] bf16 device, topk_weights [M*k] fp32 device (read only when
 *       apply_router_weight_on_input, else may be NULL).
 *  out: sorted_ids [S] int32 (S = moe_m_sum_bound): routed item per padded
 *         row, ascending r within an expert, padding = M*k;
 *       block_expert_ids [S/block_size] int32: expert of each block, -1 past
 *         the used blocks;
 *       expert_offsets [E+1] int32: first padded row of each expert, [E] = total;
 *       num_post_padded [1] int32: used rows (a multiple of block_size);
 *       inv_perm [M*k] int32: padded row of each routed item, -1 for skipped;
 *       x_perm [S,H]: x[token] per used row, zero rows for padding; bf16 for
 *         MOE_Q_BF16, e4m3fn codes (uint8) for the quantised modes;
 *       x_perm_scale [S,H/128] fp32 (quantised modes only, else may be NULL):
 *         one scale per 1x128 group, 0 for padding rows.
 *       x and x_perm may both be NULL to run the routing half only.
 *  workspace: >= moe_align_workspace_bytes(p) bytes of device scratch. */
moe_status moe_align_permute(const moe_problem* p, const void* x, const int32_t* topk_ids,
                             const float* topk_weights, int32_t* sorted_ids,
                             int32_t* block_expert_ids, int32_t* expert_offsets,
                             int32_t* num_post_padded, int32_t* inv_perm, void* x_perm,
                             float* x_perm_scale, void* workspace, size_t workspace_bytes,
                             void* stream);

/* The batched (masked) expert layout, for decode steps captured in CUDA
 * graphs (page "fused_moe.py 分析", activation formats Standard [M, K] and
 * BatchedExperts [E, max_tokens, K]; page "Blackwell 上的 DeepGEMM FusedMoE（vLLM）",
 * §2.5: DeepEP low-latency dispatch hands over [E_local, max_tokens, K] with
 * the per-expert token counts, and the experts run a masked grouped GEMM; the
 * expected_m hint of the same pages).  For each expert e and each row
 * r < expert_num_tokens[e]:
 *   y[e, r, :] = W2_e( SiLU(W1gate_e x[e, r, :]) * (W1up_e x[e, r, :]) )
 * with the path's roundings (bf16 GEMM outputs; in the quantised modes x and
 * the activation are quantised per 1x128 group as in stages 1 and 3).  No
 * router weight is applied (the combine after the experts applies it).
 *  - p: E, H, I, block_size (must be 128), quant, act_scale_fmt as for
 *    fused_experts; p->M, p->topk and apply_router_weight_on_input are ignored.
 *  - x, y: device, [E, max_tokens, H] bf16, row-major; rows of y at or past a
 *    count are left as they were or hold values of no meaning.
 *  - expert_num_tokens: device, E int32, read on the device (a graph replay
 *    sees the counts of the moment); each is clamped to [0, max_tokens].
 *  - max_tokens: a positive multiple of 128, E * max_tokens <= MOE_MAX_TOKENS *
 *    MOE_MAX_TOPK.
 *  - expected_m: expected tokens per expert (0 if unknown); picks the tile
 *    form of the bf16 GEMMs (SM pairs from 256 up), never the results.
 *  - workspace: device, at least moe_batched_workspace_bytes(p, max_tokens).
 * Nothing is allocated and the host never waits on the device, so a call can
 * be captured in a CUDA graph once a first call has run outside capture.
 * Errors: MOE_ERR_INVALID_ARG (bad sizes or NULL pointers),
 * MOE_ERR_UNSUPPORTED (as for fused_experts), MOE_ERR_WORKSPACE_TOO_SMALL,
 * MOE_ERR_CUDA. */
size_t moe_batched_workspace_bytes(const moe_problem* p, int max_tokens);
moe_status fused_experts_batched(const moe_problem* p, const void* x,
                                 const int32_t* expert_num_tokens, int max_tokens,
                                 int expected_m, const void* w13, const void* w13_scale,
                                 const void* w2, const void* w2_scale, void* y, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* Router: the step before the path (page "fused_moe.py 分析", section
 * "topk_ids, topk_weights 的由来以及内容": fused_topk with scoring_func softmax
 * or sigmoid and renormalize; expert_map from the same page).  For each of M
 * tokens (one row of logits[M, E], device, row-major, fp32 or bf16 with
 * logits_bf16 != 0):
 *  - the k experts with the largest logits -- the largest scores, since both
 *    scores increase with the logit; equal logits in ascending expert order --
 *    go to topk_ids[t, 0..k) in that order;
 *  - their scores (softmax over the row's E logits, or sigmoid of the logit)
 *    go to topk_weights[t, 0..k) (fp32), divided by the k scores' sum when
 *    renormalize != 0;
 *  - token_expert_indices[t, i] = t*k + i, the routed-item index (may be NULL);
 *  - with expert_map (device, E int32: the expert's id on this expert-parallel
 *    shard, or -1 when it lives elsewhere; may be NULL) the ids written are
 *    expert_map[id]; -1 ids are skipped by every stage of the path.
 * All outputs are device buffers of M*k elements, written on `stream`.
 * Errors: MOE_ERR_INVALID_ARG when M < 0 or M > MOE_MAX_TOKENS, E < 1 or
 * E > MOE_MAX_EXPERTS, topk < 1 or topk > min(E, MOE_MAX_TOPK), scoring is
 * not a moe_scoring value, or logits / topk_weights / topk_ids is NULL with
 * M > 0.  M = 0 returns MOE_OK without launching. */
typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_scoring;
moe_status moe_topk_router(int M, int E, int topk, const void* logits, int logits_bf16,
                           int scoring, int renormalize, const int32_t* expert_map,
                           float* topk_weights, int32_t* topk_ids,
                           int32_t* token_expert_indices, void* stream);

/* Stage 1 without a workspace, for callers that cannot allocate device memory
 * when they call the library -- for example a serving engine that reserves the
 * whole device for its own memory pool and does not let plug-ins call
 * cudaMalloc, or a latency-critical loop that cannot accept cudaMalloc's
 * implicit device synchronisation.  The paper has no counterpart: this is a
 * deployment convenience, not a stage of the method.
 *
 * Same arguments, outputs and errors as moe_align_permute, minus the
 * workspace: its scratch (per-segment expert histograms) is a fixed array of
 * MOE_NOALLOC_SCRATCH_BYTES that the library keeps in each GPU's memory for
 * the life of the process.  The entry point allocates nothing (no cudaMalloc,
 * cudaFree or allocating library call).
 *  - Limit: problems whose moe_align_workspace_bytes(p) exceeds
 *    MOE_NOALLOC_SCRATCH_BYTES (more than 262144 segment x expert counters,
 *    e.g. M*k > 131072 with E = 1024) are rejected with
 *    MOE_ERR_WORKSPACE_TOO_SMALL before anything is enqueued; use
 *    moe_align_permute with a workspace for those.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls on a device share the one array and it keeps the last call's
 *    contents (each call overwrites what it reads, so nothing carries over).
 *    Calls whose work overlaps on the GPU (different streams without
 *    ordering between them) race on it: order them on one stream. */
#define MOE_NOALLOC_SCRATCH_BYTES (1u << 20)
moe_status moe_align_permute_noalloc(const moe_problem* p, const void* x,
                                     const int32_t* topk_ids, const float* topk_weights,
                                     int32_t* sorted_ids, int32_t* block_expert_ids,
                                     int32_t* expert_offsets, int32_t* num_post_padded,
                                     int32_t* inv_perm, void* x_perm, float* x_perm_scale,
                                     void* stream);

/* Stage 2: grouped GEMM1, H1[row, n] = sum_k x_perm[row, k] * w13[e, n, k] for
 * every used block (page "fused_moe.py 分析", §1.3 routed GEMM and
 * "fused_moe_kernel 的核心原理"; FP8 blocks: "FP8 W8A8").  fp32 accumulation.
 *  in : x_perm [S,H] (+ x_scale [S,H/128] fp32 for quantised modes; [S,H/32]
 *       for MOE_Q_MXFP8_1X32),
 *       w13 [E,2I,H] (+ w13_scale), block_expert_ids, num_post_padded (device).
 *  out: fuse_act == 0: h1 [S,2I] bf16.
 *       fuse_act == 1: the gated activation (p->act_recipe) written directly
 *       (MOE_Q_BF16: z [S,I] bf16; quantised modes: out = z [S,I] e4m3fn
 *       codes and out_scale = z_scale [S,I/group] fp32, exactly as
 *       act_mul_quant would write them from h1; MOE_Q_FP8_BLOCK128 and
 *       MOE_Q_MXFP4_W4A8: 1x128 groups, MOE_Q_MXFP8_1X32: 1x32).  out_scale
 *       is only read when a quantised mode fuses the activation (then
 *       required).  fused_experts runs GEMM1 this way except for
 *       MOE_Q_FP8_BLOCK128, whose promotion epilogue bounds the GEMM (two
 *       steps measured faster there).
 *  Rows of blocks past num_post_padded are not written. */
moe_status grouped_gemm_w13(const moe_problem* p, const void* x_perm, const float* x_scale,
                            const void* w13, const void* w13_scale,
                            const int32_t* block_expert_ids, const int32_t* num_post_padded,
                            void* out, float* out_scale, int fuse_act, void* stream);

/* Stage 3: SiLU-and-mul, z = SiLU(h1[:, :I]) * h1[:, I:] (or the recipe of
 * p->act_recipe), computed in fp32 from the bf16 h1 (page "Blackwell 上的
 * DeepGEMM FusedMoE（vLLM）", §2.6.4; page "fused_moe.py 分析",
 * _silu_and_mul_kernel).  MOE_Q_BF16: z [S,I] bf16.
 * Quantised modes: z [S,I] e4m3fn codes + z_scale [S,I/128] fp32 (dynamic
 * per 1x128 group; [S,I/32] per 1x32 for MOE_Q_MXFP8_1X32).  Only rows below
 * num_post_padded are written. */
moe_status act_mul_quant(const moe_problem* p, const void* h1, const int32_t* num_post_padded,
                         void* z, float* z_scale, void* stream);

/* Stage 4: grouped GEMM2, Y2[row, h] = sum_j z[row, j] * w2[e, h, j] (same
 * passages as stage 2).  out: y2 [S,H] bf16.
 *
 * Concurrency of stages 2 and 4 in MOE_Q_BF16: at prefill sizes the GEMM runs
 * on SM pairs whose tiles are handed out by a device counter.  These entry
 * points take the counter from a library-owned ring of 64 per device, so
 * launches of them that overlap on the GPU (other streams, or graph replays
 * running beside them) must number fewer than 64, and a launch captured in a
 * CUDA graph keeps its counter at every replay: order such replays with the
 * other stage-2/4 launches on one stream.  fused_experts and its variants
 * keep their counters in the caller's workspace and have no such limit. */
moe_status grouped_gemm_w2(const moe_problem* p, const void* z, const float* z_scale,
                           const void* w2, const void* w2_scale,
                           const int32_t* block_expert_ids, const int32_t* num_post_padded,
                           void* y2, void* stream);

/* Stage 5: weighted unpermute + top-k reduce (page "Blackwell 上的 DeepGEMM
 * FusedMoE（vLLM）", §2.6.5 ep_gather): y[t,:] = bf16( sum_{i, inv_perm[t,i] >= 0}
 * w'[t,i] * y2[inv_perm[t,i], :] ), fp32 accumulation in slot order,
 * w' = 1 when apply_router_weight_on_input or router_weight_in_gemm2 (the
 * weight is then already in y2).  y [M,H] bf16. */
moe_status unpermute_reduce(const moe_problem* p, const void* y2, const int32_t* inv_perm,
                            const float* topk_weights, void* y, void* stream);

/* Stages 4 and 5 in K slices (decode-sized bf16 problems; no counterpart on
 * the pages, which run one program per output block).  With few routed rows
 * per expert, GEMM2's 128 x 256 output tiles (used blocks x H/256) number
 * fewer than the SMs; cutting K into `splits` slices gives every SM work.
 *  - moe_gemm2_splits(p): the slice count fused_experts uses for p on the
 *    current device: 1 (no slicing: bf16 SM-pair form, quantised modes,
 *    H % 256 != 0, or enough tiles) up to 8.  0 for an invalid problem.
 *  - moe_gemm2_partial_bytes(p, splits): bytes of `partial`,
 *    splits * M * topk * H * 4.
 *  - grouped_gemm_w2_split: z [S,I] bf16 (MOE_Q_BF16 only, as from
 *    grouped_gemm_w13 with fuse_act), w2 [E,H,I], block ids,
 *    num_post_padded and sorted_ids from moe_align_permute; writes the fp32
 *    sums of slice s for routed item r = sorted_ids[row] < M*topk at
 *    partial[(s * M*topk + r) * H + h] (padding rows are not written).
 *    `splits` (1 to 8) must leave no slice empty, as the counts
 *    moe_gemm2_splits returns do (else MOE_ERR_INVALID_ARG).
 *  - unpermute_reduce_split: y[t,:] = bf16( sum_i w[t,i] * bf16( sum_s
 *    partial[s, t*topk+i, :] ) ), fp32, slices and slots in order; slots
 *    with inv_perm < 0 are skipped.  The bf16 rounding of the slice sum is
 *    the rounding of the stored Y2 of the unsliced form.  Not for
 *    apply_router_weight_on_input or router_weight_in_gemm2
 *    (MOE_ERR_INVALID_ARG). */
int moe_gemm2_splits(const moe_problem* p);
size_t moe_gemm2_partial_bytes(const moe_problem* p, int splits);
moe_status grouped_gemm_w2_split(const moe_problem* p, const void* z, const void* w2,
                                 const int32_t* block_expert_ids,
                                 const int32_t* num_post_padded, const int32_t* sorted_ids,
                                 int splits, float* partial, void* stream);
moe_status unpermute_reduce_split(const moe_problem* p, const float* partial, int splits,
                                  const int32_t* inv_perm, const float* topk_weights, void* y,
                                  void* stream);

/* All five stages (page 1, FusedMoEKernelModularImpl.apply: prepare ->
 * experts -> finalize; inplace when y == x, page "fused_moe.py 分析",
 * "对外入口").  Weights as described for moe_quant; w13_scale/w2_scale NULL
 * for MOE_Q_BF16.  workspace: >= moe_workspace_bytes(p) device bytes. */
moe_status fused_experts(const moe_problem* p, const void* x, const void* w13,
                         const void* w13_scale, const void* w2, const void* w2_scale,
                         const float* topk_weights, const int32_t* topk_ids, void* y,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Stages 2 and 4 and the whole forward with per-expert biases (page
 * "fused_moe.py 分析", fused_moe_kernel post-processing: dequant -> bias ->
 * router weight -> cast; the pages' bias inputs of the expert GEMMs):
 *  - w13_bias: device, [E, 2I] bf16 (gate columns then up columns), added in
 *    fp32 to GEMM1's sums before H1 is rounded; may be NULL.
 *  - w2_bias: device, [E, H] bf16, added to GEMM2's sums before the router
 *    weight (router_weight_in_gemm2) and the bf16 cast; may be NULL.
 *  - grouped_gemm_w2_ex also takes sorted_ids (from moe_align_permute) and
 *    topk_weights [M, topk] fp32, used (and then required) only when
 *    p->router_weight_in_gemm2 is set.
 * Otherwise as grouped_gemm_w13 / grouped_gemm_w2 / fused_experts, which are
 * these entry points with NULL biases. */
moe_status grouped_gemm_w13_ex(const moe_problem* p, const void* x_perm, const float* x_scale,
                               const void* w13, const void* w13_scale, const void* w13_bias,
                               const int32_t* block_expert_ids,
                               const int32_t* num_post_padded, void* out, float* out_scale,
                               int fuse_act, void* stream);
moe_status grouped_gemm_w2_ex(const moe_problem* p, const void* z, const float* z_scale,
                              const void* w2, const void* w2_scale, const void* w2_bias,
                              const int32_t* block_expert_ids, const int32_t* num_post_padded,
                              const int32_t* sorted_ids, const float* topk_weights, void* y2,
                              void* stream);
moe_status fused_experts_ex(const moe_problem* p, const void* x, const void* w13,
                            const void* w13_scale, const void* w13_bias, const void* w2,
                            const void* w2_scale, const void* w2_bias,
                            const float* topk_weights, const int32_t* topk_ids, void* y,
                            void* workspace, size_t workspace_bytes, void* stream);

/* fused_experts fed from host memory, all on `stream`; weights stay device
 * pointers.  topk_ids and topk_weights are copied into the staging part of
 * `workspace`.  x [M,H] bf16 and y [M,H] bf16: when a buffer is page-locked
 * host memory mapped for the device (cudaHostAlloc / cudaHostRegister, as
 * torch's pin_memory gives) and 16-byte aligned, the permute kernel reads
 * x and the reduce kernel writes y in place over the host link, each row
 * once; otherwise x is copied in and y copied out through the workspace.
 * host_x and host_y must stay valid and untouched until `stream` has
 * finished this call.  workspace: >= moe_host_workspace_bytes(p) device
 * bytes. */
size_t moe_host_workspace_bytes(const moe_problem* p);
moe_status fused_experts_from_host(const moe_problem* p, const void* host_x,
                                   const int32_t* host_topk_ids,
                                   const float* host_topk_weights, void* host_y,
                                   const void* w13, const void* w13_scale, const void* w2,
                                   const void* w2_scale, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* Synchronises `stream`, reads and clears the device error word, and returns
 * MOE_OK, MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_DEVICE_BAD_INDEX or MOE_ERR_CUDA. */
moe_status moe_sync_status(void* stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* moe_status_string(moe_status s);

/* Name and description of the CUDA error behind the calling thread's most
 * recent MOE_ERR_CUDA from a launch ("" if none yet).  Thread-local storage,
 * valid until the thread's next failing call. */
const char* moe_last_error_string(void);

/* Test hook for the device watchdog: with limit_ns > 0, every bounded wait in
 * the GEMM kernels gives up after limit_ns nanoseconds instead of the default
 * (2 s); with never_arrive != 0 the GEMM producer skips its first copy, so the
 * consumer wait runs out.  The kernel then records MOE_ERR_DEVICE_TIMEOUT,
 * drains what it issued, frees its tensor memory and returns.  Call with
 * (0, 0) to restore the defaults.  Not thread-safe; affects later launches. */
void moe_debug_set_watchdog(int64_t limit_ns, int never_arrive);

/* Test hook for the grouped GEMMs (stages 2 and 4), which come in two forms
 * with identical results up to fp32 summation order: 128 x 256 tiles on one
 * SM, and 256 x 256 tiles on SM pairs (cta_group::2).  By default bf16 uses
 * the pair form when the experts average at least two 128-row blocks
 * (M * topk >= 256 * E); FP8-block, MXFP4 and MXFP8 always use one SM (their
 * pair forms measured no faster; the FP8 GEMM1 with the activation fused has
 * the single-SM form only, the block-scaled pair form needs prepacked weight
 * scales).  The pair forms take block size 128 only.  mode 0 restores the
 * default, 1 forces the single-SM form, 2 the pair form where one exists.
 * Not thread-safe; affects later launches.  No counterpart on the pages: it
 * only lets tests reach both forms at any size. */
void moe_debug_set_bf16_gemm_form(int mode);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H_ */
