// bf16 grouped GEMM over the padded expert layout on 5th-generation tensor
// cores (stages 2 and 4).
//
// What it computes: page "fused_moe.py 分析", §1.3, C[r, n] = sum_k A[t(r), k]
// * B[e(r), n, k] with B stored [E, N, K] ("NT"); "fused_moe_kernel 的核心原理":
// one program owns one expert's block of BLOCK_SIZE_M routed rows times a
// column strip, fp32 accumulation, cast to bf16 on the way out; blocks whose
// expert id is -1 are not computed.  Page "Blackwell 上的 DeepGEMM FusedMoE
// （vLLM）", §2.6.3: the contiguous layout is read block by block with the
// block's expert id; the block height must equal the padding granularity.
//
// GB300 design (not the pages' Triton/DeepGEMM kernels):
//  * persistent CTAs (one per SM), tiles 128 x 256 walked expert by expert
//    (tile_sched.cuh): the CTAs running together share one expert, so each
//    weight tile is read from HBM once for all of that expert's m-blocks and
//    the expert's activation blocks stay in L2;
//  * warp 0 lane 0: TMA producer, 4-stage ring of (A 128x64, B 256x64) bf16
//    tiles, 128-byte swizzle;
//  * warp 1 lane 0: issues tcgen05.mma (M=128, N=256, K=16) into one of two
//    256-column fp32 accumulators in tensor memory, tcgen05.commit frees the
//    smem stage / publishes the accumulator;
//  * warps 2-5: epilogue, tcgen05.ld of their 32 TMEM lanes, bf16 convert,
//    and (GEMM1) the SiLU-and-mul fused in: the B tile holds 128 gate rows and
//    the matching 128 up rows, so one tile yields 128 columns of z.
//  * every wait is bounded (wall clock); on a timeout the kernel records the
//    error, drains its own copies and MMAs, frees tensor memory and returns.
#include <mutex>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "tile_sched.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;
constexpr int NUM_THREADS = 192;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/ + kSchedBytes;

struct GemmArgs {
  const int32_t* block_expert_ids;
  const int32_t* num_post_padded;
  __nv_bfloat16* out;
  int ldo;                // output row stride (elements)
  int num_kb;             // K / BK
  int n_tiles;            // column tiles
  int b_rows_per_expert;  // rows of B per expert
  int second_box_off;     // row offset of the second 128-row B box
  int n_tile_rows;        // B rows advanced per column tile
  int out_cols_per_tile;  // output columns per tile (256, or 128 when fused)
  int blocks_cap;         // blocks of blk_rows rows the A / output buffers hold
  int blk_rows;           // rows per block of the padded layout (16, 32, 64, 128)
  int num_experts;
  int group_max;          // m-tiles per scheduling group (L2 budget)
  uint64_t limit_ns;
  int never_arrive;
  int* err;
  Epilogue ep;            // bias, router weight, activation recipe
  // split-K (GEMM2 when its tiles would leave SMs idle): unit u is K slice
  // u % splits of tile u / splits; part != nullptr stores each live row's raw
  // fp32 sums at part[(slice * part_R + routed item) * ldo + column]
  int splits;
  int kb_per_split;
  float* part;
  const int32_t* part_ids;   // row -> routed item (sorted ids); >= part_R: padding
  int part_R;
};

template <bool FUSE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_ggemm_bf16(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // bars[0..S) full, [S..2S) empty, 2S..2S+1 tmem_full, 2S+2..2S+3 tmem_empty, 2S+4 drain
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_sched = reinterpret_cast<int*>(smem + STAGES * STAGE_BYTES + 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_u32(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  // never walk past the buffers, whatever the routing wrote
  const int nb_valid = min(*args.num_post_padded / args.blk_rows, args.blocks_cap);
  const TileSched sched =
      sched_build(args.block_expert_ids, nb_valid, args.blk_rows, args.num_experts, s_sched,
                  reinterpret_cast<int*>(smem), args.n_tiles, args.group_max);
  const int total = sched_mtiles(sched) * args.n_tiles * args.splits;   // work units

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_a = l2_policy(MOE_GEMM_L2_A);
    const uint64_t pol_b = l2_policy(MOE_GEMM_L2_B);
    uint32_t stage = 0, phase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;
    bool skip_first = args.never_arrive != 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const int t = u / args.splits, ks = u - t * args.splits;
      const Tile T = sched_tile(sched, t);
      const int e = T.e;
      const int brow = e * args.b_rows_per_expert + T.n_tile * args.n_tile_rows;
      const int kb0 = ks * args.kb_per_split;
      const int kb1 = min(args.num_kb, kb0 + args.kb_per_split);
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1, abort_flag, args.limit_ns, args.err)) {
          ok = false;
          break;
        }
        if (skip_first) {
          skip_first = false;   // watchdog test: leave this stage unarmed
        } else {
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          mbar_arrive_expect_tx(full_bar(stage), STAGE_BYTES);
          tma_load_2d(sa, &tmA, full_bar(stage), kb * BK, T.row0, pol_a);
          tma_load_2d(sb, &tmB, full_bar(stage), kb * BK, brow, pol_b);
          tma_load_2d(sb + 128 * 128, &tmB, full_bar(stage), kb * BK, brow + args.second_box_off,
                      pol_b);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
    }
    // drain: every copy this thread issued must land before the CTA exits
    for (int s = 0; s < STAGES; ++s)
      if (issued_mask & (1u << s))
        mbar_wait_bounded(full_bar(s), (issued_parity >> s) & 1, nullptr, args.limit_ns, args.err);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = make_idesc(kFmtBF16, kFmtBF16, BM, BN);
    uint32_t stage = 0, phase = 0;
    int local = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const int ks = u % args.splits;
      if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1, abort_flag, args.limit_ns, args.err)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      const int kb0 = ks * args.kb_per_split;
      const int kb1 = min(args.num_kb, kb0 + args.kb_per_split);
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, args.limit_ns, args.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_base + stage * STAGE_BYTES;
        const uint64_t adesc = sdesc_k_sw128(sa);
        const uint64_t bdesc = sdesc_k_sw128(sa + A_BYTES);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          // +32 bytes along K inside the 128-byte swizzled row = +2 in the
          // (address >> 4) field of the descriptor
          umma_f16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kb != kb0) || k != 0);
        }
        tc_commit(empty_bar(stage));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      tc_commit(tfull_bar(acc));
      ++local;
    }
    // drain: all MMAs issued by this thread complete before TMEM is freed
    tc_commit(drain_bar);
    mbar_wait_bounded(drain_bar, 0, nullptr, args.limit_ns, args.err);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;   // TMEM lane quadrant this warp may access
    const int row_in_tile = q * 32 + lane;
    int local = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const int t = u / args.splits, ks = u - t * args.splits;
      const Tile T = sched_tile(sched, t);
      const int e = T.e, n_tile = T.n_tile;
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      int ok = 0;
      if (lane == 0) ok = mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, args.limit_ns, args.err);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      // rows past the expert's segment (a partial last m-tile) are not stored
      const bool live = row_in_tile < T.rows;
      const size_t row = (size_t)T.row0 + row_in_tile;
      __nv_bfloat16* out_row = args.out + row * args.ldo + (size_t)n_tile * args.out_cols_per_tile;
      if (FUSE) {
        const int gcol = n_tile * 128;          // gate columns of the tile; up at + I
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(taddr + c * 32, g);
          tmem_ld_32x32b_x32(taddr + 128 + c * 32, u);
          tmem_ld_wait();
          if (live)
            epi_glu_store32(args.ep, e, gcol + c * 32, args.ldo + gcol + c * 32, g, u,
                            out_row + c * 32);
        }
      } else if (args.part != nullptr) {
        // split-K slice: raw fp32 sums of live rows, by routed item
        const int item = live ? args.part_ids[row] : args.part_R;
        float* prow = args.part + ((size_t)ks * args.part_R + (item < args.part_R ? item : 0)) *
                                      args.ldo + (size_t)n_tile * BN;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c * 32, r);
          tmem_ld_wait();
          if (item < args.part_R) {
            float4* d4 = reinterpret_cast<float4*>(prow + c * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              d4[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                  __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
          }
        }
      } else {
        const float w = live ? epi_row_weight(args.ep, row) : 0.0f;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c * 32, r);
          tmem_ld_wait();
          if (live) epi_store32(args.ep, e, n_tile * BN + c * 32, w, r, out_row + c * 32);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      ++local;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

// 2-D K-major tensor map over a [rows, k_elems] matrix with a (128-byte wide)
// x 128-row box and 128-byte swizzle.  elem_bytes is 1 (e4m3) or 2 (bf16).
bool make_tmap_k_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t k_elems,
                       int elem_bytes, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {k_elems, rows};
  const cuuint64_t strides[1] = {k_elems * (uint64_t)elem_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)(128 / elem_bytes), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D K-major tensor map over packed E2M1 values ([rows, k_elems / 2] bytes,
// low nibble first) that lands each 16 values as 8 bytes followed by an
// 8-byte gap, so a 128-value K row fills one 128-byte swizzled smem row --
// the layout the 8-bit-container f8f6f4 MMAs read for 4-bit operands.
bool make_tmap_fp4_k_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t k_elems,
                           uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {k_elems, rows};
  const cuuint64_t strides[1] = {k_elems / 2};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D tensor map over a byte matrix [rows, row_bytes] (row_bytes a multiple
// of 16) with a box of box_bytes x box_rows, no swizzle: the box lands row
// after row, box_bytes apart.
bool make_tmap_u8_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_bytes,
                       uint32_t box_bytes, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || row_bytes % 16 != 0 || box_bytes % 16 != 0) return false;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_bytes, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_ggemm_bf16(const void* A, int cap, int K, const void* B, int b_rows_total,
                              int b_rows_per_expert, int n_out, const int32_t* block_expert_ids,
                              const int32_t* num_post_padded, void* out, bool fuse_act,
                              const Epilogue& ep, cudaStream_t stream, int splits, float* part,
                              const int32_t* part_ids, int part_R, int blk_rows) {
  if (cap <= 0) return cudaSuccess;
  if (blk_rows <= 0 || blk_rows > BM || cap % blk_rows != 0) return cudaErrorInvalidValue;
  // partial mode (part != nullptr): fp32 slice sums instead of bf16 out
  if ((part != nullptr && (fuse_act || part_ids == nullptr || part_R <= 0)) ||
      (part == nullptr && (splits > 1 || out == nullptr)))
    return cudaErrorInvalidValue;
  CUtensorMap tmA, tmB;
  if (!make_tmap_k_sw128(&tmA, A, (uint64_t)cap, (uint64_t)K, 2, 128) ||
      !make_tmap_k_sw128(&tmB, B, (uint64_t)b_rows_total, (uint64_t)K, 2, 128))
    return cudaErrorInvalidValue;
  GemmArgs a;
  a.block_expert_ids = block_expert_ids;
  a.num_post_padded = num_post_padded;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.num_kb = K / BK;
  a.b_rows_per_expert = b_rows_per_expert;
  a.blocks_cap = cap / blk_rows;
  a.blk_rows = blk_rows;
  a.num_experts = b_rows_total / b_rows_per_expert;
  a.group_max = sched_group_max(K, 2);
  if (fuse_act) {
    const int I = b_rows_per_expert / 2;
    a.ldo = I;
    a.n_tiles = I / 128;
    a.second_box_off = I;        // up rows sit I rows below the gate rows
    a.n_tile_rows = 128;
    a.out_cols_per_tile = 128;
  } else {
    a.ldo = n_out;
    a.n_tiles = n_out / BN;
    a.second_box_off = 128;
    a.n_tile_rows = BN;
    a.out_cols_per_tile = BN;
  }
  watchdog_params(&a.limit_ns, &a.never_arrive);
  a.err = dev_error_word();
  if (a.err == nullptr) return cudaErrorInvalidDevice;   // no usable current device
  a.ep = ep;
  // K slices of kb_per_split steps each; the caller sizes and reads the
  // partials by `splits`, so a count that would leave a slice empty is an
  // error rather than silently reduced
  a.splits = splits > 1 ? splits : 1;
  a.kb_per_split = (a.num_kb + a.splits - 1) / a.splits;
  if ((a.num_kb + a.kb_per_split - 1) / a.kb_per_split != a.splits) return cudaErrorInvalidValue;
  a.part = part;
  a.part_ids = part_ids;
  a.part_R = part_R;
  const int grid = num_sms();
  if (fuse_act) {
    static DeviceOnce attr;
    const cudaError_t ea = attr.call([] {
      return cudaFuncSetAttribute(k_ggemm_bf16<true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    });
    if (ea != cudaSuccess) return ea;
    k_ggemm_bf16<true><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(tmA, tmB, a);
  } else {
    static DeviceOnce attr;
    const cudaError_t ea = attr.call([] {
      return cudaFuncSetAttribute(k_ggemm_bf16<false>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    });
    if (ea != cudaSuccess) return ea;
    k_ggemm_bf16<false><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(tmA, tmB, a);
  }
  return cudaGetLastError();
}

}  // namespace moe
