// FP8 (e4m3) grouped GEMM with fp32 block scales (stages 2 and 4 of
// MOE_Q_FP8_BLOCK128).
//
// What it computes: page "fused_moe.py 分析", "FP8 W8A8": block-wise scales are
// read per K block and C_block = dot(qA_block, qB_block) * a_scale * b_scale,
// accumulated over K blocks; here activation scales are per (row, 128-column
// group) and weight scales per 128x128 block (page "Blackwell 上的 DeepGEMM
// FusedMoE（vLLM）", TL;DR: "FP8 block 128x128", dynamic 128 activations):
//   C[r, n] = sum_kb sa[r, kb] * sb[e, n/128, kb] * sum_{k in kb} qa[r,k] qb[e,n,k].
//
// The hardware block-scaled MMA takes power-of-two (UE8M0) scales only, and
// these scales are arbitrary fp32, so the scales are applied on the CUDA
// cores ("promotion"):
//  * warp 0 lane 0: TMA producer, 4-stage ring of (A 128x128, B 256x128) e4m3
//    tiles -- one stage is exactly one 128-wide K block;
//  * warp 1 lane 0: four kind::f8f6f4 MMAs (M=128, N=256, K=32) per K block
//    into one of two 256-column tensor-memory partials, alternating, and one
//    tcgen05.commit (partial full).  (128x128 MMAs ran at about half the
//    tensor rate on GB300; N=256 keeps the pipe fed.)
//  * warps 4-11 (warpgroups 1 and 2): warp w owns TMEM lane quadrant w%4 (32
//    rows) and one 128-column half of the tile -- exactly one 128x128
//    weight-scale block, so one scale product sa[row,kb]*sb[kb] per thread
//    and K block; it reads the partial with tcgen05.ld (four 16-column loads
//    per wait), releases it, and accumulates in fp32 registers (the first of
//    these warps also returns the K block's operand stage to the producer
//    once the partial is complete); at the end of
//    the tile the sum is rounded to bf16 and stored.  The 128 accumulators a
//    thread holds need the register split below (setmaxnreg): warpgroup 0
//    (producer, MMA issuer, two idle warps) gives registers up.
//  * a last column tile narrower than 256 (N % 256 == 128) computes its upper
//    half on whatever the weight box held and never stores it.
//  * tiles are walked expert by expert (tile_sched.cuh), so each weight tile
//    is fetched once for all of the expert's m-blocks and the expert's
//    activations stay in L2.
//  * every wait is bounded, as in the bf16 kernel.
#include <mutex>

#include "e4m3_pack.cuh"
#include "moe_common.cuh"
#include "moe_internal.h"
#include "tile_sched.cuh"

namespace moe {

bool make_tmap_k_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t k_elems,
                       int elem_bytes, uint32_t box_rows);

namespace {

constexpr int BM = 128, BN = 256, BK = 128, STAGES = 4, NPART = 2;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = NPART * BN;
constexpr int NUM_EPI_WARPS = 8;
constexpr int EPI_WARP0 = 4;                      // epilogue = warpgroups 1 and 2
constexpr int NUM_THREADS = (EPI_WARP0 + NUM_EPI_WARPS) * 32;
// Register split (setmaxnreg): launched at LAUNCH_REGS a thread (3 warps on
// each register-file partition -> at most 168); warpgroup 0 (producer, MMA
// issuer, two idle warps) drops to CTRL_REGS, the epilogue warpgroups rise to
// EPI_REGS.  The increases can only be met if the sum fits the launch pool.
constexpr int LAUNCH_REGS = 168, CTRL_REGS = 56, EPI_REGS = 216;
static_assert(128 * CTRL_REGS + 256 * EPI_REGS <= NUM_THREADS * LAUNCH_REGS,
              "register split exceeds the launch allocation");
static_assert(32 * (CTRL_REGS + 2 * EPI_REGS) <= 16384, "register-file partition");
constexpr int AMAX_BYTES = 2 * 2 * BM * 4;      // fused epilogue: [tile parity][half][row]
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256 + kSchedBytes + AMAX_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct Fp8Args {
  const int32_t* block_expert_ids;
  const int32_t* num_post_padded;
  const float* a_scale;   // [cap, K/128]
  const float* b_scale;   // [E, N/128, K/128]
  __nv_bfloat16* out;     // [cap, N]
  int ldo;                // N
  int num_kb;             // K / 128
  int n_tiles;            // ceil(N / 256)
  int n_blocks;           // N / 128 (weight-scale blocks per expert)
  int b_rows_per_expert;  // N
  int blocks_cap;         // blocks of blk_rows rows the buffers hold
  int blk_rows;           // rows per block of the padded layout
  int num_experts;
  int group_max;          // m-tiles per scheduling group (L2 budget)
  uint64_t limit_ns;
  int never_arrive;
  int* err;
  Epilogue ep;            // bias, router weight, gated activation recipe
  // fused GEMM1 epilogue (FUSE): z codes [cap, I] e4m3, scales [cap, I/128]
  uint8_t* zq;
  float* zs;
  int I;
  int ue8m0;
};

template <bool FUSE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_ggemm_fp8(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const Fp8Args args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // full[S], empty[S], pfull[P], pempty[P], drain, amax exchange[4]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 2 * NPART + 1 + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_sched = reinterpret_cast<int*>(smem + STAGES * STAGE_BYTES + 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_u32(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto pfull_bar = [&](int b) { return bar_base + 8u * (2 * STAGES + b); };
  auto pempty_bar = [&](int b) { return bar_base + 8u * (2 * STAGES + NPART + b); };
  const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 2 * NPART);
  auto amax_bar = [&](int q) { return bar_base + 8u * (2 * STAGES + 2 * NPART + 1 + q); };
  float* s_amax = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 256 + kSchedBytes);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < NPART; ++b) {
      mbar_init(pfull_bar(b), 1);
      mbar_init(pempty_bar(b), NUM_EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    for (int qq = 0; qq < 4; ++qq) mbar_init(amax_bar(qq), 2);   // the two halves' lane 0
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

  const int nb_valid = min(*args.num_post_padded / args.blk_rows, args.blocks_cap);
  const TileSched sched =
      sched_build(args.block_expert_ids, nb_valid, args.blk_rows, args.num_experts, s_sched,
                  reinterpret_cast<int*>(smem), args.n_tiles, args.group_max);
  const int total = sched_mtiles(sched) * args.n_tiles;

  if (warp < EPI_WARP0) {
   setmaxnreg_dec<CTRL_REGS>();     // all of warpgroup 0, before its role split
   if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_a = l2_policy(MOE_GEMM_L2_A);
    const uint64_t pol_b = l2_policy(MOE_GEMM_L2_B);
    uint32_t stage = 0, phase = 0, issued_mask = 0, issued_parity = 0;
    bool skip_first = args.never_arrive != 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile T = sched_tile(sched, t);
      const int e = T.e, n_tile = T.n_tile;
      // B tile: 256 consecutive weight rows, or (FUSE) gate rows
      // [128 j, 128 j + 128) and the matching up rows I + 128 j ...
      const int brow = FUSE ? e * args.b_rows_per_expert + n_tile * 128
                            : e * args.b_rows_per_expert + n_tile * BN;
      const int brow2 = FUSE ? brow + args.I : brow + 128;
      bool ok = true;
      for (int kb = 0; kb < args.num_kb; ++kb) {
        if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1, abort_flag, args.limit_ns, args.err)) {
          ok = false;
          break;
        }
        if (skip_first) {
          skip_first = false;
        } else {
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          mbar_arrive_expect_tx(full_bar(stage), STAGE_BYTES);
          tma_load_2d(sa, &tmA, full_bar(stage), kb * BK, T.row0, pol_a);
          tma_load_2d(sa + A_BYTES, &tmB, full_bar(stage), kb * BK, brow, pol_b);
          tma_load_2d(sa + A_BYTES + 128 * BK, &tmB, full_bar(stage), kb * BK, brow2, pol_b);
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
    for (int s = 0; s < STAGES; ++s)
      if (issued_mask & (1u << s))
        mbar_wait_bounded(full_bar(s), (issued_parity >> s) & 1, nullptr, args.limit_ns, args.err);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = make_idesc(kFmtE4M3, kFmtE4M3, BM, BN);
    uint32_t stage = 0, phase = 0, pc = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      for (int kb = 0; kb < args.num_kb; ++kb, ++pc) {
        const uint32_t buf = pc % NPART, pphase = (pc / NPART) & 1;
        if (!mbar_wait_bounded(pempty_bar(buf), pphase ^ 1, abort_flag, args.limit_ns, args.err) ||
            !mbar_wait_bounded(full_bar(stage), phase, abort_flag, args.limit_ns, args.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_base + stage * STAGE_BYTES;
        const uint64_t adesc = sdesc_k_sw128(sa);
        const uint64_t bdesc = sdesc_k_sw128(sa + A_BYTES);
        const uint32_t d_tmem = tmem_base + buf * BN;
#pragma unroll
        for (int k = 0; k < BK / 32; ++k) umma_f8(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, k);
        tc_commit(pfull_bar(buf));     // also frees the stage: see the epilogue
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    tc_commit(drain_bar);
    mbar_wait_bounded(drain_bar, 0, nullptr, args.limit_ns, args.err);
   }
  } else {
    setmaxnreg_inc<EPI_REGS>();      // all of warpgroups 1 and 2
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;               // TMEM lane quadrant
    const int half = (warp - EPI_WARP0) >> 2;   // 128-column half of the tile
    const int row_in_tile = q * 32 + lane;
    uint32_t pc = 0, xpar = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile T = sched_tile(sched, t);
      const int e = T.e, n_tile = T.n_tile;
      // weight-scale block of this warp's columns (FUSE: its 64 gate columns
      // lie in block n_tile, the matching up columns in block I/128 + n_tile)
      const int nblk = FUSE ? n_tile : 2 * n_tile + half;
      const bool active = FUSE || nblk < args.n_blocks;   // false: past N on a ragged last tile
      // rows past the expert's segment (a partial last m-tile) are computed
      // on other rows' data and not stored; their scales are read from the
      // tile's first row, inside the buffers
      const bool live = row_in_tile < T.rows;
      const size_t row = (size_t)T.row0 + row_in_tile;
      const float* sa_row = args.a_scale + (live ? row : (size_t)T.row0) * args.num_kb;
      const float* sb_blk =
          args.b_scale + ((size_t)e * args.n_blocks + (active ? nblk : 0)) * (size_t)args.num_kb;
      const float* sb_up =
          FUSE ? sb_blk + (size_t)(args.I / 128) * args.num_kb : sb_blk;
      float acc[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
      constexpr int SCALE_AHEAD = FUSE ? 2 : 4;   // FUSE holds two weight-scale streams
      float ra[SCALE_AHEAD], rb[SCALE_AHEAD], ru[SCALE_AHEAD];
#pragma unroll
      for (int j = 0; j < SCALE_AHEAD; ++j) {
        ra[j] = j < args.num_kb ? __ldg(sa_row + j) : 0.0f;
        rb[j] = j < args.num_kb ? __ldg(sb_blk + j) : 0.0f;
        ru[j] = FUSE && j < args.num_kb ? __ldg(sb_up + j) : 0.0f;
      }
      for (int kb0 = 0; kb0 < args.num_kb && ok; kb0 += SCALE_AHEAD) {
#pragma unroll
        for (int j = 0; j < SCALE_AHEAD; ++j) {
          const int kb = kb0 + j;
          if (kb >= args.num_kb) break;
          const float s = ra[j] * rb[j];
          const float su = FUSE ? ra[j] * ru[j] : s;       // up columns' scale product
          if (kb + SCALE_AHEAD < args.num_kb) {
            ra[j] = __ldg(sa_row + kb + SCALE_AHEAD);
            rb[j] = __ldg(sb_blk + kb + SCALE_AHEAD);
            if (FUSE) ru[j] = __ldg(sb_up + kb + SCALE_AHEAD);
          }
          const uint32_t buf = pc % NPART, pphase = (pc / NPART) & 1;
          int got = 0;
          if (lane == 0)
            got = mbar_wait_bounded(pfull_bar(buf), pphase, abort_flag, args.limit_ns, args.err);
          got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) {
            ok = false;
            break;
          }
          // The K block's MMAs have completed, so they are done reading its
          // operand stage (one stage per K block, in the same order): hand
          // it back to the producer from here rather than with a second
          // tcgen05.commit per K block (that commit cost ~45 cycles of
          // the tensor pipe's 512 a K block).
          if (warp == EPI_WARP0 && lane == 0) mbar_arrive(empty_bar(pc % STAGES));
          tc_fence_after();
          // FUSE: columns [64 half, +64) of the gate half, then of the up half
          const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN +
                                 (FUSE ? half * 64 : half * 128);
#pragma unroll
          for (int c = 0; c < 2; ++c) {     // two rounds of four 16-column loads
            uint32_t p0[16], p1[16], p2[16], p3[16];
            const uint32_t tc = taddr + (FUSE ? c * 128 : c * 64);
            const float sc = c == 0 ? s : su;
            tmem_ld_32x32b_x16(tc, p0);
            tmem_ld_32x32b_x16(tc + 16, p1);
            tmem_ld_32x32b_x16(tc + 32, p2);
            tmem_ld_32x32b_x16(tc + 48, p3);
            tmem_ld_wait();
            if (c == 1) {     // every read of this buffer by this warp is done
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(pempty_bar(buf));
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              acc[c * 64 + i] = fmaf(sc, __uint_as_float(p0[i]), acc[c * 64 + i]);
              acc[c * 64 + 16 + i] = fmaf(sc, __uint_as_float(p1[i]), acc[c * 64 + 16 + i]);
              acc[c * 64 + 32 + i] = fmaf(sc, __uint_as_float(p2[i]), acc[c * 64 + 32 + i]);
              acc[c * 64 + 48 + i] = fmaf(sc, __uint_as_float(p3[i]), acc[c * 64 + 48 + i]);
            }
          }
          ++pc;
        }
      }
      if (!ok) break;
      if (FUSE) {
        // acc[0, 64): gate sums, acc[64, 128): up sums of columns 64 half ..
        // of n-block n_tile.  z = act(bf16 g, bf16 u) in fp32 as act_mul_quant
        // computes it from a stored H1; the 1x128 group's amax is combined
        // with the other half's warp through shared memory.
        const int gcol0 = n_tile * 128 + half * 64, ucol0 = args.I + gcol0;
        const bool bias = args.ep.bias != nullptr;
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          float gs = acc[j], us = acc[64 + j];
          if (bias) {
            gs += epi_bias(args.ep, e, gcol0 + j);
            us += epi_bias(args.ep, e, ucol0 + j);
          }
          acc[j] = act_glu(args.ep, bf16_round(gs), bf16_round(us));
          amax = fmaxf(amax, fabsf(acc[j]));
        }
        const uint32_t par = xpar & 1;
        float* sx = s_amax + (par * 2) * BM;
        sx[half * BM + row_in_tile] = amax;
        __syncwarp();
        int got = 1;
        if (lane == 0) {
          mbar_arrive(amax_bar(q));
          got = mbar_wait_bounded(amax_bar(q), par, abort_flag, args.limit_ns, args.err);
        }
        got = __shfl_sync(0xffffffffu, got, 0);
        __syncwarp();                                 // lane 0's acquire covers the warp
        ++xpar;
        if (!got) {
          ok = false;
          break;
        }
        amax = fmaxf(sx[row_in_tile], sx[BM + row_in_tile]);
        const float sc = act_scale(amax, args.ue8m0 != 0);
        const float rc = __frcp_rn(sc);
        uint4* zdst = reinterpret_cast<uint4*>(args.zq + row * (size_t)args.I + (size_t)gcol0);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint32_t wd[4];
#pragma unroll
          for (int qd = 0; qd < 4; ++qd) {
            uint32_t word = 0;
#pragma unroll
            for (int bb = 0; bb < 4; ++bb)
              word |= (uint32_t)f32_to_e4m3(quot_rn(acc[16 * v + 4 * qd + bb], sc, rc))
                      << (8 * bb);
            wd[qd] = word;
          }
          if (live) zdst[v] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        }
        if (half == 0 && live) args.zs[row * (size_t)(args.I / 128) + n_tile] = sc;
      } else if (active && live) {
        __nv_bfloat16* dst = args.out + row * args.ldo + (size_t)nblk * 128;
        const float w = epi_row_weight(args.ep, row);
        const bool bias = args.ep.bias != nullptr;
#pragma unroll
        for (int v = 0; v < 4; ++v) {                // 32 columns per 64-byte store
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int c = v * 32 + 2 * j;
            float x0 = acc[c], x1 = acc[c + 1];
            if (bias) {
              x0 += epi_bias(args.ep, e, nblk * 128 + c);
              x1 += epi_bias(args.ep, e, nblk * 128 + c + 1);
            }
            pk[j] = bf16x2_bits(__float2bfloat16_rn(x0 * w), __float2bfloat16_rn(x1 * w));
          }
          st_row64(dst + v * 32, pk);
        }
      }
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

}  // namespace

namespace {
template <bool FUSE>
cudaError_t launch_fp8_form(const CUtensorMap& tmA, const CUtensorMap& tmB, const Fp8Args& a,
                            cudaStream_t stream) {
  static DeviceOnce setup;
  const cudaError_t es = setup.call([] {
    cudaError_t e = cudaFuncSetAttribute(k_ggemm_fp8<FUSE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // the register split above is only safe at exactly LAUNCH_REGS a thread
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, k_ggemm_fp8<FUSE>);
    if (e != cudaSuccess) return e;
    return fa.numRegs == LAUNCH_REGS ? cudaSuccess : cudaErrorInvalidConfiguration;
  });
  if (es != cudaSuccess) return es;
  k_ggemm_fp8<FUSE><<<num_sms(), NUM_THREADS, SMEM_BYTES, stream>>>(tmA, tmB, a);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_ggemm_fp8(const void* A, const float* a_scale, int cap, int K, const void* B,
                             const float* b_scale, int b_rows_total, int b_rows_per_expert,
                             int n_out, const int32_t* block_expert_ids,
                             const int32_t* num_post_padded, void* out, const Epilogue& ep,
                             cudaStream_t stream, float* z_scale, bool fuse_act, bool ue8m0,
                             int blk_rows) {
  if (cap <= 0) return cudaSuccess;
  if (blk_rows <= 0 || blk_rows > BM || cap % blk_rows != 0) return cudaErrorInvalidValue;
  // fused GEMM1: B rows per expert = 2I (gate then up), I a multiple of 128
  if (fuse_act && (z_scale == nullptr || b_rows_per_expert % 256 != 0 ||
                   n_out != b_rows_per_expert))
    return cudaErrorInvalidValue;
  CUtensorMap tmA, tmB;
  if (!make_tmap_k_sw128(&tmA, A, (uint64_t)cap, (uint64_t)K, 1, 128) ||
      !make_tmap_k_sw128(&tmB, B, (uint64_t)b_rows_total, (uint64_t)K, 1, 128))
    return cudaErrorInvalidValue;
  Fp8Args a;
  a.ep = ep;
  a.block_expert_ids = block_expert_ids;
  a.num_post_padded = num_post_padded;
  a.a_scale = a_scale;
  a.b_scale = b_scale;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ldo = n_out;
  a.num_kb = K / BK;
  a.n_blocks = n_out / 128;
  a.I = b_rows_per_expert / 2;
  // fused: one tile per 128-column block of z (gate rows j + up rows I + j)
  a.n_tiles = fuse_act ? a.I / 128 : (n_out + BN - 1) / BN;
  a.zq = fuse_act ? static_cast<uint8_t*>(out) : nullptr;
  a.zs = z_scale;
  a.ue8m0 = ue8m0 ? 1 : 0;
  a.b_rows_per_expert = b_rows_per_expert;
  a.blocks_cap = cap / blk_rows;
  a.blk_rows = blk_rows;
  a.num_experts = b_rows_total / b_rows_per_expert;
  a.group_max = sched_group_max(K, 1);
  watchdog_params(&a.limit_ns, &a.never_arrive);
  a.err = dev_error_word();
  if (a.err == nullptr) return cudaErrorInvalidDevice;   // no usable current device
  return fuse_act ? launch_fp8_form<true>(tmA, tmB, a, stream)
                  : launch_fp8_form<false>(tmA, tmB, a, stream);
}

}  // namespace moe
