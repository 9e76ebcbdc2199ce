// FP8 (e4m3) grouped GEMM with fp32 block scales on SM pairs (tcgen05
// cta_group::2), stages 2 and 4 of MOE_Q_FP8_BLOCK128 at prefill sizes.
//
// Same computation as k_ggemm_fp8 (page "fused_moe.py 分析", "FP8 W8A8": one
// product of the two scales per K block; page "Blackwell 上的 DeepGEMM
// FusedMoE（vLLM）", TL;DR: 128x128 weight blocks, dynamic 1x128 activations):
//   C[r, n] = sum_kb sa[r, kb] * sb[e, n/128, kb] * sum_{k in kb} qa[r,k] qb[e,n,k],
// issued as 256 x 256 tiles over a cluster of two CTAs, as the bf16 pair
// kernel does:
//  * the pair computes two 128-row m-blocks of one expert; each CTA stages
//    its own 128 activation rows and one 128-row half of the 256-row weight
//    tile per 128-deep K block (32 KB a stage, against 48 KB in the
//    single-SM kernel for the same MMA work per SM: the TMA writes and the
//    MMA operand reads share each SM's shared-memory bandwidth);
//  * the leader's MMA thread issues four tcgen05.mma.cta_group::2
//    .kind::f8f6f4 (M=256, N=256, K=32) per K block into one of two
//    256-column fp32 partials in each CTA's tensor memory (rows 0-127 in the
//    leader's, 128-255 in the peer's), and its commits arrive on both CTAs'
//    barriers;
//  * in each CTA eight promotion warps (two per TMEM lane quadrant, one
//    per 128-column weight-scale block) read the K block's partial, release
//    it to the leader (remote mbarrier arrive; the MMA waits for all 16
//    warps of the pair), and accumulate sa * sb * partial in fp32
//    registers; at the end of the tile the sums are rounded to bf16 and
//    stored (the pages' per-K-block promotion);
//  * tiles are handed out at run time through the leader's producer and a
//    4-slot tile-index ring read by both CTAs, walking expert by expert as in
//    tile_sched.cuh; an expert with an odd block count ends with a pair
//    whose peer half repeats the leader's block and is not stored;
//  * a last column tile narrower than 256 (N % 256 == 128) computes its
//    upper half on whatever the weight box held and never stores it;
//  * every wait is bounded (device error word + CTA abort flag).
#include <atomic>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "tile_sched.cuh"

namespace moe {

bool make_tmap_k_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t k_elems,
                       int elem_bytes, uint32_t box_rows);

namespace {

constexpr int BM = 128, BN = 256, BK = 128, STAGES = 6, NPART = 2;
constexpr int A_BYTES = BM * BK;              // this CTA's activation rows (e4m3)
constexpr int B_BYTES = (BN / 2) * BK;        // this CTA's half of the weight tile
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int PAIR_TX = 2 * STAGE_BYTES;      // bytes landing per stage on the leader's barrier
constexpr int TMEM_COLS = NPART * BN;
constexpr int NUM_EPI_WARPS = 8;
constexpr int EPI_WARP0 = 4;                  // promotion warps = warpgroups 1 and 2
constexpr int NUM_THREADS = (EPI_WARP0 + NUM_EPI_WARPS) * 32;
// Register split as in k_ggemm_fp8: launched at LAUNCH_REGS a thread,
// warpgroup 0 (producer, MMA issuer, two idle warps) drops to CTRL_REGS, the
// promotion warpgroups rise to EPI_REGS (128 fp32 sums a thread).
constexpr int LAUNCH_REGS = 168, CTRL_REGS = 56, EPI_REGS = 216;
static_assert(128 * CTRL_REGS + 256 * EPI_REGS <= NUM_THREADS * LAUNCH_REGS,
              "register split exceeds the launch allocation");
static_assert(32 * (CTRL_REGS + 2 * EPI_REGS) <= 16384, "register-file partition");
constexpr int RING = 4;                       // tile-index slots
// leader MMA issuer + peer producer + the promotion warps of both CTAs
constexpr int RING_READERS = 2 + 2 * NUM_EPI_WARPS;
constexpr int SCHED_BYTES = kSchedBytes + 4 * (kSchedMaxRuns + 1);   // + pairs per segment
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256 + SCHED_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct Fp8PairArgs {
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
  int m_blocks_cap;
  int num_experts;
  uint64_t limit_ns;
  int never_arrive;
  int* err;
  int* tile_ctr;          // {next tile, CTAs finished}, zero at launch
  Epilogue ep;            // bias, router weight
};

__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_ggemm_fp8_2sm(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const Fp8PairArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // full[S], empty[S], pfull[P], pempty[P], drain, ring_full[RING], ring_empty[RING]
  uint32_t* tmem_holder =
      reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 2 * NPART + 1 + 2 * RING);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_ring = reinterpret_cast<int*>(tmem_holder + 2);   // RING tile indices
  int* s_sched = reinterpret_cast<int*>(smem + STAGES * STAGE_BYTES + 256);
  int* s_pairs = s_sched + kSchedBytes / 4;    // prefix of pairs per segment

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_u32(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto pfull_bar = [&](int b) { return bar_base + 8u * (2 * STAGES + b); };
  auto pempty_bar = [&](int b) { return bar_base + 8u * (2 * STAGES + NPART + b); };
  const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 2 * NPART);
  auto ring_full = [&](int i) { return bar_base + 8u * (2 * STAGES + 2 * NPART + 1 + i); };
  auto ring_empty = [&](int i) {
    return bar_base + 8u * (2 * STAGES + 2 * NPART + 1 + RING + i);
  };
  const uint32_t ring_base = smem_u32(s_ring);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < NPART; ++b) {
      mbar_init(pfull_bar(b), 1);
      mbar_init(pempty_bar(b), 2 * NUM_EPI_WARPS);   // both CTAs' warps (leader's is used)
    }
    mbar_init(drain_bar, 1);
    for (int i = 0; i < RING; ++i) {
      mbar_init(ring_full(i), 1);
      mbar_init(ring_empty(i), RING_READERS);        // only the leader's are waited on
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc_pair(smem_u32(tmem_holder), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();        // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  // 128-row blocks (the pair forms take no other block size)
  const int nb_valid = min(*args.num_post_padded / BM, args.m_blocks_cap);
  const TileSched sched =
      sched_build(args.block_expert_ids, nb_valid, BM, args.num_experts, s_sched,
                  reinterpret_cast<int*>(smem), args.n_tiles, 1 << 20);
  sched_pairs_build(sched, s_pairs);
  __syncthreads();
  const int total = s_pairs[sched.nruns] * args.n_tiles;

  // Tile ring: the leader's producer publishes tile j in slot j % RING (-1:
  // no tiles left); every reader takes the slots in the same order.
  auto ring_put = [&](int j, int t) -> bool {
    const int slot = j & (RING - 1);
    if (!mbar_wait_bounded<true>(ring_empty(slot), ((j / RING) & 1) ^ 1, abort_flag,
                                 args.limit_ns, args.err))
      return false;
    s_ring[slot] = t;
    st_shared_cluster(mapa_shared(ring_base + 4u * slot, 1), t);
    mbar_arrive(ring_full(slot));
    mbar_arrive_cluster(mapa_shared(ring_full(slot), 1));
    return true;
  };
  auto ring_take = [&](int j) -> int {   // -2 when the wait ran out
    const int slot = j & (RING - 1);
    if (!mbar_wait_bounded<true>(ring_full(slot), (j / RING) & 1, abort_flag, args.limit_ns,
                                 args.err))
      return -2;
    const int t = reinterpret_cast<volatile int*>(s_ring)[slot];
    mbar_arrive_cluster(mapa_shared(ring_empty(slot), 0));
    return t;
  };

  if (warp < EPI_WARP0) {
   setmaxnreg_dec<CTRL_REGS>();     // all of warpgroup 0, before its role split
   if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producers
    const uint64_t pol_a = l2_policy(MOE_GEMM_L2_A);
    const uint64_t pol_b = l2_policy(MOE_GEMM_L2_B);
    uint32_t stage = 0, phase = 0, issued_mask = 0, issued_parity = 0;
    bool skip_first = leader && args.never_arrive != 0;
    // The leader publishes tile j + 1 as it starts issuing tile j, so the
    // peer has its next index before it reaches the tile boundary.
    int t_lead = -1, pending = 0;
    bool ring_ok = true;
    if (leader) {
      const int f = atomicAdd(args.tile_ctr, 1);
      t_lead = f < total ? f : -1;
      ring_ok = ring_put(0, t_lead);
      if (t_lead >= 0) pending = atomicAdd(args.tile_ctr, 1);
    }
    for (int j = 0;; ++j) {
      int t;
      if (leader) {
        t = t_lead;
        if (!ring_ok || t < 0) break;
        t_lead = pending < total ? pending : -1;
        ring_ok = ring_put(j + 1, t_lead);
        if (t_lead >= 0) pending = atomicAdd(args.tile_ctr, 1);
      } else {
        t = ring_take(j);
        if (t < 0) break;
      }
      const PairTile P = sched_pair_tile(sched, s_pairs, t);
      const int e = P.e, n_tile = P.n_tile;
      const int my_row = leader ? P.row0 : P.row1;
      // weight rows [brow, brow + 128): the leader's half, the peer's the next 128
      const int brow = e * args.b_rows_per_expert + n_tile * BN + (leader ? 0 : BN / 2);
      bool ok = true;
      for (int kb = 0; kb < args.num_kb; ++kb) {
        if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1, abort_flag, args.limit_ns, args.err)) {
          ok = false;
          break;
        }
        if (skip_first) {
          skip_first = false;   // watchdog test: leave this stage unarmed
        } else {
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          const uint32_t bar = mapa_shared(full_bar(stage), 0);
          if (leader) {
            mbar_arrive_expect_tx(full_bar(stage), PAIR_TX);
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
          tma_load_2d_pair(sa, &tmA, bar, kb * BK, my_row, pol_a);
          tma_load_2d_pair(sa + A_BYTES, &tmB, bar, kb * BK, brow, pol_b);
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
    }
    // the leader's barrier counts both CTAs' copies: once its issued phases
    // complete, every copy of the pair has landed
    if (leader)
      for (int s = 0; s < STAGES; ++s)
        if (issued_mask & (1u << s))
          mbar_wait_bounded(full_bar(s), (issued_parity >> s) & 1, nullptr, args.limit_ns,
                            args.err);
   } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = make_idesc(kFmtE4M3, kFmtE4M3, 2 * BM, BN);
    uint32_t stage = 0, phase = 0, pc = 0;
    bool ok = true;
    for (int j = 0; ok; ++j) {
      const int t = ring_take(j);
      if (t < 0) break;
      for (int kb = 0; kb < args.num_kb; ++kb, ++pc) {
        const uint32_t buf = pc % NPART, pphase = (pc / NPART) & 1;
        if (!mbar_wait_bounded(pempty_bar(buf), pphase ^ 1, abort_flag, args.limit_ns,
                               args.err) ||
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
        for (int k = 0; k < BK / 32; ++k)
          umma_f8_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, k);
        tc_commit_pair(empty_bar(stage), 0x3);
        tc_commit_pair(pfull_bar(buf), 0x3);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    tc_commit_pair(drain_bar, 0x1);
    mbar_wait_bounded(drain_bar, 0, nullptr, args.limit_ns, args.err);
   }
  } else {
    setmaxnreg_inc<EPI_REGS>();      // all of warpgroups 1 and 2
    // ------------------------------------------------------------ promotion
    const int q = warp & 3;                       // TMEM lane quadrant
    const int half = (warp - EPI_WARP0) >> 2;     // 128-column half of the tile
    const int row_in_tile = q * 32 + lane;
    uint32_t pc = 0;
    bool ok = true;
    for (int j = 0; ok; ++j) {
      int t = 0;
      if (lane == 0) t = ring_take(j);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t < 0) break;
      const PairTile P = sched_pair_tile(sched, s_pairs, t);
      const int e = P.e, n_tile = P.n_tile;
      const bool has1 = P.has1;
      const bool store = leader || has1;          // a lone block's peer half is a repeat
      const int nblk = 2 * n_tile + half;
      const bool active = nblk < args.n_blocks;   // false: past N on a ragged last tile
      const size_t row = (size_t)(leader ? P.row0 : P.row1) + row_in_tile;
      const float* sa_row = args.a_scale + row * args.num_kb;
      const float* sb_blk =
          args.b_scale + ((size_t)e * args.n_blocks + (active ? nblk : 0)) * (size_t)args.num_kb;
      float acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
      constexpr int SCALE_AHEAD = 4;
      float ra[SCALE_AHEAD], rb[SCALE_AHEAD];
#pragma unroll
      for (int i = 0; i < SCALE_AHEAD; ++i) {
        ra[i] = i < args.num_kb ? __ldg(sa_row + i) : 0.0f;
        rb[i] = i < args.num_kb ? __ldg(sb_blk + i) : 0.0f;
      }
      for (int kb0 = 0; kb0 < args.num_kb && ok; kb0 += SCALE_AHEAD) {
#pragma unroll
        for (int i = 0; i < SCALE_AHEAD; ++i) {
          const int kb = kb0 + i;
          if (kb >= args.num_kb) break;
          const float s = ra[i] * rb[i];
          if (kb + SCALE_AHEAD < args.num_kb) {
            ra[i] = __ldg(sa_row + kb + SCALE_AHEAD);
            rb[i] = __ldg(sb_blk + kb + SCALE_AHEAD);
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
          tc_fence_after();
          const uint32_t taddr =
              tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN + half * 128;
#pragma unroll
          for (int c = 0; c < 2; ++c) {     // two rounds of four 16-column loads
            uint32_t p0[16], p1[16], p2[16], p3[16];
            const uint32_t tc = taddr + c * 64;
            tmem_ld_32x32b_x16(tc, p0);
            tmem_ld_32x32b_x16(tc + 16, p1);
            tmem_ld_32x32b_x16(tc + 32, p2);
            tmem_ld_32x32b_x16(tc + 48, p3);
            tmem_ld_wait();
            if (c == 1) {     // every read of this buffer by this warp is done
              tc_fence_before();
              __syncwarp();
              // no data passes through memory (the reads have completed into
              // registers), so no release: a cluster-scope release here put a
              // memory barrier into every K block (ncu: membar the top stall)
              if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(pempty_bar(buf), 0));
            }
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) {
              acc[c * 64 + i2] = fmaf(s, __uint_as_float(p0[i2]), acc[c * 64 + i2]);
              acc[c * 64 + 16 + i2] = fmaf(s, __uint_as_float(p1[i2]), acc[c * 64 + 16 + i2]);
              acc[c * 64 + 32 + i2] = fmaf(s, __uint_as_float(p2[i2]), acc[c * 64 + 32 + i2]);
              acc[c * 64 + 48 + i2] = fmaf(s, __uint_as_float(p3[i2]), acc[c * 64 + 48 + i2]);
            }
          }
          ++pc;
        }
      }
      if (!ok) break;
      if (store && active) {
        __nv_bfloat16* dst = args.out + row * args.ldo + (size_t)nblk * 128;
        const float w = epi_row_weight(args.ep, row);
        const bool bias = args.ep.bias != nullptr;
#pragma unroll
        for (int v = 0; v < 4; ++v) {                // 32 columns per 64-byte store
          uint32_t pk[16];
#pragma unroll
          for (int i2 = 0; i2 < 16; ++i2) {
            const int c = v * 32 + 2 * i2;
            float x0 = acc[c], x1 = acc[c + 1];
            if (bias) {
              x0 += epi_bias(args.ep, e, nblk * 128 + c);
              x1 += epi_bias(args.ep, e, nblk * 128 + c + 1);
            }
            pk[i2] = bf16x2_bits(__float2bfloat16_rn(x0 * w), __float2bfloat16_rn(x1 * w));
          }
          st_row64(dst + v * 32, pk);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) {
    // after a timeout, give copies the other CTA may still have in flight
    // into this CTA's shared memory time to land before the pair exits
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
  }
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
  if (threadIdx.x == 0) {
    // this CTA's counter updates (thread 0 is the leader's producer) are
    // done; the last CTA of the grid zeroes the counter for the next launch
    __threadfence();
    if (atomicAdd(args.tile_ctr + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(args.tile_ctr, 0);
      atomicExch(args.tile_ctr + 1, 0);
    }
  }
}

}  // namespace

cudaError_t launch_ggemm_fp8_2sm(const void* A, const float* a_scale, int cap, int K,
                                 const void* B, const float* b_scale, int b_rows_total,
                                 int b_rows_per_expert, int n_out,
                                 const int32_t* block_expert_ids,
                                 const int32_t* num_post_padded, void* out, const Epilogue& ep,
                                 cudaStream_t stream, int* tile_ctr) {
  if (cap <= 0) return cudaSuccess;
  if (n_out != b_rows_per_expert || n_out % 128 != 0) return cudaErrorInvalidValue;
  CUtensorMap tmA, tmB;
  if (!make_tmap_k_sw128(&tmA, A, (uint64_t)cap, (uint64_t)K, 1, BM) ||
      !make_tmap_k_sw128(&tmB, B, (uint64_t)b_rows_total, (uint64_t)K, 1, BN / 2))
    return cudaErrorInvalidValue;
  Fp8PairArgs a;
  a.block_expert_ids = block_expert_ids;
  a.num_post_padded = num_post_padded;
  a.a_scale = a_scale;
  a.b_scale = b_scale;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ldo = n_out;
  a.num_kb = K / BK;
  a.n_tiles = (n_out + BN - 1) / BN;
  a.n_blocks = n_out / 128;
  a.b_rows_per_expert = b_rows_per_expert;
  a.m_blocks_cap = cap / BM;
  a.num_experts = b_rows_total / b_rows_per_expert;
  watchdog_params(&a.limit_ns, &a.never_arrive);
  a.err = dev_error_word();
  if (a.err == nullptr) return cudaErrorInvalidDevice;   // no usable current device
  a.ep = ep;
  a.tile_ctr = tile_ctr != nullptr ? tile_ctr : next_tile_counter();
  if (a.tile_ctr == nullptr) return cudaErrorInvalidDevice;

  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  static DeviceOnce setup;
  static int max_pairs[kMaxDevices];
  const int dev = device_index();
  const cudaError_t es = setup.call([&] {
    cudaError_t e = cudaFuncSetAttribute(k_ggemm_fp8_2sm,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // the register split is only safe at exactly LAUNCH_REGS a thread
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, k_ggemm_fp8_2sm);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != LAUNCH_REGS) return cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3(num_sms(), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, k_ggemm_fp8_2sm, &cfg);
    if (e != cudaSuccess) return e;
    max_pairs[dev] = n;
    return cudaSuccess;
  });
  if (es != cudaSuccess) return es;
  if (max_pairs[dev] <= 0) return cudaErrorInvalidConfiguration;
  // one wave of persistent pairs (as many as fit on the GPU at once)
  cfg.gridDim = dim3(2 * max_pairs[dev], 1, 1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, k_ggemm_fp8_2sm, tmA, tmB, a);
}

}  // namespace moe
