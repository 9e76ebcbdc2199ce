// bf16 grouped GEMM on SM pairs (tcgen05 cta_group::2), stages 2 and 4.
//
// Same computation as k_ggemm_bf16 (page "fused_moe.py 分析", §1.3 and
// "fused_moe_kernel 的核心原理"; page "Blackwell 上的 DeepGEMM FusedMoE（vLLM）",
// §2.6.3), issued as 256 x 256 tiles over a cluster of two CTAs:
//  * the pair computes two 128-row m-blocks of the same expert; each CTA
//    loads its own 128 activation rows and one half (128 rows) of the
//    256-row weight tile -- GEMM1: the gate rows in the leader, the matching
//    up rows in the peer -- so a CTA takes in 32 KB per K step instead of
//    48 KB for the same MMA work per SM; the tensor core reads the other
//    half of the weights from the peer SM.  (The single-CTA kernel was fed
//    too slowly: with four 48 KB stages it ran ~18% slower on three.)
//  * a 6-stage ring per CTA; the peer's copies complete on the leader's
//    barrier (cp.async.bulk.tensor ... .cta_group::2), the leader's MMA thread
//    issues tcgen05.mma.cta_group::2 (M=256, N=256, K=16) into the pair's
//    accumulator (rows 0-127 in the leader's TMEM, 128-255 in the peer's), and
//    its tcgen05.commit multicasts to both CTAs' barriers;
//  * each CTA's epilogue (warps 2-5) drains its own TMEM rows; the peer's
//    warps arrive on the leader's accumulator-empty barrier;
//  * tiles walk expert by expert, n-tile major, so the pairs working at the
//    same time share weight tiles in L2; an expert with an odd number of
//    blocks ends with a pair whose peer half repeats the leader's block and
//    is not stored.
//  * tiles are handed out at run time: the leader's producer takes the next
//    tile index from a global counter and publishes it through a 4-slot ring
//    to its own MMA and epilogue warps and to the peer's producer and
//    epilogue (remote store + remote mbarrier arrive); a slot is rewritten
//    only after all ten readers have released it.  A statically strided
//    order let the pairs drift apart by several tiles, so that pairs meant to
//    share a weight tile read it from DRAM at different times.  The counter
//    is the caller's (two ints in the fused_experts workspace, zeroed on its
//    stream before the launch) or, for the stage entry points, one of a
//    library-owned ring of slots, one per launch in flight; the last CTA to
//    finish resets it.
//  * every wait is bounded; the final cluster barrier is reached by both CTAs
//    after their bounded loops.
#include <atomic>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "tile_sched.cuh"

namespace moe {

bool make_tmap_k_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t k_elems,
                       int elem_bytes, uint32_t box_rows);

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;          // this CTA's activation rows
constexpr int B_BYTES = (BN / 2) * BK * 2;    // this CTA's half of the weight tile
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int PAIR_TX = 2 * STAGE_BYTES;      // bytes landing per stage on the leader's barrier
constexpr int TMEM_COLS = 2 * BN;
constexpr int NUM_THREADS = 192;
constexpr int SCHED_BYTES = kSchedBytes + 4 * (kSchedMaxRuns + 1);   // + pairs per segment
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256 + SCHED_BYTES;
constexpr int RING = 4;                       // tile-index slots
constexpr int RING_READERS = 10;              // leader MMA + 4 epilogue warps, peer producer + 4
constexpr int CTR_SLOTS = 64;                 // tile counters: launches that may be in flight

// {next tile, CTAs finished} per counter slot; zero between launches.
__device__ int g_pair_tile_ctr[CTR_SLOTS * 2];

struct Pair2Args {
  const int32_t* block_expert_ids;
  const int32_t* num_post_padded;
  __nv_bfloat16* out;
  int ldo;
  int num_kb;
  int n_tiles;
  int b_rows_per_expert;
  int second_box_off;     // row offset of the peer's weight half
  int n_tile_rows;
  int out_cols_per_tile;
  int m_blocks_cap;
  int num_experts;
  uint64_t limit_ns;
  int never_arrive;
  int* err;
  int* tile_ctr;          // {next tile, CTAs finished}, zero at launch
  Epilogue ep;            // bias, router weight, activation recipe
};

template <bool FUSE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_ggemm_bf16_2sm(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const Pair2Args args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // full[S], empty[S], tfull[2], tempty[2], drain, ring_full[RING], ring_empty[RING]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5 + 2 * RING);
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
  auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 4);
  auto ring_full = [&](int i) { return bar_base + 8u * (2 * STAGES + 5 + i); };
  auto ring_empty = [&](int i) { return bar_base + 8u * (2 * STAGES + 5 + RING + i); };
  const uint32_t ring_base = smem_u32(s_ring);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 8);     // 4 epilogue warps in each CTA (leader's is used)
    }
    mbar_init(drain_bar, 1);
    for (int i = 0; i < RING; ++i) {
      mbar_init(ring_full(i), 1);
      mbar_init(ring_empty(i), RING_READERS);   // only the leader's are waited on
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

  // Tile ring.  The leader's producer publishes tile j in slot j % RING
  // (-1: no tiles left); every reader takes the slots in the same order.
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

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producers
    const uint64_t pol_a = l2_policy(MOE_GEMM_L2_A);
    const uint64_t pol_b = l2_policy(MOE_GEMM_L2_B);
    uint32_t stage = 0, phase = 0, issued_mask = 0, issued_parity = 0;
    bool skip_first = leader && args.never_arrive != 0;
    // The leader publishes tile j + 1 as it starts issuing tile j, so the
    // peer has its next index before it reaches the tile boundary; the
    // counter read for tile j + 2 is in flight meanwhile.
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
      const int brow = e * args.b_rows_per_expert + n_tile * args.n_tile_rows +
                       (leader ? 0 : args.second_box_off);
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
    constexpr uint32_t idesc = make_idesc(kFmtBF16, kFmtBF16, 2 * BM, BN);
    uint32_t stage = 0, phase = 0;
    int local = 0;
    for (int j = 0;; ++j) {
      const int t = ring_take(j);
      if (t < 0) break;
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1, abort_flag, args.limit_ns, args.err))
        break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      bool ok = true;
      for (int kb = 0; kb < args.num_kb; ++kb) {
        if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, args.limit_ns, args.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_base + stage * STAGE_BYTES;
        const uint64_t adesc = sdesc_k_sw128(sa);
        const uint64_t bdesc = sdesc_k_sw128(sa + A_BYTES);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          umma_f16_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0);
        tc_commit_pair(empty_bar(stage), 0x3);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      tc_commit_pair(tfull_bar(acc), 0x3);
      ++local;
    }
    tc_commit_pair(drain_bar, 0x1);
    mbar_wait_bounded(drain_bar, 0, nullptr, args.limit_ns, args.err);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int row_in_tile = q * 32 + lane;
    int local = 0;
    for (int j = 0;; ++j) {
      int t = 0;
      if (lane == 0) t = ring_take(j);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t < 0) break;
      const PairTile P = sched_pair_tile(sched, s_pairs, t);
      const int e = P.e, n_tile = P.n_tile;
      const bool has1 = P.has1;
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      int ok = 0;
      if (lane == 0)
        ok = mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, args.limit_ns, args.err);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const bool store = leader || has1;      // a lone block's peer half is a repeat
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      const size_t row = (size_t)(leader ? P.row0 : P.row1) + row_in_tile;
      __nv_bfloat16* out_row = args.out + row * args.ldo + (size_t)n_tile * args.out_cols_per_tile;
      if (FUSE) {
        const int gcol = n_tile * 128;          // gate columns of the tile; up at + I
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(taddr + c * 32, g);
          tmem_ld_32x32b_x32(taddr + 128 + c * 32, u);
          tmem_ld_wait();
          if (!store) continue;
          epi_glu_store32(args.ep, e, gcol + c * 32, args.ldo + gcol + c * 32, g, u,
                          out_row + c * 32);
        }
      } else {
        const float w = store ? epi_row_weight(args.ep, row) : 0.0f;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c * 32, r);
          tmem_ld_wait();
          if (!store) continue;
          epi_store32(args.ep, e, n_tile * BN + c * 32, w, r, out_row + c * 32);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
      ++local;
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

template <bool FUSE>
cudaError_t launch_pairs(const CUtensorMap& tmA, const CUtensorMap& tmB, const Pair2Args& a,
                         cudaStream_t stream) {
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
    cudaError_t e = cudaFuncSetAttribute(k_ggemm_bf16_2sm<FUSE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(num_sms(), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, k_ggemm_bf16_2sm<FUSE>, &cfg);
    if (e != cudaSuccess) return e;
    max_pairs[dev] = n;
    return cudaSuccess;
  });
  if (es != cudaSuccess) return es;
  if (max_pairs[dev] <= 0) return cudaErrorInvalidConfiguration;
  // one wave of persistent pairs (as many as fit on the GPU at once)
  cfg.gridDim = dim3(2 * max_pairs[dev], 1, 1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, k_ggemm_bf16_2sm<FUSE>, tmA, tmB, a);
}

}  // namespace

// A tile counter for the next launch that brings none of its own (the stage
// entry points): slots of a library-owned ring rotate, so launches in flight
// at the same time (other streams) use different counters as long as fewer
// than CTR_SLOTS of them overlap.  The device address of the ring is looked
// up once per device under a lock.
int* next_tile_counter() {
  static DeviceOnce once;
  static int* base[kMaxDevices] = {};
  static std::atomic<unsigned> seq{0};
  const int dev = device_index();
  const cudaError_t e = once.call([&] {
    void* p = nullptr;
    const cudaError_t r = cudaGetSymbolAddress(&p, g_pair_tile_ctr);
    if (r == cudaSuccess) base[dev] = static_cast<int*>(p);
    return r;
  });
  if (e != cudaSuccess || dev < 0) return nullptr;
  return base[dev] + 2 * (seq.fetch_add(1) % CTR_SLOTS);
}

cudaError_t launch_ggemm_bf16_2sm(const void* A, int cap, int K, const void* B, int b_rows_total,
                                  int b_rows_per_expert, int n_out,
                                  const int32_t* block_expert_ids,
                                  const int32_t* num_post_padded, void* out, bool fuse_act,
                                  const Epilogue& ep, cudaStream_t stream, int* tile_ctr) {
  if (cap <= 0) return cudaSuccess;
  CUtensorMap tmA, tmB;
  if (!make_tmap_k_sw128(&tmA, A, (uint64_t)cap, (uint64_t)K, 2, 128) ||
      !make_tmap_k_sw128(&tmB, B, (uint64_t)b_rows_total, (uint64_t)K, 2, 128))
    return cudaErrorInvalidValue;
  Pair2Args a;
  a.block_expert_ids = block_expert_ids;
  a.num_post_padded = num_post_padded;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.num_kb = K / BK;
  a.b_rows_per_expert = b_rows_per_expert;
  a.m_blocks_cap = cap / BM;
  a.num_experts = b_rows_total / b_rows_per_expert;
  if (fuse_act) {
    const int I = b_rows_per_expert / 2;
    a.ldo = I;
    a.n_tiles = I / 128;
    a.second_box_off = I;        // the peer loads the up rows matching the leader's gate rows
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
  a.tile_ctr = tile_ctr != nullptr ? tile_ctr : next_tile_counter();
  if (a.tile_ctr == nullptr) return cudaErrorInvalidDevice;
  return fuse_act ? launch_pairs<true>(tmA, tmB, a, stream)
                  : launch_pairs<false>(tmA, tmB, a, stream);
}

}  // namespace moe
