// Block-scaled (E8M0 per 32) grouped GEMM on SM pairs (tcgen05 cta_group::2):
// MXFP4 W4A8 and MXFP8 1x32, stages 2 and 4, with prepacked weight scales
// (moe_prepack_weights) and 128-row blocks.
//
// Same computation as k_ggemm_mxfp4 (page "Blackwell 上的 DeepGEMM FusedMoE
// （vLLM）", TL;DR table, W4A8 MXFP4 and MXFP8 1x32 rows):
//   C[r, n] = sum_k (qa[r,k] * sa[r, k/g]) * (qb[e,n,k] * 2^(sb[e,n,k/32]-127)),
// issued as 256 x 256 tiles over a cluster of two CTAs, as the bf16 pair
// kernel does:
//  * the pair computes two 128-row m-tiles of one expert; each CTA stages its
//    own 128 activation rows and one 128-row half of the weight tile per
//    128-deep K block (GEMM1 with the activation: the leader the gate rows,
//    the peer the matching up rows), 32 KB a stage instead of 48 KB in the
//    single-SM kernel for the same MMA work per SM;
//  * block-scale operands: each CTA's ring slot holds the activation-scale
//    operand of its own 128 rows and the weight-scale operand of all 256
//    weight rows of the tile (copied from the prepacked scales); the leader's
//    scale writers fill both CTAs' slots; the leader's MMA thread copies the slots into
//    tensor memory with tcgen05.cp.cta_group::2 -- each CTA's slot into its
//    own tensor memory -- and issues tcgen05.mma.cta_group::2
//    .kind::mxf8f6f4.block_scale (M=256, N=256, K=32); each CTA's half of the
//    MMA reads its rows' scales and the full weight-scale operand from its own
//    tensor memory (found by a probe of the two placements: with only each
//    CTA's half of the weight scales, the columns of the other half came out
//    with the wrong scales);
//  * the peer's slot is written with shared::cluster stores and a proxy fence,
//    so no signal per K block crosses the pair;
//  * each CTA's four epilogue warps drain its 128 rows of the accumulator
//    (mx_row_epilogue: the fused activation + quantisation, or bf16 stores)
//    and release it to the leader;
//  * tiles are handed out at run time (a tile counter and a 4-slot ring, as
//    in the other pair kernels); an expert with an odd block count ends with a
//    pair whose peer half repeats the leader's block and is not stored;
//  * every wait is bounded.
#include <atomic>
#include <type_traits>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "mx_common.cuh"
#include "tile_sched.cuh"

namespace moe {

bool make_tmap_k_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t k_elems,
                       int elem_bytes, uint32_t box_rows);
bool make_tmap_fp4_k_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t k_elems,
                           uint32_t box_rows);

namespace {

constexpr int BM = 128, BN = 256, BK = 128, STAGES = 6, SSLOTS = 6;
constexpr int A_BYTES = BM * BK;              // this CTA's activation rows (e4m3)
constexpr int B_BYTES = (BN / 2) * BK;        // this CTA's weight rows (4-bit values padded to bytes)
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SF_A_BYTES = 512;               // 128 rows x 4 K chunks
constexpr int SF_BYTES = SF_A_BYTES + 2 * 512;   // + the weight operand, 256 rows
constexpr int SF_COL0 = BN;                   // tensor-memory scale slots after the accumulator
constexpr int TMEM_COLS = 512;
static_assert(SF_COL0 + 32 * (STAGES - 1) + 16 + 8 <= TMEM_COLS, "tensor memory");
constexpr int EPI_WARP0 = 4, NUM_THREADS = 256;
constexpr int RING = 4;                       // tile-index slots
constexpr int BAR_BYTES = 512;
constexpr int SCHED_BYTES = kSchedBytes + 4 * (kSchedMaxRuns + 1);
constexpr int SMEM_BYTES =
    STAGES * STAGE_BYTES + SSLOTS * SF_BYTES + 1024 + BAR_BYTES + SCHED_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct MxPairArgs {
  const int32_t* block_expert_ids;
  const int32_t* num_post_padded;
  const float* a_scale;     // [cap, K/g] fp32 powers of two
  const uint8_t* b_scale;   // prepacked: [E][K/128][N/128] blocks of 512 bytes
  __nv_bfloat16* out;       // [cap, N]
  int ldo;                  // N
  int num_kb;               // K / 128
  int n_tiles;
  int b_rows_per_expert;    // N
  int m_blocks_cap;
  int num_experts;
  uint64_t limit_ns;
  int never_arrive;
  int* err;
  int* tile_ctr;            // {next tile, CTAs finished}, zero at launch
  Epilogue ep;
  uint8_t* zq;              // fused GEMM1: z codes [cap, I], scales [cap, I / group]
  float* zs;
  int I;
  int ue8m0;
};

template <bool MX8, bool FUSE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_ggemm_mx_2sm(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const MxPairArgs args) {
  // scale-writer warps per CTA: MXFP8 warp 2 (activations) + warp 3
  // (weights); W4A8 warp 3 writes both
  constexpr int WRITERS = MX8 ? 2 : 1;
  // leader MMA issuer + peer producer + the leader's writers + both CTAs'
  // epilogue warps
  constexpr int RING_READERS = 2 + WRITERS + 2 * 4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sf_ring = smem + STAGES * STAGE_BYTES;            // SSLOTS x SF_BYTES
  uint64_t* bars = reinterpret_cast<uint64_t*>(sf_ring + SSLOTS * SF_BYTES);
  // full[S], empty[S], sfull[SS], sempty[SS], tfull, tempty, drain, ring_full[R], ring_empty[R]
  constexpr int NBARS = 2 * STAGES + 2 * SSLOTS + 3 + 2 * RING;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_ring = reinterpret_cast<int*>(tmem_holder + 2);
  static_assert(NBARS * 8 + 8 + 4 * RING <= BAR_BYTES, "barrier area");
  int* s_sched = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + BAR_BYTES);
  int* s_pairs = s_sched + kSchedBytes / 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_u32(bars);
  const uint32_t sf_base = smem_u32(sf_ring);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto sfull_bar = [&](int s) { return bar_base + 8u * (2 * STAGES + s); };
  auto sempty_bar = [&](int s) { return bar_base + 8u * (2 * STAGES + SSLOTS + s); };
  const uint32_t tfull_bar = bar_base + 8u * (2 * STAGES + 2 * SSLOTS);
  const uint32_t tempty_bar = bar_base + 8u * (2 * STAGES + 2 * SSLOTS + 1);
  const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 2 * SSLOTS + 2);
  auto ring_full = [&](int i) { return bar_base + 8u * (2 * STAGES + 2 * SSLOTS + 3 + i); };
  auto ring_empty = [&](int i) {
    return bar_base + 8u * (2 * STAGES + 2 * SSLOTS + 3 + RING + i);
  };
  const uint32_t ring_base = smem_u32(s_ring);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int s = 0; s < SSLOTS; ++s) {
      mbar_init(sfull_bar(s), WRITERS);           // the leader's writers (leader's is used)
      mbar_init(sempty_bar(s), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, 8);                     // 4 epilogue warps in each CTA
    mbar_init(drain_bar, 1);
    for (int i = 0; i < RING; ++i) {
      mbar_init(ring_full(i), 1);
      mbar_init(ring_empty(i), RING_READERS);     // only the leader's are waited on
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

  const int nb_valid = min(*args.num_post_padded / BM, args.m_blocks_cap);
  const TileSched sched =
      sched_build(args.block_expert_ids, nb_valid, BM, args.num_experts, s_sched,
                  reinterpret_cast<int*>(smem), args.n_tiles, 1 << 20);
  sched_pairs_build(sched, s_pairs);
  __syncthreads();
  const int total = s_pairs[sched.nruns] * args.n_tiles;
  const int N = args.b_rows_per_expert;

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
  // a warp's ring read: lane 0 takes the slot, the warp gets its tile index
  auto warp_take = [&](int j) -> int {
    int t = 0;
    if (lane == 0) t = ring_take(j);
    return __shfl_sync(0xffffffffu, t, 0);
  };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producers
    const uint64_t pol_a = l2_policy(MOE_GEMM_L2_A);
    const uint64_t pol_b = l2_policy(MOE_GEMM_L2_B);
    constexpr int TX = A_BYTES + (MX8 ? B_BYTES : B_BYTES / 2);   // packed 4-bit bytes count
    uint32_t stage = 0, phase = 0, issued_mask = 0, issued_parity = 0;
    bool skip_first = leader && args.never_arrive != 0;
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
      const int my_row = leader ? P.row0 : P.row1;
      // weight rows: GEMM1 with the activation, the gate rows [128 j, +128)
      // (leader) and the matching up rows I + 128 j (peer); else 256
      // consecutive rows, 128 each
      const int brow = FUSE ? P.e * N + P.n_tile * 128 + (leader ? 0 : args.I)
                            : P.e * N + P.n_tile * BN + (leader ? 0 : BN / 2);
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
            mbar_arrive_expect_tx(full_bar(stage), 2 * TX);
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
    if (leader)
      for (int s = 0; s < STAGES; ++s)
        if (issued_mask & (1u << s))
          mbar_wait_bounded(full_bar(s), (issued_parity >> s) & 1, nullptr, args.limit_ns,
                            args.err);
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t stage = 0, phase = 0, sslot = 0, sphase = 0;
    int local = 0;
    bool ok = true;
    for (int j = 0; ok; ++j) {
      const int t = ring_take(j);
      if (t < 0) break;
      if (!mbar_wait_bounded<true>(tempty_bar, (local & 1) ^ 1, abort_flag, args.limit_ns,
                                   args.err))
        break;
      tc_fence_after();
      for (int kb = 0; kb < args.num_kb; ++kb) {
        if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, args.limit_ns, args.err) ||
            !mbar_wait_bounded(sfull_bar(sslot), sphase, abort_flag, args.limit_ns, args.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_base + stage * STAGE_BYTES;
        const uint64_t adesc = sdesc_k_sw128(sa);
        const uint64_t bdesc = sdesc_k_sw128(sa + A_BYTES);
        const uint32_t sfa = tmem_base + SF_COL0 + 32 * stage, sfb = sfa + 16;
        const uint32_t src = sf_base + sslot * SF_BYTES;
        tmem_cp_pair_32x128b_x4(sfa, sdesc_rows16(src));
        tmem_cp_pair_32x128b_x4(sfb, sdesc_rows16(src + SF_A_BYTES));
        tmem_cp_pair_32x128b_x4(sfb + 4, sdesc_rows16(src + SF_A_BYTES + 512));
#pragma unroll
        for (int k = 0; k < BK / 32; ++k)
          umma_mxf8f6f4_pair(tmem_base, adesc + 2 * k, bdesc + 2 * k,
                             make_idesc_block_scaled(kFmtE4M3, MX8 ? kFmtE4M3 : kFmtE2M1,
                                                     2 * BM, BN, k),
                             sfa, sfb, (kb | k) != 0);
        tc_commit_pair(empty_bar(stage), 0x3);
        tc_commit_pair(sempty_bar(sslot), 0x3);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
        if (++sslot == SSLOTS) {
          sslot = 0;
          sphase ^= 1;
        }
      }
      if (!ok) break;
      tc_commit_pair(tfull_bar, 0x3);
      ++local;
    }
    tc_commit_pair(drain_bar, 0x1);
    mbar_wait_bounded(drain_bar, 0, nullptr, args.limit_ns, args.err);
  } else if (leader && ((MX8 && warp == 2) || warp == 3)) {
    // ------------------------------------------------------------ scale writers
    // The leader's writers fill the ring slots of both CTAs: per K block the
    // activation operand of each CTA's 128 rows (lane l: rows l + 32 c, one
    // 16-byte word) and, in both slots, the weight operand of the tile's 256
    // weight rows (16 bytes per lane and 128-row group, copied from the
    // prepacked blocks).  The peer's slot is written with shared::cluster
    // stores, so every signal per K block stays inside the leader CTA (a
    // handshake from the peer per K block measured twice as slow).
    // MXFP8: warp 2 the leader's rows, warp 3 the peer's rows and the weight
    // operand; W4A8: warp 3 everything.
    const int G = N / 128;
    uint32_t sslot = 0, sphase = 0;
    bool ok = true;
    auto writer = [&](auto own_tag, auto peer_tag) {
      constexpr bool OWN_A = decltype(own_tag)::value;     // the leader's activation rows
      constexpr bool PEER = decltype(peer_tag)::value;     // the peer's rows + weight operand
      for (int j = 0; ok; ++j) {
        const int t = warp_take(j);
        if (t < 0) break;
        const PairTile P = sched_pair_tile(sched, s_pairs, t);
        const int g0 = FUSE ? P.n_tile : 2 * P.n_tile;
        const int g1 = FUSE ? args.I / 128 + P.n_tile : 2 * P.n_tile + 1;
        const bool two = g1 < G;                 // false: a 128-row last tile of GEMM2
        const uint4* bsrc = reinterpret_cast<const uint4*>(args.b_scale) + lane;
        auto bblock = [&](int kb, int g) {       // uint4 index of group g's block, K block kb
          return ((size_t)(P.e * args.num_kb + kb) * G + g) * 32;
        };
        AGroup<MX8> a_own, a_peer;
        uint4 b0[4], b1[4];
        for (int kb0 = 0; kb0 < args.num_kb && ok; kb0 += 4) {
          if (OWN_A)
            load_ascales<MX8>(a_own, args.a_scale, (size_t)P.row0, BM, lane, args.num_kb, kb0);
          if (PEER) {
            load_ascales<MX8>(a_peer, args.a_scale, (size_t)P.row1, BM, lane, args.num_kb, kb0);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const int kb = min(kb0 + jj, args.num_kb - 1);
              b0[jj] = __ldg(bsrc + bblock(kb, g0));
              b1[jj] = two ? __ldg(bsrc + bblock(kb, g1))
                           : make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
            }
          }
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            if (kb0 + jj >= args.num_kb) break;
            int got = 1;
            if (lane == 0)
              got = mbar_wait_bounded(sempty_bar(sslot), sphase ^ 1, abort_flag, args.limit_ns,
                                      args.err);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
              ok = false;
              break;
            }
            uint4* slot = reinterpret_cast<uint4*>(sf_ring + sslot * SF_BYTES);
            const uint32_t peer_slot = mapa_shared(sf_base + sslot * SF_BYTES, 1);
            if (OWN_A) {
              uint32_t aw[4];
#pragma unroll
              for (int c = 0; c < 4; ++c) aw[c] = a_word<MX8>(a_own, c, jj);
              slot[lane] = make_uint4(aw[0], aw[1], aw[2], aw[3]);
            }
            if (PEER) {
              uint32_t aw[4];
#pragma unroll
              for (int c = 0; c < 4; ++c) aw[c] = a_word<MX8>(a_peer, c, jj);
              st_shared_cluster_v4(peer_slot + 16u * lane, make_uint4(aw[0], aw[1], aw[2], aw[3]));
              slot[32 + lane] = b0[jj];
              slot[64 + lane] = b1[jj];
              st_shared_cluster_v4(peer_slot + SF_A_BYTES + 16u * lane, b0[jj]);
              st_shared_cluster_v4(peer_slot + SF_A_BYTES + 512 + 16u * lane, b1[jj]);
            }
            fence_proxy_async_all();
            __syncwarp();
            if (lane == 0) mbar_arrive(sfull_bar(sslot));
            if (++sslot == SSLOTS) {
              sslot = 0;
              sphase ^= 1;
            }
          }
        }
      }
    };
    if constexpr (MX8) {
      if (warp == 2)
        writer(std::true_type{}, std::false_type{});
      else
        writer(std::false_type{}, std::true_type{});
    } else {
      writer(std::true_type{}, std::true_type{});
    }
  } else if (warp >= EPI_WARP0) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int row_in_tile = q * 32 + lane;
    int local = 0;
    for (int j = 0;; ++j) {
      const int t = warp_take(j);
      if (t < 0) break;
      const PairTile P = sched_pair_tile(sched, s_pairs, t);
      int ok = 0;
      if (lane == 0) ok = mbar_wait_bounded(tfull_bar, local & 1, abort_flag, args.limit_ns, args.err);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const bool live = leader || P.has1;        // a lone block's peer half is a repeat
      const size_t row = (size_t)(leader ? P.row0 : P.row1) + row_in_tile;
      mx_row_epilogue<MX8, FUSE>(tmem_base + ((uint32_t)(q * 32) << 16), row, live, args.ep,
                                 P.e, P.n_tile, args.I, args.ue8m0 != 0, args.zq, args.zs,
                                 args.out, args.ldo, N, [&] {
                                   tc_fence_before();
                                   __syncwarp();
                                   if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar, 0));
                                 });
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
    __threadfence();
    if (atomicAdd(args.tile_ctr + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(args.tile_ctr, 0);
      atomicExch(args.tile_ctr + 1, 0);
    }
  }
}

template <bool MX8, bool FUSE>
cudaError_t launch_mx_pairs(const CUtensorMap& tmA, const CUtensorMap& tmB, const MxPairArgs& a,
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
    cudaError_t e = cudaFuncSetAttribute(k_ggemm_mx_2sm<MX8, FUSE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(num_sms(), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, k_ggemm_mx_2sm<MX8, FUSE>, &cfg);
    if (e != cudaSuccess) return e;
    max_pairs[dev] = n;
    return cudaSuccess;
  });
  if (es != cudaSuccess) return es;
  if (max_pairs[dev] <= 0) return cudaErrorInvalidConfiguration;
  cfg.gridDim = dim3(2 * max_pairs[dev], 1, 1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, k_ggemm_mx_2sm<MX8, FUSE>, tmA, tmB, a);
}

}  // namespace

cudaError_t launch_ggemm_mx_2sm(const void* A, const float* a_scale, int cap, int K, const void* B,
                                const uint8_t* b_scale_packed, int b_rows_total,
                                int b_rows_per_expert, int n_out,
                                const int32_t* block_expert_ids, const int32_t* num_post_padded,
                                void* out, bool b_e4m3, const Epilogue& ep, cudaStream_t stream,
                                float* z_scale, bool fuse_act, bool ue8m0, int* tile_ctr) {
  if (cap <= 0) return cudaSuccess;
  if ((reinterpret_cast<uintptr_t>(B) & (b_e4m3 ? 15u : 31u)) != 0 ||
      (reinterpret_cast<uintptr_t>(b_scale_packed) & 15u) != 0)
    return cudaErrorInvalidValue;
  if (b_rows_per_expert % 128 != 0 || K % 128 != 0 || n_out != b_rows_per_expert ||
      cap % BM != 0)
    return cudaErrorInvalidValue;
  if (fuse_act && (z_scale == nullptr || b_rows_per_expert % 256 != 0)) return cudaErrorInvalidValue;
  CUtensorMap tmA, tmB;
  if (!make_tmap_k_sw128(&tmA, A, (uint64_t)cap, (uint64_t)K, 1, BM) ||
      !(b_e4m3 ? make_tmap_k_sw128(&tmB, B, (uint64_t)b_rows_total, (uint64_t)K, 1, BN / 2)
               : make_tmap_fp4_k_sw128(&tmB, B, (uint64_t)b_rows_total, (uint64_t)K, BN / 2)))
    return cudaErrorInvalidValue;
  MxPairArgs a;
  a.block_expert_ids = block_expert_ids;
  a.num_post_padded = num_post_padded;
  a.a_scale = a_scale;
  a.b_scale = b_scale_packed;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ldo = n_out;
  a.num_kb = K / BK;
  a.I = b_rows_per_expert / 2;
  a.n_tiles = fuse_act ? a.I / 128 : (n_out + BN - 1) / BN;
  a.zq = fuse_act ? static_cast<uint8_t*>(out) : nullptr;
  a.zs = z_scale;
  a.ue8m0 = ue8m0 ? 1 : 0;
  a.b_rows_per_expert = b_rows_per_expert;
  a.m_blocks_cap = cap / BM;
  a.num_experts = b_rows_total / b_rows_per_expert;
  a.ep = ep;
  watchdog_params(&a.limit_ns, &a.never_arrive);
  a.err = dev_error_word();
  if (a.err == nullptr) return cudaErrorInvalidDevice;   // no usable current device
  a.tile_ctr = tile_ctr != nullptr ? tile_ctr : next_tile_counter();
  if (a.tile_ctr == nullptr) return cudaErrorInvalidDevice;
  if (b_e4m3)
    return fuse_act ? launch_mx_pairs<true, true>(tmA, tmB, a, stream)
                    : launch_mx_pairs<true, false>(tmA, tmB, a, stream);
  return fuse_act ? launch_mx_pairs<false, true>(tmA, tmB, a, stream)
                  : launch_mx_pairs<false, false>(tmA, tmB, a, stream);
}

}  // namespace moe
