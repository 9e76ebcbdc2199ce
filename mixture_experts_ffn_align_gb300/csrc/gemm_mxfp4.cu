// Block-scaled (E8M0 per 32) grouped GEMM: MXFP4 x FP8 (W4A8, stages 2 and 4 of
// MOE_Q_MXFP4_W4A8) and MXFP8 x MXFP8 (MOE_Q_MXFP8_1X32: e4m3 weights with an
// E8M0 scale per 1x32, activations e4m3 with a UE8M0 scale per 1x32 -- page
// "Blackwell 上的 DeepGEMM FusedMoE（vLLM）", TL;DR table, MXFP8 (1x32) row and
// §2.9: the same GEMM with recipe (1, 32)).  The MXFP8 form (template MX8)
// loads the weights with the ordinary byte tensor map (one e4m3 per byte, the
// same smem footprint as the padded E2M1 tile), tells the MMA that B is e4m3,
// and builds each activation scale word from four 1x32 exponents instead of
// one 1x128 exponent repeated.
//
// What it computes: page "Blackwell 上的 DeepGEMM FusedMoE（vLLM）", TL;DR table,
// W4A8 MXFP4 row: weights E2M1 with one E8M0 scale per 32 along K, activations
// e4m3 with dynamic 128-element scales (here rounded up to powers of two,
// UE8M0, so that the tensor core can apply them); §2.8(d): weights stay packed
// two per byte.  For every used 128-row block with expert e:
//   C[r, n] = sum_k (qa[r,k] * sa[r, k/128]) * (e2m1(qb[e,n,k]) * 2^(sb[e,n,k/32]-127)).
// All scales are powers of two, so the block-scaled MMA
// (tcgen05.mma kind::mxf8f6f4.block_scale.scale_vec::1X) applies them in
// hardware and accumulates the whole K range in one fp32 TMEM accumulator.
//
//  * warp 0 lane 0: TMA producer, 4-stage ring; per 128-wide K block an e4m3
//    A tile (128 x 128 B) and an E2M1 B tile of 256 rows loaded with the
//    padded 4-bit TMA type (each 16 values -> 8 bytes + 8-byte gap, so a row
//    of 128 values fills one 128-byte swizzled smem row; the copy counts the
//    packed bytes toward the barrier), 128-byte swizzle;
//  * scale writers: MXFP8, warps 2 and 3 (warp 2 the A operand, warp 3 the
//    B operand; one warp doing both measured busy ~90 % of the kernel and
//    stalled the MMA issuer ~27 % of the DeepSeek-shaped MXFP8 GEMM1); W4A8,
//    warp 3 alone (warp 2 copies the slots into tensor memory, below).  Per
//    K block they build the two scale operands in
//    a shared-memory ring of SSLOTS slots: the A operand (each row's UE8M0
//    exponent in all 4 bytes: one scale covers 128 = 4 x 32) and the B
//    operand (the 4 E8M0 bytes of each column's 4 K chunks), each 128-row
//    group as 32 rows of 16 bytes -- row r at byte 16 (r % 32) + 4 (r / 32),
//    byte j of the word for K chunk j, which is the tensor-memory layout the
//    block-scaled MMA reads (32 lanes x 4 columns, row r at lane r % 32,
//    column r / 32, repeated in every lane quadrant; byte j picked by the
//    scale-ID field of MMA j).  When K % 512 == 0 (weight-scale rows are
//    16-byte multiples) the weight scales of 4 K blocks x the tile's 256 rows
//    come in as one TMA box, two groups ahead, and are transposed from
//    shared memory; otherwise every lane loads them 16 bytes (4 K blocks) at
//    a time, one group ahead.  The staged form took the DeepSeek-shaped GEMM1
//    from 1.08 to 0.88 ms: each weight-scale row is read once from HBM, and
//    register loads one group ahead left that latency exposed.  (4-byte
//    cp.async copies straight into the packed places were slower still:
//    four times the L1 wavefronts.)
//  * warp 1 lane 0: copies the K block's scale operands into tensor memory
//    with tcgen05.cp (32x128b, repeated to the four lane quadrants), then
//    issues four MMAs (M=128, N=256, K=32) into the 256-column accumulator
//    (N=128 MMAs run at about half the tensor rate); copy and MMAs run in
//    issue order in the tensor pipe, so no thread waits between them, and
//    one tcgen05.commit frees the stage and its scale slot.  W4A8: lane 0 of
//    warp 2 (no scale writing to do there) makes the copies and commits
//    each slot's readiness, and the MMA issuer only waits for it: a thread's
//    shared-memory waits stall behind its own copies still queued in the
//    tensor pipe (~80 cycles a K block, measured), so they are better taken
//    off the issuer.  (Writing the scales
//    into tensor memory with tcgen05.st from four warps cost 0.34 of 1.13 ms
//    on the DeepSeek-shaped GEMM1.)  Each smem stage has its own tensor-memory
//    scale slot (16-column aligned: an odd-column scale address raised a
//    misaligned-address fault), rewritten only after the stage's producer
//    wait has seen that slot's MMAs complete;
//  * warps 4-7: epilogue, one warp per TMEM lane quadrant, 128 columns at a
//    time: tcgen05.ld -> bf16 -> global.  Tensor memory holds one 256-column
//    accumulator plus the scale slots, so the next tile's MMAs wait for the
//    epilogue to have read it.  (Eight warps of 128 columns each measured
//    slower on both GEMMs.)
//  * a last column tile narrower than 256 (N % 256 == 128) is computed on
//    whatever the weight box held above N and its upper half is not stored.
//  * tiles walked expert by expert (tile_sched.cuh); every wait is bounded.
#include <algorithm>
#include <mutex>

#include "../../include/moe_ffn.h"
#include "e4m3_pack.cuh"
#include "moe_common.cuh"
#include "moe_internal.h"
#include "mx_common.cuh"
#include "tile_sched.cuh"

namespace moe {

bool make_tmap_k_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t k_elems,
                       int elem_bytes, uint32_t box_rows);
bool make_tmap_fp4_k_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t k_elems,
                           uint32_t box_rows);
bool make_tmap_u8_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_bytes,
                       uint32_t box_bytes, uint32_t box_rows);

namespace {

// Where the weight-scale operand of each K block comes from: built by warp 3
// from E8M0 bytes it loads to registers (any K), transposed from TMA boxes of
// 4 K blocks (K % 512 == 0), or copied in ready-made from scales that
// moe_prepack_weights rewrote into the operand layout.
enum : int { SRC_REGS = 0, SRC_STAGED = 1, SRC_PACKED = 2 };

constexpr int BM = 128, BN = 256, BK = 128, STAGES = 4, SSLOTS = 4;
// Staged weight scales (K % 512 == 0): 16 bytes = 4 K blocks of each of the
// tile's 256 rows per TMA box, NSTG groups in flight.
constexpr int NSTG = 2, STG_BYTES = 16 * BN;
constexpr int A_BYTES = BM * BK;          // e4m3
constexpr int B_BYTES = BN * BK;          // 4-bit values padded to one byte each in smem
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TX_BYTES = A_BYTES + B_BYTES / 2;   // bytes the copies of one stage count
constexpr int SF_A_BYTES = 512;           // 128 rows x 4 K chunks
constexpr int SF_BYTES = SF_A_BYTES + 2 * 512;    // + 256 columns x 4 K chunks
constexpr int SF_COL0 = BN;               // tensor-memory scale slots after the accumulator
constexpr int SF_SLOT = 16;               // stage s: A at SF_COL0 + 32 s, B at + 16
constexpr int TMEM_COLS = 512;
constexpr int NUM_EPI_WARPS = 4, EPI_WARP0 = 4;
constexpr int NUM_THREADS = (EPI_WARP0 + NUM_EPI_WARPS) * 32;
constexpr int SMEM_BYTES =
    STAGES * STAGE_BYTES + SSLOTS * SF_BYTES + NSTG * STG_BYTES + 1024 + 512 + kSchedBytes;
static_assert(SF_COL0 + SF_SLOT * (2 * SSLOTS - 1) + BN / 32 <= TMEM_COLS, "tensor memory");
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct Mx4Args {
  const int32_t* block_expert_ids;
  const int32_t* num_post_padded;
  const float* a_scale;     // [cap, K/128] fp32 powers of two
  const uint8_t* b_scale;   // [E, N, K/32] E8M0
  __nv_bfloat16* out;       // [cap, N]
  int ldo;                  // N
  int num_kb;               // K / 128
  int n_tiles;              // ceil(N / 256)
  int b_rows_per_expert;    // N
  int blocks_cap;           // blocks of blk_rows rows the buffers hold
  int blk_rows;             // rows per block of the padded layout
  int num_experts;
  int group_max;
  uint64_t limit_ns;
  int never_arrive;
  int* err;
  Epilogue ep;              // bias, router weight, gated activation recipe
  // fused GEMM1 epilogue (FUSE): z codes [cap, I] e4m3 and z scales
  // [cap, I / group] fp32 (powers of two when ue8m0)
  uint8_t* zq;
  float* zs;
  int I;
  int ue8m0;
};

template <int SRC, bool MX8, bool FUSE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_ggemm_mxfp4(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmS, const Mx4Args args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr bool COPIER = !MX8;   // warp 2 copies the scales into tensor memory (W4A8)
  uint8_t* sf_ring = smem + STAGES * STAGE_BYTES;    // SSLOTS x SF_BYTES, 16-byte aligned
  uint8_t* stg_ring = sf_ring + SSLOTS * SF_BYTES;     // NSTG x STG_BYTES (SRC_STAGED)
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg_ring + NSTG * STG_BYTES);
  // full[S], empty[S], sfull[SS], (SS unused), tfull, tempty, drain, stg_full[NSTG],
  // sready[SS], cdrain
  uint32_t* tmem_holder =
      reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 3 * SSLOTS + 4 + NSTG);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_sched = reinterpret_cast<int*>(stg_ring + NSTG * STG_BYTES + 512);
  static_assert(8 * (2 * STAGES + 3 * SSLOTS + 4 + NSTG) + 8 <= 512, "barrier area");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_u32(bars);
  const uint32_t sf_base = smem_u32(sf_ring);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto sfull_bar = [&](int s) { return bar_base + 8u * (2 * STAGES + s); };
  // A scale slot is free once the MMAs of its K block have completed, which
  // is when the operand stage of that K block is (one slot per stage): the
  // stage's barrier serves both, one tcgen05.commit per K block.
  static_assert(SSLOTS == STAGES, "one scale slot per operand stage");
  auto sempty_bar = [&](int s) { return empty_bar(s); };
  const uint32_t tfull_bar = bar_base + 8u * (2 * STAGES + 2 * SSLOTS);
  const uint32_t tempty_bar = bar_base + 8u * (2 * STAGES + 2 * SSLOTS + 1);
  const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 2 * SSLOTS + 2);
  auto stg_full = [&](int s) { return bar_base + 8u * (2 * STAGES + 2 * SSLOTS + 3 + s); };
  auto sready_bar = [&](int s) {
    return bar_base + 8u * (2 * STAGES + 2 * SSLOTS + 3 + NSTG + s);
  };
  const uint32_t cdrain_bar = bar_base + 8u * (2 * STAGES + 3 * SSLOTS + 3 + NSTG);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int s = 0; s < SSLOTS; ++s) {
      mbar_init(sfull_bar(s), MX8 ? 2 : 1);   // one arrival per scale writer
      mbar_init(sready_bar(s), 1);
    }
    mbar_init(cdrain_bar, 1);
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, NUM_EPI_WARPS);
    for (int s = 0; s < NSTG; ++s) mbar_init(stg_full(s), 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (SRC == SRC_STAGED) tma_prefetch_desc(&tmS);
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
  const int N = args.b_rows_per_expert;

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
      const int brow = FUSE ? e * N + n_tile * 128 : e * N + n_tile * BN;
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
          mbar_arrive_expect_tx(full_bar(stage), MX8 ? A_BYTES + B_BYTES : TX_BYTES);
          tma_load_2d(sa, &tmA, full_bar(stage), kb * BK, T.row0, pol_a);
          tma_load_2d(sa + A_BYTES, &tmB, full_bar(stage), kb * BK, brow, pol_b);
          tma_load_2d(sa + A_BYTES + B_BYTES / 2, &tmB, full_bar(stage), kb * BK, brow2, pol_b);
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
  } else if (COPIER && warp == 2) {
    // ------------------------------------------------------------ scale copier
    // W4A8 (one scale writer, warp 3): lane 0 of warp 2 copies each complete
    // slot into its tensor-memory scale slot (tcgen05.cp) and commits
    // sready, so the MMA issuer only waits for ready scales.  When the
    // issuer made the copies, each of its later shared-memory waits stalled
    // behind its own copies still queued in the tensor pipe (~80 cycles of a
    // 512-cycle K block); a thread with no other work can take that stall.
    // The tensor memory of slot s is free: the slot was rewritten only after
    // its MMAs of SSLOTS K blocks earlier completed (sempty).
    if (lane == 0) {
      uint32_t cslot = 0, cphase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        for (int kb = 0; kb < args.num_kb; ++kb) {
          if (!mbar_wait_bounded(sfull_bar(cslot), cphase, abort_flag, args.limit_ns, args.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa = tmem_base + SF_COL0 + SF_SLOT * 2 * cslot;
          const uint32_t src = sf_base + cslot * SF_BYTES;
          tmem_cp_32x128b_x4(sfa, sdesc_rows16(src));
          tmem_cp_32x128b_x4(sfa + SF_SLOT, sdesc_rows16(src + SF_A_BYTES));
          tmem_cp_32x128b_x4(sfa + SF_SLOT + 4, sdesc_rows16(src + SF_A_BYTES + 512));
          tc_commit(sready_bar(cslot));
          if (++cslot == SSLOTS) {
            cslot = 0;
            cphase ^= 1;
          }
        }
      }
      tc_commit(cdrain_bar);   // this thread's copies complete before the CTA tears down
      mbar_wait_bounded(cdrain_bar, 0, nullptr, args.limit_ns, args.err);
    }
  } else if ((MX8 && warp == 2) || warp == 3) {
    // ------------------------------------------------------------ scale writers
    // Warp 3 builds the weight-scale operand of each K block (the E8M0 bytes
    // as given).  MXFP8: warp 2 builds the activation-scale operand (A words
    // from four 1x32 fp32 scales of each of this lane's rows); each writes its
    // part of the ring slot and arrives on the slot's full barrier.  (One warp
    // doing both was busy ~90 % of the MXFP8 GEMM1 and held the MMA issuer
    // back.)  W4A8: one 1x128 scale per row and K block is little work, a
    // second writer measured 3-5 % slower, so warp 3 writes both parts.
    const bool wa = warp == 2;
    uint32_t sslot = 0, sphase = 0;
    // lane l: 16 bytes at row l of the A block (warp 2; W4A8: aw from warp
    // 3) or of both B blocks (warp 3)
    auto put_slot = [&](const uint32_t (&w)[8], const uint32_t (&aw)[4]) {
      int got = 1;
      if (lane == 0)
        got = mbar_wait_bounded(sempty_bar(sslot), sphase ^ 1, abort_flag, args.limit_ns,
                                args.err);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) return false;
      uint4* dst = reinterpret_cast<uint4*>(sf_ring + sslot * SF_BYTES) + lane;
      if (wa || !MX8) dst[0] = make_uint4(aw[0], aw[1], aw[2], aw[3]);
      if (!wa) {
        dst[32] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[64] = make_uint4(w[4], w[5], w[6], w[7]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(sfull_bar(sslot));
      if (++sslot == SSLOTS) {
        sslot = 0;
        sphase ^= 1;
      }
      return true;
    };
    if constexpr (SRC == SRC_STAGED) {
      // Warp 3: the weight scales of 4 K blocks x the tile's 256 rows arrive
      // as one TMA box (row n at byte 16 n) NSTG groups ahead.  Warp 2: the
      // activation scales (in L2: the permute/act kernel just wrote them)
      // are loaded to registers one group ahead.
      const int ngroups = args.num_kb / 4;
      const uint64_t pol_s = l2_policy(MOE_GEMM_L2_B);
      const uint32_t stg_base = smem_u32(stg_ring);
      struct Cursor {
        int t, g, row0, rows, n_tile, e;
      };
      auto seek = [&](Cursor& c) {             // the tile at c.t, if any
        for (; c.t < total; c.t += gridDim.x) {
          const Tile T = sched_tile(sched, c.t);
          c.row0 = T.row0;
          c.rows = T.rows;
          c.n_tile = T.n_tile;
          c.e = T.e;
          {
            c.g = 0;
            return true;
          }
        }
        return false;
      };
      auto step = [&](Cursor& c) {
        if (++c.g < ngroups) return true;
        c.t += gridDim.x;
        return seek(c);
      };
      Cursor use{(int)blockIdx.x, 0, 0, 0, 0};
      bool use_ok = seek(use);
      bool ok = true;
      if (wa) {
        auto load_a = [&](const Cursor& c, AGroup<MX8>& A) {
          load_ascales<MX8>(A, args.a_scale, (size_t)c.row0, c.rows, lane, args.num_kb, 4 * c.g);
        };
        Cursor anext = use;
        bool anext_ok = use_ok;
        AGroup<MX8> a_cur, a_nxt;
        if (use_ok) {
          load_a(use, a_cur);
          anext_ok = step(anext);
          if (anext_ok) load_a(anext, a_nxt);
        }
        while (use_ok && ok) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t w[8] = {}, aw[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) aw[c] = a_word<MX8>(a_cur, c, j);
            if (!put_slot(w, aw)) {
              ok = false;
              break;
            }
          }
          if (!ok) break;
          use_ok = step(use);
          a_cur = a_nxt;
          if (anext_ok) {
            anext_ok = step(anext);
            if (anext_ok) load_a(anext, a_nxt);
          }
        }
      } else {
        auto stage_group = [&](const Cursor& c, int slot) {   // lane 0
          mbar_arrive_expect_tx(stg_full(slot), STG_BYTES);
          if (FUSE) {   // gate rows, then the matching up rows (128-row boxes)
            tma_load_2d(stg_base + slot * STG_BYTES, &tmS, stg_full(slot), 16 * c.g,
                        c.e * N + c.n_tile * 128, pol_s);
            tma_load_2d(stg_base + slot * STG_BYTES + STG_BYTES / 2, &tmS, stg_full(slot),
                        16 * c.g, c.e * N + args.I + c.n_tile * 128, pol_s);
          } else {
            tma_load_2d(stg_base + slot * STG_BYTES, &tmS, stg_full(slot), 16 * c.g,
                        c.e * N + c.n_tile * BN, pol_s);
          }
        };
        Cursor fill = use;
        bool fill_ok = use_ok;
        int nfill = 0, nuse = 0;
        for (; nfill < NSTG && fill_ok; ++nfill) {
          if (lane == 0) stage_group(fill, nfill);
          fill_ok = step(fill);
        }
        // W4A8: this warp also builds the A words, scales one group ahead
        AGroup<MX8> a_cur, a_nxt;
        Cursor anext = use;
        bool anext_ok = use_ok;
        auto load_a = [&](const Cursor& c, AGroup<MX8>& A) {
          load_ascales<MX8>(A, args.a_scale, (size_t)c.row0, c.rows, lane, args.num_kb, 4 * c.g);
        };
        if constexpr (!MX8) {
          if (use_ok) {
            load_a(use, a_cur);
            anext_ok = step(anext);
            if (anext_ok) load_a(anext, a_nxt);
          }
        }
        while (use_ok && ok) {
          const int slot = nuse % NSTG;
          int got = 1;
          if (lane == 0)
            got = mbar_wait_bounded(stg_full(slot), (nuse / NSTG) & 1, abort_flag, args.limit_ns,
                                    args.err);
          got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) break;
          const uint32_t stg = stg_base + slot * STG_BYTES;
          const int n0 = use.n_tile * BN + lane;    // this lane's rows: n0 + 32 c
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t w[8], aw[4] = {};
#pragma unroll
            for (int c = 0; c < 8; ++c)   // rows past N (ragged last tile): 2^0
              w[c] = FUSE || n0 + 32 * c < N ? ld_shared_u32(stg + 16 * (lane + 32 * c) + 4 * j)
                                              : 0x7F7F7F7Fu;
            if constexpr (!MX8) {
#pragma unroll
              for (int c = 0; c < 4; ++c) aw[c] = a_word<MX8>(a_cur, c, j);
            }
            if (!put_slot(w, aw)) {
              ok = false;
              break;
            }
          }
          if (!ok) break;
          ++nuse;
          // this warp's reads of the staging slot come before the copy that refills it
          fence_proxy_async_smem();
          __syncwarp();
          if (fill_ok) {
            if (lane == 0) stage_group(fill, nfill % NSTG);
            ++nfill;
            fill_ok = step(fill);
          }
          use_ok = step(use);
          if constexpr (!MX8) {
            a_cur = a_nxt;
            if (anext_ok) {
              anext_ok = step(anext);
              if (anext_ok) load_a(anext, a_nxt);
            }
          }
        }
        // copies issued but not consumed (a wait ran out) land before the CTA exits
        if (lane == 0)
          for (int k = nuse; k < nfill; ++k)
            mbar_wait_bounded(stg_full(k % NSTG), (k / NSTG) & 1, nullptr, args.limit_ns,
                              args.err);
      }
    } else if constexpr (SRC == SRC_PACKED) {
      // Prepacked weight scales ([E][K/128][N/128] blocks of 512 bytes, each
      // the 32 x 16-byte operand of one 128-row group and K block): lane 0 of
      // warp 3 copies a K block's weight operand (two groups: 256 rows, or
      // the gate group and its up group) straight into the slot with bulk
      // copies that complete on the slot's full barrier.  The activation
      // words are built as in the other forms (warp 2 for MXFP8, warp 3 for
      // W4A8), one group of 4 K blocks ahead.
      const int G = N / 128;                     // 128-row scale groups per expert
      constexpr int SCALE_PF = 8;                // K blocks ahead for the L2 prefetch
      const bool writes_a = wa || !MX8;
      const bool writes_b = !wa;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile T = sched_tile(sched, t);
        const int e = T.e, n_tile = T.n_tile;
        auto load_a = [&](AGroup<MX8>& A, int g) {
          load_ascales<MX8>(A, args.a_scale, (size_t)T.row0, T.rows, lane, args.num_kb, g);
        };
        AGroup<MX8> a_cur, a_nxt;
        if (writes_a) {
          load_a(a_cur, 0);
          if (args.num_kb > 4) load_a(a_nxt, 4);
        }
        // group offsets (in 512-byte blocks) of the operand's two halves
        const int g0 = FUSE ? n_tile : 2 * n_tile;
        const int g1 = FUSE ? args.I / 128 + n_tile : 2 * n_tile + 1;
        const bool two = g1 < G;                   // false: a 128-row last tile
        for (int kb0 = 0; kb0 < args.num_kb && ok; kb0 += 4) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int kb = kb0 + j;
            if (kb >= args.num_kb) break;
            int got = 1;
            if (lane == 0)
              got = mbar_wait_bounded(sempty_bar(sslot), sphase ^ 1, abort_flag, args.limit_ns,
                                      args.err);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
              ok = false;
              break;
            }
            uint8_t* slot = sf_ring + sslot * SF_BYTES;
            if (writes_b && lane == 0) {
              const uint8_t* src = args.b_scale + ((size_t)e * args.num_kb + kb) * G * 512;
              // The slot's copy waits for these bytes a few K blocks from now,
              // and they are read once from HBM (at W4A8 rates that latency
              // showed through the slot ring): ask for those of K block
              // kb + SCALE_PF in L2 already.  (Running on into the CTA's next
              // tile measured slower on GEMM1.)
              if (kb + SCALE_PF < args.num_kb) {
                const uint8_t* pf = src + (size_t)SCALE_PF * G * 512;
                if (FUSE || !two) {
                  bulk_prefetch_l2(pf + (size_t)g0 * 512, 512);
                  if (two) bulk_prefetch_l2(pf + (size_t)g1 * 512, 512);
                } else {
                  bulk_prefetch_l2(pf + (size_t)g0 * 512, 1024);
                }
              }
              const uint32_t dst = smem_u32(slot + SF_A_BYTES);
              const uint32_t bytes = two ? 1024u : 512u;
              // MXFP8: this arrival is warp 3's; W4A8: warp 3 arrives below
              if (MX8)
                mbar_arrive_expect_tx(sfull_bar(sslot), bytes);
              else
                mbar_expect_tx(sfull_bar(sslot), bytes);
              if (FUSE || !two) {
                bulk_load(dst, src + (size_t)g0 * 512, 512, sfull_bar(sslot));
                if (two) bulk_load(dst + 512, src + (size_t)g1 * 512, 512, sfull_bar(sslot));
              } else {
                bulk_load(dst, src + (size_t)g0 * 512, 1024, sfull_bar(sslot));
              }
            }
            if (writes_a) {
              uint32_t aw[4];
#pragma unroll
              for (int c = 0; c < 4; ++c) aw[c] = a_word<MX8>(a_cur, c, j);
              reinterpret_cast<uint4*>(slot)[lane] = make_uint4(aw[0], aw[1], aw[2], aw[3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(sfull_bar(sslot));
            }
            if (++sslot == SSLOTS) {
              sslot = 0;
              sphase ^= 1;
            }
          }
          if (writes_a) {
            a_cur = a_nxt;
            if (kb0 + 8 < args.num_kb) load_a(a_nxt, kb0 + 8);
          }
        }
      }
    } else {
      const int kq = args.num_kb * 4;            // E8M0 bytes per weight row
      const bool vec = (args.num_kb & 3) == 0;   // rows 16-byte aligned: vector loads
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile T = sched_tile(sched, t);
        const int e = T.e, n_tile = T.n_tile;
        auto load_a = [&](AGroup<MX8>& A, int g) {
          load_ascales<MX8>(A, args.a_scale, (size_t)T.row0, T.rows, lane, args.num_kb, g);
        };
        // activation scales of 4 K blocks per load (W4A8, built by warp 3
        // with the weight operand: one group ahead; MXFP8, warp 2: its 4x
        // larger scales at the group's start)
        AGroup<MX8> a_cur, a_nxt;
        if constexpr (!MX8) {
          load_a(a_cur, 0);
          if (args.num_kb > 4) load_a(a_nxt, 4);
        }
        if (wa) {
          for (int kb0 = 0; kb0 < args.num_kb && ok; kb0 += 4) {
            load_a(a_cur, kb0);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (kb0 + j >= args.num_kb) break;
              uint32_t w[8] = {}, aw[4];
#pragma unroll
              for (int c = 0; c < 4; ++c) aw[c] = a_word<MX8>(a_cur, c, j);
              if (!put_slot(w, aw)) {
                ok = false;
                break;
              }
            }
          }
        } else {
          // lane l builds rows l + 32 c (c < 8) of the weight operand; rows
          // past N (ragged last tile) read nothing.  Scales of 4 K blocks per
          // load, one group of 4 in flight ahead.
          const size_t row0 = FUSE ? (size_t)e * N + (size_t)n_tile * 128 + lane
                                   : (size_t)e * N + (size_t)n_tile * BN + lane;
          const uint8_t* sb_base = args.b_scale + row0 * kq;
          const size_t sb_step = (size_t)32 * kq;                    // bytes per 32 rows
          // FUSE: operand rows 128..255 are the up rows, I - 128 further on
          const size_t sb_up = FUSE ? (size_t)(args.I - 128) * kq : 0;
          const int n_valid = FUSE ? 256 : N - n_tile * BN - lane;   // row c valid if 32c < this
          auto load_b = [&](int g, uint4 (&B)[8]) {
            const int n = args.num_kb - g;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t* pb =
                  reinterpret_cast<const uint32_t*>(sb_base + c * sb_step + (c >= 4 ? sb_up : 0)) + g;
              if (32 * c >= n_valid) {
                B[c] = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
              } else if (vec) {
                B[c] = __ldg(reinterpret_cast<const uint4*>(pb));
              } else {
                B[c] = make_uint4(__ldg(pb), n > 1 ? __ldg(pb + 1) : 0u,
                                  n > 2 ? __ldg(pb + 2) : 0u, n > 3 ? __ldg(pb + 3) : 0u);
              }
            }
          };
          uint4 b_cur[8], b_nxt[8];
          load_b(0, b_cur);
          if (args.num_kb > 4) load_b(4, b_nxt);
          for (int kb0 = 0; kb0 < args.num_kb && ok; kb0 += 4) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (kb0 + j >= args.num_kb) break;
              uint32_t w[8], aw[4] = {};
#pragma unroll
              for (int c = 0; c < 8; ++c)
                w[c] = j == 0 ? b_cur[c].x : j == 1 ? b_cur[c].y : j == 2 ? b_cur[c].z : b_cur[c].w;
              if constexpr (!MX8) {
#pragma unroll
                for (int c = 0; c < 4; ++c) aw[c] = a_word<MX8>(a_cur, c, j);
              }
              if (!put_slot(w, aw)) {
                ok = false;
                break;
              }
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) b_cur[c] = b_nxt[c];
            if (kb0 + 8 < args.num_kb) load_b(kb0 + 8, b_nxt);
            if constexpr (!MX8) {
              a_cur = a_nxt;
              if (kb0 + 8 < args.num_kb) load_a(a_nxt, kb0 + 8);
            }
          }
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t stage = 0, phase = 0, sslot = 0, sphase = 0;
    int local = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      if (!mbar_wait_bounded(tempty_bar, (local & 1) ^ 1, abort_flag, args.limit_ns, args.err))
        break;
      tc_fence_after();
      for (int kb = 0; kb < args.num_kb; ++kb) {
        if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, args.limit_ns, args.err) ||
            !mbar_wait_bounded(COPIER ? sready_bar(sslot) : sfull_bar(sslot), sphase, abort_flag,
                               args.limit_ns, args.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_base + stage * STAGE_BYTES;
        const uint64_t adesc = sdesc_k_sw128(sa);
        const uint64_t bdesc = sdesc_k_sw128(sa + A_BYTES);
        const uint32_t sfa = tmem_base + SF_COL0 + SF_SLOT * 2 * sslot;
        if constexpr (!COPIER) {
          const uint32_t sf_src = sf_base + sslot * SF_BYTES;
          tmem_cp_32x128b_x4(sfa, sdesc_rows16(sf_src));
          tmem_cp_32x128b_x4(sfa + SF_SLOT, sdesc_rows16(sf_src + SF_A_BYTES));
          tmem_cp_32x128b_x4(sfa + SF_SLOT + 4, sdesc_rows16(sf_src + SF_A_BYTES + 512));
        }
#pragma unroll
        for (int j = 0; j < BK / 32; ++j) {
          umma_mxf8f6f4(tmem_base, adesc + 2 * j, bdesc + 2 * j,
                        make_idesc_block_scaled(kFmtE4M3, MX8 ? kFmtE4M3 : kFmtE2M1, BM, BN, j),
                        sfa,
                        sfa + SF_SLOT, (kb | j) != 0);
        }
        tc_commit(empty_bar(stage));   // frees the stage and its scale slot
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
      tc_commit(tfull_bar);
      ++local;
    }
    tc_commit(drain_bar);
    mbar_wait_bounded(drain_bar, 0, nullptr, args.limit_ns, args.err);
  } else if (warp >= EPI_WARP0) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                         // TMEM lane quadrant
    const int row_in_tile = q * 32 + lane;
    int local = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile T = sched_tile(sched, t);
      const int e = T.e, n_tile = T.n_tile;
      int ok = 0;
      if (lane == 0)
        ok = mbar_wait_bounded(tfull_bar, local & 1, abort_flag, args.limit_ns, args.err);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      // rows past the expert's segment (a partial last m-tile) are not stored
      const bool live = row_in_tile < T.rows;
      const size_t row = (size_t)T.row0 + row_in_tile;
      mx_row_epilogue<MX8, FUSE>(tmem_base + ((uint32_t)(q * 32) << 16), row, live, args.ep, e,
                                 n_tile, args.I, args.ue8m0 != 0, args.zq, args.zs, args.out,
                                 args.ldo, N, [&] {
                                   tc_fence_before();   // the accumulator is read: hand it back
                                   __syncwarp();
                                   if (lane == 0) mbar_arrive(tempty_bar);
                                 });
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

}  // namespace

namespace {
template <int SRC, bool MX8, bool FUSE>
void launch_form(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmS,
                 const Mx4Args& a, cudaStream_t stream) {
  // a failed opt-in shows as the launch's error (cudaGetLastError in the caller)
  static DeviceOnce attr;
  (void)attr.call([] {
    return cudaFuncSetAttribute(k_ggemm_mxfp4<SRC, MX8, FUSE>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  k_ggemm_mxfp4<SRC, MX8, FUSE><<<num_sms(), NUM_THREADS, SMEM_BYTES, stream>>>(tmA, tmB, tmS, a);
}
template <bool FUSE>
void launch_forms(int src, bool mx8, const CUtensorMap& tmA, const CUtensorMap& tmB,
                  const CUtensorMap& tmS, const Mx4Args& a, cudaStream_t stream) {
  if (src == SRC_PACKED)
    mx8 ? launch_form<SRC_PACKED, true, FUSE>(tmA, tmB, tmS, a, stream)
        : launch_form<SRC_PACKED, false, FUSE>(tmA, tmB, tmS, a, stream);
  else if (src == SRC_STAGED)
    mx8 ? launch_form<SRC_STAGED, true, FUSE>(tmA, tmB, tmS, a, stream)
        : launch_form<SRC_STAGED, false, FUSE>(tmA, tmB, tmS, a, stream);
  else
    mx8 ? launch_form<SRC_REGS, true, FUSE>(tmA, tmB, tmS, a, stream)
        : launch_form<SRC_REGS, false, FUSE>(tmA, tmB, tmS, a, stream);
}
}  // namespace

cudaError_t launch_ggemm_mxfp4(const void* A, const float* a_scale, int cap, int K, const void* B,
                               const uint8_t* b_scale, int b_rows_total, int b_rows_per_expert,
                               int n_out, const int32_t* block_expert_ids,
                               const int32_t* num_post_padded, void* out, bool b_e4m3,
                               const Epilogue& ep, cudaStream_t stream, float* z_scale,
                               bool fuse_act, bool ue8m0, bool scales_prepacked, int blk_rows) {
  if (cap <= 0) return cudaSuccess;
  if (blk_rows <= 0 || blk_rows > BM || cap % blk_rows != 0) return cudaErrorInvalidValue;
  // packed E2M1 tensor maps want 32-byte aligned bases, byte maps 16; bulk
  // copies of prepacked scales 16
  if ((reinterpret_cast<uintptr_t>(B) & (b_e4m3 ? 15u : 31u)) != 0 ||
      (reinterpret_cast<uintptr_t>(b_scale) & (scales_prepacked ? 15u : 3u)))
    return cudaErrorInvalidValue;
  if (scales_prepacked && (b_rows_per_expert % 128 != 0 || K % 128 != 0))
    return cudaErrorInvalidValue;
  // fused GEMM1: B rows per expert = 2I (gate then up), I a multiple of 128
  if (fuse_act && (z_scale == nullptr || b_rows_per_expert % 256 != 0 ||
                   n_out != b_rows_per_expert))
    return cudaErrorInvalidValue;
  CUtensorMap tmA, tmB;
  if (!make_tmap_k_sw128(&tmA, A, (uint64_t)cap, (uint64_t)K, 1, 128) ||
      !(b_e4m3 ? make_tmap_k_sw128(&tmB, B, (uint64_t)b_rows_total, (uint64_t)K, 1, 128)
               : make_tmap_fp4_k_sw128(&tmB, B, (uint64_t)b_rows_total, (uint64_t)K, 128)))
    return cudaErrorInvalidValue;
  Mx4Args a;
  a.ep = ep;
  a.block_expert_ids = block_expert_ids;
  a.num_post_padded = num_post_padded;
  a.a_scale = a_scale;
  a.b_scale = b_scale;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ldo = n_out;
  a.num_kb = K / BK;
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
  // weight scales: prepacked operands by bulk copy; else staged by TMA when
  // their rows are 16-byte multiples; else loaded to registers
  const bool staged = !scales_prepacked && K % 512 == 0 &&
                      (reinterpret_cast<uintptr_t>(b_scale) & 15u) == 0;
  const int src = scales_prepacked ? SRC_PACKED : (staged ? SRC_STAGED : SRC_REGS);
  CUtensorMap tmS = tmB;        // used by the staged form only
  if (staged && !make_tmap_u8_rows(&tmS, b_scale, (uint64_t)b_rows_total, (uint64_t)(K / 32), 16,
                                   fuse_act ? 128 : BN))
    return cudaErrorInvalidValue;
  if (fuse_act)
    launch_forms<true>(src, b_e4m3, tmA, tmB, tmS, a, stream);
  else
    launch_forms<false>(src, b_e4m3, tmA, tmB, tmS, a, stream);
  return cudaGetLastError();
}

namespace {
// One thread per (expert, K block, 128-row group, lane l): the 16 bytes of
// operand row l -- the E8M0 bytes of rows l, l + 32, l + 64, l + 96 of the
// group for the K block's 4 chunks of 32, row r's 4 bytes at 4 (r / 32).
__global__ void k_prepack_mx_scales(const uint8_t* __restrict__ scale, int E, int N, int K,
                                    uint4* __restrict__ packed) {
  const int KB = K / 128, G = N / 128, KQ = K / 32;
  const size_t total = (size_t)E * KB * G * 32;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int l = (int)(i % 32);
    size_t r = i / 32;
    const int g = (int)(r % G);
    r /= G;
    const int kb = (int)(r % KB);
    const int e = (int)(r / KB);
    uint32_t w[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const size_t row = (size_t)e * N + (size_t)g * 128 + l + 32 * c;
      w[c] = *reinterpret_cast<const uint32_t*>(scale + row * KQ + 4 * kb);
    }
    packed[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}
}  // namespace

cudaError_t launch_prepack_mx_scales(const uint8_t* scale, int E, int N, int K, void* packed,
                                     cudaStream_t stream) {
  if (E <= 0) return cudaSuccess;
  const size_t total = (size_t)E * (K / 128) * (N / 128) * 32;
  const int threads = 256;
  const size_t want = (total + threads - 1) / threads;
  const int grid = (int)std::min<size_t>(want, (size_t)num_sms() * 8);
  k_prepack_mx_scales<<<grid, threads, 0, stream>>>(scale, E, N, K,
                                                      static_cast<uint4*>(packed));
  return cudaGetLastError();
}

}  // namespace moe
