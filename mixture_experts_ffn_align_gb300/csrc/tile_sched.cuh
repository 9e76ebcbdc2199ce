// Tile order of the persistent grouped GEMMs.
//
// The padded layout puts each expert's rows in one segment of consecutive
// blocks (block_size rows each: 16, 32, 64 or 128), segments in expert order.
// The GEMMs compute 128-row m-tiles: each expert's segment is cut into
// ceil(rows / 128) m-tiles from its first row, so an m-tile never mixes two
// experts; when the block size is below 128 the last m-tile of a segment may
// be partial, and its rows past the segment (the next expert's, or none) are
// computed but never stored.  With 128-row blocks the m-tiles are the blocks.
//
// Tiles are numbered expert by expert: all (m-tile, n-tile) pairs of one
// expert, n-tile major with the expert's m-tiles inner, before the next
// expert.  CTAs that run at the same time then share one expert: every weight
// tile is fetched by all of that expert's m-tiles within a few microseconds
// (one DRAM read, the rest hit L2) and the expert's activation rows stay in
// L2 across all its n-tiles.  An expert with more m-tiles than `group_max`
// (whose activations would not fit the L2 budget) is split into chunks of at
// most `group_max` m-tiles.
//
// Every CTA derives the segments from block_expert_ids itself at kernel
// start, so the scheduler needs no extra input from the host.
#pragma once

#include <stdint.h>

namespace moe {

constexpr int kSchedMaxRuns = 1025;     // segments <= E <= 1024
// Shared memory of the schedule: a header, then the m-tile prefix [runs + 1],
// first row, end row and expert of each segment.
constexpr int kSchedBytes = 16 + 4 * (4 * kSchedMaxRuns + 1);

struct TileSched {
  const int* mt0;    // first m-tile of each segment; mt0[nruns] = m-tiles in all
  const int* row0;   // first row of each segment
  const int* rend;   // end row (exclusive) of each segment
  const int* exp;    // expert of each segment
  int nruns;
  int n_tiles;
  int group_max;
};

// One tile: rows [row0, row0 + rows) of expert e (rows <= 128), column tile
// n_tile; run / mt_local locate the m-tile inside its segment.
struct Tile {
  int e, row0, rows, n_tile, run, mt_local;
};

// Builds the schedule from the block ids of `nb` blocks of blk_rows rows.
// mem: kSchedBytes of shared memory kept for the kernel's life; scratch:
// 2 * num_experts ints of shared memory that are free until this returns (the
// pipeline stages).  Every thread of the CTA must call it; it contains
// __syncthreads.  Block ids outside [0, num_experts) are skipped; rows stay
// inside [0, nb * blk_rows) whatever the ids hold.
__device__ __forceinline__ TileSched sched_build(const int32_t* __restrict__ block_ids, int nb,
                                                 int blk_rows, int num_experts, int* mem,
                                                 int* scratch, int n_tiles, int group_max) {
  int* hdr = mem;
  int* mt0 = mem + 4;
  int* row0 = mt0 + kSchedMaxRuns + 1;
  int* rend = row0 + kSchedMaxRuns;
  int* exp = rend + kSchedMaxRuns;
  int* s_first = scratch;
  int* s_end = scratch + num_experts;
  for (int e = threadIdx.x; e < num_experts; e += blockDim.x) {
    s_first[e] = -1;
    s_end[e] = -1;
  }
  __syncthreads();
  for (int b = threadIdx.x; b < nb; b += blockDim.x) {
    const int e = block_ids[b];
    if (e < 0 || e >= num_experts) continue;
    if (b == 0 || block_ids[b - 1] != e) s_first[e] = b;
    if (b + 1 == nb || block_ids[b + 1] != e) s_end[e] = b + 1;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int nr = 0, mt = 0;
    for (int base = 0; base < num_experts; base += 32) {
      const int e = base + lane;
      const int f = e < num_experts ? s_first[e] : -1;
      const int en = e < num_experts ? s_end[e] : -1;
      const bool has = f >= 0 && en > f;
      const int cnt = has ? ((en - f) * blk_rows + 127) / 128 : 0;
      const unsigned m = __ballot_sync(0xffffffffu, has);
      int inc = cnt;                                   // inclusive scan of the m-tiles
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      if (has) {
        const int r = nr + __popc(m & ((1u << lane) - 1u));
        mt0[r] = mt + inc - cnt;
        row0[r] = f * blk_rows;
        rend[r] = en * blk_rows;
        exp[r] = e;
      }
      nr += __popc(m);
      mt += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) {
      mt0[nr] = mt;
      hdr[0] = nr;
    }
  }
  __syncthreads();
  TileSched s;
  s.mt0 = mt0;
  s.row0 = row0;
  s.rend = rend;
  s.exp = exp;
  s.nruns = hdr[0];
  s.n_tiles = n_tiles;
  s.group_max = group_max;
  return s;
}

// m-tiles of the whole schedule (tiles = m-tiles * n_tiles).
__device__ __forceinline__ int sched_mtiles(const TileSched& s) { return s.mt0[s.nruns]; }

// Segment holding global m-tile q.
__device__ __forceinline__ int sched_run_of(const TileSched& s, int q) {
  int lo = 0, hi = s.nruns - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s.mt0[mid] <= q) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Rows of m-tile mt_local of segment r.
__device__ __forceinline__ void sched_rows(const TileSched& s, int r, int mt_local, int& row0,
                                           int& rows) {
  row0 = s.row0[r] + 128 * mt_local;
  rows = min(128, s.rend[r] - row0);
}

// Tile t (0 <= t < sched_mtiles * n_tiles).
__device__ __forceinline__ Tile sched_tile(const TileSched& s, int t) {
  Tile T;
  const int q = t / s.n_tiles;            // mt0[r] <= q < mt0[r + 1] for the owning segment
  const int r = sched_run_of(s, q);
  const int m0 = s.mt0[r], nm = s.mt0[r + 1] - m0;
  const int local = t - m0 * s.n_tiles;
  const int chunk_tiles = s.group_max * s.n_tiles;
  const int c = local / chunk_tiles;
  const int gm = min(s.group_max, nm - c * s.group_max);
  const int l2 = local - c * chunk_tiles;
  T.n_tile = l2 / gm;
  T.mt_local = c * s.group_max + (l2 - T.n_tile * gm);
  T.run = r;
  T.e = s.exp[r];
  sched_rows(s, r, T.mt_local, T.row0, T.rows);
  return T;
}

// SM-pair schedules (the cta_group::2 GEMMs): the m-tiles of each segment go
// two by two, a lone last one paired with itself.  pairs: kSchedMaxRuns + 1
// ints of shared memory, the prefix of pairs per segment; thread 0 fills it,
// so a __syncthreads must follow before it is read.
__device__ __forceinline__ void sched_pairs_build(const TileSched& s, int* pairs) {
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int r = 0; r < s.nruns; ++r) {
      pairs[r] = acc;
      acc += (s.mt0[r + 1] - s.mt0[r] + 1) >> 1;
    }
    pairs[s.nruns] = acc;
  }
}

// Pair tile t (0 <= t < pairs[nruns] * n_tiles): expert e, the leader's
// m-tile at row0, the peer's at row1 (== row0 for a lone m-tile, !has1),
// column tile n_tile.  Tiles walk segment by segment, n-tile major.
struct PairTile {
  int e, row0, row1, n_tile;
  bool has1;
};
__device__ __forceinline__ PairTile sched_pair_tile(const TileSched& s, const int* pairs,
                                                    int t) {
  PairTile P;
  const int q = t / s.n_tiles;
  int lo = 0, hi = s.nruns - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pairs[mid] <= q) lo = mid; else hi = mid - 1;
  }
  const int np = pairs[lo + 1] - pairs[lo];
  const int local = t - pairs[lo] * s.n_tiles;
  P.n_tile = local / np;
  const int m0 = 2 * (local - P.n_tile * np);               // m-tile inside the segment
  P.has1 = s.mt0[lo] + m0 + 1 < s.mt0[lo + 1];
  P.e = s.exp[lo];
  P.row0 = s.row0[lo] + 128 * m0;
  P.row1 = P.has1 ? P.row0 + 128 : P.row0;
  return P;
}

// m-tiles of 128 rows x K elements of `elem_bytes` that fit the L2 budget.
inline int sched_group_max(int K, int elem_bytes) {
#ifndef MOE_GEMM_GROUP_BYTES
#define MOE_GEMM_GROUP_BYTES (48ll << 20)
#endif
  const long long blk = 128ll * K * elem_bytes;
  const long long g = MOE_GEMM_GROUP_BYTES / blk;
  return (int)(g < 1 ? 1 : (g > 1 << 20 ? 1 << 20 : g));
}

}  // namespace moe
