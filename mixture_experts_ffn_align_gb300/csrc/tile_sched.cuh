// Tile order of the persistent grouped GEMMs.
//
// The padded layout puts each expert's rows in consecutive 128-row blocks.
// Tiles are numbered expert by expert: all (m-block, n-tile) pairs of one
// expert, n-tile major with the expert's m-blocks inner, before the next
// expert.  CTAs that run at the same time then share one expert: every weight
// tile is fetched by all of that expert's m-blocks within a few microseconds
// (one DRAM read, the rest hit L2) and the expert's activation blocks stay in
// L2 across all its n-tiles.  An expert with more m-blocks than `group_max`
// (whose activations would not fit the L2 budget) is split into chunks of at
// most `group_max` blocks.
//
// Every CTA derives the expert runs from block_expert_ids itself at kernel
// start (block ids staged in shared memory, one warp finds the run starts
// with ballots), so the scheduler needs no extra input from the host.
#pragma once

#include <stdint.h>

namespace moe {

constexpr int kSchedMaxBlocks = 4096;   // >= m_sum bound / 128 for every valid problem
constexpr int kSchedMaxRuns = 1025;     // <= E + 1

struct TileSched {
  const int* runs;   // shared: first block of each run; runs[nruns] = nb_valid
  int nruns;
  int n_tiles;
  int group_max;
};

// Stage block ids (all threads) and compute the runs (warp 0).  Must be called
// by every thread of the CTA; contains two __syncthreads.
__device__ __forceinline__ int sched_build(const int32_t* __restrict__ block_ids, int nb_valid,
                                           int* s_ids, int* s_runs, int* s_nruns) {
  for (int b = threadIdx.x; b < nb_valid; b += blockDim.x) s_ids[b] = block_ids[b];
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int count = 0;
    for (int base = 0; base < nb_valid; base += 32) {
      const int b = base + lane;
      const bool start = b < nb_valid && (b == 0 || s_ids[b] != s_ids[b - 1]);
      const unsigned m = __ballot_sync(0xffffffffu, start);
      if (start) s_runs[count + __popc(m & ((1u << lane) - 1u))] = b;
      count += __popc(m);
    }
    if (lane == 0) {
      s_runs[count] = nb_valid;
      *s_nruns = count;
    }
  }
  __syncthreads();
  return *s_nruns;
}

// Tile t (0 <= t < nb_valid * n_tiles) -> (m-block, n-tile).
__device__ __forceinline__ void sched_tile(const TileSched& s, int t, int& m_blk, int& n_tile) {
  const int q = t / s.n_tiles;          // runs[r] <= q < runs[r + 1] for the owning run
  int lo = 0, hi = s.nruns - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s.runs[mid] <= q) lo = mid; else hi = mid - 1;
  }
  const int b0 = s.runs[lo], nb = s.runs[lo + 1] - b0;
  const int local = t - b0 * s.n_tiles;
  const int chunk_tiles = s.group_max * s.n_tiles;
  const int c = local / chunk_tiles;
  const int gm = min(s.group_max, nb - c * s.group_max);
  const int l2 = local - c * chunk_tiles;
  n_tile = l2 / gm;
  m_blk = b0 + c * s.group_max + (l2 - n_tile * gm);
}

// Blocks of 128 rows x K elements of `elem_bytes` that fit the L2 budget.
inline int sched_group_max(int K, int elem_bytes) {
#ifndef MOE_GEMM_GROUP_BYTES
#define MOE_GEMM_GROUP_BYTES (48ll << 20)
#endif
  const long long blk = 128ll * K * elem_bytes;
  const long long g = MOE_GEMM_GROUP_BYTES / blk;
  return (int)(g < 1 ? 1 : (g > kSchedMaxBlocks ? kSchedMaxBlocks : g));
}

}  // namespace moe
