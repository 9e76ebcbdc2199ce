// Pieces shared by the block-scaled (E8M0 per 32) grouped GEMMs, on one SM
// (gemm_mxfp4.cu) and on SM pairs (gemm_mx_2sm.cu): the activation-scale
// words of the MMA's scale operand, and the epilogue of one accumulator row.
#pragma once

#include "e4m3_pack.cuh"
#include "moe_common.cuh"

namespace moe {

// Activation scales of 4 K blocks for this lane's rows (lane + 32 c):
// W4A8: one fp32 per K block (a 1x128 group covers the 4 chunks of 32);
// MXFP8: four fp32 per K block (one per 1x32 chunk).
template <bool MX8>
struct AGroup {
  float4 v[4][MX8 ? 4 : 1];
};
// Loads the scales of K blocks g .. g+3 (those past num_kb read as 2^0) of
// this lane's rows lane + 32 c of the m-tile starting at tile_row0; rows at
// or past `rows` (past the expert's segment: their results are not stored)
// read the tile's first row instead, inside the buffer.
template <bool MX8>
__device__ __forceinline__ void load_ascales(AGroup<MX8>& A, const float* a_scale,
                                             size_t tile_row0, int rows, int lane, int num_kb,
                                             int g) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const size_t row = tile_row0 + (lane + 32 * c < rows ? lane + 32 * c : 0);
    if constexpr (MX8) {
      const float* pa = a_scale + row * (size_t)(4 * num_kb);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        A.v[c][j] = g + j < num_kb ? __ldg(reinterpret_cast<const float4*>(pa + 4 * (g + j)))
                                   : make_float4(1.0f, 1.0f, 1.0f, 1.0f);
    } else {
      const float* pa = a_scale + row * (size_t)num_kb + g;
      const int n = num_kb - g;
      if ((num_kb & 3) == 0)
        A.v[c][0] = __ldg(reinterpret_cast<const float4*>(pa));
      else
        A.v[c][0] = make_float4(__ldg(pa), n > 1 ? __ldg(pa + 1) : 1.0f,
                                n > 2 ? __ldg(pa + 2) : 1.0f, n > 3 ? __ldg(pa + 3) : 1.0f);
    }
  }
}
// a power-of-two fp32 scale 2^(x-127) has biased exponent x = its E8M0 code
__device__ __forceinline__ uint32_t e8m0_of(float s) { return (__float_as_uint(s) >> 23) & 0xFFu; }
// The scale word of row c for K block j of the group: byte q for chunk q.
template <bool MX8>
__device__ __forceinline__ uint32_t a_word(const AGroup<MX8>& A, int c, int j) {
  if constexpr (MX8) {
    const float4 f = A.v[c][j];
    return e8m0_of(f.x) | e8m0_of(f.y) << 8 | e8m0_of(f.z) << 16 | e8m0_of(f.w) << 24;
  } else {
    const float4 f = A.v[c][0];
    return e8m0_of(j == 0 ? f.x : j == 1 ? f.y : j == 2 ? f.z : f.w) * 0x01010101u;
  }
}

// Epilogue of one row of a 128 x 256 fp32 accumulator tile, one thread per
// row: taddr is the tensor-memory address of the row's lane quadrant at
// column 0 (the warp reads its 32 rows).  release() is called by the whole
// warp once its last read of the accumulator is done (the tile's MMAs for
// the next tile may then overwrite it).
//  FUSE (GEMM1 with the activation): columns [0, 128) hold the row's gate
//    sums of n-block n_tile, [128, 256) the matching up sums; each is rounded
//    to bf16 as a stored H1 would be (all of them read before the
//    accumulator is released), z = act(g, u) in fp32 (as act_mul_quant
//    computes it), then e4m3 codes with one scale per group of 32 (MXFP8) or
//    128 columns into zq [rows, I] / zs [rows, I / group].
//  otherwise: bf16((sum + bias) * router weight) into out [rows, ldo], 256
//    columns of n-tile n_tile, or 128 when N - 256 n_tile == 128.
// Rows that are not live (past the expert's segment) are read, not stored.
template <bool MX8, bool FUSE, class Release>
__device__ __forceinline__ void mx_row_epilogue(uint32_t taddr, size_t row, bool live,
                                                const Epilogue& ep, int e, int n_tile, int I,
                                                bool ue8m0, uint8_t* zq, float* zs,
                                                __nv_bfloat16* out, int ldo, int N,
                                                Release&& release) {
  constexpr int BN = 256;
  if constexpr (FUSE) {
    const int gcol0 = n_tile * 128, ucol0 = I + n_tile * 128;
    const bool bias = ep.bias != nullptr;
    uint4* zdst = reinterpret_cast<uint4*>(zq + row * (size_t)I + (size_t)gcol0);
    constexpr int ZG = MX8 ? 32 : 128;                  // quantisation group
    float* zs_row = zs + row * (size_t)(I / ZG) + (size_t)n_tile * (128 / ZG);
    // First read the whole accumulator row, keeping each (gate, up) pair as
    // the two bf16 roundings the activation takes (what a stored H1 would
    // hold), and hand the accumulator back: the next tile's MMAs then wait
    // only for these loads, not for the activation arithmetic.
    uint32_t w[128];                                   // column c: g low, u high
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t g[32], u[32];
      tmem_ld_32x32b_x32(taddr + c * 32, g);
      tmem_ld_32x32b_x32(taddr + 128 + c * 32, u);
      tmem_ld_wait();
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        float gs = __uint_as_float(g[jj]), us = __uint_as_float(u[jj]);
        if (bias) {
          gs += epi_bias(ep, e, gcol0 + c * 32 + jj);
          us += epi_bias(ep, e, ucol0 + c * 32 + jj);
        }
        w[c * 32 + jj] = bf16x2_bits(__float2bfloat16_rn(gs), __float2bfloat16_rn(us));
      }
    }
    release();                                         // the accumulator is read
    // z = act(g, u) in fp32 (as act_mul_quant computes it), in place
    auto zval = [&](uint32_t gu) {
      return act_glu(ep, __uint_as_float(gu << 16), __uint_as_float(gu & 0xFFFF0000u));
    };
    // 16 codes -> uint4; power-of-two scales: v * (1/s) is the exact quotient
    auto quant16 = [&](const uint32_t* zb, float sc, float rc) {
      float qv[16];
#pragma unroll
      for (int b = 0; b < 16; ++b) {
        const float z = __uint_as_float(zb[b]);
        qv[b] = ue8m0 ? z * rc : quot_rn(z, sc, rc);
      }
      return make_uint4(e4m3x4(qv[0], qv[1], qv[2], qv[3]), e4m3x4(qv[4], qv[5], qv[6], qv[7]),
                        e4m3x4(qv[8], qv[9], qv[10], qv[11]),
                        e4m3x4(qv[12], qv[13], qv[14], qv[15]));
    };
    if constexpr (MX8) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {                    // one 1x32 group per chunk
        float amax = 0.0f;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const float z = zval(w[c * 32 + jj]);
          w[c * 32 + jj] = __float_as_uint(z);
          amax = fmaxf(amax, fabsf(z));
        }
        const float sc = act_scale(amax, ue8m0);
        const float rc = __frcp_rn(sc);
        if (live) {
          zdst[2 * c] = quant16(w + c * 32, sc, rc);
          zdst[2 * c + 1] = quant16(w + c * 32 + 16, sc, rc);
          zs_row[c] = sc;
        }
      }
    } else {
      float amax = 0.0f;
#pragma unroll
      for (int j = 0; j < 128; ++j) {
        const float z = zval(w[j]);
        w[j] = __float_as_uint(z);
        amax = fmaxf(amax, fabsf(z));
      }
      const float sc = act_scale(amax, ue8m0);
      const float rc = __frcp_rn(sc);
      if (live) {
#pragma unroll
        for (int v = 0; v < 8; ++v) zdst[v] = quant16(w + 16 * v, sc, rc);
        zs_row[0] = sc;
      }
    }
  } else {
    const float w = live ? epi_row_weight(ep, row) : 0.0f;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {            // 128 columns at a time
      __nv_bfloat16* out_row = out + row * ldo + (size_t)n_tile * BN + half * 128;
      // 256 columns, or 128 if ragged; live rows only
      const bool store = live && half * 128 < N - n_tile * BN;
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(taddr + half * 128 + c * 32, r[c]);
      tmem_ld_wait();
      if (half == 1) release();                       // the accumulator is read: hand it back
      if (store) {
        const int col0 = n_tile * BN + half * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) epi_store32(ep, e, col0 + 32 * c, w, r[c], out_row + 32 * c);
      }
    }
  }
}

}  // namespace moe
