// quant.cuh -- NVFP4 1x16 block quantization on the device.
//
// Recipe (Megatron-LM PR #8262, "Background" and "What is added"): E2M1
// elements, one E4M3 scale per 16 consecutive elements, round to nearest, no
// 2D blocks / Hadamard transform / stochastic rounding; one fp32 scale per
// token with the global recipe constant 1/(448*6); weights get one fp32 scale
// per expert.  Operation order inside a block (the pages do not print one):
//   sf   = E4M3_rn(fl(fl(amax_b / 6) * enc))
//   r    = fl(enc / dec(sf))            (block of +0 codes when dec(sf) == 0)
//   code = E2M1_rn(fl(v * r))
// All divisions and products are single IEEE operations (__fdiv_rn /
// __fmul_rn), so the result is a deterministic function of the inputs.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace moe {

// Encode scale (2688 / amax) and decode scale (amax * fl(1/2688)).
constexpr float kRecipeMax = 2688.0f;           // 448 * 6
constexpr float kRecipeInv = 1.0f / 2688.0f;    // folded by the compiler, correctly rounded

// Byte offset of block scale (row r, scale column j) in a 128x4-swizzled plane
// whose rows carry c16 = D/16 scale columns (c16 % 4 == 0): 512-byte atoms of
// 128 rows x 4 scale columns, atom byte (r%32)*16 + ((r/32)%4)*4 + (j%4).
__device__ __forceinline__ uint64_t sf_offset(uint64_t r, uint32_t j, uint32_t c16) {
  return ((r >> 7) * (c16 >> 2) + (j >> 2)) * 512u + (r & 31u) * 16u + ((r >> 5) & 3u) * 4u +
         (j & 3u);
}

// Quantize one block of 16 fp32 values with encode scale `enc`.
// Returns the E4M3 scale byte; writes the 8 packed code bytes (element 2i in
// the low nibble) to `codes` as a uint2.
__device__ __forceinline__ uint32_t quant_block16(const float (&v)[16], float enc, uint2& codes) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const float sf_f = __fmul_rn(__fdiv_rn(amax, 6.0f), enc);
  const uint32_t sf = cvt_e4m3(sf_f);
  const float sfd = e4m3_to_f32(sf);
  if (sfd == 0.0f) {
    codes = make_uint2(0u, 0u);
    return sf;
  }
  const float r = __fdiv_rn(enc, sfd);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t byte = cvt_e2m1x2(__fmul_rn(v[2 * i], r), __fmul_rn(v[2 * i + 1], r));
    w[i >> 2] |= byte << (8 * (i & 3));
  }
  codes = make_uint2(w[0], w[1]);
  return sf;
}

// 16 bf16 values (two 16-byte vectors) -> fp32.
__device__ __forceinline__ void bf16x16_to_f32(const uint4& a, const uint4& b, float (&v)[16]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float bf16x8_absmax(const uint4& a) {
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, fabsf(__uint_as_float(w[i] << 16)));
    m = fmaxf(m, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
  }
  return m;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// FC2-input requantization of one activated fp32 row (I values) by one warp:
// per-row NVFP4 with the recipe constant (Megatron-LM PR #8262, "How to
// extend": fc2_input_scale = 1/(448*6)), or with a static encode scale (the
// per-tensor recipe: fc2_input_scale = a2_scale, row scale 1).  Writes the I/2
// code bytes of permuted row p, its block scales into the 128x4-swizzled plane
// and its row scale.  Lane l owns blocks l, l+32, ... (16 consecutive values
// each, 64 contiguous bytes).  A row of up to G * 2048 values is loaded once
// into registers (all its loads in flight together); longer rows are read in
// groups of 128 blocks, twice.  The fused GEMM's requant uses the same
// quant_block16 and amax, so both give the same bits.
template <int G>
__device__ __forceinline__ void requant_group_load(const float4* __restrict__ r4, int b0, int nb,
                                                   int lane, float (&v)[4 * G][16]) {
#pragma unroll
  for (int k = 0; k < 4 * G; ++k) {
    const int b = b0 + lane + 32 * k;
    if (b < nb) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 f = __ldcs(r4 + 4 * b + i);  // streamed: read once
        v[k][4 * i] = f.x;
        v[k][4 * i + 1] = f.y;
        v[k][4 * i + 2] = f.z;
        v[k][4 * i + 3] = f.w;
      }
    }
  }
}
template <int G>
__device__ __forceinline__ void requant_row_warp(const float* __restrict__ row, int I, uint64_t p,
                                                 uint8_t* __restrict__ qc,
                                                 uint8_t* __restrict__ qsf,
                                                 float* __restrict__ qs,
                                                 const float* __restrict__ static_enc, int lane) {
  constexpr int kGroup = 128 * G;  // blocks held in registers at once
  const float4* r4 = reinterpret_cast<const float4*>(row);
  const int nb = I / 16;  // a multiple of 16: lanes come in groups of four in range
  const uint32_t c16 = (uint32_t)nb;
  float v[4 * G][16];
  float m = 1.0f;
  if (!static_enc) {
    m = 0.0f;
    for (int b0 = 0; b0 < nb; b0 += kGroup) {
      requant_group_load<G>(r4, b0, nb, lane, v);
#pragma unroll
      for (int k = 0; k < 4 * G; ++k)
        if (b0 + lane + 32 * k < nb) {
#pragma unroll
          for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[k][i]));
        }
    }
    m = warp_max(m);
  }
  uint2* crow = reinterpret_cast<uint2*>(qc + p * (uint64_t)(I / 2));
  if (m == 0.0f) {
    for (int b = lane; b < nb; b += 32) {
      crow[b] = make_uint2(0u, 0u);
      if ((b & 3) == 0) *reinterpret_cast<uint32_t*>(qsf + sf_offset(p, b, c16)) = 0u;
    }
    if (lane == 0) qs[p] = 0.0f;
    return;
  }
  const float enc = static_enc ? *static_enc : __fdiv_rn(kRecipeMax, m);
  for (int b0 = 0; b0 < nb; b0 += kGroup) {
    // a row of one group (and the static-scale path) is still in registers
    if (nb > kGroup || static_enc) requant_group_load<G>(r4, b0, nb, lane, v);
#pragma unroll
    for (int k = 0; k < 4 * G; ++k) {
      const int b = b0 + lane + 32 * k;
      uint32_t sfb = 0;
      if (b < nb) {
        uint2 q;
        sfb = quant_block16(v[k], enc, q);
        crow[b] = q;
      }
      // a group of four lanes holds four consecutive blocks: one 4-byte store of
      // their scale bytes (consecutive in the swizzled plane)
      const uint32_t w = sfb | (__shfl_down_sync(0xFFFFFFFFu, sfb, 1) << 8) |
                         (__shfl_down_sync(0xFFFFFFFFu, sfb, 2) << 16) |
                         (__shfl_down_sync(0xFFFFFFFFu, sfb, 3) << 24);
      if ((lane & 3) == 0 && b < nb) *reinterpret_cast<uint32_t*>(qsf + sf_offset(p, b, c16)) = w;
    }
  }
  if (lane == 0) qs[p] = static_enc ? 1.0f : __fmul_rn(m, kRecipeInv);
}

}  // namespace moe
