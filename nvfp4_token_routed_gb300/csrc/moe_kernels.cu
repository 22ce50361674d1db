// moe_kernels.cu -- the bandwidth-bound stages of the routed NVFP4 MoE layer:
// per-token quantization, weight preparation, the routing permutation (count,
// scan, scatter + gather), the FC2-input requantization and the deterministic
// top-k finalize.  Every kernel moves data in 16-byte vectors, one warp per row.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace moe {

// ============================================================== token quantization
// Megatron-LM PR #8262, "What is added": quantize_routed_nvfp4_input quantizes
// activations per token with the recipe constant 1/(448*6) as global scale.
// One warp per token: warp-shuffle amax, then one 16-element block per lane.
// Rows of H values are written with Hp = round_up(H, 256) columns; the blocks
// past H are zero (zero codes, zero scale bytes), which leaves every dot product
// with a zero-padded weight row unchanged (Megatron-LM PR #8262, "Why CuTe DSL":
// hidden sizes are padded to 256).
// With `static_enc` (the per-tensor recipe, Megatron-LM PR #8262, "How to
// extend": nvfp4_quantize(x, a1_scale) with a fixed scale tensor) every row uses
// that encode scale and no per-token scale is written.
// Rows of up to 512 * NB values (NB blocks of 16 per lane) are loaded once into
// registers, all their loads in flight together; longer rows are read twice.
// NB: blocks of 16 values a lane holds in registers (0: rows of any length, read
// twice); S: warps sharing a row (S = 2 halves the registers a warp needs for
// rows of 4097-8192 values, so that twice the rows are in flight).
template <int NB, int S>
__global__ void __launch_bounds__(256) quantize_tokens_kernel(int T, int H, int Hp,
                                                              const uint4* __restrict__ x,
                                                              uint8_t* __restrict__ codes,
                                                              uint8_t* __restrict__ sf,
                                                              float* __restrict__ scale,
                                                              const float* __restrict__ static_enc) {
  __shared__ float s_max[8];
  pdl_wait();
  pdl_trigger();
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int t = gw / S;          // row; warp gw % S of its S holds its blocks lane + 32 (S j + part)
  const int part = gw % S;
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const uint4* row = x + (size_t)t * (H / 8);
  const int nb = H / 16;
  if (NB > 0 && nb <= 32 * NB * S) {
    // lane l holds blocks l + 32 (S j + part): two 16-byte vectors each
    uint4 r[NB > 0 ? NB : 1][2];
    float m = 0.0f;
    if (t < T) {
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        const int b = lane + 32 * (S * j + part);
        if (b < nb) {
          r[j][0] = __ldcs(row + 2 * b);
          r[j][1] = __ldcs(row + 2 * b + 1);
        }
      }
#pragma unroll
      for (int j = 0; j < NB; ++j)
        if (lane + 32 * (S * j + part) < nb)
          m = fmaxf(m, fmaxf(bf16x8_absmax(r[j][0]), bf16x8_absmax(r[j][1])));
    }
    m = warp_max(m);
    if (S > 1) {
      // the row's warps are neighbours in the block: exchange their maxima
      if (lane == 0) s_max[wib] = m;
      __syncthreads();
#pragma unroll
      for (int i = 0; i < S; ++i) m = fmaxf(m, s_max[(wib / S) * S + i]);
    }
    if (t >= T) return;
    if (static_enc) m = 1.0f;  // any non-zero value: the static path quantizes every real block
    uint2* crow = reinterpret_cast<uint2*>(codes + (size_t)t * (Hp / 2));
    uint8_t* srow = sf + (size_t)t * (Hp / 16);
    for (int b = (m == 0.0f ? 0 : nb) + lane + 32 * part; b < Hp / 16; b += 32 * S) {
      crow[b] = make_uint2(0u, 0u);
      srow[b] = 0;
    }
    if (m == 0.0f) {
      if (lane == 0 && part == 0) scale[t] = 0.0f;
      return;
    }
    const float enc = static_enc ? *static_enc : __fdiv_rn(kRecipeMax, m);
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int b = lane + 32 * (S * j + part);
      if (b < nb) {
        float v[16];
        bf16x16_to_f32(r[j][0], r[j][1], v);
        uint2 q;
        srow[b] = (uint8_t)quant_block16(v, enc, q);
        crow[b] = q;
      }
    }
    if (lane == 0 && part == 0 && !static_enc) scale[t] = __fmul_rn(m, kRecipeInv);
    return;
  }
  if (S > 1 || t >= T) return;  // (S > 1 launches only when rows fit the registers)
  float m = 1.0f;  // any non-zero value: the static path quantizes every real block
  if (!static_enc) {
    m = 0.0f;
    for (int i = lane; i < H / 8; i += 32) m = fmaxf(m, bf16x8_absmax(__ldg(row + i)));
    m = warp_max(m);
  }
  uint2* crow = reinterpret_cast<uint2*>(codes + (size_t)t * (Hp / 2));
  uint8_t* srow = sf + (size_t)t * (Hp / 16);
  for (int b = (m == 0.0f ? 0 : H / 16) + lane; b < Hp / 16; b += 32) {
    crow[b] = make_uint2(0u, 0u);
    srow[b] = 0;
  }
  if (m == 0.0f) {
    if (lane == 0) scale[t] = 0.0f;
    return;
  }
  const float enc = static_enc ? *static_enc : __fdiv_rn(kRecipeMax, m);
  for (int b = lane; b < H / 16; b += 32) {
    float v[16];
    bf16x16_to_f32(__ldg(row + 2 * b), __ldg(row + 2 * b + 1), v);
    uint2 q;
    srow[b] = (uint8_t)quant_block16(v, enc, q);
    crow[b] = q;
  }
  if (lane == 0 && !static_enc) scale[t] = __fmul_rn(m, kRecipeInv);
}

void launch_quantize_tokens(int T, int H, int Hp, const void* x, uint8_t* codes, uint8_t* sf,
                            float* scale, const float* static_enc, cudaStream_t s) {
  const int warps = 8;
  // rows of up to 2048 values: one warp, 4 blocks a lane; up to 8192: two warps
  // per row, 8 blocks a lane each; beyond: one warp, the row read twice
  const int S = H <= 2048 ? 1 : H <= 8192 ? 2 : 1;
  const int blocks = (int)(((int64_t)T * S + warps - 1) / warps);
  auto* k = H <= 2048 ? quantize_tokens_kernel<4, 1>
                      : H <= 8192 ? quantize_tokens_kernel<8, 2> : quantize_tokens_kernel<0, 1>;
  launch_pdl(k, dim3(blocks), dim3(warps * 32), 0, s, T, H, Hp, static_cast<const uint4*>(x),
             codes, sf, scale, static_enc);
}

// ============================================================== weight preparation
// Megatron-LM PR #8262, "What is added": prepare_routed_nvfp4_weights -> packed
// E2M1, 128x4-swizzled E4M3 block scales, one fp32 alpha per expert; "How to
// extend": alpha = 1 / w_scale.  Stage 1: per-expert amax (order-free max,
// accumulated as the bit pattern of a non-negative float into alpha[]).
__global__ void __launch_bounds__(256) expert_amax_kernel(const uint4* __restrict__ w,
                                                          int64_t vec_per_expert,
                                                          uint32_t* __restrict__ amax_bits) {
  const int e = blockIdx.y;
  const uint4* base = w + (size_t)e * vec_per_expert;
  float m = 0.0f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < vec_per_expert;
       i += (int64_t)gridDim.x * blockDim.x)
    m = fmaxf(m, bf16x8_absmax(__ldg(base + i)));
  m = warp_max(m);
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) r = fmaxf(r, red[i]);
    atomicMax(amax_bits + e, __float_as_uint(r));
  }
}

// Stage 2: one warp per stored row.  The source [N][D] rows are stored as
// [Np][Dp] with zero rows and zero blocks past the source (padding to 256,
// Megatron-LM PR #8262, "Why CuTe DSL"); SwiGLU pads each half separately.  For
// SwiGLU the stored FC1 row order interleaves 64-row blocks [gate f0..f0+63 |
// up f0..f0+63] of the padded halves, so one 128-row GEMM tile holds matching
// gate and up rows; canonical order is [gate; up].
__global__ void __launch_bounds__(256) quantize_weights_kernel(
    const uint4* __restrict__ w, int E, int N, int D, int Np, int Dp, int swiglu_I,
    const uint32_t* __restrict__ amax_bits, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ sf, uint64_t sf_expert_bytes) {
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= (int64_t)E * Np) return;
  const int e = (int)(gw / Np);
  const int ir = (int)(gw % Np);
  int src = ir < N ? ir : -1;  // source row of stored row ir, -1 for a padding row
  if (swiglu_I > 0) {
    const int b = ir >> 6;
    const int half = b & 1, f = (b >> 1) * 64 + (ir & 63);
    src = f < swiglu_I ? half * swiglu_I + f : -1;
  }
  const float amax = __uint_as_float(amax_bits[e]);
  uint2* crow = reinterpret_cast<uint2*>(codes + ((size_t)e * Np + ir) * (Dp / 2));
  uint8_t* plane = sf + (size_t)e * sf_expert_bytes;
  const uint32_t c16 = (uint32_t)(Dp / 16);
  const int real_blocks = (amax == 0.0f || src < 0) ? 0 : D / 16;
  for (int b = real_blocks + lane; b < Dp / 16; b += 32) {
    crow[b] = make_uint2(0u, 0u);
    plane[sf_offset(ir, b, c16)] = 0;
  }
  if (real_blocks == 0) return;
  const uint4* row = w + ((size_t)e * N + src) * (D / 8);
  const float enc = __fdiv_rn(kRecipeMax, amax);
  for (int b = lane; b < D / 16; b += 32) {
    float v[16];
    bf16x16_to_f32(__ldg(row + 2 * b), __ldg(row + 2 * b + 1), v);
    uint2 q;
    plane[sf_offset(ir, b, c16)] = (uint8_t)quant_block16(v, enc, q);
    crow[b] = q;
  }
}

// Stage 3: alpha = 1 / w_scale with w_scale = 2688 / amax (0 for an all-zero
// expert); with a static input scale a (per-tensor recipe, "How to extend":
// fc_alpha = 1 / (w_scale * a_scale)) alpha = 1 / (w_scale * a).
__global__ void expert_alpha_kernel(int E, float* alpha, const float* a_scale) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const float amax = alpha[e];  // still holds the amax bit pattern
  const float w_scale = __fdiv_rn(kRecipeMax, amax);
  alpha[e] = amax == 0.0f ? 0.0f
                          : __fdiv_rn(1.0f, a_scale ? __fmul_rn(w_scale, *a_scale) : w_scale);
}

void launch_prepare_fc(int E, int N, int D, int Np, int Dp, int swiglu_I, const void* w,
                       uint8_t* codes, uint8_t* sf, float* alpha, const float* a_scale,
                       cudaStream_t s) {
  cudaMemsetAsync(alpha, 0, sizeof(float) * E, s);
  const int64_t vec = (int64_t)N * D / 8;
  int bx = (int)((vec + 256 * 8 - 1) / (256 * 8));
  if (bx > 64) bx = 64;
  expert_amax_kernel<<<dim3(bx, E), 256, 0, s>>>(static_cast<const uint4*>(w), vec,
                                                 reinterpret_cast<uint32_t*>(alpha));
  const int64_t warps = (int64_t)E * Np;
  const uint64_t sf_bytes = (uint64_t)Np * (Dp / 16);  // Np % 128 == 0 and Dp/16 % 4 == 0: no pad
  quantize_weights_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(
      static_cast<const uint4*>(w), E, N, D, Np, Dp, swiglu_I,
      reinterpret_cast<const uint32_t*>(alpha), codes, sf, sf_bytes);
  expert_alpha_kernel<<<(E + 255) / 256, 256, 0, s>>>(E, alpha, a_scale);
}

// ============================================================== routing permutation
// Stable counting sort of the (token, slot) routes by expert: per-chunk
// histograms, a per-expert scan over chunks plus an exclusive scan of the
// 128-row-padded group sizes, a stable scatter of the route ids, then a gather
// of the token rows into expert-contiguous order.
constexpr int kChunk = 256;

// Expert id of route idx from int32 ids, or from int64 ids ([FI] Tensor and
// numerical contract: signed int32/int64 ids) read as two words; an int64 value
// outside the int32 range is returned as -2, an invalid id.
__device__ __forceinline__ int load_id(const int32_t* __restrict__ ids, int idx, int ids64) {
  if (!ids64) return ids[idx];
  const int2 v = reinterpret_cast<const int2*>(ids)[idx];
  return v.y == (v.x >> 31) ? v.x : -2;
}

__global__ void __launch_bounds__(kChunk) route_count_kernel(const int32_t* __restrict__ ids,
                                                             int ids64, int TK, int E,
                                                             int32_t* __restrict__ chunk_counts) {
  extern __shared__ int s_cnt[];
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < E; i += blockDim.x) s_cnt[i] = 0;
  __syncthreads();
  const int idx = blockIdx.x * kChunk + threadIdx.x;
  int bad = 0;
  if (idx < TK) {
    const int e = load_id(ids, idx, ids64);
    if (e >= 0 && e < E)
      atomicAdd(&s_cnt[e], 1);
    else if (e != -1)
      bad = 1;
  }
  bad = __syncthreads_or(bad);
  // row of E counts plus one flag word: the chunk held an id outside [-1, E)
  int32_t* row = chunk_counts + (size_t)blockIdx.x * (E + 1);
  for (int i = threadIdx.x; i < E; i += blockDim.x) row[i] = s_cnt[i];
  if (threadIdx.x == 0) row[E] = bad;
}

__global__ void __launch_bounds__(1024) route_scan_kernel(
    int nchunks, int E, const int32_t* __restrict__ chunk_counts, int32_t* __restrict__ chunk_prefix,
    int32_t* __restrict__ counts, int32_t* __restrict__ group_row0, int4* __restrict__ tiles,
    int32_t* __restrict__ status, int32_t* __restrict__ tile_sync, int tile_sync_words) {
  pdl_wait();
  pdl_trigger();
  // per-token-tile counters of the fused FC1 -> FC2 GEMM start at zero
  for (int i = threadIdx.x; i < tile_sync_words; i += blockDim.x) tile_sync[i] = 0;
  // (1) per-expert exclusive prefix over the chunks: P threads per expert (the
  // largest power of two with E * P <= 1024, P <= 32, adjacent lanes), each
  // summing a contiguous range of chunks, then a scan across the P partial sums
  __shared__ int s_total[1024];
  {
    int P = 1;
    while (P < 32 && E * P * 2 <= (int)blockDim.x) P *= 2;
    const int t = threadIdx.x, ea = t / P, part = t % P;
    const int cs = (nchunks + P - 1) / P;
    const int c0 = min(part * cs, nchunks), c1 = min(c0 + cs, nchunks);
    int local = 0;
    if (ea < E)
      for (int c = c0; c < c1; ++c) local += chunk_counts[(size_t)c * (E + 1) + ea];
    int incl = local;  // inclusive scan across the P parts of this expert
    for (int o = 1; o < P; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o, P);
      if (part >= o) incl += y;
    }
    if (ea < E) {
      int run = incl - local;
      int c = c0;
      for (; c + 4 <= c1; c += 4) {  // four loads in flight ahead of their stores
        int v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = chunk_counts[(size_t)(c + u) * (E + 1) + ea];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          chunk_prefix[(size_t)(c + u) * E + ea] = run;
          run += v[u];
        }
      }
      for (; c < c1; ++c) {
        chunk_prefix[(size_t)c * E + ea] = run;
        run += chunk_counts[(size_t)c * (E + 1) + ea];
      }
      if (part == P - 1) s_total[ea] = incl;
    }
  }
  __syncthreads();
  const int e = threadIdx.x;
  const int total = e < E ? s_total[e] : 0;
  int bad = 0;
  for (int c = e; c < nchunks; c += blockDim.x) bad |= chunk_counts[(size_t)c * (E + 1) + E];
  bad = __syncthreads_or(bad);
  const int ntiles = (total + kTileRows - 1) / kTileRows;
  // block-wide exclusive scan of ntiles, and the largest tile
  __shared__ int warp_sum[32];
  __shared__ int max_rows;
  if (e == 0) max_rows = 0;
  const int lane = e & 31, wid = e >> 5;
  int incl = ntiles;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sum[wid] = incl;
  __syncthreads();
  if (total > 0) atomicMax(&max_rows, min(kTileRows, total));
  if (wid == 0) {
    int v = (lane < (int)(blockDim.x >> 5)) ? warp_sum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, v, o);
      if (lane >= o) v += y;
    }
    warp_sum[lane] = v;  // inclusive over warps
  }
  __syncthreads();
  const int base = incl - ntiles + (wid > 0 ? warp_sum[wid - 1] : 0);
  if (e < E) {
    counts[e] = total;
    group_row0[e] = base * kTileRows;
    for (int j = 0; j < ntiles; ++j) tiles[base + j] = make_int4(e, base, ntiles, total);
  }
  if (e == (int)blockDim.x - 1) {
    status[kStatusFlags] = bad ? kFlagBadExpertId : 0;
    status[kStatusTiles] = base + ntiles;
    status[kStatusRows] = (base + ntiles) * kTileRows;
    status[kStatusMaxRows] = max_rows;
    status[kStatusItemCtr] = 0;
    status[kStatusItemCtr + 1] = 0;
  }
}

__global__ void __launch_bounds__(kChunk) route_scatter_kernel(
    const int32_t* __restrict__ ids, int ids64, int TK, int E,
    const int32_t* __restrict__ chunk_prefix,
    const int32_t* __restrict__ group_row0, int32_t* __restrict__ inv, int32_t* __restrict__ perm) {
  extern __shared__ int s_wcnt[];  // [kChunk/32][E]
  constexpr int kWarps = kChunk / 32;
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) s_wcnt[i] = 0;
  __syncthreads();
  const int idx = blockIdx.x * kChunk + threadIdx.x;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = idx < TK ? load_id(ids, idx, ids64) : -1;
  const bool valid = e >= 0 && e < E;
  // stable rank: earlier lanes of this warp with the same expert, then earlier warps
  const unsigned peers = __match_any_sync(0xFFFFFFFFu, valid ? e : -1);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (valid && rank == 0) s_wcnt[w * E + e] = __popc(peers);
  __syncthreads();
  int p = -1;
  if (valid) {
    int before = 0;
    for (int v = 0; v < w; ++v) before += s_wcnt[v * E + e];
    p = group_row0[e] + chunk_prefix[(size_t)blockIdx.x * E + e] + before + rank;
    perm[p] = idx;
  }
  if (idx < TK) inv[idx] = p;
}

// One warp: a bf16 row of n8 x 8 values -> f16 times 2^-k, k chosen from the
// row's largest magnitude so that it lands in [2^14, 2^15) (no scaling for a
// zero row or an Inf/NaN); returns 2^k, the row's scale.  Every value of
// magnitude at least 2^-14 after the scaling (all within 2^28 of the largest)
// is exact in f16; smaller ones round to f16's subnormal step, far below the
// rounding of the fp32 accumulation they meet.  dst may be src.
__device__ __forceinline__ float bf16_row_to_f16(const uint4* src, uint4* dst, int n8, int lane) {
  // largest magnitude (bf16 bits without the sign order like the magnitudes;
  // halves compared separately)
  uint32_t m = 0;
  for (int i = lane; i < n8; i += 32) {
    const uint4 v = src[i];
    m = __vmaxu2(m, __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                             __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
  }
  uint32_t mx = max(m & 0xFFFFu, m >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  // largest in [2^(e-127), 2^(e-126)) for biased exponent e: k = e - 141,
  // with 2^-k kept a normal fp32
  const int e = (int)(mx >> 7);
  const int k = (mx == 0 || e == 255) ? 0 : max(e - 141, -126);
  const float down = __uint_as_float((uint32_t)(127 - k) << 23);
  // four vectors per lane in flight before their stores
  for (int i0 = 0; i0 < n8; i0 += 128) {
    uint4 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (i0 + lane + 32 * q < n8) v[q] = src[i0 + lane + 32 * q];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (i0 + lane + 32 * q >= n8) continue;
      const uint32_t in[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
      uint32_t out[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = __fmul_rn(__uint_as_float(in[j] << 16), down);
        const float hi = __fmul_rn(__uint_as_float(in[j] & 0xFFFF0000u), down);
        const __half2 h = __floats2half2_rn(lo, hi);
        out[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
      dst[i0 + lane + 32 * q] = make_uint4(out[0], out[1], out[2], out[3]);
    }
  }
  return __uint_as_float((uint32_t)(127 + k) << 23);
}

// Row gather of one route (one warp): the token's quantized row, its row scale
// and (kScales) its block scales (W4A4; rows already padded to Hp by the
// quantizer) or its bf16 row (W4A16) into permuted row p.  W4A16 rows go to the
// FC1 GEMM as f16, which it multiplies with f16-decoded weights, as
// bf16_row_to_f16 forms them, its scale 2^k in ps.  The Hp - H padding columns
// are zeroed.
struct GatherArgs {
  int K, H, Hp;
  const uint8_t* xc;
  const uint8_t* xsf;
  const float* xs;
  uint8_t* pc;
  uint8_t* psf;
  float* ps;
  const uint4* xb;
  uint4* pb;
  // W4A4 block scales by token tile (gather_tile_scales)
  const int4* tiles;
  const int32_t* status;
  const int32_t* perm;
};
template <bool kW4A16, bool kScales = true>
__device__ __forceinline__ void gather_route_row(const GatherArgs& g, int idx, int p, int lane) {
  const int t = idx / g.K;
  if constexpr (kW4A16) {
    const uint4* src = g.xb + (size_t)t * (g.H / 8);
    uint4* dst = g.pb + (size_t)p * (g.Hp / 8);
    const float rs = bf16_row_to_f16(src, dst, g.H / 8, lane);
    for (int i = g.H / 8 + lane; i < g.Hp / 8; i += 32) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    if (lane == 0) g.ps[p] = rs;
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(g.xc + (size_t)t * (g.Hp / 2));
    uint4* dst = reinterpret_cast<uint4*>(g.pc + (size_t)p * (g.Hp / 2));
    for (int i = lane; i < g.Hp / 32; i += 32) dst[i] = __ldg(src + i);
    if constexpr (kScales) {
      const uint32_t* ssrc = reinterpret_cast<const uint32_t*>(g.xsf + (size_t)t * (g.Hp / 16));
      const uint32_t c16 = (uint32_t)(g.Hp / 16);
      for (int j = lane; j < g.Hp / 64; j += 32)
        *reinterpret_cast<uint32_t*>(g.psf + sf_offset(p, 4 * j, c16)) = __ldg(ssrc + j);
    }
    if (lane == 0) g.ps[p] = g.xs ? g.xs[t] : 1.0f;  // per-tensor tokens carry no row scale
  }
}

// W4A4 block scales of token tile tt, scale words jw0 .. jw0 + kTileScaleWords - 1
// of its rows (word j: the E4M3 scales of columns 4j .. 4j + 3), one warp.  In
// the 128x4-swizzled plane the 16-byte chunk `lane` of a 512-byte atom holds
// word j of rows lane, lane + 32, lane + 64 and lane + 96 of the tile (the
// layout sf_offset maps), so the lane assembles that chunk from the four rows'
// tokens and the warp stores the atom whole: one coalesced store instead of 32
// scattered 4-byte ones.  Padding rows of the tile get zero scales.
constexpr int kTileScaleWords = 4;
__device__ __forceinline__ void gather_tile_scales(const GatherArgs& g, int tt, int jw0, int lane) {
  const int4 tl = g.tiles[tt];  // {expert, expert's first tile, expert's tiles, routes}
  const int rows = min(kTileRows, tl.w - kTileRows * (tt - tl.y));
  const int nw = g.Hp / 64;     // scale words per row = atoms per 128-row block
  const uint32_t* src[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int r = lane + 32 * q;
    src[q] = r < rows ? reinterpret_cast<const uint32_t*>(
                            g.xsf + (size_t)(g.perm[tt * kTileRows + r] / g.K) * (g.Hp / 16))
                      : nullptr;
  }
  uint4 v[kTileScaleWords];
#pragma unroll
  for (int u = 0; u < kTileScaleWords; ++u) {
    const int j = jw0 + u;
    if (j < nw) {
      v[u].x = src[0] ? __ldg(src[0] + j) : 0u;
      v[u].y = src[1] ? __ldg(src[1] + j) : 0u;
      v[u].z = src[2] ? __ldg(src[2] + j) : 0u;
      v[u].w = src[3] ? __ldg(src[3] + j) : 0u;
    }
  }
  uint8_t* chunk = g.psf + (size_t)tt * nw * 512 + lane * 16;
#pragma unroll
  for (int u = 0; u < kTileScaleWords; ++u)
    if (jw0 + u < nw) *reinterpret_cast<uint4*>(chunk + (size_t)(jw0 + u) * 512) = v[u];
}

// Small batches (TK <= kSmallRoutes): count, scan and scatter in one block of
// 1024 threads, saving two launches.  Same outputs as the three kernels: the
// histogram and the tile table as the scan writes them, then the stable
// scatter in 1024-route chunks (earlier warps of the chunk, then the lane's
// rank among earlier lanes with the same expert, on top of a running
// per-expert cursor).  Dynamic shared memory: hist[E], cursor[E], wcnt[32][E].
// Up to kInlineGatherRoutes routes it also gathers the rows (one warp per
// route), saving the gather launch.
constexpr int kSmallRoutes = 2048;  // measured: one block is slower than three kernels at 4096
constexpr int kInlineGatherRoutes = 32;
__global__ void __launch_bounds__(1024) route_small_kernel(
    const int32_t* __restrict__ ids, int ids64, int TK, int E, int32_t* __restrict__ counts,
    int32_t* __restrict__ group_row0, int4* __restrict__ tiles, int32_t* __restrict__ status,
    int32_t* __restrict__ tile_sync, int tile_sync_words, int32_t* __restrict__ inv,
    int32_t* __restrict__ perm, const GatherArgs ga, int gather, int w4a16) {
  extern __shared__ int s_small[];
  int* hist = s_small;
  int* cursor = s_small + E;
  int* wcnt = s_small + 2 * E;  // [32][E]
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  for (int i = tid; i < tile_sync_words; i += blockDim.x) tile_sync[i] = 0;
  for (int i = tid; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  // (1) histogram of valid ids, and the invalid-id flag
  int bad = 0;
  for (int i = tid; i < TK; i += blockDim.x) {
    const int e = load_id(ids, i, ids64);
    if (e >= 0 && e < E)
      atomicAdd(&hist[e], 1);
    else if (e != -1)
      bad = 1;
  }
  bad = __syncthreads_or(bad);
  // (2) exclusive scan of the 128-row-padded group sizes, the tile table and
  // the largest tile (thread e owns expert e, E <= 1024)
  const int total = tid < E ? hist[tid] : 0;
  const int ntiles = (total + kTileRows - 1) / kTileRows;
  __shared__ int warp_sum[32];
  __shared__ int max_rows;
  if (tid == 0) max_rows = 0;
  int incl = ntiles;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sum[wid] = incl;
  __syncthreads();
  if (total > 0) atomicMax(&max_rows, min(kTileRows, total));
  if (wid == 0) {
    int v = (lane < (int)(blockDim.x >> 5)) ? warp_sum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, v, o);
      if (lane >= o) v += y;
    }
    warp_sum[lane] = v;  // inclusive over warps
  }
  __syncthreads();
  const int base = incl - ntiles + (wid > 0 ? warp_sum[wid - 1] : 0);
  if (tid < E) {
    counts[tid] = total;
    group_row0[tid] = base * kTileRows;
    cursor[tid] = base * kTileRows;
    for (int j = 0; j < ntiles; ++j) tiles[base + j] = make_int4(tid, base, ntiles, total);
  }
  if (tid == (int)blockDim.x - 1) {
    status[kStatusFlags] = bad ? kFlagBadExpertId : 0;
    status[kStatusTiles] = base + ntiles;
    status[kStatusRows] = (base + ntiles) * kTileRows;
    status[kStatusMaxRows] = max_rows;
    status[kStatusItemCtr] = 0;
    status[kStatusItemCtr + 1] = 0;
  }
  // (3) stable scatter, one 1024-route chunk after another
  for (int c0 = 0; c0 < TK; c0 += blockDim.x) {
    for (int i = tid; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    const int idx = c0 + tid;
    const int e = idx < TK ? load_id(ids, idx, ids64) : -1;
    const bool valid = e >= 0 && e < E;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, valid ? e : -1);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (valid && rank == 0) wcnt[wid * E + e] = __popc(peers);
    __syncthreads();
    int p = -1;
    if (valid) {
      int before = 0;
      for (int v = 0; v < wid; ++v) before += wcnt[v * E + e];
      p = cursor[e] + before + rank;
      perm[p] = idx;
    }
    if (idx < TK) inv[idx] = p;
    __syncthreads();
    for (int i = tid; i < E; i += blockDim.x) {
      int n = 0;
      for (int v = 0; v < 32; ++v) n += wcnt[v * E + i];
      cursor[i] += n;
    }
    __syncthreads();  // the next chunk clears wcnt only after every thread has read it
  }
  // (4) tiny batches: the row gather too, warp w copying route w's row
  if (gather && wid < TK) {
    const int p = inv[wid];
    if (p >= 0) {
      if (w4a16)
        gather_route_row<true>(ga, wid, p, lane);
      else
        gather_route_row<false>(ga, wid, p, lane);
    }
  }
}

// Gather: one warp per route copies its token's row to the route's permuted row.
// W4A4 rows are already padded to Hp by the quantizer; W4A16 copies H bf16
// values and zero-fills the Hp - H padding columns.  W4A4 launches start with
// `scale_blocks` blocks whose warps write the block scales tile by tile
// (gather_tile_scales), ahead of the route blocks so that their chains of
// dependent loads overlap the row copies: warp w takes tile w / jchunks and
// words kTileScaleWords * (w % jchunks) onwards; warps past the scan's tile
// count have nothing to do.
template <bool kW4A16>
__global__ void __launch_bounds__(128) gather_rows_kernel(int TK, const int32_t* __restrict__ inv,
                                                          const GatherArgs g, int scale_blocks,
                                                          int jchunks) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  if (!kW4A16 && (int)blockIdx.x < scale_blocks) {
    const int w = ((int)blockIdx.x * (int)blockDim.x + (int)threadIdx.x) >> 5;
    const int tt = w / jchunks;
    if (tt >= g.status[kStatusTiles]) return;
    gather_tile_scales(g, tt, kTileScaleWords * (w % jchunks), lane);
    return;
  }
  const int idx = (((int)blockIdx.x - scale_blocks) * (int)blockDim.x + (int)threadIdx.x) >> 5;
  if (idx >= TK) return;
  const int p = inv[idx];
  if (p < 0) return;
  gather_route_row<kW4A16, false>(g, idx, p, lane);
}

// Kernels launch_route issues for TK routes: routing and the row gather.
int route_kernel_launches(int64_t TK) {
  return TK <= kInlineGatherRoutes ? 1 : TK <= kSmallRoutes ? 2 : 4;
}

static GatherArgs gather_args(const RouteArgs& a) {
  return GatherArgs{a.K,   a.H,   a.Hp, a.xc, a.xsf, a.xs, a.pc, a.psf, a.ps,
                    static_cast<const uint4*>(a.xb), static_cast<uint4*>(a.pb),
                    a.tiles, a.status, a.perm};
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
  if (a.TK <= kSmallRoutes) {
    const size_t smem = sizeof(int) * 34 * (size_t)a.E;  // hist, cursor, 32 warp rows
    static std::atomic<uint64_t> configured{0};  // per device
    cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(route_small_kernel),
                                        (int)(sizeof(int) * 34 * 1024), configured);
    if (err != cudaSuccess) return err;
    launch_pdl(route_small_kernel, dim3(1), dim3(1024), smem, s, a.ids, a.ids64, a.TK, a.E,
               a.counts, a.group_row0, a.tiles, a.status, a.tile_sync, a.tile_sync_words, a.inv,
               a.perm, gather_args(a), a.TK <= kInlineGatherRoutes ? 1 : 0, a.w4a16);
    if (a.TK <= kInlineGatherRoutes) return cudaGetLastError();  // rows gathered by the same block
  } else {
    const int nchunks = (a.TK + kChunk - 1) / kChunk;
    launch_pdl(route_count_kernel, dim3(nchunks), dim3(kChunk), sizeof(int) * a.E, s, a.ids,
               a.ids64, a.TK, a.E, a.chunk_counts);
    launch_pdl(route_scan_kernel, dim3(1), dim3(1024), 0, s, nchunks, a.E,
               (const int32_t*)a.chunk_counts, a.chunk_prefix, a.counts, a.group_row0, a.tiles,
               a.status, a.tile_sync, a.tile_sync_words);
    const size_t smem = sizeof(int) * (kChunk / 32) * a.E;
    launch_pdl(route_scatter_kernel, dim3(nchunks), dim3(kChunk), smem, s, a.ids, a.ids64, a.TK,
               a.E, (const int32_t*)a.chunk_prefix, (const int32_t*)a.group_row0, a.inv, a.perm);
  }
  // 4-warp blocks: small enough in registers to share an SM with a GEMM CTA,
  // which can then start (programmatic launch) before the gather is done
  const int gblocks = (a.TK + 3) / 4;
  if (a.w4a16) {
    launch_pdl(gather_rows_kernel<true>, dim3(gblocks), dim3(128), 0, s, a.TK,
               (const int32_t*)a.inv, gather_args(a), 0, 1);
  } else {
    // the scale warps cover every tile the workspace can hold: its rows are TK
    // plus up to 127 padding rows for each of min(TK, E) experts, in whole tiles
    const int64_t pad_groups = std::min<int64_t>(a.TK, a.E);
    const int64_t tiles_cap = (a.TK + pad_groups * (kTileRows - 1) + kTileRows - 1) / kTileRows;
    const int jchunks = (a.Hp / 64 + kTileScaleWords - 1) / kTileScaleWords;
    const int64_t sblocks = (tiles_cap * jchunks + 3) / 4;
    launch_pdl(gather_rows_kernel<false>, dim3((unsigned)(gblocks + sblocks)), dim3(128), 0, s,
               a.TK, (const int32_t*)a.inv, gather_args(a), (int)sblocks, jchunks);
  }
  return cudaGetLastError();
}

// ============================================================== W4A16 FC2 operand
// Each valid route's bf16 activated row (the FC1 handoff) as f16 times a power
// of two, its scale 2^k (bf16_row_to_f16), for the f16 FC2 GEMM.  One warp per
// route.
__global__ void __launch_bounds__(256) act_f16_kernel(int TK, int Ip, const int32_t* __restrict__ inv,
                                                      const uint4* act, uint4* act16,
                                                      float* __restrict__ scale) {
  pdl_wait();
  pdl_trigger();
  const int idx = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (idx >= TK) return;
  const int p = inv[idx];
  if (p < 0) return;
  const float rs = bf16_row_to_f16(act + (size_t)p * (Ip / 8), act16 + (size_t)p * (Ip / 8),
                                   Ip / 8, lane);
  if (lane == 0) scale[p] = rs;
}

void launch_act_f16(int TK, int Ip, const int32_t* inv, const void* act, void* act16,
                    float* scale, cudaStream_t s) {
  launch_pdl(act_f16_kernel, dim3((TK + 7) / 8), dim3(256), 0, s, TK, Ip, inv,
             static_cast<const uint4*>(act), static_cast<uint4*>(act16), scale);
}

// ============================================================== FC2-input requant
// Megatron-LM PR #8262, "How to extend": fc2_input_scale = 1/(448*6) for the
// per-token recipe; the FC2 input is quantized per routed row.  One warp per
// route reads the fp32 activated row written by the FC1 epilogue.
// With `static_enc` (per-tensor recipe: fc2_input_scale = a2_scale) every row
// uses that encode scale and its row scale is 1.
// G: rows of up to G * 2048 values are read once, into registers.
template <int G>
__global__ void __launch_bounds__(256) requant_kernel(int TK, int I, const int32_t* __restrict__ inv,
                                                      const float* __restrict__ act,
                                                      uint8_t* __restrict__ qc,
                                                      uint8_t* __restrict__ qsf,
                                                      float* __restrict__ qs,
                                                      const float* __restrict__ static_enc) {
  pdl_wait();
  pdl_trigger();
  const int idx = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (idx >= TK) return;
  const int p = inv[idx];
  if (p < 0) return;
  requant_row_warp<G>(act + (size_t)p * I, I, (uint64_t)p, qc, qsf, qs, static_enc, lane);
}

void launch_requant(int TK, int I, const int32_t* inv, const float* act, uint8_t* qc, uint8_t* qsf,
                    float* qs, const float* static_enc, cudaStream_t s) {
  // Large batches: 2-warp blocks (91 registers a thread), small enough to share
  // an SM with a GEMM CTA, so FC2 can start (programmatic launch) before the
  // long pass is done (ReLU2 H7168 E256 T=4096: -11 us); small batches keep
  // 8-warp blocks (the many tiny blocks cost more than they overlap there).
  const int warps = TK > kSmallRoutes ? 2 : 8;
  if (I <= 2048)
    launch_pdl(requant_kernel<1>, dim3((TK + warps - 1) / warps), dim3(warps * 32), 0, s, TK, I,
               inv, act, qc, qsf, qs, static_enc);
  else
    launch_pdl(requant_kernel<2>, dim3((TK + warps - 1) / warps), dim3(warps * 32), 0, s, TK, I,
               inv, act, qc, qsf, qs, static_enc);
}

// ============================================================== finalize
// Megatron-LM PR #8262, "What is added": the two-stage finalize reduces each
// token's top-k routes in a fixed order; FlashInfer PR #5019, "Tensor and
// numerical contract": bf16 per-route terms times fp32 scores, one final bf16
// conversion.  fp32 accumulator from +0, k ascending, one fma per term.
__global__ void __launch_bounds__(128) finalize_kernel(int K, int H, int Hp,
                                                       const int32_t* __restrict__ inv,
                                                       const float* __restrict__ w,
                                                       const uint4* __restrict__ route,
                                                       uint4* __restrict__ out) {
  __shared__ int s_p[32];
  __shared__ float s_w[32];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  if (threadIdx.x < K) {
    s_p[threadIdx.x] = inv[(size_t)t * K + threadIdx.x];
    s_w[threadIdx.x] = w[(size_t)t * K + threadIdx.x];
  }
  __syncthreads();
  const int v = blockIdx.y * blockDim.x + threadIdx.x;
  if (v >= H / 8) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  for (int k0 = 0; k0 < K; k0 += 8) {
    uint4 r[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // issue the loads of 8 routes before using any
      const int p = k0 + j < K ? s_p[k0 + j] : -1;
      r[j] = p >= 0 ? route[(size_t)p * (Hp / 8) + v] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (k0 + j >= K || s_p[k0 + j] < 0) continue;
      const float wk = s_w[k0 + j];
      const uint32_t q[4] = {r[j].x, r[j].y, r[j].z, r[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fmaf_rn(wk, __uint_as_float(q[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = __fmaf_rn(wk, __uint_as_float(q[i] & 0xFFFF0000u), acc[2 * i + 1]);
      }
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    o[i] = *reinterpret_cast<const uint32_t*>(&b2);
  }
  out[(size_t)t * (H / 8) + v] = make_uint4(o[0], o[1], o[2], o[3]);
}

void launch_finalize(int T, int K, int H, int Hp, const int32_t* inv, const float* w,
                     const void* route, void* out, cudaStream_t s) {
  const int threads = 128;
  dim3 grid(T, (H / 8 + threads - 1) / threads);
  launch_pdl(finalize_kernel, grid, dim3(threads), 0, s, K, H, Hp, inv, w,
             static_cast<const uint4*>(route), static_cast<uint4*>(out));
}

}  // namespace moe
