// gemm_w4a4.cu -- block-scaled NVFP4 x NVFP4 grouped GEMMs (FC1 with fused
// activation, FC2) on tcgen05 tensor cores.
//
// Megatron-LM PR #8262, "Background" / "What is added": FC1 and FC2 are block-
// scaled grouped GEMMs over expert groups; FC1's epilogue applies the expert
// alpha and the per-token scale, then squared-ReLU or SwiGLU.  The FC2 input
// requantization of each route row needs the row's amax over all of I, so the
// FC1 epilogue writes the fp32 activated row and a row-parallel pass quantizes it.
//
// Structure (swap-AB: weights are the M=128 operand, tokens the N operand, so a
// decode-sized group of 1..128 tokens does not waste a 128-row MMA):
//   * persistent CTAs, one per SM; work item = (token tile, 256-row weight tile)
//   * warp 0: TMA producer -- weight tile halves (2 x 128 rows x 128 B, 128-byte
//     swizzle), token tile (16-row boxes), scale atoms via bulk copies
//   * warp 1: TMEM allocator and single-thread MMA issuer:
//     tcgen05.cp of the scale atoms into TMEM, then
//     tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (K = 64 per instruction)
//   * warps 2-5: epilogue, one TMEM lane (= one weight row) per thread
//   * 4-stage shared-memory ring guarded by mbarriers; every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace w4a4 {
constexpr int kStages = 4;
constexpr int kBK = 256;                        // K elements per stage
constexpr int kRowBytes = kBK / 2;              // packed FP4 bytes per row per stage
constexpr int kAHalfBytes = 128 * kRowBytes;    // 16 KB
constexpr int kABytes = 2 * kAHalfBytes;        // 32 KB
constexpr int kBBytes = kTileRows * kRowBytes;  // 16 KB
constexpr int kAtom = 512;                      // 128 rows x 4 scale columns
constexpr int kSfaBytes = 2 * 4 * kAtom;        // two row halves x 4 K-atoms
constexpr int kSfbBytes = 4 * kAtom;
constexpr int kOffB = kABytes;
constexpr int kOffSfa = kOffB + kBBytes;
constexpr int kOffSfb = kOffSfa + kSfaBytes;
constexpr int kStageBytes = kOffSfb + kSfbBytes;  // 55296, a multiple of 1024
constexpr int kBarOff = kStages * kStageBytes;
constexpr int kSmemBytes = kBarOff + 256 + 1024;  // + barriers + alignment slack
constexpr int kTmemCols = 512;
constexpr int kAccCols = 256;            // two 128-column accumulators (row halves)
constexpr int kSfColsPerStage = 48;      // SFA 2 x 4 atoms x 4 cols + SFB 4 atoms x 4 cols
constexpr int kThreads = 192;
static_assert(kStageBytes % 1024 == 0, "stage must keep 1024-byte alignment");
static_assert(kAccCols + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
}  // namespace w4a4

struct Smem {
  uint8_t* base;
  __device__ uint32_t bar(int i) const { return smem_u32(base + w4a4::kBarOff + 8 * i); }
};

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicOr(status + kStatusFlags, kFlagWaitTimeout);
      return false;
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(w4a4::kThreads, 1)
    gemm_w4a4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmArgs a) {
  using namespace w4a4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const Smem S{smem};
  // barrier indices: full[s] = s, empty[s] = kStages + s, acc_full, acc_empty, drain
  const int kFull = 0, kEmpty = kStages, kAccFull = 2 * kStages, kAccEmpty = 2 * kStages + 1,
            kDrain = 2 * kStages + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + 8 * (2 * kStages + 3));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int n_tiles = a.status[kStatusTiles];
  const int n_items = n_tiles * a.m_tiles;
  if ((int)blockIdx.x >= n_items) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(S.bar(kFull + s), 1);
      mbar_init(S.bar(kEmpty + s), 1);
    }
    mbar_init(S.bar(kAccFull), 1);
    mbar_init(S.bar(kAccEmpty), 128);
    mbar_init(S.bar(kDrain), 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int kblocks = a.K / kBK;
  const int atoms = a.K / 64;            // scale atoms per 128-row block
  const size_t plane = (size_t)a.w_rows * (a.K / 16);  // weight scale bytes per expert

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int last_par[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) last_par[s] = -1;
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int tt = item / a.m_tiles, mt = item % a.m_tiles;
        const int e = a.tile_expert[tt];
        const int rows = a.tile_rows[tt];
        const int n16 = (rows + 15) & ~15;
        const int a_row = e * a.w_rows + mt * 256;
        const int b_row = tt * kTileRows;
        const uint8_t* sfa0 = a.sfa + (size_t)e * plane + (size_t)(2 * mt) * atoms * kAtom;
        const uint8_t* sfb0 = a.sfb + (size_t)tt * atoms * kAtom;
        const uint32_t tx = kABytes + kSfaBytes + kSfbBytes + n16 * kRowBytes;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_or_abort(S.bar(kEmpty + stage), phase ^ 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          uint8_t* sb = smem + stage * kStageBytes;
          const uint32_t full = S.bar(kFull + stage);
          mbar_expect_tx(full, tx);
          tma_load_2d_hint(smem_u32(sb), &tmA, full, kb * kRowBytes, a_row, pol_w);
          tma_load_2d_hint(smem_u32(sb + kAHalfBytes), &tmA, full, kb * kRowBytes, a_row + 128,
                           pol_w);
          for (int c = 0; c < n16 / 16; ++c)
            tma_load_2d_hint(smem_u32(sb + kOffB + c * 16 * kRowBytes), &tmB, full, kb * kRowBytes,
                             b_row + 16 * c, pol_x);
          bulk_load(smem_u32(sb + kOffSfa), sfa0 + (size_t)(kb * 4) * kAtom, 4 * kAtom, full);
          bulk_load(smem_u32(sb + kOffSfa + 4 * kAtom), sfa0 + (size_t)(atoms + kb * 4) * kAtom,
                    4 * kAtom, full);
          bulk_load(smem_u32(sb + kOffSfb), sfb0 + (size_t)(kb * 4) * kAtom, 4 * kAtom, full);
          last_par[stage] = (int)phase;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // let every copy still in flight land before the CTA's shared memory goes away
        for (int s = 0; s < kStages; ++s)
          if (last_par[s] >= 0) mbar_wait(S.bar(kFull + s), (uint32_t)last_par[s]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc_phase = 0;
      bool ok = true, issued = false;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int tt = item / a.m_tiles;
        const int rows = a.tile_rows[tt];
        const int n16 = (rows + 15) & ~15;
        const uint32_t idesc = idesc_mxf4nvf4(128, n16);
        if (!wait_or_abort(S.bar(kAccEmpty), acc_phase ^ 1, abort_flag, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_or_abort(S.bar(kFull + stage), phase, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* sb = smem + stage * kStageBytes;
          const uint32_t sf_col = tmem + kAccCols + stage * kSfColsPerStage;
#pragma unroll
          for (int i = 0; i < 8; ++i)  // SFA: half i/4, K-atom i%4 -> columns 4*i
            tc_cp_sf_atom(sf_col + 4 * i, smem_desc(smem_u32(sb + kOffSfa + i * kAtom), 0, 128, 0));
#pragma unroll
          for (int i = 0; i < 4; ++i)
            tc_cp_sf_atom(sf_col + 32 + 4 * i,
                          smem_desc(smem_u32(sb + kOffSfb + i * kAtom), 0, 128, 0));
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t bdesc = smem_desc(smem_u32(sb + kOffB + ks * 32), 16, 1024, 2);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint64_t adesc =
                  smem_desc(smem_u32(sb + h * kAHalfBytes + ks * 32), 16, 1024, 2);
              mma_mxf4nvf4(tmem + h * 128, adesc, bdesc, idesc, sf_col + 16 * h + 4 * ks,
                           sf_col + 32 + 4 * ks, (kb | ks) != 0 ? 1u : 0u);
            }
          }
          issued = true;
          tc_commit(S.bar(kEmpty + stage));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(S.bar(kAccFull));
        acc_phase ^= 1;
      }
      if (!ok && issued) {
        // drain the tensor-core work issued so far before TMEM is released
        tc_commit(S.bar(kDrain));
        mbar_wait(S.bar(kDrain), 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                  // TMEM lane quadrant of this warp
    const int r = q * 32 + lane;             // row within a 128-row half
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    uint32_t acc_phase = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const int tt = item / a.m_tiles, mt = item % a.m_tiles;
      const int e = a.tile_expert[tt];
      const int rows = a.tile_rows[tt];
      const int n16 = (rows + 15) & ~15;
      const int row0 = tt * kTileRows;
      if (!wait_or_abort(S.bar(kAccFull), acc_phase, abort_flag, a.status)) break;
      tc_fence_after();
      const float alpha = a.alpha[e];
      for (int c0 = 0; c0 < n16; c0 += 16) {
        float g[16], u[16];
        tmem_ld16(tmem + lane_addr + c0, g);
        tmem_ld16(tmem + lane_addr + 128 + c0, u);
        tmem_wait_ld();
#pragma unroll 4
        for (int j = 0; j < 16; ++j) {
          const int col = c0 + j;
          if (col >= rows) break;
          const size_t p = (size_t)row0 + col;
          const float s = a.row_scale[p];
          if constexpr (MODE == kFc1Swiglu) {
            const float yg = __fmul_rn(__fmul_rn(g[j], alpha), s);
            const float yu = __fmul_rn(__fmul_rn(u[j], alpha), s);
            const float act = __fmul_rn(__fdiv_rn(yg, __fadd_rn(1.0f, expf(-yg))), yu);
            a.act_out[p * a.I + mt * 128 + r] = act;
          } else if constexpr (MODE == kFc1Relu2) {
            const float y0 = fmaxf(__fmul_rn(__fmul_rn(g[j], alpha), s), 0.0f);
            const float y1 = fmaxf(__fmul_rn(__fmul_rn(u[j], alpha), s), 0.0f);
            float* dst = a.act_out + p * a.I + mt * 256 + r;
            dst[0] = __fmul_rn(y0, y0);
            dst[128] = __fmul_rn(y1, y1);
          } else {
            const float z0 = __fmul_rn(__fmul_rn(g[j], alpha), s);
            const float z1 = __fmul_rn(__fmul_rn(u[j], alpha), s);
            uint16_t* dst = a.route_out + p * a.H + mt * 256 + r;
            dst[0] = __bfloat16_as_ushort(__float2bfloat16_rn(z0));
            dst[128] = __bfloat16_as_ushort(__float2bfloat16_rn(z1));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(S.bar(kAccEmpty));
      acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int MODE>
static cudaError_t launch_mode(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                               int grid, cudaStream_t s) {
  static bool configured = false;  // per process; the attribute is per function
  if (!configured) {
    cudaError_t err = cudaFuncSetAttribute(gemm_w4a4_kernel<MODE>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           w4a4::kSmemBytes);
    if (err != cudaSuccess) return err;
    configured = true;
  }
  gemm_w4a4_kernel<MODE><<<grid, w4a4::kThreads, w4a4::kSmemBytes, s>>>(tmA, tmB, a);
  return cudaGetLastError();
}

cudaError_t launch_gemm_w4a4(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                             int grid, cudaStream_t s) {
  switch (a.mode) {
    case kFc1Relu2: return launch_mode<kFc1Relu2>(tmA, tmB, a, grid, s);
    case kFc1Swiglu: return launch_mode<kFc1Swiglu>(tmA, tmB, a, grid, s);
    default: return launch_mode<kFc2>(tmA, tmB, a, grid, s);
  }
}

}  // namespace moe
