// gemm_w4a4.cu -- block-scaled NVFP4 x NVFP4 grouped GEMMs (FC1 with fused
// activation, FC2) on tcgen05 tensor cores, as separate launches or as one
// persistent FC1 -> requant -> FC2 launch.
//
// Megatron-LM PR #8262, "Background" / "What is added": FC1 and FC2 are block-
// scaled grouped GEMMs over expert groups; FC1's epilogue applies the expert
// alpha and the per-token scale, then squared-ReLU or SwiGLU.  The FC2 input
// requantization of each route row needs the row's amax over all of I, so the
// FC1 epilogue writes the fp32 activated row and the row is quantized once the
// whole tile is written: by a row-parallel pass between two launches, or, in
// the fused launch, by a requant work item of the tile that waits for the
// tile's FC1 items (the pages' MegaMoE keeps FC1 and FC2 in one persistent
// kernel, FlashInfer PR #5019).
//
// Structure (swap-AB: weights are the M=128 operand, tokens the N operand, so a
// decode-sized group of a few tokens does not waste a 128-row MMA):
//   * persistent CTAs, one per SM; work item = (token tile of <= 128 rows of one
//     expert, 128-row weight tile of that expert) of FC1 or of FC2; FC1 items are
//     numbered first.  Each CTA starts with item blockIdx.x and then claims items
//     from a global counter, and its roles receive them through a shared-memory
//     ring
//   * two TMA producers, each one thread, both filling every stage: warp 0
//     claims the items and loads the weight tile (128 rows x 128 B, 128-byte
//     swizzle) and its scale atoms; warp 10 loads the token tile (one to three
//     boxes of 128/64/32/16 rows) and its scale atoms.  Each copy costs its
//     issuing thread a few hundred cycles, so a stage is split between two
//     threads and issued in as few copies as its shape allows.  In the fused
//     launch the token producer of an FC2 item first waits for its tile's
//     requantized rows (the weight producer keeps streaming meanwhile).
//   * warps 6-9: scale staging -- move each stage's E4M3 scale atoms from shared
//     memory into that stage's TMEM scale slot with tcgen05.st, in the layout the
//     block-scaled MMA reads (row r of a 128-row atom at lane r%32, column r/32,
//     replicated in all four lane quadrants)
//   * warp 1: TMEM allocator and MMA issuer (whole warp, elect.sync issues):
//     tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X, K = 64 per
//     instruction, N = the tile's token count rounded up to 16
//   * warps 2-5: epilogue, one TMEM lane (= one weight row) per thread; each
//     chunk of up to 32 tokens is staged in shared memory as [token][feature]
//     rows and one thread writes it with TMA tensor stores (two 16 KB staging
//     buffers; one 8 KB buffer of 16-token chunks in squared-ReLU FC1 launches
//     with tiles of more than 96 tokens)
//   * the shared-memory stage ring is sized at run time from the largest token
//     tile of the launch and the staging buffers (5 stages at 128 tokens, 6 in
//     those squared-ReLU FC1 launches, 8 at 16); two accumulator buffers (four
//     when no tile exceeds 64 tokens) let the epilogue of one tile overlap the
//     MMAs of the next ones.
//   * every wait is bounded; on timeout the CTA records an error flag, drains its
//     own copies and MMAs, frees TMEM and returns.
// SwiGLU: the stored FC1 rows interleave 64-row blocks [gate | up], so TMEM
// lanes 0-63 hold gate rows and 64-127 the matching up rows; both halves are
// staged in shared memory and all four epilogue warps apply silu(gate) * up.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace moe {

namespace w4a4 {
constexpr int kBK = 256;                    // K elements per stage
constexpr int kRowBytes = kBK / 2;          // packed FP4 bytes per row per stage
constexpr int kABytes = 128 * kRowBytes;    // 16 KB weight tile per stage
constexpr int kAtom = 512;                  // 128 rows x 4 scale columns
constexpr int kSfaBytes = 4 * kAtom;        // 4 K-atoms of the 128-row weight tile
constexpr int kMaxStages = 12;
constexpr int kMaxAcc = 4;                  // accumulator buffers (4 when tiles <= 64 tokens)
constexpr int kTmemCols = 512;
// Epilogue output staging: two buffers, each one chunk of up to 32 tokens x the
// tile's output features (fp32 x 128, or SwiGLU gate + up fp32 x 64 each, or
// bf16 x 128), written to global memory by TMA stores of 16-row boxes.
constexpr int kEpiBufBytes = 16384;
constexpr int kEpiBytes = 2 * kEpiBufBytes;
constexpr int kBarBytes = 2048;             // barriers, flags, item ring; then 128 row scales
constexpr int kSmemBytes = 227 * 1024;      // dynamic shared memory of every launch
constexpr int kThreads = 352;               // 11 warps
// barrier indices
constexpr int kBarFull = 0;
constexpr int kBarEmpty = kMaxStages;
constexpr int kBarSfReady = 2 * kMaxStages;
constexpr int kBarAccFull = 3 * kMaxStages;
constexpr int kBarAccEmpty = kBarAccFull + kMaxAcc;
constexpr int kBarItemFull = kBarAccEmpty + kMaxAcc;
constexpr int kBarItemEmpty = kBarItemFull + kItemSlots;
constexpr int kBarDrain = kBarItemEmpty + kItemSlots;
constexpr int kNumBars = kBarDrain + 1;
constexpr int kFlagsOff = 8 * kNumBars;     // tmem slot, abort flag, epilogue stop flag, requant flag
constexpr int kRingOff = 768;               // kItemSlots int4
static_assert(kFlagsOff + 16 <= kRingOff && kRingOff + 16 * kItemSlots <= 1024, "flag area");
}  // namespace w4a4

// ---------------------------------------------------------------- work items
// FC1 items [0, n1), then (fused launch) one requant item per token tile
// [n1, n1 + nr), then FC2 items [n1 + nr, n1 + nr + n2).  Within a GEMM phase
// the numbering of tile_decode (an expert's token tiles for one weight tile side
// by side).  Every item waits only on lower-numbered items.  (Interleaving the
// phases per tile was measured slower: a CTA whose FC2 item waits holds FC1
// items it has already claimed, and the waits chain up.)  The phase (0 FC1, 1
// FC2, 2 requant) rides in bits 16.. of TileInfo::mt.
constexpr int kPhaseRequant = 2;
struct ItemSpace {
  int n1, nr, n2, m1, m2;
};
__device__ __forceinline__ int4 item_raw(const W4A4Args& a, const ItemSpace& sp, int item) {
  if (item >= sp.n1 + sp.nr + sp.n2) return make_int4(0, 0, 1, 0);
  if (item < sp.n1) return a.tiles[item / sp.m1];
  if (item < sp.n1 + sp.nr) return a.tiles[item - sp.n1];
  return a.tiles[(item - sp.n1 - sp.nr) / sp.m2];
}
__device__ __forceinline__ TileInfo item_decode(const ItemSpace& sp, int item, const int4& t) {
  if (item >= sp.n1 + sp.nr + sp.n2) return TileInfo{0, 0, 0, 0};
  if (item >= sp.n1 && item < sp.n1 + sp.nr) {
    const int tt = item - sp.n1;
    return TileInfo{t.x, tt, kPhaseRequant << 16, min(kTileRows, t.w - kTileRows * (tt - t.y))};
  }
  const int ph = item >= sp.n1 ? 1 : 0;
  const int m = ph ? sp.m2 : sp.m1;
  const int local = (ph ? item - sp.n1 - sp.nr : item) - m * t.y;
  const int j = local % t.z;
  return TileInfo{t.x, t.y + j, (local / t.z) | (ph << 16), min(kTileRows, t.w - kTileRows * j)};
}

// Block pass of the fused requant: the tile's rows x Ip/16 blocks of 16 values
// spread over 128 threads, two blocks in flight per thread (loads first, then the
// quantization and the stores).  row_amax: per-row amax, or anything non-zero
// for the static-scale recipe.  Same arithmetic as requant_row_warp.
__device__ __forceinline__ void requant_blocks(const float* __restrict__ act0, int Ip, int rows,
                                               int row0, const float* __restrict__ row_amax,
                                               const float* __restrict__ static_enc,
                                               uint8_t* __restrict__ qc, uint8_t* __restrict__ qsf,
                                               int et) {
  const int nb = Ip / 16;  // blocks per row
  const uint32_t c16 = (uint32_t)nb;
  const int total = rows * nb;
  for (int b0 = et; b0 < total; b0 += 256) {
    float v[2][16];
    int rr[2], jj[2];
    bool have[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int b = b0 + 128 * u;
      have[u] = b < total;
      rr[u] = have[u] ? b / nb : 0;
      jj[u] = have[u] ? b - rr[u] * nb : 0;
      if (have[u]) {
        const float4* src = reinterpret_cast<const float4*>(act0 + (size_t)rr[u] * Ip) + 4 * jj[u];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 f = src[i];
          v[u][4 * i] = f.x;
          v[u][4 * i + 1] = f.y;
          v[u][4 * i + 2] = f.z;
          v[u][4 * i + 3] = f.w;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (!have[u]) continue;
      const uint64_t p = (uint64_t)(row0 + rr[u]);
      const float mm = row_amax[rr[u]];
      uint2* crow = reinterpret_cast<uint2*>(qc + p * (uint64_t)(Ip / 2));
      if (mm == 0.0f) {
        crow[jj[u]] = make_uint2(0u, 0u);
        qsf[sf_offset(p, jj[u], c16)] = 0;
        continue;
      }
      const float enc = static_enc ? *static_enc : __fdiv_rn(kRecipeMax, mm);
      uint2 qv;
      qsf[sf_offset(p, jj[u], c16)] = (uint8_t)quant_block16(v[u], enc, qv);
      crow[jj[u]] = qv;
    }
  }
}

// Bounded wait for another CTA's flag to reach `target` (acquire); records a
// timeout like the mbarrier waits.
__device__ __forceinline__ bool wait_flag_geq(const int32_t* flag, int target,
                                              volatile int* abort_flag, int32_t* status) {
  if (ld_acquire_gpu(flag) >= target) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    __nanosleep(128);
    if (ld_acquire_gpu(flag) >= target) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicOr(status + kStatusFlags, kFlagWaitTimeout);
      return false;
    }
  }
}

template <int ACT>
__global__ void __launch_bounds__(w4a4::kThreads, 1)
    gemm_w4a4_kernel(const __grid_constant__ W4A4Maps maps, const __grid_constant__ W4A4Args a) {
  using namespace w4a4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const Ring R{smem};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kFlagsOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_stop = reinterpret_cast<volatile int*>(tmem_slot + 2);
  volatile int* rq_flag = reinterpret_cast<volatile int*>(tmem_slot + 3);
  const ItemQueue Q{reinterpret_cast<int4*>(smem + kRingOff), R.bar(kBarItemFull),
                    R.bar(kBarItemEmpty)};
  float* s_scale = reinterpret_cast<float*>(smem + 1024);  // row scales of the current tile (128)
  uint8_t* epi_buf = smem + kBarBytes;               // epilogue staging, 1024-aligned

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // prologue that reads nothing the previous kernel writes: barriers, TMEM
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(R.bar(kBarFull + s), 2);  // the weight and the token producer
      mbar_init(R.bar(kBarEmpty + s), 1);
      mbar_init(R.bar(kBarSfReady + s), 4);
    }
    for (int b = 0; b < kMaxAcc; ++b) {
      mbar_init(R.bar(kBarAccFull + b), 1);
      mbar_init(R.bar(kBarAccEmpty + b), 128);
    }
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(R.bar(kBarItemFull + s), 1);
      mbar_init(R.bar(kBarItemEmpty + s), 1 + 4 + 4 + 1);  // MMA, staging, epilogue, token producer
    }
    mbar_init(R.bar(kBarDrain), 1);
    *abort_flag = 0;
    *epi_stop = 0;
    *rq_flag = 0;
    fence_barrier_init();
    for (int p = 0; p < 2; ++p) {
      if (!(p ? a.run_fc2 : a.run_fc1)) continue;
      prefetch_tmap(&maps.a[p]);
      for (int i = 0; i < 4; ++i) prefetch_tmap(&maps.b[p].box[i]);
      prefetch_tmap(&maps.o[p]);
    }
  }
  __syncwarp();  // thread 0's set-up branch rejoins its warp before the barrier
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_trigger();
  if (a.span && threadIdx.x == 0) atomicMin(a.span, (unsigned long long)globaltimer());

  const int n_tiles = a.status[kStatusTiles];
  const ItemSpace sp{a.run_fc1 ? n_tiles * a.ph[0].m_tiles : 0, a.fused ? n_tiles : 0,
                     a.run_fc2 ? n_tiles * a.ph[1].m_tiles : 0, a.ph[0].m_tiles,
                     a.ph[1].m_tiles};

  // ---- geometry from the largest token tile (<= 128 rows) of this launch
  const int max_n16 = (a.status[kStatusMaxRows] + 15) & ~15;
  const int b_bytes = max_n16 * kRowBytes;                // multiple of 2048
  const int stage_bytes = kABytes + kSfaBytes + b_bytes + 4 * kAtom;  // multiple of 1024
  const int off_sfa = kABytes, off_b = kABytes + kSfaBytes, off_sfb = off_b + b_bytes;
  const int acc_stride = (max_n16 + 31) & ~31;            // TMEM columns per accumulator
  const int nbuf = max_n16 <= 64 ? 4 : 2;                 // accumulator buffers
  const int slot_cols = 32;                               // scale columns per stage (A 16, B 16)
  const int sf_base = nbuf * acc_stride;
  // Squared-ReLU FC1 launches with 97-128-token tiles stage the epilogue through
  // one 8 KB buffer in 16-token chunks: that leaves room for a sixth 36 KB
  // stage, 108 KB of weights in flight instead of 90 KB.  Every other launch
  // uses two 16 KB buffers in 32-token chunks (FC2's short items and the
  // SwiGLU pairing were measured slower with the single buffer).
  const bool narrow_epi =
      ACT == kFc1Relu2 && a.run_fc1 && !a.run_fc2 && max_n16 > 96;
  const int epi_bytes = narrow_epi ? kEpiBufBytes / 2 : kEpiBytes;  // multiple of 1024
  const int cw = narrow_epi ? 16 : 32;                // tokens per epilogue chunk
  uint8_t* stages = smem + kBarBytes + epi_bytes;     // 1024-aligned
  int n_stages = (kSmemBytes - 1024 - kBarBytes - epi_bytes) / stage_bytes;
  if (n_stages > kMaxStages) n_stages = kMaxStages;
  while (n_stages > 2 && sf_base + n_stages * slot_cols > kTmemCols) --n_stages;

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      int last_par[kMaxStages];
#pragma unroll
      for (int s = 0; s < kMaxStages; ++s) last_par[s] = -1;
      const uint64_t pol_w = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      QueuePos qp;
      bool ok = true;
      // The next item is claimed when the current one starts (its copies hide
      // the atomic's latency) and its table entry is read when the current one's
      // copies are out; the ring is about one item deep, so that read does not
      // starve the MMAs.  Claiming only one item ahead keeps the CTAs' finish
      // times within about one item of each other.
      int item = blockIdx.x;
      TileInfo cur = item_decode(sp, item, item_raw(a, sp, item));  // rows == 0 past the end
      while (ok) {
        if (!queue_push(Q, qp, cur, abort_flag, a.status) || cur.rows == 0) break;
        const int claim = atomicAdd(a.item_counter, 1);  // the next item: gridDim.x + claim
        const int ph = cur.mt >> 16, mt = cur.mt & 0xFFFF;
        if (ph != kPhaseRequant) {  // a requant item has no stages: the epilogue warps do it
          const W4A4Phase& P = a.ph[ph];
          const int kblocks = P.K / kBK;
          const int atoms = P.K / 64;                              // scale atoms per 128-row block
          const size_t plane = (size_t)P.w_rows * (P.K / 16);      // weight scale bytes per expert
          const int a_row = cur.e * P.w_rows + mt * 128;
          const uint8_t* sfa0 = P.sfa + (size_t)cur.e * plane + (size_t)mt * atoms * kAtom;
          const CUtensorMap* tmA = &maps.a[ph];
          constexpr uint32_t tx = kABytes + kSfaBytes;
          for (int kb = 0; kb < kblocks; ++kb) {
            if (!wait_or_abort(R.bar(kBarEmpty + stage), phase ^ 1, abort_flag, a.status)) {
              ok = false;
              break;
            }
            uint8_t* sb = stages + stage * stage_bytes;
            const uint32_t full = R.bar(kBarFull + stage);
            mbar_expect_tx(full, tx);
            tma_load_2d_hint(smem_u32(sb), tmA, full, kb * kRowBytes, a_row, pol_w);
            bulk_load(smem_u32(sb + off_sfa), sfa0 + (size_t)(kb * 4) * kAtom, 4 * kAtom, full);
            last_par[stage] = (int)phase;
            if (++stage == n_stages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
        item = (int)gridDim.x + claim;
        cur = item_decode(sp, item, item_raw(a, sp, item));
      }
      if (!ok || *abort_flag) drain_stages(R, kBarFull, last_par, kMaxStages);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ token producer
    if (lane == 0) {
      int last_par[kMaxStages];
#pragma unroll
      for (int s = 0; s < kMaxStages; ++s) last_par[s] = -1;
      const uint64_t pol_x = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      QueuePos qp;
      bool ok = true;
      while (ok) {
        const TileInfo cur = queue_pop_thread(Q, qp, abort_flag, a.status);
        if (cur.rows == 0) break;
        const int ph = cur.mt >> 16;
        if (ph == kPhaseRequant) continue;
        const W4A4Phase& P = a.ph[ph];
        if (a.fused && ph == 1) {
          // the tile's FC2 input is written by another CTA's epilogue (generic
          // stores); acquire it, then order it before this thread's TMA reads
          if (!wait_flag_geq(a.rq_done + cur.tt, 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
        }
        const int kblocks = P.K / kBK;
        const int atoms = P.K / 64;
        const int n16 = (cur.rows + 15) & ~15;
        const int b_row = cur.tt * kTileRows;
        const uint8_t* sfb0 = P.sfb + (size_t)cur.tt * atoms * kAtom;
        const uint32_t tx = n16 * kRowBytes + 4 * kAtom;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_or_abort(R.bar(kBarEmpty + stage), phase ^ 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          uint8_t* sb = stages + stage * stage_bytes;
          const uint32_t full = R.bar(kBarFull + stage);
          mbar_expect_tx(full, tx);
          for (int r0 = 0; r0 < n16;) {
            // largest box that still fits the rows left: n16 in 1-3 copies
            const int rem = n16 - r0;
            const int lg = rem >= 128 ? 3 : rem >= 64 ? 2 : rem >= 32 ? 1 : 0;
            tma_load_2d_hint(smem_u32(sb + off_b + r0 * kRowBytes), &maps.b[ph].box[lg], full,
                             kb * kRowBytes, b_row + r0, pol_x);
            r0 += 16 << lg;
          }
          bulk_load(smem_u32(sb + off_sfb), sfb0 + (size_t)(kb * 4) * kAtom, 4 * kAtom, full);
          last_par[stage] = (int)phase;
          if (++stage == n_stages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok || *abort_flag) drain_stages(R, kBarFull, last_par, kMaxStages);
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------------ scale staging
    // Atom bytes [16l, 16l+16) hold rows l, l+32, l+64, l+96 (4 scales each);
    // lane l of every quadrant gets them in 4 consecutive columns.
    const uint32_t lane_q = (uint32_t)((warp & 3) * 32) << 16;
    int stage = 0;
    uint32_t phase = 0;
    QueuePos qp;
    bool ok = true;
    while (ok) {
      const TileInfo cur = queue_pop_warp(Q, qp, abort_flag, a.status);
      if (cur.rows == 0) break;
      if ((cur.mt >> 16) == kPhaseRequant) continue;
      const int kblocks = a.ph[cur.mt >> 16].K / kBK;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!wait_or_abort(R.bar(kBarFull + stage), phase, abort_flag, a.status)) {
          ok = false;
          break;
        }
        const uint32_t sb = smem_u32(stages + stage * stage_bytes);
        const uint32_t col0 = tmem + lane_q + sf_base + stage * slot_cols;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          tmem_st4(col0 + 4 * ks, lds128(sb + off_sfa + ks * kAtom + lane * 16));
          tmem_st4(col0 + 16 + 4 * ks, lds128(sb + off_sfb + ks * kAtom + lane * 16));
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(R.bar(kBarSfReady + stage));
        if (++stage == n_stages) {
          stage = 0;
          phase ^= 1;
        }
      }
      ok = __all_sync(0xFFFFFFFFu, ok);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (waits and descriptors are warp-uniform) and
    // elect.sync picks the lane that issues each MMA and commit: a single-lane
    // loop pays ~60 ns of issue latency per MMA, the warp form ~13 ns.
    int stage = 0, local = 0;
    uint32_t phase = 0;
    QueuePos qp;
    bool ok = true, issued = false;
    while (ok) {
      const TileInfo cur = queue_pop_warp(Q, qp, abort_flag, a.status);
      if (cur.rows == 0) break;
      if ((cur.mt >> 16) == kPhaseRequant) continue;
      const int kblocks = a.ph[cur.mt >> 16].K / kBK;
      const int n16 = (cur.rows + 15) & ~15;
      const uint32_t idesc = idesc_mxf4nvf4(128, n16);
      const int buf = local % nbuf;
      const uint32_t acc_par = ((uint32_t)(local / nbuf) & 1u) ^ 1u;
      ok = __all_sync(0xFFFFFFFFu,
                      wait_or_abort(R.bar(kBarAccEmpty + buf), acc_par, abort_flag, a.status));
      if (!ok) break;
      tc_fence_after();
      const uint32_t acc = tmem + buf * acc_stride;
      for (int kb = 0; kb < kblocks; ++kb) {
        // scales staged (which implies the stage's copies landed); the full
        // barrier is re-checked so this warp observes the TMA writes itself
        ok = __all_sync(0xFFFFFFFFu,
                        wait_or_abort(R.bar(kBarSfReady + stage), phase, abort_flag, a.status) &&
                            wait_or_abort(R.bar(kBarFull + stage), phase, abort_flag, a.status));
        if (!ok) break;
        tc_fence_after();
        const uint32_t sb = smem_u32(stages + stage * stage_bytes);
        const uint32_t col0 = tmem + sf_base + stage * slot_cols;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t adesc = smem_desc(sb + ks * 32, 16, 1024, 2);
          const uint64_t bdesc = smem_desc(sb + off_b + ks * 32, 16, 1024, 2);
          mma_mxf4nvf4_warp(acc, adesc, bdesc, idesc, col0 + 4 * ks, col0 + 16 + 4 * ks,
                            (kb | ks) != 0 ? 1u : 0u);
        }
        issued = true;
        tc_commit_warp(R.bar(kBarEmpty + stage));
        if (++stage == n_stages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      tc_commit_warp(R.bar(kBarAccFull + buf));
      ++local;
    }
    if ((!ok || *abort_flag) && issued) {
      // drain the tensor-core work issued so far before TMEM is released
      tc_commit_warp(R.bar(kBarDrain));
      mbar_wait(R.bar(kBarDrain), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Per item: one TMEM lane (weight row r) per thread; 32-token chunks are
    // scaled, activated and written to a shared-memory staging buffer laid out
    // [token][feature], which one thread stores with TMA (16-row boxes).  The
    // next item and its per-token scales are fetched while this one runs.
    const int q = warp & 3;                  // TMEM lane quadrant of this warp
    const int r = q * 32 + lane;             // weight row within the 128-row tile
    const int et = threadIdx.x - 64;         // epilogue thread 0..127
    const bool issuer = et == 0;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    int local = 0;
    int eb = 0;                              // staging buffer of the next chunk
    QueuePos qp;
    // row scale of this thread's token column in an item; in the fused launch the
    // FC2 row scales come from another CTA and are read once the tile is released
    auto row_scale = [&](const TileInfo& t) -> float {
      const int ph = t.mt >> 16;
      if (!t.rows || r >= ((t.rows + 15) & ~15) || ph == kPhaseRequant || (a.fused && ph == 1))
        return 0.0f;
      return a.ph[ph].row_scale[(size_t)t.tt * kTileRows + r];
    };
    TileInfo cur = queue_pop_warp(Q, qp, abort_flag, a.status);
    float s_r = row_scale(cur);
    while (true) {
      if ((cur.mt >> 16) == kPhaseRequant) {
        // FC2-input requant of one token tile: wait until all its FC1 items are
        // stored (their epilogues also folded every row's amax), then quantize
        // the 16-element blocks spread over the 128 threads; the arithmetic of
        // requant_row_warp.
        const int tt = cur.tt, rows = cur.rows, row0 = tt * kTileRows, Ip = a.Ip;
        if (issuer)
          *rq_flag = wait_flag_geq(a.fc1_done + tt, a.ph[0].m_tiles, abort_flag, a.status);
        named_bar_sync(1, 128);
        if (!*rq_flag) break;  // timed out: the abort flag is set
        fence_acq_rel_gpu();
        const float* act0 = a.act + (size_t)row0 * Ip;
        if (et < rows) {
          // the row amax that the tile's FC1 epilogues folded together
          const float mm = a.a2_static ? 1.0f : __uint_as_float(ld_acquire_gpu(
                                                    reinterpret_cast<const int32_t*>(a.row_amax) +
                                                    row0 + et));
          s_scale[et] = mm;
          a.qs[row0 + et] = a.a2_static ? 1.0f : (mm == 0.0f ? 0.0f : __fmul_rn(mm, kRecipeInv));
        }
        named_bar_sync(1, 128);
        requant_blocks(act0, Ip, rows, row0, s_scale, a.a2_static, a.qc, a.qsf, et);
        fence_proxy_async_global();  // the FC2 producers read these rows with TMA
        named_bar_sync(1, 128);
        if (issuer) {
          fence_acq_rel_gpu();
          st_release_gpu(a.rq_done + tt, 1);
        }
        cur = queue_pop_warp(Q, qp, abort_flag, a.status);
        s_r = row_scale(cur);
        continue;
      }
      const int ph = cur.mt >> 16;
      const int mt = cur.mt & 0xFFFF;
      const int tt = cur.tt;
      const int rows = cur.rows;
      const int n16 = (rows + 15) & ~15;
      const int row0 = tt * kTileRows;
      const int buf = local % nbuf;
      const uint32_t acc_par = (uint32_t)(local / nbuf) & 1u;
      const float alpha = rows ? a.ph[ph].alpha[cur.e] : 0.0f;
      // all four epilogue warps take the same stop decision, so none is left
      // waiting alone at a named barrier; the first barrier also ends every
      // read of the previous tile's staged scales
      if (rows == 0 || !wait_or_abort(R.bar(kBarAccFull + buf), acc_par, abort_flag, a.status))
        *epi_stop = 1;
      if (rows && a.fused && ph == 1 && r < n16) {
        // the tile's FC2 input (and its row scales) were released before its
        // MMAs ran; acquire the release on this thread too
        if (wait_flag_geq(a.rq_done + tt, 1, abort_flag, a.status))
          s_r = a.ph[1].row_scale[(size_t)row0 + r];
        else
          *epi_stop = 1;
      }
      named_bar_sync(1, 128);
      s_scale[r] = s_r;
      const bool stop = *epi_stop != 0;
      named_bar_sync(1, 128);
      if (stop) break;
      cur = queue_pop_warp(Q, qp, abort_flag, a.status);  // the next item (rows 0: end)
      s_r = row_scale(cur);
      tc_fence_after();
      const uint32_t acc = tmem + lane_addr + buf * acc_stride;
      for (int c0 = 0; c0 < n16; c0 += cw) {
        const int ncol = min(cw, n16 - c0);
        float v[32];
        tmem_ld16(acc + c0, *reinterpret_cast<float(*)[16]>(v));
        if (ncol > 16) tmem_ld16(acc + c0 + 16, *reinterpret_cast<float(*)[16]>(v + 16));
        tmem_wait_ld();
        if (c0 + cw >= n16) {
          // every TMEM read of this accumulator is done: the MMA may reuse it
          tc_fence_before();
          mbar_arrive(R.bar(kBarAccEmpty + buf));
        }
        // staging buffer eb is free once the store issued from it two chunks ago (one
        // chunk ago with the single buffer) has read it
        if (issuer) {
          if (narrow_epi)
            bulk_wait_group_read<0>();
          else
            bulk_wait_group_read<1>();
        }
        named_bar_sync(1, 128);
        uint8_t* ob = epi_buf + eb * kEpiBufBytes;
        // the chunk's token scales, read up front (32; a 16-token chunk uses the
        // first 16), so the loops below hold no shared-memory load behind a store
        float y[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float4 sc = reinterpret_cast<const float4*>(s_scale + c0)[k];
          y[4 * k + 0] = __fmul_rn(__fmul_rn(v[4 * k + 0], alpha), sc.x);
          y[4 * k + 1] = __fmul_rn(__fmul_rn(v[4 * k + 1], alpha), sc.y);
          y[4 * k + 2] = __fmul_rn(__fmul_rn(v[4 * k + 2], alpha), sc.z);
          y[4 * k + 3] = __fmul_rn(__fmul_rn(v[4 * k + 3], alpha), sc.w);
        }
        int out_x;                           // first output feature of the tile
        uint32_t box_bytes;                  // bytes of one staged token row
        if (ph == 1) {
          uint16_t* o = reinterpret_cast<uint16_t*>(ob);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < ncol) o[j * 128 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(y[j]));
          out_x = mt * 128;
          box_bytes = 128 * 2;
        } else if constexpr (ACT == kFc1Swiglu) {
          // lanes 0-63: gate rows of features mt*64 + (r & 63); lanes 64-127: up rows
          float* g = reinterpret_cast<float*>(ob);
          float* u = g + cw * 64;
          float* dst = r < 64 ? g : u;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < ncol) dst[j * 64 + (r & 63)] = y[j];
          named_bar_sync(1, 128);
          // thread et: feature et & 63 of tokens et/64, et/64 + 2, ...
          const int f = et & 63, jb = et >> 6;
          float yg[16], yu[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            if (jb + 2 * k < ncol) {
              yg[k] = g[(jb + 2 * k) * 64 + f];
              yu[k] = u[(jb + 2 * k) * 64 + f];
            }
          if (a.swiglu_limit > 0.0f) {  // clamped SwiGLU: cap the gate, clip the up value
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              yg[k] = fminf(yg[k], a.swiglu_limit);
              yu[k] = fmaxf(fminf(yu[k], a.swiglu_limit), -a.swiglu_limit);
            }
          }
#pragma unroll
          for (int k = 0; k < 16; ++k)
            if (jb + 2 * k < ncol)
              g[(jb + 2 * k) * 64 + f] =
                  __fmul_rn(__fdividef(yg[k], __fadd_rn(1.0f, __expf(-yg[k]))), yu[k]);
          out_x = mt * 64;
          box_bytes = 64 * 4;
        } else {
          float* o = reinterpret_cast<float*>(ob);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < ncol) {
              const float t = fmaxf(y[j], 0.0f);
              o[j * 128 + r] = __fmul_rn(t, t);
            }
          out_x = mt * 128;
          box_bytes = 128 * 4;
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (issuer) {
          for (int p = 0; p < ncol; p += 16)
            tma_store_2d(&maps.o[ph], smem_u32(ob + p * box_bytes), out_x, row0 + c0 + p);
          bulk_commit_group();
        }
        if (a.fused && ph == 0 && !a.a2_static) {
          // this item's part of each token's row amax (the FC2-input scale): four
          // threads per staged token row, |value| maxima folded with fmaxf as the
          // stand-alone requant does, then one atomic max per row (non-negative
          // floats order like their bit patterns)
          const int j = et >> 2, part = et & 3;
          const int nf = box_bytes / 4;  // staged features per token: 64 or 128
          const float* srow = reinterpret_cast<const float*>(ob) + j * nf + part * (nf / 4);
          float mx = 0.0f;
          for (int k = 0; k < nf / 4; ++k) mx = fmaxf(mx, fabsf(srow[k]));
          mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
          if (part == 0 && j < ncol && c0 + j < rows)
            atomicMax(reinterpret_cast<unsigned int*>(a.row_amax) + row0 + c0 + j,
                      __float_as_uint(mx));
        }
        if (!narrow_epi) eb ^= 1;
      }
      ++local;
      if (a.fused && ph == 0) {
        // count this FC1 item of the tile once its rows (and its part of the row
        // maxima) are in global memory
        named_bar_sync(1, 128);
        if (issuer) {
          bulk_wait_group<0>();
          fence_proxy_async_global();
          atom_add_acq_rel_gpu(a.fc1_done + tt, 1);
        }
      }
    }
    if (issuer) bulk_wait_group<0>();  // every store has completed before the CTA ends
  }

  // Lane 0 of warps 0, 1 and 10 ran its role alone; the warp reconverges before
  // the CTA barrier (bar.sync is a per-warp, aligned barrier), so TMEM is
  // released only after every role has finished.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (a.span && threadIdx.x == 0) atomicMax(a.span + 1, (unsigned long long)globaltimer());
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Self-test of the bounded waits: one thread waits on an mbarrier that nothing
// arrives on, then on a flag that nothing sets, with the same helpers the GEMM
// roles use.  Each wait gives up after its time limit and records
// kFlagWaitTimeout in status[]; the kernel then returns normally.
__global__ void selftest_wait_kernel(const int32_t* never_set, int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_barrier_init();
  abort_flag = 0;
  volatile int* ab = &abort_flag;
  const bool mbar_ok = wait_or_abort(b, 0, ab, status);  // no arrival: times out
  *ab = 0;
  const bool flag_ok = wait_flag_geq(never_set, 1, ab, status);  // never set: times out
  if (mbar_ok || flag_ok) status[kStatusFlags] = 0;  // a wait that "succeeded" fails the test
}

cudaError_t launch_selftest_wait(const int32_t* never_set, int32_t* status, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(never_set, status);
  return cudaGetLastError();
}

template <int ACT>
static cudaError_t launch_act(const W4A4Maps& maps, const W4A4Args& a, int grid, cudaStream_t s) {
  static std::atomic<uint64_t> configured{0};  // per device
  cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(gemm_w4a4_kernel<ACT>),
                                      w4a4::kSmemBytes, configured);
  if (err != cudaSuccess) return err;
  return launch_pdl(gemm_w4a4_kernel<ACT>, dim3(grid), dim3(w4a4::kThreads),
                    (size_t)w4a4::kSmemBytes, s, maps, a);
}

cudaError_t launch_gemm_w4a4(const W4A4Maps& maps, const W4A4Args& a, int act, int grid,
                             cudaStream_t s) {
  return act == kFc1Swiglu ? launch_act<kFc1Swiglu>(maps, a, grid, s)
                           : launch_act<kFc1Relu2>(maps, a, grid, s);
}

}  // namespace moe
