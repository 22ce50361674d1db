// gemm_w4a16.cu -- BF16-activation x NVFP4-weight grouped GEMMs (FC1 with fused
// activation and bf16 handoff, FC2) on tcgen05 tensor cores.
//
// Megatron-LM PR #8262, "How to extend" (BF16 x NVFP4, 'weight_only'): bf16
// hidden states meet the same prepared NVFP4 weights and alphas, no activation
// quantization.  FlashInfer PR #5019, "Tensor and numerical contract": decode
// E2M1 x E4M3 to BF16, accumulate in FP32, then apply the expert alpha; FC1's
// activation comes before a BF16 handoff; FC2 applies alpha before BF16 output.
//
// Operand types: both GEMMs multiply in f16, with the products of the bf16
// contract.  The decoded weights (code x scale: at most 6 significant bits,
// between 2^-10 and 2688) are exact in f16.  The bf16 rows (FC1: the token
// rows, from the gather; FC2: the bf16 handoff rows, converted after FC1) arrive
// in f16, each times a power of two 2^-k that puts its largest magnitude in
// [2^14, 2^15), so every value down to 2^-28 of the row's largest is exact; the
// epilogue multiplies by 2^k.  Scaling a row by a power of two changes no
// rounding of the fp32 accumulation, so the result is that of the bf16
// product.  f16 is chosen because the conversion instructions decode E2M1 and
// E4M3 to f16 directly: about 15 cycles per eight codes and SM sub-partition,
// against 26 for an integer decode to bf16 (measured on GB300).
//
// Structure (swap-AB as in the W4A4 kernel; weights are the M=128 operand and
// are decoded on chip, never written back to global or shared memory):
//   * warp 0: weight producer -- claims items and streams packed E2M1 weight
//     slots (128 rows x 128 B = 256 K elements, 128-byte swizzle, so each row is
//     read in 128-byte runs) with their E4M3 scale atoms (bulk copy)
//   * the last warp: token producer -- one 3-D tiled copy per 256-K block: four
//     64-element K chunks of the tile's 16-bit rows (128-byte swizzle),
//     chunk-major, in the smallest 16/32/64/96/128-row box that covers the item
//   * warps 6..5+kDecodeWarps: decode -- kDecodeWarps/4 warps per TMEM lane
//     quadrant; thread r of quadrant q owns weight row 32q+r: for each 128-K
//     half of a packed slot its warps read the packed bytes and their scales
//     from shared memory, form the exact f16 values of code x scale with the
//     conversion instructions (decode8_f16) and write them into a TMEM A slot
//     (lane = row, 2 K elements per column); the packed slot is released once
//     read
//   * warp 1 (also the TMEM allocator) and warp 6+kDecodeWarps: MMA issuers --
//     tcgen05.mma.kind::f16 with A from TMEM and B from shared memory, K = 16
//     per instruction, N = the tile's token count rounded up to 16; the first
//     issues the even K steps into one partial sum, the second the odd ones
//     into another, each from a whole warp with elect.sync (a single-lane loop
//     is bound by issue latency at small N)
//   * warps 2-5: epilogue (alpha, the row scales 2^k, activation, bf16
//     rounding), one TMEM lane per thread; SwiGLU pairs gate and up rows through
//     shared memory as in W4A4
//   * rings: packed-weight slots (4-9 of 18 KB, as many as shared memory holds
//     next to a few token stages, each released as soon as the decode warps have
//     read it into registers), TMEM slots of decoded weights (1-3 blocks of
//     256 K) and token stages (2-8 blocks of 256 K, loaded ahead of the MMAs
//     independently of the decode); each item's accumulator is split into even
//     / odd K-step partial sums; two items in flight (launches with tiles of
//     more than 96 tokens run each tile as two items of up to 64 rows); every
//     wait bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace w4a16 {
constexpr int kRawK = 256;                  // K elements per packed-weight slot
constexpr int kRawBytes = 128 * kRawK / 2;  // 16 KB: 128 rows x 128 B (128-byte swizzle)
constexpr int kAtom = 512;
constexpr int kSfaBytes = 4 * kAtom;        // 4 K-atoms (4 scale columns each)
constexpr int kRawSlotBytes = kRawBytes + kSfaBytes;
constexpr int kBK = kRawK;                  // K elements per token stage / decoded TMEM slot
constexpr int kChunks = kBK / 64;           // 64-element (128-byte) K chunks per token stage
constexpr int kChunkRowBytes = 128;         // 64 f16 per row per K chunk
constexpr int kACols = kBK / 2;             // TMEM columns of one decoded A slot
constexpr int kMaxRaw = 10;                 // packed-weight slots (released once read)
constexpr int kMaxRing = 3;                 // TMEM slots of decoded A (blocks being decoded / multiplied)
constexpr int kMaxTok = 8;                  // token stages (each one 256-K block of the token tile)
constexpr int kMaxAcc = 2;
constexpr int kTmemCols = 512;
constexpr int kXchgFloats = 2 * 64 * 33;
constexpr int kXchgBytes = (kXchgFloats * 4 + 1023) / 1024 * 1024;
constexpr int kBarBytes = 2048;
constexpr int kSmemBytes = 227 * 1024;
constexpr int kRingBudget = kSmemBytes - 1024 - kBarBytes - kXchgBytes;
constexpr int kDecodeWarps = 8;             // warps 6.., kDecodeWarps / 4 per TMEM lane quadrant
constexpr int kDecodePerQuad = kDecodeWarps / 4;
constexpr int kChunksPerWarp = 4 / kDecodePerQuad;  // 16-byte chunks of a 128-K half per warp
constexpr int kIssuers = 2;                 // MMA issuers: even and odd K steps
constexpr int kIssuerWarp1 = 6 + kDecodeWarps;      // warp of the second issuer
constexpr int kTokenWarp = 7 + kDecodeWarps;        // token-stage producer
constexpr int kThreads = (8 + kDecodeWarps) * 32;
static_assert(kDecodePerQuad * 4 == kDecodeWarps && kChunksPerWarp * kDecodePerQuad == 4 &&
                  kChunksPerWarp <= 2, "decode: a warp's chunks share one scale atom");
constexpr int kBarRawFull = 0;
constexpr int kBarRawEmpty = kBarRawFull + kMaxRaw;
constexpr int kBarFull = kBarRawEmpty + kMaxRaw;          // token stage landed (TMA bytes)
constexpr int kBarTokEmpty = kBarFull + kMaxTok;          // token stage's MMAs are done
constexpr int kBarReady = kBarTokEmpty + kMaxTok;         // A slot decoded
constexpr int kBarFree = kBarReady + kMaxRing;            // A slot's MMAs are done
constexpr int kBarAccFull = kBarFree + kMaxRing;
constexpr int kBarAccEmpty = kBarAccFull + kMaxAcc;
constexpr int kBarItemFull = kBarAccEmpty + kMaxAcc;
constexpr int kBarItemEmpty = kBarItemFull + kItemSlots;
constexpr int kBarDrain = kBarItemEmpty + kItemSlots;
constexpr int kNumBars = kBarDrain + kIssuers;
constexpr int kFlagsOff = 8 * kNumBars;
constexpr int kRingOff = 768;
static_assert(kFlagsOff + 16 <= kRingOff && kRingOff + 16 * kItemSlots <= 1024, "flag area");
// Token boxes: the smallest of 16/32/64/96/128 rows >= n16; box_map(n16) is its
// tensor map (maps 0-3: 16 << i rows, map 4: 96 rows).
__device__ __forceinline__ int box_map(int n16) {
  return n16 <= 16 ? 0 : n16 <= 32 ? 1 : n16 <= 64 ? 2 : n16 <= 96 ? 4 : 3;
}
// Work items of a launch whose token tiles are split in halves (split = 2):
// item = base x split + h, base numbered as tile_decode numbers items, half h
// the tile's rows 64 h .. 64 h + 63.  The second half of a tile of at most 64
// rows decodes with rows -1 (no work); past the end, rows 0.  The half rides
// in bits 16.. of TileInfo::mt.
constexpr int kSplitRows = 64;
__device__ __forceinline__ int4 split_raw(const GemmArgs& a, int item, int n_items, int split) {
  return tile_raw(a, item / split, n_items / split);
}
__device__ __forceinline__ TileInfo split_decode(const GemmArgs& a, int item, int n_items,
                                                 int split, const int4& raw) {
  TileInfo t = tile_decode(a, item / split, n_items / split, raw);
  if (split == 1 || t.rows == 0) return t;
  const int h = item % split;
  const int rows = h == 0 ? min(kSplitRows, t.rows) : t.rows - kSplitRows;
  t.rows = rows > 0 ? rows : -1;
  t.mt |= h << 16;
  return t;
}
__device__ __forceinline__ int box_rows(int n16) {
  return n16 <= 16 ? 16 : n16 <= 32 ? 32 : n16 <= 64 ? 64 : n16 <= 96 ? 96 : 128;
}
}  // namespace w4a16

template <int MODE>
__global__ void __launch_bounds__(w4a16::kThreads, 1)
    gemm_w4a16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ TokenMaps tmB,
                      const GemmArgs a) {
  using namespace w4a16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const Ring R{smem};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kFlagsOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_stop = reinterpret_cast<volatile int*>(tmem_slot + 2);
  const ItemQueue Q{reinterpret_cast<int4*>(smem + kRingOff), R.bar(kBarItemFull),
                    R.bar(kBarItemEmpty)};
  float* xchg = reinterpret_cast<float*>(smem + kBarBytes);
  float* s_rs = reinterpret_cast<float*>(smem + 1024);  // row scales of the current tile (128)
  uint8_t* rings = smem + kBarBytes + kXchgBytes;     // 1024-aligned

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxRaw; ++s) {
      mbar_init(R.bar(kBarRawFull + s), 1);
      mbar_init(R.bar(kBarRawEmpty + s), kDecodeWarps);
    }
    for (int j = 0; j < kMaxTok; ++j) {
      mbar_init(R.bar(kBarFull + j), 1);
      mbar_init(R.bar(kBarTokEmpty + j), kIssuers);
    }
    for (int j = 0; j < kMaxRing; ++j) {
      mbar_init(R.bar(kBarReady + j), kDecodeWarps);
      mbar_init(R.bar(kBarFree + j), kIssuers);
    }
    for (int b = 0; b < kMaxAcc; ++b) {
      mbar_init(R.bar(kBarAccFull + b), kIssuers);
      mbar_init(R.bar(kBarAccEmpty + b), 128);
    }
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(R.bar(kBarItemFull + s), 1);
      mbar_init(R.bar(kBarItemEmpty + s), kIssuers + kDecodeWarps + 4 + 1);
    }
    for (int i = 0; i < kIssuers; ++i) mbar_init(R.bar(kBarDrain + i), 1);
    *abort_flag = 0;
    *epi_stop = 0;
    fence_barrier_init();
    prefetch_tmap(&tmA);
    for (int i = 0; i < 5; ++i) prefetch_tmap(&tmB.box[i]);
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

  // Launches with tiles of more than 96 tokens run each tile as two items of up
  // to kSplitRows rows (the weight tile decoded once per half, its second read
  // an L2 hit on a neighbouring CTA), so that two items are in flight next to
  // two decoded A slots in TMEM.  Measured on GB300: H7168/I2048/E256 top-8
  // T=4096 (128-token tiles) FC2 1268 -> 1104 us; at 65-96-token tiles two
  // whole items and one A slot are faster (E384 T=4096 FC1 2291 vs 2630 us).
  const int max_rows = a.status[kStatusMaxRows];
  const int split = max_rows > 96 ? 2 : 1;
  const int n_items = a.status[kStatusTiles] * a.m_tiles * split;
  const int max_n16 = (min(max_rows, kSplitRows * (3 - split)) + 15) & ~15;
  // A token stage is one 3-D box: kChunks 64-K chunks of box_rows(n16) rows
  // each, chunk-major, so chunk c of a tile starts c x box_rows x 128 bytes in.
  const int stage_bytes = kChunks * box_rows(max_n16) * kChunkRowBytes;  // multiple of 1024
  // Each item accumulates into two partial sums (even and odd K steps, each
  // issued by its own warp), added in a fixed order in the epilogue.  The
  // split never depends on the batch, so results stay bitwise batch invariant.
  // Two items are in flight (the epilogue of one overlaps the MMAs of the
  // next) up to 96-token tiles, where the accumulators leave TMEM room for a
  // single decoded A slot (measured on GB300 at 65-96-token tiles: FC1 and FC2
  // 16% and 17% faster than two A slots with one item in flight); one item
  // beyond.
  const int acc_cols = (max_n16 + 31) & ~31;
  const int nacc = kIssuers;
  const int acc_stride = nacc * acc_cols;                  // TMEM columns per item
  const int nbuf = max_n16 <= 96 ? 2 : 1;                  // accumulator buffers
  const int a_base = nbuf * acc_stride;                    // decoded A slots follow the accumulators
  // Shared memory goes first to packed-weight slots: the weight stream needs
  // its bytes in flight to cover the memory latency under load (measured on
  // GB300: with 6 slots of 18 KB the decode warps waited for weights 80% of the
  // time), then to token stages (at least 4, or 2 for 128-row tiles).
  const int tok_min = max_n16 <= 64 ? 4 : 2;
  const int n_raw = min(kMaxRaw, (kRingBudget - tok_min * stage_bytes) / kRawSlotBytes);
  uint8_t* raw_ring = rings;
  uint8_t* stage_ring = rings + n_raw * kRawSlotBytes;     // multiple of 1024 past rings
  // Block b of the CTA's K stream uses TMEM A slot b % n_ring and token stage
  // b % n_tok, so token loads run ahead of the MMAs independently of the decode.
  const int n_ring = min(kMaxRing, (kTmemCols - a_base) / kACols);
  const int n_tok = min(kMaxTok, (kRingBudget - n_raw * kRawSlotBytes) / stage_bytes);

  const int kraw = a.K / kRawK;                        // packed-weight slots per item
  const int atoms = a.K / 64;
  const size_t plane = (size_t)a.w_rows * (a.K / 16);

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    // Claims items, publishes them to the other roles and streams the packed
    // weight slots (one tiled copy of 128 rows x 256 K and one bulk copy of
    // their scale atoms per slot).
    if (lane == 0) {
      int last_raw[kMaxRaw];
#pragma unroll
      for (int s = 0; s < kMaxRaw; ++s) last_raw[s] = -1;
      const uint64_t pol_w = policy_evict_first();
      int rs = 0;
      uint32_t rphase = 0;
      QueuePos qp;
      bool ok = true;
      // Items are claimed two ahead and their table entries loaded one ahead;
      // the raw values are only used an item later, so neither the atomic's nor
      // the load's latency stalls the copy stream.
      int item = blockIdx.x;
      // rows == 0 past the end, -1 for an empty half (neither published nor loaded)
      TileInfo cur = split_decode(a, item, n_items, split, split_raw(a, item, n_items, split));
      int next = (int)gridDim.x + (item < n_items ? atomicAdd(a.item_counter, 1) : n_items);
      int4 next_raw = split_raw(a, next, n_items, split);
      int claim = next < n_items ? atomicAdd(a.item_counter, 1) : n_items;  // raw counter value
      while (ok) {
        if (cur.rows >= 0 && (!queue_push(Q, qp, cur, abort_flag, a.status) || cur.rows == 0))
          break;
        const int next2 = (int)gridDim.x + claim;         // claimed one item ago
        const int4 next2_raw = split_raw(a, next2, n_items, split);
        claim = next2 < n_items ? atomicAdd(a.item_counter, 1) : n_items;
        const TileInfo nxt = split_decode(a, next, n_items, split, next_raw);  // loaded one item ago
        const int mt = cur.mt & 0xFFFF;
        const int a_row = cur.e * a.w_rows + mt * 128;
        const uint8_t* sfa0 = a.sfa + (size_t)cur.e * plane + (size_t)mt * atoms * kAtom;
        for (int kr = 0; kr < (cur.rows > 0 ? kraw : 0); ++kr) {
          if (!wait_or_abort(R.bar(kBarRawEmpty + rs), rphase ^ 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          uint8_t* rb = raw_ring + rs * kRawSlotBytes;
          const uint32_t rfull = R.bar(kBarRawFull + rs);
          mbar_expect_tx(rfull, kRawSlotBytes);
          tma_load_2d_hint(smem_u32(rb), &tmA, rfull, kr * (kRawK / 2), a_row, pol_w);
          bulk_load(smem_u32(rb + kRawBytes), sfa0 + (size_t)(kr * 4) * kAtom, kSfaBytes, rfull);
          last_raw[rs] = (int)rphase;
          if (++rs == n_raw) {
            rs = 0;
            rphase ^= 1;
          }
        }
        cur = nxt;
        next = next2;
        next_raw = next2_raw;
      }
      if (!ok || *abort_flag) {
        for (int s = 0; s < kMaxRaw; ++s)
          if (last_raw[s] >= 0) mbar_wait(R.bar(kBarRawFull + s), (uint32_t)last_raw[s]);
      }
    }
  } else if (warp == kTokenWarp) {
    // ------------------------------------------------------------ token producer
    // One 3-D tiled copy per token stage: the kChunks 64-K chunks of the tile's
    // rows, in the smallest of the 16/32/64/128-row boxes that covers them.  A
    // stage is refilled once both MMA issuers have finished with it.
    if (lane == 0) {
      int last_stg[kMaxTok];
#pragma unroll
      for (int s = 0; s < kMaxTok; ++s) last_stg[s] = -1;
      const uint64_t pol_x = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      QueuePos qp;
      bool ok = true;
      while (ok) {
        const TileInfo cur = queue_pop_thread(Q, qp, abort_flag, a.status);
        if (cur.rows == 0) break;
        const int n16 = (cur.rows + 15) & ~15;
        const int bl = box_map(n16);
        const uint32_t tx = (uint32_t)(kChunks * box_rows(n16) * kChunkRowBytes);
        const int b_row = cur.tt * kTileRows + kSplitRows * (cur.mt >> 16);
        for (int kb = 0; kb < a.K / kBK; ++kb) {
          if (!wait_or_abort(R.bar(kBarTokEmpty + stage), phase ^ 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          const uint32_t full = R.bar(kBarFull + stage);
          mbar_expect_tx(full, tx);
          tma_load_3d_hint(smem_u32(stage_ring + stage * stage_bytes), &tmB.box[bl], full, 0,
                           b_row, kChunks * kb, pol_x);
          last_stg[stage] = (int)phase;
          if (++stage == n_tok) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok || *abort_flag) {
        for (int s = 0; s < kMaxTok; ++s)
          if (last_stg[s] >= 0) mbar_wait(R.bar(kBarFull + s), (uint32_t)last_stg[s]);
      }
    }
  } else if (warp >= 6 && warp < 6 + kDecodeWarps) {
    // ------------------------------------------------------------ decode into TMEM
    // Packed row m: 128 B per slot (256 K), 16-byte chunk c stored at chunk
    // c ^ (m & 7) (128-byte swizzle).  A packed slot becomes one TMEM A slot:
    // half h (K 128h..128h+127, chunks 4h..4h+3) goes to columns 64h..64h+63;
    // the kDecodePerQuad warps of a quadrant split each half's four chunks.
    const int q = warp & 3;
    const int wq = (warp - 6) >> 2;            // warp within its quadrant
    const int m = q * 32 + lane;                 // weight row of this thread
    const uint32_t lane_q = (uint32_t)(q * 32) << 16;
    const uint32_t swz = (uint32_t)(m & 7);
    int rs = 0, slot = 0;
    uint32_t rphase = 0, aphase = 0;
    QueuePos qp;
    bool ok = true;
    while (ok) {
      const TileInfo cur = queue_pop_warp(Q, qp, abort_flag, a.status);
      if (cur.rows == 0) break;
      for (int kr = 0; kr < kraw && ok; ++kr) {
        // the packed slot has landed: read this warp's part of it into
        // registers (row m's chunks and their block-scale words) and release it
        // at once, before waiting for a TMEM slot
        if (!wait_or_abort(R.bar(kBarRawFull + rs), rphase, abort_flag, a.status)) {
          ok = false;
          break;
        }
        const uint32_t rb = smem_u32(raw_ring + rs * kRawSlotBytes);
        uint32_t sw[2];
        uint4 raws[2][kChunksPerWarp];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // row m's block scales of this warp's chunks: one 4-scale word of atom
          // 2h (chunks 0-1) or 2h+1 (chunks 2-3)
          const int atom = 2 * h + (kChunksPerWarp * wq >= 2 ? 1 : 0);
          sw[h] = lds32(rb + kRawBytes + atom * kAtom + (m & 31) * 16 + (m >> 5) * 4);
#pragma unroll
          for (int cc = 0; cc < kChunksPerWarp; ++cc) {
            const int c = kChunksPerWarp * wq + cc;
            raws[h][cc] = lds128(rb + m * 128 + (((uint32_t)(4 * h + c) ^ swz) << 4));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(R.bar(kBarRawEmpty + rs));
        if (++rs == n_raw) {
          rs = 0;
          rphase ^= 1;
        }
        // decode into registers while the TMEM slot may still be in use
        uint32_t o[2][kChunksPerWarp][16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int cc = 0; cc < kChunksPerWarp; ++cc) {  // 32 elements per 16-byte chunk
            const int c = kChunksPerWarp * wq + cc;        // chunk within the half
            const uint4 raw = raws[h][cc];
            uint32_t sc0, sc1;
            e4m3x2_scale_f16x2(sw[h] >> (16 * (c & 1)), sc0, sc1);
            decode8_f16(raw.x, sc0, o[h][cc]);
            decode8_f16(raw.y, sc0, o[h][cc] + 4);
            decode8_f16(raw.z, sc1, o[h][cc] + 8);
            decode8_f16(raw.w, sc1, o[h][cc] + 12);
          }
        }
        // the TMEM slot's previous MMAs are done
        if (!wait_or_abort(R.bar(kBarFree + slot), aphase ^ 1, abort_flag, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acol = tmem + lane_q + a_base + slot * kACols;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int cc = 0; cc < kChunksPerWarp; ++cc)
            tmem_st16(acol + 64 * h + 16 * (kChunksPerWarp * wq + cc), o[h][cc]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(R.bar(kBarReady + slot));
        if (++slot == n_ring) {
          slot = 0;
          aphase ^= 1;
        }
      }
      ok = __all_sync(0xFFFFFFFFu, ok);
    }
  } else if (warp == 1 || warp == kIssuerWarp1) {
    // ------------------------------------------------------------ MMA issuers
    // Issuer `part` (warp 1: 0, the last warp: 1) issues the K steps of its
    // parity into its partial sum.  The whole warp runs the loop (waits and
    // descriptors are warp-uniform) and elect.sync picks the lane that issues
    // each MMA and commit: that keeps the MMA rate near the tensor pipe's even
    // for 16-token tiles, where a single-lane loop is bound by issue latency.
    const int part = warp == 1 ? 0 : 1;
    int slot = 0, local = 0, ts = 0;
    uint32_t aphase = 0, tphase = 0;
    QueuePos qp;
    bool ok = true, issued = false;
    const int kblocks = a.K / kBK;
    while (ok) {
      const TileInfo cur = queue_pop_warp(Q, qp, abort_flag, a.status);
      if (cur.rows == 0) break;
      const int n16 = (cur.rows + 15) & ~15;
      const uint32_t idesc = idesc_f16(128, n16);  // f16 weights and f16 rows
      const int chunk_bytes = box_rows(n16) * kChunkRowBytes;  // this tile's chunk stride
      const int buf = local % nbuf;
      const uint32_t acc_par = ((uint32_t)(local / nbuf) & 1u) ^ 1u;
      ok = __all_sync(0xFFFFFFFFu,
                      wait_or_abort(R.bar(kBarAccEmpty + buf), acc_par, abort_flag, a.status));
      if (!ok) break;
      tc_fence_after();
      const uint32_t acc = tmem + buf * acc_stride + part * acc_cols;
      for (int kb = 0; kb < kblocks; ++kb) {
        // the block's decoded weights and its token stage
        ok = __all_sync(0xFFFFFFFFu,
                        wait_or_abort(R.bar(kBarReady + slot), aphase, abort_flag, a.status) &&
                            wait_or_abort(R.bar(kBarFull + ts), tphase, abort_flag, a.status));
        if (!ok) break;
        tc_fence_after();
        const uint32_t sb = smem_u32(stage_ring + ts * stage_bytes);
        const uint32_t acol = tmem + a_base + slot * kACols;
#pragma unroll
        for (int kp = 0; kp < kBK / 32; ++kp) {
          const int ks = 2 * kp + part;
          const uint64_t bdesc = smem_desc(sb + (ks >> 2) * chunk_bytes + (ks & 3) * 32, 16, 1024, 2);
          mma_f16_ts_warp(acc, acol + 8 * ks, bdesc, idesc, (kb == 0 && kp == 0) ? 0u : 1u);
        }
        issued = true;
        tc_commit_warp(R.bar(kBarFree + slot));
        tc_commit_warp(R.bar(kBarTokEmpty + ts));
        if (++slot == n_ring) {
          slot = 0;
          aphase ^= 1;
        }
        if (++ts == n_tok) {
          ts = 0;
          tphase ^= 1;
        }
      }
      if (!ok) break;
      tc_commit_warp(R.bar(kBarAccFull + buf));
      ++local;
    }
    if ((!ok || *abort_flag) && issued) {
      tc_commit_warp(R.bar(kBarDrain + part));
      mbar_wait(R.bar(kBarDrain + part), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    int local = 0;
    QueuePos qp;
    while (true) {
      const TileInfo cur = queue_pop_warp(Q, qp, abort_flag, a.status);
      const int mt = cur.mt & 0xFFFF;
      const int rows = cur.rows;
      const int n16 = (rows + 15) & ~15;
      const int row0 = cur.tt * kTileRows + kSplitRows * (cur.mt >> 16);
      const int buf = local % nbuf;
      const uint32_t acc_par = (uint32_t)(local / nbuf) & 1u;
      // each token column's f16 row was multiplied by a power of two 2^-k when
      // it was formed; 2^k, the row scale, undoes it exactly
      const float alpha = rows ? a.alpha[cur.e] : 0.0f;
      const float rs = r < rows ? a.row_scale[(size_t)row0 + r] : 0.0f;
      if (rows == 0 || !wait_or_abort(R.bar(kBarAccFull + buf), acc_par, abort_flag, a.status))
        *epi_stop = 1;
      named_bar_sync(1, 128);
      // every thread is past the previous tile's reads of s_rs
      s_rs[r] = rs;
      const bool stop = *epi_stop != 0;
      named_bar_sync(1, 128);
      if (stop) break;
      tc_fence_after();
      const uint32_t acc = tmem + lane_addr + buf * acc_stride;
      if constexpr (MODE == kFc1Swiglu) {
        // Rows 0-63 of the weight tile are the gate rows and 64-127 the up rows
        // of the same 64 features.  For each chunk of 32 tokens every thread
        // publishes its row's alpha-scaled sums in shared memory; then thread r
        // forms the activations of feature r % 64 for tokens 16 (r / 64) ..
        // 16 (r / 64) + 15 of the chunk, so that all 128 threads share the
        // activation work.
        const int fl = r & 63;
        const int j0 = 16 * (r >> 6);
        const int f = mt * 64 + fl;
        const float* xg = xchg + fl * 33;             // gate sums of feature fl
        const float* xu = xchg + (64 + fl) * 33;      // up sums of feature fl
        float* mine = xchg + r * 33;
        for (int c0 = 0; c0 < n16; c0 += 32) {
          float v[32];
          tmem_ld16(acc + c0, *reinterpret_cast<float(*)[16]>(v));
          if (c0 + 16 < n16) tmem_ld16(acc + c0 + 16, *reinterpret_cast<float(*)[16]>(v + 16));
          if (nacc == 2) {
            float w[32];
            tmem_ld16(acc + acc_cols + c0, *reinterpret_cast<float(*)[16]>(w));
            if (c0 + 16 < n16)
              tmem_ld16(acc + acc_cols + c0 + 16, *reinterpret_cast<float(*)[16]>(w + 16));
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __fadd_rn(v[j], w[j]);
          }
          tmem_wait_ld();
          const int ncol = min(32, n16 - c0);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < ncol) mine[j] = __fmul_rn(__fmul_rn(v[j], alpha), s_rs[c0 + j]);
          named_bar_sync(1, 128);
          const int jend = min(j0 + 16, min(ncol, rows - c0));
          for (int j = j0; j < jend; ++j) {
            const size_t p = (size_t)row0 + c0 + j;
            float yg = xg[j];
            float yu = xu[j];
            if (a.swiglu_limit > 0.0f) {  // clamped SwiGLU: cap the gate, clip the up value
              yg = fminf(yg, a.swiglu_limit);
              yu = fmaxf(fminf(yu, a.swiglu_limit), -a.swiglu_limit);
            }
            const float act = __fmul_rn(__fdiv_rn(yg, __fadd_rn(1.0f, expf(-yg))), yu);
            a.route_out[p * a.I + f] = __bfloat16_as_ushort(__float2bfloat16_rn(act));
          }
          named_bar_sync(1, 128);  // the chunk's sums are read before the next one lands
        }
      } else {
        for (int c0 = 0; c0 < n16; c0 += 16) {
          float v[16];
          tmem_ld16(acc + c0, v);
          if (nacc == 2) {
            float w[16];
            tmem_ld16(acc + acc_cols + c0, w);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __fadd_rn(v[j], w[j]);
          }
          tmem_wait_ld();
#pragma unroll 4
          for (int j = 0; j < 16; ++j) {
            const int col = c0 + j;
            if (col >= rows) break;
            const size_t p = (size_t)row0 + col;
            const float y = __fmul_rn(__fmul_rn(v[j], alpha), s_rs[col]);
            if constexpr (MODE == kFc1Relu2) {
              const float t = fmaxf(y, 0.0f);
              a.route_out[p * a.I + mt * 128 + r] =
                  __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(t, t)));
            } else {
              a.route_out[p * a.H + mt * 128 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(R.bar(kBarAccEmpty + buf));
      ++local;
    }
  }

  // Lane 0 of warps 0 and 1 ran its role alone; the warp reconverges before
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

template <int MODE>
static cudaError_t launch_w4a16_mode(const CUtensorMap& tmA, const TokenMaps& tmB,
                                     const GemmArgs& a, int grid, cudaStream_t s) {
  static std::atomic<uint64_t> configured{0};  // per device
  cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(gemm_w4a16_kernel<MODE>),
                                      w4a16::kSmemBytes, configured);
  if (err != cudaSuccess) return err;
  return launch_pdl(gemm_w4a16_kernel<MODE>, dim3(grid), dim3(w4a16::kThreads),
                    (size_t)w4a16::kSmemBytes, s, tmA, tmB, a);
}

cudaError_t launch_gemm_w4a16(const CUtensorMap& tmA, const TokenMaps& tmB, const GemmArgs& a,
                              int grid, cudaStream_t s) {
  switch (a.mode) {
    case kFc1Relu2: return launch_w4a16_mode<kFc1Relu2>(tmA, tmB, a, grid, s);
    case kFc1Swiglu: return launch_w4a16_mode<kFc1Swiglu>(tmA, tmB, a, grid, s);
    default: return launch_w4a16_mode<kFc2>(tmA, tmB, a, grid, s);
  }
}

}  // namespace moe
