// internal.h -- declarations shared by the host runtime and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <utility>

namespace moe {

// Rows of one token tile of the grouped GEMMs.  Every expert group in the
// permuted buffers starts at a multiple of this, so a tile has one expert.
constexpr int kTileRows = 128;
// Batches of at most this many routes, and at most kFusedRoutesPerExpert routes
// per expert on average, run FC1 -> requant -> FC2 as one launch (measured on
// GB300: 2-11% faster at 1-4 routes per expert, 4% slower at 16).
constexpr int64_t kFusedMaxRoutes = 2048;
constexpr int64_t kFusedRoutesPerExpert = 8;

// Workspace status words (int32).
constexpr int kStatusFlags = 0;   // error bits, see below
constexpr int kStatusTiles = 1;   // number of token tiles after the scan
constexpr int kStatusRows = 2;    // padded rows in use after the scan
constexpr int kStatusMaxRows = 3; // largest token tile (rows) after the scan
constexpr int kStatusItemCtr = 4; // two work-item counters (FC1, FC2), zeroed by the scan
constexpr int kStatusWords = 16;

constexpr int kFlagBadExpertId = 1;   // an id outside [-1, E) was seen (slot ignored)
// The routing scan rewrites every status word each forward (no separate reset).
constexpr int kFlagWaitTimeout = 2;   // a bounded in-kernel wait gave up

struct RouteArgs {
  int TK, K, E, H;
  int Hp;  // H rounded up to 256: row length of the permuted token rows
  int w4a16;
  const int32_t* ids;
  int ids64;  // ids are int64 (read as two int32 words)
  int32_t* status;
  int32_t* chunk_counts;
  int32_t* chunk_prefix;
  int32_t* counts;
  int32_t* group_row0;
  int4* tiles;  // per token tile: {expert, expert's first tile, expert's tiles, expert's routes}
  int32_t* tile_sync;     // fused GEMM: per-tile counters zeroed by the scan (or null)
  int tile_sync_words;
  int32_t* inv;
  int32_t* perm;
  // W4A4 gather
  const uint8_t* xc;
  const uint8_t* xsf;
  const float* xs;
  uint8_t* pc;
  uint8_t* psf;
  float* ps;
  // W4A16 gather
  const void* xb;
  void* pb;
};

// Grouped GEMM over the token tiles produced by the routing scan.
// A = weights (rows of one expert, K-major), B = permuted token rows (K-major).
enum GemmMode { kFc1Relu2 = 0, kFc1Swiglu = 1, kFc2 = 2 };

struct GemmArgs {
  int mode;            // GemmMode
  int K;               // reduction length (H for FC1, I for FC2)
  int m_tiles;         // 128-row weight tiles per expert
  int w_rows;          // weight rows per expert (N1 for FC1, H for FC2)
  const uint8_t* sfa;  // weight scales, swizzled, [E][w_rows * K/16]
  const uint8_t* sfb;  // token scales, swizzled over permuted rows
  const float* alpha;  // [E]
  const float* row_scale;  // per permuted row: s_t (FC1) or s2 (FC2)
  const int4* tiles;   // per token tile: {expert, first tile, tiles, routes} of its expert
  int32_t* status;
  int32_t* item_counter;  // work items claimed beyond the first gridDim.x (zeroed by the scan)
  float* act_out;      // FC1: [rows][I] fp32
  int I;
  uint16_t* route_out; // FC2: [rows][H] bf16
  int H;
  float swiglu_limit;  // > 0: clamped SwiGLU (W4A16 FC1)
  unsigned long long* span;  // profiling: [0] min CTA start, [1] max CTA end (%globaltimer), or null
};

// Launch with programmatic stream serialization: the kernel may start while the
// previous kernel of the stream finishes; it calls pdl_wait() before reading
// anything that kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current device,
// once per device: the attribute belongs to the function on each device, so a
// process that uses several devices sets it on each.  `done` holds one bit per
// device (devices 0-63) and is only set after the call succeeded; two threads
// racing on the first launch both make the (idempotent) call.
inline cudaError_t ensure_smem_limit(const void* fn, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const uint64_t bit = uint64_t(1) << dev;
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// static_enc: null for the per-token recipe, else the device encode scale a1 of
// the per-tensor recipe (scale is then not written).
void launch_quantize_tokens(int T, int H, int Hp, const void* x, uint8_t* codes, uint8_t* sf,
                            float* scale, const float* static_enc, cudaStream_t s);
// a_scale: null, or the device static input scale folded into alpha.
void launch_prepare_fc(int E, int N, int D, int Np, int Dp, int swiglu_I, const void* w,
                       uint8_t* codes, uint8_t* sf, float* alpha, const float* a_scale,
                       cudaStream_t s);
cudaError_t launch_route(const RouteArgs& a, cudaStream_t s);
// W4A16: the bf16 activated rows of the valid routes as f16 rows times 2^-k,
// 2^k per row in scale (the f16 FC2 GEMM's operand).
void launch_act_f16(int TK, int Ip, const int32_t* inv, const void* act, void* act16,
                    float* scale, cudaStream_t s);
void launch_route_topk(int T, int E, int K, const float* logits, int32_t* ids, float* w,
                       cudaStream_t s);
void launch_requant(int TK, int I, const int32_t* inv, const float* act, uint8_t* qc, uint8_t* qsf,
                    float* qs, const float* static_enc, cudaStream_t s);
void launch_finalize(int T, int K, int H, int Hp, const int32_t* inv, const float* w,
                     const void* route, void* out, cudaStream_t s);
// One GEMM of the W4A4 kernel (FC1 or FC2).
struct W4A4Phase {
  int K;                   // reduction length (Hp for FC1, Ip for FC2)
  int m_tiles;             // 128-row weight tiles per expert
  int w_rows;              // weight rows per expert
  const uint8_t* sfa;      // weight scales, swizzled, [E][w_rows * K/16]
  const uint8_t* sfb;      // token scales, swizzled over permuted rows
  const float* alpha;      // [E]
  const float* row_scale;  // per permuted row: s_t (FC1) or s2 (FC2)
};

// Arguments of one W4A4 GEMM launch: FC1 items, FC2 items, or both.  Fused
// (both phases, one launch): the epilogue that stores a token tile's last FC1
// item requantizes that tile's rows and releases rq_done[tile]; the token
// producer of an FC2 item waits for it.  Items are claimed in order, FC1 items
// first, and every wait is on a lower-numbered item, so the launch always makes
// progress while its CTAs are resident.
struct W4A4Args {
  W4A4Phase ph[2];          // [0] FC1, [1] FC2
  int run_fc1, run_fc2, fused;
  const int4* tiles;        // per token tile: {expert, first tile, tiles, routes}
  int32_t* status;
  int32_t* item_counter;    // items claimed beyond the first gridDim.x (zeroed by the scan)
  int32_t* fc1_done;        // fused: per token tile, FC1 items whose rows are stored
  int32_t* rq_done;         // fused: per token tile, 1 once its FC2 input is quantized
  float* row_amax;          // fused: per permuted row, amax of the activated row (atomic max)
  const float* act;         // fused requant: fp32 activated rows [rows][Ip]
  int Ip;
  uint8_t* qc;              // FC2-input codes [rows][Ip/2]
  uint8_t* qsf;             // FC2-input scales, swizzled
  float* qs;                // FC2-input row scales
  const float* a2_static;   // per-tensor recipe: static FC2-input encode scale (else null)
  float swiglu_limit;       // > 0: clamped SwiGLU (gate <= L, |up| <= L)
  unsigned long long* span; // profiling: [0] min CTA start, [1] max CTA end (%globaltimer), or null
};

// Token-tile tensor maps of one operand: the same [rows][row_bytes] buffer with
// boxes of 16, 32, 64 and 128 rows (128-byte swizzle), so that a tile of n rows
// (a multiple of 16) arrives in at most three copies.
struct TokenMaps {
  CUtensorMap box[5];  // 16, 32, 64, 128 rows; [4] 96 rows (W4A16 only)
};
// Tensor maps of both phases: weights, tokens (four box heights) and the output
// rows as TMA store target, 16-row boxes of the tile's features (FC1 ReLU2: fp32
// x 128 of act; SwiGLU: fp32 x 64 of act; FC2: bf16 x 128 of the route rows).
struct W4A4Maps {
  CUtensorMap a[2];
  TokenMaps b[2];
  CUtensorMap o[2];
};
// act: kFc1Relu2 or kFc1Swiglu (the FC1 epilogue; FC2 items need no choice).
cudaError_t launch_gemm_w4a4(const W4A4Maps& maps, const W4A4Args& a, int act, int grid,
                             cudaStream_t s);
// Test hook of the bounded in-kernel waits (moe_nvfp4_selftest_wait_timeout).
cudaError_t launch_selftest_wait(const int32_t* never_set, int32_t* status, cudaStream_t s);
// W4A16: tmA over packed weights (128-byte boxes, 128-byte swizzle), tmB over bf16
// token rows (128-byte boxes, 128-byte swizzle); route_out receives the bf16
// activated rows (FC1, row stride I) or the bf16 route rows (FC2, stride H).
cudaError_t launch_gemm_w4a16(const CUtensorMap& tmA, const TokenMaps& tmB, const GemmArgs& a,
                              int grid, cudaStream_t s);

}  // namespace moe
