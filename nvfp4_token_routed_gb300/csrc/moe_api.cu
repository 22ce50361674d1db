// moe_api.cu -- host runtime behind include/moe_nvfp4.h: argument validation,
// workspace layout, tensor-map construction and the launch sequence of each
// entry point.  No allocation, no host synchronisation on the forward path.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <algorithm>

#include "../../include/moe_nvfp4.h"
#include "internal.h"

using namespace moe;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  // 0 unknown, 1 ok, -1 unsupported; published with release after `sms` is set,
  // so a thread that reads it with acquire also sees `sms`
  std::atomic<int> checked{0};
  int sms = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

moe_status check_device(int* sms_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  DeviceInfo& di = g_dev[dev];
  int state = di.checked.load(std::memory_order_acquire);
  if (state == 0) {
    std::lock_guard<std::mutex> lock(g_mu);
    state = di.checked.load(std::memory_order_acquire);
    if (state == 0) {
      int major = 0, minor = 0, sms = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
      di.sms = sms;
      state = (major == 10 && minor == 3) ? 1 : -1;
      di.checked.store(state, std::memory_order_release);
    }
  }
  if (state < 0) return MOE_ERR_UNSUPPORTED_DEVICE;
  if (sms_out) *sms_out = di.sms;
  return MOE_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// H and I are multiples of 64 (whole 128x4 scale atoms); the library stores and
// computes them zero-padded to multiples of 256 (one GEMM K stage).
bool dim_ok(int32_t x) { return x >= 64 && x <= 65536 && x % 64 == 0; }
int64_t pad256(int64_t x) { return (x + 255) / 256 * 256; }

moe_status check_dims(const moe_dims* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->act != MOE_ACT_RELU2 && d->act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  if (d->E < 1 || d->E > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!dim_ok(d->H) || !dim_ok(d->I)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

moe_status check_tk(const moe_dims* d, int32_t T, int32_t K) {
  if (T < 0 || K < 1) return MOE_ERR_INVALID_ARG;
  if (K > 32 || K > d->E) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((int64_t)T * K > (int64_t(1) << 26)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

int64_t hp_of(const moe_dims* d) { return pad256(d->H); }
int64_t ip_of(const moe_dims* d) { return pad256(d->I); }
// stored FC1 rows per expert: Ip, or 2 * Ip for SwiGLU (each half padded)
int64_t n1p_of(const moe_dims* d) { return d->act == MOE_ACT_SWIGLU ? 2 * ip_of(d) : ip_of(d); }

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

void compute_layout(const moe_dims* d, int32_t T, int32_t K, int32_t w4a16, moe_ws_layout* L) {
  std::memset(L, 0, sizeof(*L));
  const int64_t TK = (int64_t)T * K;
  const int64_t E = d->E, H = hp_of(d), I = ip_of(d);
  const int64_t pad_groups = TK < E ? TK : E;
  int64_t rows = TK + pad_groups * (kTileRows - 1);
  rows = (rows + kTileRows - 1) / kTileRows * kTileRows;
  const int64_t tiles = rows / kTileRows;
  const int64_t nchunks = (TK + 255) / 256;
  L->rows_cap = rows;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = up256(off + bytes);
    return o;
  };
  L->status = take(sizeof(int32_t) * kStatusWords);
  L->counts = take(sizeof(int32_t) * E);
  L->group_row0 = take(sizeof(int32_t) * E);
  L->tiles = take(sizeof(int32_t) * 4 * (tiles ? tiles : 1));
  L->chunk_counts = take(sizeof(int32_t) * nchunks * (E + 1));
  L->chunk_prefix = take(sizeof(int32_t) * nchunks * E);
  L->inv = take(sizeof(int32_t) * TK);
  L->perm = take(sizeof(int32_t) * rows);
  if (!w4a16) {
    L->xq_codes = take((size_t)rows * (H / 2));
    L->xq_sf = take((size_t)rows * (H / 16));
    L->xq_scale = take(sizeof(float) * rows);
    L->act = take(sizeof(float) * (size_t)rows * I);
    L->fc2q_codes = take((size_t)rows * (I / 2));
    L->fc2q_sf = take((size_t)rows * (I / 16));
    L->fc2q_scale = take(sizeof(float) * rows);
  } else {
    L->x_perm = take(sizeof(uint16_t) * (size_t)rows * H);
    L->xq_scale = take(sizeof(float) * rows);
    L->act_bf16 = take(sizeof(uint16_t) * (size_t)rows * I);
    L->act_f16 = take(sizeof(uint16_t) * (size_t)rows * I);
    L->act_scale = take(sizeof(float) * rows);
  }
  L->route = take(sizeof(uint16_t) * (size_t)rows * H);
  L->tile_sync = take(sizeof(int32_t) * (2 * (size_t)(tiles ? tiles : 1) + (size_t)rows));
  L->total = off;
}

// ---------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 lookup_encode_fn() {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  return nullptr;
}
// looked up once per process (a function-local static is initialised once,
// thread-safely)
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = lookup_encode_fn();
  return fn;
}

// 2-D byte tensor [rows][row_bytes] (row stride = row_bytes), box of
// box_rows x box_bytes with the 128-byte (box_bytes 128) or 64-byte (64) swizzle.
bool make_tmap_bytes(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows,
                     uint32_t box_rows, uint32_t box_bytes = 128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_bytes, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D tensor of `elem_bytes`-byte elements [rows][inner], unswizzled boxes of
// box_rows x box_inner elements (TMA store targets).
bool make_tmap_out(CUtensorMap* m, const void* base, CUtensorMapDataType dtype, uint32_t elem_bytes,
                   uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * elem_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The four token-tile maps of a [rows][row_bytes] buffer (rows >= 128: the
// buffer holds whole 128-row tiles).
bool make_token_maps(TokenMaps* t, const void* base, uint64_t row_bytes, uint64_t rows) {
  for (int i = 0; i < 4; ++i)
    if (!make_tmap_bytes(&t->box[i], base, row_bytes, rows, 16u << i)) return false;
  return true;
}

// The five token-stage maps of a 16-bit [rows][row_bytes] buffer for the W4A16
// GEMM: a 3-D view (128-byte chunk of a row, row, chunk index) whose box
// (128 B, 16/32/64/128/96 rows, 4 chunks) lands chunk-major in shared memory,
// i.e. four 128-byte-swizzled K-major chunks (256 K) of box-height rows, in one
// copy.
bool make_token_maps_3d(TokenMaps* t, const void* base, uint64_t row_bytes, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  for (int i = 0; i < 5; ++i) {
    cuuint64_t dims[3] = {128, rows, row_bytes / 128};
    cuuint64_t strides[2] = {row_bytes, 128};
    cuuint32_t box[3] = {128, i < 4 ? 16u << i : 96u, 4};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(&t->box[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
  }
  return true;
}

moe_status check_weights(const moe_nvfp4_weights* w) {
  if (!w || !w->fc1_codes || !w->fc1_sf || !w->fc1_alpha || !w->fc2_codes || !w->fc2_sf ||
      !w->fc2_alpha)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(w->fc1_codes, 16) || !aligned(w->fc1_sf, 16) || !aligned(w->fc2_codes, 16) ||
      !aligned(w->fc2_sf, 16) || !aligned(w->fc1_alpha, 4) || !aligned(w->fc2_alpha, 4))
    return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Profiling events (moe_nvfp4_profile_events) and GEMM spans
// (moe_nvfp4_profile_spans).
constexpr int kMaxProfileEvents = 8;
cudaEvent_t g_prof[kMaxProfileEvents];
int g_nprof = 0;
unsigned long long* g_span = nullptr;

// Stage boundaries of a forward: 0 before routing, 1 before FC1, 2 before the
// requant, 3 before FC2, 4 before the finalize, 5 at the end.  Each stage is an
// NVTX range (host-side enqueue; a no-op unless a profiler is attached), and the
// events registered with moe_nvfp4_profile_events are recorded at the boundaries.
void mark(int i, cudaStream_t s) {
  static const char* const kStage[5] = {"moe.route", "moe.fc1", "moe.requant", "moe.fc2",
                                        "moe.finalize"};
  if (i > 0) nvtxRangePop();
  if (i < 5) nvtxRangePushA(kStage[i]);
  if (i >= g_nprof || !g_prof[i]) return;
  // inside stream capture the record must become an event-record node of the graph
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(g_prof[i], s, cudaEventRecordExternal);
  else
    cudaEventRecord(g_prof[i], s);
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

}  // namespace

namespace moe {
int route_kernel_launches(int64_t TK);  // routing + gather launches; next to those kernels
}  // namespace moe

extern "C" {

int32_t moe_nvfp4_abi_version(void) { return MOE_NVFP4_ABI_VERSION; }

const char* moe_nvfp4_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_MISALIGNED: return "misaligned pointer";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_BAD_EXPERT_ID: return "expert id outside [-1, E) (slot ignored)";
    case MOE_ERR_DEVICE_TIMEOUT: return "an in-kernel wait timed out";
  }
  return "unknown status";
}

moe_status moe_nvfp4_weight_sizes(const moe_dims* d, size_t bytes_out[6]) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (!bytes_out) return MOE_ERR_INVALID_ARG;
  const size_t E = d->E, H = (size_t)hp_of(d), I = (size_t)ip_of(d), N1 = (size_t)n1p_of(d);
  bytes_out[0] = E * N1 * (H / 2);
  bytes_out[1] = E * N1 * (H / 16);
  bytes_out[2] = E * sizeof(float);
  bytes_out[3] = E * H * (I / 2);
  bytes_out[4] = E * H * (I / 16);
  bytes_out[5] = E * sizeof(float);
  return MOE_OK;
}

static moe_status prepare_impl(const moe_dims* d, const void* fc1_bf16, const void* fc2_bf16,
                               const float* a1_scale, const float* a2_scale,
                               const moe_nvfp4_weights* out, moe_stream_t stream) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if (!fc1_bf16 || !fc2_bf16) return MOE_ERR_INVALID_ARG;
  if (!aligned(fc1_bf16, 16) || !aligned(fc2_bf16, 16)) return MOE_ERR_MISALIGNED;
  if ((st = check_weights(out)) != MOE_OK) return st;
  if ((st = check_device(nullptr)) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool swiglu = d->act == MOE_ACT_SWIGLU;
  const int N1 = swiglu ? 2 * d->I : d->I;
  launch_prepare_fc(d->E, N1, d->H, (int)n1p_of(d), (int)hp_of(d), swiglu ? d->I : 0, fc1_bf16,
                    out->fc1_codes, out->fc1_sf, out->fc1_alpha, a1_scale, s);
  launch_prepare_fc(d->E, d->H, d->I, (int)hp_of(d), (int)ip_of(d), 0, fc2_bf16, out->fc2_codes,
                    out->fc2_sf, out->fc2_alpha, a2_scale, s);
  return cuda_status(cudaGetLastError());
}

moe_status moe_nvfp4_prepare_weights(const moe_dims* d, const void* fc1_bf16,
                                     const void* fc2_bf16, const moe_nvfp4_weights* out,
                                     moe_stream_t stream) {
  return prepare_impl(d, fc1_bf16, fc2_bf16, nullptr, nullptr, out, stream);
}

moe_status moe_nvfp4_prepare_weights_per_tensor(const moe_dims* d, const void* fc1_bf16,
                                                const void* fc2_bf16, const float* a1_scale,
                                                const float* a2_scale,
                                                const moe_nvfp4_weights* out,
                                                moe_stream_t stream) {
  if (!a1_scale || !a2_scale) return MOE_ERR_INVALID_ARG;
  if (!aligned(a1_scale, 4) || !aligned(a2_scale, 4)) return MOE_ERR_MISALIGNED;
  return prepare_impl(d, fc1_bf16, fc2_bf16, a1_scale, a2_scale, out, stream);
}

static moe_status quantize_impl(int32_t T, int32_t H, const void* x_bf16, uint8_t* codes,
                                uint8_t* sf, float* scale, const float* a1_scale,
                                moe_stream_t stream) {
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (!dim_ok(H)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return MOE_OK;
  if (!x_bf16 || !codes || !sf || (!scale && !a1_scale)) return MOE_ERR_INVALID_ARG;
  if (!aligned(x_bf16, 16) || !aligned(codes, 16) || !aligned(sf, 16) ||
      (scale && !aligned(scale, 4)) || (a1_scale && !aligned(a1_scale, 4)))
    return MOE_ERR_MISALIGNED;
  moe_status st = check_device(nullptr);
  if (st != MOE_OK) return st;
  launch_quantize_tokens(T, H, (int)pad256(H), x_bf16, codes, sf, scale, a1_scale,
                         reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

moe_status moe_nvfp4_quantize_tokens(int32_t T, int32_t H, const void* x_bf16, uint8_t* codes,
                                     uint8_t* sf, float* scale, moe_stream_t stream) {
  if (T > 0 && !scale) return MOE_ERR_INVALID_ARG;
  return quantize_impl(T, H, x_bf16, codes, sf, scale, nullptr, stream);
}

moe_status moe_nvfp4_quantize_tokens_static(int32_t T, int32_t H, const void* x_bf16,
                                            const float* a1_scale, uint8_t* codes, uint8_t* sf,
                                            moe_stream_t stream) {
  if (T > 0 && !a1_scale) return MOE_ERR_INVALID_ARG;
  return quantize_impl(T, H, x_bf16, codes, sf, nullptr, a1_scale, stream);
}

int32_t moe_nvfp4_forward_kernel_count(const moe_dims* d, int32_t T, int32_t K, int32_t w4a16) {
  if (check_dims(d) != MOE_OK || check_tk(d, T, K) != MOE_OK) return -1;
  if (T == 0) return 0;
  const int64_t TK = (int64_t)T * K;
  const bool fused = !w4a16 && TK <= kFusedMaxRoutes && TK <= kFusedRoutesPerExpert * d->E;
  // W4A4 three: FC1, requant, FC2; W4A16 three: FC1, the f16 FC2 operand, FC2
  const int gemms = w4a16 ? 3 : fused ? 1 : 3;
  return route_kernel_launches(TK) + gemms + 1;  // routing and gather, GEMMs, finalize
}

size_t moe_nvfp4_workspace_bytes(const moe_dims* d, int32_t T_max, int32_t K, int32_t w4a16) {
  if (check_dims(d) != MOE_OK || check_tk(d, T_max, K) != MOE_OK) return 0;
  moe_ws_layout L;
  compute_layout(d, T_max, K, w4a16 ? 1 : 0, &L);
  return L.total;
}

moe_status moe_nvfp4_workspace_layout(const moe_dims* d, int32_t T, int32_t K, int32_t w4a16,
                                      moe_ws_layout* out) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if ((st = check_tk(d, T, K)) != MOE_OK) return st;
  if (!out) return MOE_ERR_INVALID_ARG;
  compute_layout(d, T, K, w4a16 ? 1 : 0, out);
  return MOE_OK;
}

static const moe_forward_opts kDefaultOpts = {0, 0.0f};

static moe_status forward_common(const moe_dims* d, const moe_nvfp4_weights* w, int32_t T,
                                 int32_t K, const void* topk_ids, const float* topk_w,
                                 void* out_bf16, void* ws, size_t ws_bytes, int w4a16,
                                 const moe_forward_opts& o, moe_ws_layout* L, int* sms) {
  moe_status st = check_dims(d);
  if (st != MOE_OK) return st;
  if ((st = check_tk(d, T, K)) != MOE_OK) return st;
  if ((st = check_weights(w)) != MOE_OK) return st;
  if ((o.ids_int64 != 0 && o.ids_int64 != 1) || !(o.swiglu_limit >= 0.0f) ||
      (o.swiglu_limit > 0.0f && d->act != MOE_ACT_SWIGLU) || o.swiglu_limit > 3.0e38f)
    return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!topk_ids || !topk_w || !out_bf16 || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(topk_ids, o.ids_int64 ? 8 : 4) || !aligned(topk_w, 4) || !aligned(out_bf16, 16) ||
      !aligned(ws, 256))
    return MOE_ERR_MISALIGNED;
  compute_layout(d, T, K, w4a16, L);
  if (ws_bytes < L->total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return check_device(sms);
}

static RouteArgs route_args(const moe_dims* d, int32_t T, int32_t K, const void* ids, int ids64,
                            void* ws, const moe_ws_layout& L, int w4a16) {
  RouteArgs r{};
  r.ids64 = ids64;
  r.TK = T * K;
  r.K = K;
  r.E = d->E;
  r.H = d->H;
  r.Hp = (int)hp_of(d);
  r.w4a16 = w4a16;
  r.ids = static_cast<const int32_t*>(ids);
  r.status = at<int32_t>(ws, L.status);
  r.chunk_counts = at<int32_t>(ws, L.chunk_counts);
  r.chunk_prefix = at<int32_t>(ws, L.chunk_prefix);
  r.counts = at<int32_t>(ws, L.counts);
  r.group_row0 = at<int32_t>(ws, L.group_row0);
  r.tiles = at<int4>(ws, L.tiles);
  r.inv = at<int32_t>(ws, L.inv);
  r.perm = at<int32_t>(ws, L.perm);
  return r;
}

// scale: per-token row scales (per-token recipe) or null with a2_static set (the
// per-tensor recipe: no row scales, FC2 input quantized with the static scale).
static moe_status forward_w4a4_impl(const moe_dims* d, const moe_nvfp4_weights* w, int32_t T,
                                    int32_t K, const uint8_t* codes, const uint8_t* sf,
                                    const float* scale, const float* a2_static,
                                    const void* topk_ids, const float* topk_w, void* out_bf16,
                                    void* ws, size_t ws_bytes, const moe_forward_opts& o,
                                    moe_stream_t stream) {
  moe_ws_layout L;
  int sms = 0;
  if (T > 0 && (!codes || !sf || (!scale && !a2_static))) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!aligned(codes, 16) || !aligned(sf, 16) || (scale && !aligned(scale, 4)) ||
                (a2_static && !aligned(a2_static, 4))))
    return MOE_ERR_MISALIGNED;
  moe_status st =
      forward_common(d, w, T, K, topk_ids, topk_w, out_bf16, ws, ws_bytes, 0, o, &L, &sms);
  if (st != MOE_OK || T == 0) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // padded sizes: stored weights, token rows and every workspace row
  const int H = (int)hp_of(d), I = (int)ip_of(d), N1 = (int)n1p_of(d);

  W4A4Maps maps;
  const bool swiglu = d->act == MOE_ACT_SWIGLU;
  if (!make_tmap_bytes(&maps.a[0], w->fc1_codes, H / 2, (uint64_t)d->E * N1, 128) ||
      !make_token_maps(&maps.b[0], at<uint8_t>(ws, L.xq_codes), H / 2, L.rows_cap) ||
      !make_tmap_out(&maps.o[0], at<float>(ws, L.act), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, I,
                     L.rows_cap, swiglu ? 64 : 128, 16) ||
      !make_tmap_bytes(&maps.a[1], w->fc2_codes, I / 2, (uint64_t)d->E * H, 128) ||
      !make_token_maps(&maps.b[1], at<uint8_t>(ws, L.fc2q_codes), I / 2, L.rows_cap) ||
      !make_tmap_out(&maps.o[1], at<uint16_t>(ws, L.route), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H,
                     L.rows_cap, 128, 16))
    return MOE_ERR_CUDA;

  // Decode-sized batches with few routes per expert run FC1, the FC2-input
  // requant and FC2 as one persistent launch (no launch gaps, no FC1 tail before
  // FC2 starts); other batches run them as three launches, where the requant is
  // one wide pass.  Both compute the same bits.
  const int64_t tiles_cap = L.rows_cap / kTileRows;
  const int64_t TK = (int64_t)T * K;
  const bool fused = TK <= kFusedMaxRoutes && TK <= kFusedRoutesPerExpert * d->E;

  mark(0, s);
  RouteArgs r = route_args(d, T, K, topk_ids, o.ids_int64, ws, L, 0);
  r.xc = codes;
  r.xsf = sf;
  r.xs = scale;
  r.pc = at<uint8_t>(ws, L.xq_codes);
  r.psf = at<uint8_t>(ws, L.xq_sf);
  r.ps = at<float>(ws, L.xq_scale);
  if (fused) {
    r.tile_sync = at<int32_t>(ws, L.tile_sync);
    r.tile_sync_words = (int)(2 * tiles_cap + L.rows_cap);
  }
  if (launch_route(r, s) != cudaSuccess) return MOE_ERR_CUDA;
  mark(1, s);

  W4A4Args g{};
  g.ph[0] = W4A4Phase{H, N1 / 128, N1, w->fc1_sf, at<uint8_t>(ws, L.xq_sf), w->fc1_alpha,
                      at<float>(ws, L.xq_scale)};
  g.ph[1] = W4A4Phase{I, H / 128, H, w->fc2_sf, at<uint8_t>(ws, L.fc2q_sf), w->fc2_alpha,
                      at<float>(ws, L.fc2q_scale)};
  g.tiles = at<int4>(ws, L.tiles);
  g.status = at<int32_t>(ws, L.status);
  g.item_counter = g.status + kStatusItemCtr;
  g.span = g_span;  // FC1's (or the one launch's) span
  g.fc1_done = at<int32_t>(ws, L.tile_sync);
  g.rq_done = g.fc1_done + tiles_cap;
  g.row_amax = reinterpret_cast<float*>(g.rq_done + tiles_cap);
  g.act = at<float>(ws, L.act);
  g.Ip = I;
  g.qc = at<uint8_t>(ws, L.fc2q_codes);
  g.qsf = at<uint8_t>(ws, L.fc2q_sf);
  g.qs = at<float>(ws, L.fc2q_scale);
  g.a2_static = a2_static;
  g.swiglu_limit = o.swiglu_limit;
  const int act = swiglu ? kFc1Swiglu : kFc1Relu2;
  if (fused) {
    g.run_fc1 = g.run_fc2 = g.fused = 1;
    const int grid = (int)std::min<int64_t>(sms, tiles_cap * (g.ph[0].m_tiles + g.ph[1].m_tiles));
    if (launch_gemm_w4a4(maps, g, act, grid, s) != cudaSuccess) return MOE_ERR_CUDA;
    mark(2, s);
    mark(3, s);
    mark(4, s);
  } else {
    g.run_fc1 = 1;
    int grid = (int)std::min<int64_t>(sms, tiles_cap * g.ph[0].m_tiles);
    if (launch_gemm_w4a4(maps, g, act, grid, s) != cudaSuccess) return MOE_ERR_CUDA;
    mark(2, s);
    launch_requant(T * K, I, at<int32_t>(ws, L.inv), at<float>(ws, L.act),
                   at<uint8_t>(ws, L.fc2q_codes), at<uint8_t>(ws, L.fc2q_sf),
                   at<float>(ws, L.fc2q_scale), a2_static, s);
    mark(3, s);
    W4A4Args g2 = g;
    g2.run_fc1 = 0;
    g2.run_fc2 = 1;
    g2.span = g_span ? g_span + 2 : nullptr;
    g2.item_counter = g.status + kStatusItemCtr + 1;
    grid = (int)std::min<int64_t>(sms, tiles_cap * g2.ph[1].m_tiles);
    if (launch_gemm_w4a4(maps, g2, act, grid, s) != cudaSuccess) return MOE_ERR_CUDA;
    mark(4, s);
  }

  launch_finalize(T, K, d->H, H, at<int32_t>(ws, L.inv), topk_w, at<uint16_t>(ws, L.route),
                  out_bf16, s);
  mark(5, s);
  return cuda_status(cudaGetLastError());
}

moe_status moe_nvfp4_forward(const moe_dims* d, const moe_nvfp4_weights* w, int32_t T, int32_t K,
                             const uint8_t* codes, const uint8_t* sf, const float* scale,
                             const int32_t* topk_ids, const float* topk_w, void* out_bf16,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (T > 0 && !scale) return MOE_ERR_INVALID_ARG;
  return forward_w4a4_impl(d, w, T, K, codes, sf, scale, nullptr, topk_ids, topk_w, out_bf16, ws,
                           ws_bytes, kDefaultOpts, stream);
}

moe_status moe_nvfp4_forward_ex(const moe_dims* d, const moe_nvfp4_weights* w, int32_t T,
                                int32_t K, const uint8_t* codes, const uint8_t* sf,
                                const float* scale, const void* topk_ids, const float* topk_w,
                                void* out_bf16, void* ws, size_t ws_bytes,
                                const moe_forward_opts* opts, moe_stream_t stream) {
  if (T > 0 && !scale) return MOE_ERR_INVALID_ARG;
  return forward_w4a4_impl(d, w, T, K, codes, sf, scale, nullptr, topk_ids, topk_w, out_bf16, ws,
                           ws_bytes, opts ? *opts : kDefaultOpts, stream);
}

moe_status moe_nvfp4_forward_per_tensor(const moe_dims* d, const moe_nvfp4_weights* w, int32_t T,
                                        int32_t K, const uint8_t* codes, const uint8_t* sf,
                                        const float* a2_scale, const int32_t* topk_ids,
                                        const float* topk_w, void* out_bf16, void* ws,
                                        size_t ws_bytes, moe_stream_t stream) {
  if (T > 0 && !a2_scale) return MOE_ERR_INVALID_ARG;
  return forward_w4a4_impl(d, w, T, K, codes, sf, nullptr, a2_scale, topk_ids, topk_w, out_bf16,
                           ws, ws_bytes, kDefaultOpts, stream);
}

static moe_status forward_w4a16_impl(const moe_dims* d, const moe_nvfp4_weights* w, int32_t T,
                                     int32_t K, const void* x_bf16, const void* topk_ids,
                                     const float* topk_w, void* out_bf16, void* ws,
                                     size_t ws_bytes, const moe_forward_opts& o,
                                     moe_stream_t stream) {
  moe_ws_layout L;
  int sms = 0;
  if (T > 0 && !x_bf16) return MOE_ERR_INVALID_ARG;
  if (T > 0 && !aligned(x_bf16, 16)) return MOE_ERR_MISALIGNED;
  moe_status st =
      forward_common(d, w, T, K, topk_ids, topk_w, out_bf16, ws, ws_bytes, 1, o, &L, &sms);
  if (st != MOE_OK || T == 0) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // padded sizes: stored weights, token rows and every workspace row
  const int H = (int)hp_of(d), I = (int)ip_of(d), N1 = (int)n1p_of(d);

  CUtensorMap tmA1, tmA2;
  TokenMaps tmB1, tmB2;
  if (!make_tmap_bytes(&tmA1, w->fc1_codes, H / 2, (uint64_t)d->E * N1, 128) ||
      !make_token_maps_3d(&tmB1, at<uint8_t>(ws, L.x_perm), 2 * (uint64_t)H, L.rows_cap) ||
      !make_tmap_bytes(&tmA2, w->fc2_codes, I / 2, (uint64_t)d->E * H, 128) ||
      !make_token_maps_3d(&tmB2, at<uint8_t>(ws, L.act_f16), 2 * (uint64_t)I, L.rows_cap))
    return MOE_ERR_CUDA;

  mark(0, s);
  RouteArgs r = route_args(d, T, K, topk_ids, o.ids_int64, ws, L, 1);
  r.xb = x_bf16;
  r.pb = at<uint8_t>(ws, L.x_perm);
  r.ps = at<float>(ws, L.xq_scale);
  if (launch_route(r, s) != cudaSuccess) return MOE_ERR_CUDA;
  mark(1, s);

  const int64_t tiles_cap = L.rows_cap / kTileRows;
  GemmArgs g{};
  g.mode = d->act == MOE_ACT_SWIGLU ? kFc1Swiglu : kFc1Relu2;
  g.K = H;
  g.m_tiles = N1 / 128;
  g.w_rows = N1;
  g.sfa = w->fc1_sf;
  g.alpha = w->fc1_alpha;
  g.row_scale = at<float>(ws, L.xq_scale);
  g.tiles = at<int4>(ws, L.tiles);
  g.status = at<int32_t>(ws, L.status);
  g.item_counter = g.status + kStatusItemCtr;
  g.route_out = at<uint16_t>(ws, L.act_bf16);
  g.I = I;
  g.H = H;
  g.span = g_span;
  g.swiglu_limit = o.swiglu_limit;
  int grid = (int)std::min<int64_t>(sms, tiles_cap * g.m_tiles);
  if (launch_gemm_w4a16(tmA1, tmB1, g, grid, s) != cudaSuccess) return MOE_ERR_CUDA;
  mark(2, s);
  launch_act_f16(T * K, I, at<int32_t>(ws, L.inv), at<uint8_t>(ws, L.act_bf16),
                 at<uint8_t>(ws, L.act_f16), at<float>(ws, L.act_scale), s);
  mark(3, s);

  GemmArgs g2 = g;
  g2.mode = kFc2;
  g2.K = I;
  g2.m_tiles = H / 128;
  g2.w_rows = H;
  g2.sfa = w->fc2_sf;
  g2.alpha = w->fc2_alpha;
  g2.row_scale = at<float>(ws, L.act_scale);
  g2.item_counter = g.status + kStatusItemCtr + 1;
  g2.span = g_span ? g_span + 2 : nullptr;
  g2.route_out = at<uint16_t>(ws, L.route);
  grid = (int)std::min<int64_t>(sms, tiles_cap * g2.m_tiles);
  if (launch_gemm_w4a16(tmA2, tmB2, g2, grid, s) != cudaSuccess) return MOE_ERR_CUDA;
  mark(4, s);

  launch_finalize(T, K, d->H, H, at<int32_t>(ws, L.inv), topk_w, at<uint16_t>(ws, L.route),
                  out_bf16, s);
  mark(5, s);
  return cuda_status(cudaGetLastError());
}

moe_status moe_nvfp4_forward_w4a16(const moe_dims* d, const moe_nvfp4_weights* w, int32_t T,
                                   int32_t K, const void* x_bf16, const int32_t* topk_ids,
                                   const float* topk_w, void* out_bf16, void* ws,
                                   size_t ws_bytes, moe_stream_t stream) {
  return forward_w4a16_impl(d, w, T, K, x_bf16, topk_ids, topk_w, out_bf16, ws, ws_bytes,
                            kDefaultOpts, stream);
}

moe_status moe_nvfp4_forward_w4a16_ex(const moe_dims* d, const moe_nvfp4_weights* w, int32_t T,
                                      int32_t K, const void* x_bf16, const void* topk_ids,
                                      const float* topk_w, void* out_bf16, void* ws,
                                      size_t ws_bytes, const moe_forward_opts* opts,
                                      moe_stream_t stream) {
  return forward_w4a16_impl(d, w, T, K, x_bf16, topk_ids, topk_w, out_bf16, ws, ws_bytes,
                            opts ? *opts : kDefaultOpts, stream);
}

moe_status moe_nvfp4_route_topk(int32_t T, int32_t E, int32_t K, const float* logits,
                                int32_t* topk_ids, float* topk_w, moe_stream_t stream) {
  if (T < 0 || E < 1 || K < 1) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || K > 32 || K > E) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4))
    return MOE_ERR_MISALIGNED;
  moe_status st = check_device(nullptr);
  if (st != MOE_OK) return st;
  launch_route_topk(T, E, K, logits, topk_ids, topk_w, reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

moe_status moe_nvfp4_profile_events(void* const* events, int32_t n) {
  if (n < 0 || n > kMaxProfileEvents) return MOE_ERR_INVALID_ARG;
  if (!events) n = 0;
  for (int i = 0; i < kMaxProfileEvents; ++i)
    g_prof[i] = i < n ? static_cast<cudaEvent_t>(events[i]) : nullptr;
  g_nprof = n;
  return MOE_OK;
}

moe_status moe_nvfp4_profile_spans(void* device_spans) {
  if (device_spans && !aligned(device_spans, 8)) return MOE_ERR_MISALIGNED;
  g_span = static_cast<unsigned long long*>(device_spans);
  return MOE_OK;
}

moe_status moe_nvfp4_selftest_wait_timeout(void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return MOE_ERR_MISALIGNED;
  const size_t need = sizeof(int32_t) * (kStatusWords + 1);
  if (ws_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
  moe_status st = check_device(nullptr);
  if (st != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* status = static_cast<int32_t*>(ws);
  if (cudaMemsetAsync(ws, 0, need, s) != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(launch_selftest_wait(status + kStatusWords, status, s));
}

moe_status moe_nvfp4_read_status(const void* ws, moe_stream_t stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  int32_t flags = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&flags, ws, sizeof(flags), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (flags & kFlagWaitTimeout) return MOE_ERR_DEVICE_TIMEOUT;
  if (flags & kFlagBadExpertId) return MOE_ERR_BAD_EXPERT_ID;
  return MOE_OK;
}

}  // extern "C"
