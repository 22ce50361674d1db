/*
 * moe_nvfp4.h -- C ABI of libmoe_nvfp4.so: a single-GPU routed mixture-of-
 * experts expert layer in NVFP4 for GB300 (sm_103a).
 *
 * Sources (web pages, cited by title and section):
 *   [MLM] Megatron-LM PR #8262 "per-token NVFP4 squared-ReLU and SwiGLU MoE via
 *         FlashInfer CuTe DSL" -- Background, What is added, Why CuTe DSL, How
 *         to extend, What is tested.
 *   [FI]  FlashInfer PR #5019 "CuTe DSL NVFP4 W4A16 MegaMoE" -- Tensor and
 *         numerical contract.
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers of the current CUDA device unless
 *     stated otherwise; the caller owns every buffer.  The library never
 *     allocates, frees or synchronises in prepare / quantize / forward, so those
 *     calls can be captured in a CUDA graph once the device check below has run
 *     (it runs on the first call on each device; make that call outside capture).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     enqueued on it; results are valid once the stream reaches that point.
 *   - Host-side validation runs first.  On any error nothing is launched and
 *     nothing is written, and the status code says why.
 *   - bf16 is IEEE bfloat16 stored as 2 bytes; E2M1 codes are packed two per
 *     byte, element 2j in the low nibble; E4M3 scales are one byte each (the
 *     "fn" variant: bias 7, max 448, no infinities).
 *   - Shape limits of this version: 1 <= E <= 1024; H and I multiples of 64 in
 *     [64, 65536]; 1 <= K <= min(32, E) ([FI] Tensor and numerical contract,
 *     supported scope); 0 <= T and T*K <= 2^26.
 *   - Padding ([MLM] Why CuTe DSL: hidden sizes are padded to 256, e.g. 2688 ->
 *     2816; What is tested: non-256-aligned shapes exercise the padding).  The
 *     library stores and computes every hidden / intermediate dimension padded
 *     with zeros to Hp = round_up(H, 256) and Ip = round_up(I, 256); N1p = Ip
 *     (squared ReLU) or 2*Ip (SwiGLU, each half padded).  Zero codes and zero
 *     block scales in the padding leave every real dot product unchanged, and
 *     the layer output is [T][H].  When H and I are multiples of 256, Hp = H and
 *     Ip = I.
 */
#ifndef MOE_NVFP4_H_
#define MOE_NVFP4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad enum      */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* outside the shape limits above             */
  MOE_ERR_MISALIGNED = 3,         /* a pointer is not aligned as documented     */
  MOE_ERR_WORKSPACE_TOO_SMALL = 4,
  MOE_ERR_UNSUPPORTED_DEVICE = 5, /* current device is not compute capability 10.3 */
  MOE_ERR_CUDA = 6,               /* a CUDA runtime/driver call failed          */
  MOE_ERR_BAD_EXPERT_ID = 7,      /* device-reported: an id outside [-1, E)     */
  MOE_ERR_DEVICE_TIMEOUT = 8      /* device-reported: a bounded wait gave up    */
} moe_status;

typedef enum { MOE_ACT_RELU2 = 0, MOE_ACT_SWIGLU = 1 } moe_act;

/* Layer shape.  N1 = I for squared ReLU, 2I for SwiGLU ([MLM] What is added:
 * SwiGLU's FC1 has twice FC2's input width; [FI]: gate-then-up FC1).  H and I are
 * the real (unpadded) sizes. */
typedef struct {
  int32_t E; /* experts                 */
  int32_t H; /* hidden size             */
  int32_t I; /* intermediate size       */
  int32_t act; /* moe_act               */
} moe_dims;

/* Prepared NVFP4 weights ([MLM] What is added: packed E2M1, 128x4-swizzled E4M3
 * block scales, per-expert FP32 alphas; [FI] Tensor and numerical contract:
 * scale plane of P = round_up(N,128)*round_up(D/16,4) bytes per expert, alpha
 * kept separate, never folded into scales).  All device pointers, 16-byte
 * aligned (alphas 4-byte).  Stored layouts (padded sizes Hp, Ip, N1p above):
 *   fc1_codes [E][N1p][Hp/2] K-contiguous rows.  For SwiGLU the stored row order
 *                           interleaves 64-row blocks of the padded halves:
 *                           stored rows [128f, 128f+64) are gate features
 *                           [64f, 64f+64) and stored rows [128f+64, 128f+128)
 *                           the matching up features.  Squared ReLU keeps row
 *                           order.  Features >= I and columns >= H are zero.
 *   fc1_sf    [E][N1p*Hp/16] swizzled: byte of (stored row r, scale column j) is
 *                           ((r/128)*(Hp/64) + j/4)*512 + (r%32)*16 + ((r/32)%4)*4 + j%4
 *   fc1_alpha [E]           1 / w_scale, w_scale = 2688 / amax(expert FC1)
 *   fc2_codes [E][Hp][Ip/2], fc2_sf [E][Hp*Ip/16] (same swizzle), fc2_alpha [E]. */
typedef struct {
  uint8_t* fc1_codes;
  uint8_t* fc1_sf;
  float* fc1_alpha;
  uint8_t* fc2_codes;
  uint8_t* fc2_sf;
  float* fc2_alpha;
} moe_nvfp4_weights;

/* Byte offsets of the workspace regions for one (dims, T, K, variant); used by
 * tests and debuggers to read intermediate results.  Offsets are from the
 * workspace base; a region that the variant does not use has size 0. */
typedef struct {
  size_t total;
  int64_t rows_cap;      /* padded permuted rows reserved (multiple of 128);
                            each expert's group starts at a multiple of 128 */
  size_t status;         /* int32[16]: [0] error bits, [1] token tiles, [2] padded rows,
                            [3] rows of the largest token tile */
  size_t counts;         /* int32[E] routes per expert                     */
  size_t group_row0;     /* int32[E] first permuted row of each expert     */
  size_t tiles;          /* int32[rows_cap/128][4] per token tile: expert, the
                            expert's first tile, its tile count, its routes */
  size_t chunk_counts;   /* int32[ceil(T*K/256)][E+1]: routes per expert in
                            each 256-route chunk, then 1 if the chunk held an
                            id outside [-1, E)                              */
  size_t chunk_prefix;   /* int32[ceil(T*K/256)][E]                        */
  size_t inv;            /* int32[T*K] permuted row of route t*K+k, or -1   */
  size_t perm;           /* int32[rows_cap] route id t*K+k of a valid row   */
  size_t xq_codes;       /* W4A4: u8[rows_cap][Hp/2] permuted token codes   */
  size_t xq_sf;          /* W4A4: u8 swizzled over permuted rows, Hp/16 cols */
  size_t xq_scale;       /* f32[rows_cap] per-row token scale: W4A4 the
                            NVFP4 row scale; W4A16 the power of two 2^k
                            that x_perm's row was divided by              */
  size_t act;            /* W4A4: f32[rows_cap][Ip] activated FC1 rows      */
  size_t fc2q_codes;     /* W4A4: u8[rows_cap][Ip/2] requantized FC2 input  */
  size_t fc2q_sf;        /* W4A4: u8 swizzled over permuted rows, Ip/16 cols */
  size_t fc2q_scale;     /* W4A4: f32[rows_cap] FC2-input row scale s2      */
  size_t x_perm;         /* W4A16: f16[rows_cap][Hp] permuted token rows,
                            each bf16 row times 2^-k (k from its largest
                            magnitude, which lands in [2^14, 2^15))        */
  size_t act_bf16;       /* W4A16: bf16[rows_cap][Ip] activated FC1 rows
                            (the bf16 handoff)                              */
  size_t route;          /* bf16[rows_cap][Hp] per-route FC2 rows           */
  size_t tile_sync;      /* int32[2][rows_cap/128] then f32[rows_cap]: per
                            token tile the FC1 items stored and the FC2-input
                            ready flag, per row the activated row's amax, of
                            the one-launch FC1 -> FC2 path, taken when
                            T*K <= min(2048, 8*E)                           */
  size_t act_f16;        /* W4A16: f16[rows_cap][Ip] act_bf16's rows times
                            2^-k, k from each row's largest magnitude, which
                            lands in [2^14, 2^15) (the FC2 GEMM's operand)  */
  size_t act_scale;      /* W4A16: f32[rows_cap] 2^k of each act_f16 row    */
} moe_ws_layout;

/* ABI version of this header (bumped on any incompatible change). */
#define MOE_NVFP4_ABI_VERSION 3
int32_t moe_nvfp4_abi_version(void);

/* Human-readable text of a status code (static storage). */
const char* moe_nvfp4_status_string(moe_status s);

/* Byte sizes of the six prepared-weight buffers, in the order of
 * moe_nvfp4_weights' members.  Host only, no CUDA calls. */
moe_status moe_nvfp4_weight_sizes(const moe_dims* d, size_t bytes_out[6]);

/* Stage 1, weight prep ([MLM] What is added: prepare_routed_nvfp4_weights;
 * How to extend: alpha = 1/w_scale).  fc1_bf16 is [E][N1][H] in canonical row
 * order ([gate; up] for SwiGLU), fc2_bf16 is [E][H][I]; both 16-byte aligned.
 * Writes every byte of `out` (in place: re-running refreshes the same buffers,
 * so addresses captured by CUDA graphs stay valid).  Per expert and FC:
 * amax over the matrix, w_scale = 2688/amax, rows quantized with enc = w_scale,
 * alpha = 1/w_scale (0 and all-zero codes for an all-zero expert). */
moe_status moe_nvfp4_prepare_weights(const moe_dims* d, const void* fc1_bf16,
                                     const void* fc2_bf16, const moe_nvfp4_weights* out,
                                     moe_stream_t stream);

/* Stage 2, per-token activation quantization ([MLM] Background: one FP32 scale
 * per token; What is added: global scale = recipe constant 1/(448*6), no host
 * sync).  x_bf16 [T][H] -> codes [T][Hp/2], linear block scales sf [T][Hp/16]
 * (the columns past H are zero), scale [T] = amax_t / 2688 (0 for an all-zero
 * row).  x, codes, sf 16-byte aligned; scale 4-byte aligned.  T == 0 is a no-op. */
moe_status moe_nvfp4_quantize_tokens(int32_t T, int32_t H, const void* x_bf16, uint8_t* codes,
                                     uint8_t* sf, float* scale, moe_stream_t stream);

/* Workspace bytes that moe_nvfp4_forward (w4a16 = 0) or
 * moe_nvfp4_forward_w4a16 (w4a16 = 1) needs for up to T_max tokens with top-K.
 * Host only.  Returns 0 for invalid arguments. */
size_t moe_nvfp4_workspace_bytes(const moe_dims* d, int32_t T_max, int32_t K, int32_t w4a16);

/* Number of kernels one moe_nvfp4_forward (w4a16 = 0) or
 * moe_nvfp4_forward_w4a16 (w4a16 = 1) call launches for T tokens with top-K:
 * routing and the row gather (one kernel up to 32 routes, two up to 2048,
 * four beyond), the grouped GEMMs (W4A4: one launch when T*K <= min(2048, 8*E), else FC1, the
 * FC2-input requant and FC2; W4A16: FC1, the conversion of the bf16 handoff
 * rows to the f16 FC2 operand, and FC2) and the finalize; 0 for
 * T == 0.  Host only, no device work.  Returns -1 for invalid arguments. */
int32_t moe_nvfp4_forward_kernel_count(const moe_dims* d, int32_t T, int32_t K, int32_t w4a16);

/* Region offsets of the workspace for exactly T tokens (host only). */
moe_status moe_nvfp4_workspace_layout(const moe_dims* d, int32_t T, int32_t K, int32_t w4a16,
                                      moe_ws_layout* out);

/* Stages 3-6, W4A4 forward ([MLM] What is added: flashinfer_routed_nvfp4_moe
 * with the two-stage finalize; How to extend: fc1_alpha = fc2_alpha =
 * 1/w_scale, per_token_scale from the quantizer, fc2_input_scale = 1/(448*6)).
 *   codes/sf/scale: the output of moe_nvfp4_quantize_tokens for the T tokens.
 *   topk_ids int32 [T][K]: expert of each slot, -1 = empty slot; an id outside
 *     [-1, E) is treated as empty and reported by moe_nvfp4_read_status.
 *   topk_w fp32 [T][K]: routing score of each slot.
 *   out_bf16 [T][H]: out[t] = bf16( sum_{k ascending} topk_w[t,k] * route(t,k) )
 *     with route(t,k) = bf16( FC2(requant(act(FC1(x_t)))) ) of expert
 *     topk_ids[t,k]; an fp32 accumulator from +0; no route -> zeros.  The sum
 *     order and every per-route value are independent of the other tokens in
 *     the batch, so each token's output is bitwise batch invariant.
 *   ws: at least moe_nvfp4_workspace_bytes(d, T, K, 0) bytes, 256-byte aligned;
 *     one workspace per stream (concurrent calls need distinct workspaces).
 * T == 0 is a no-op. */
moe_status moe_nvfp4_forward(const moe_dims* d, const moe_nvfp4_weights* w, int32_t T, int32_t K,
                             const uint8_t* codes, const uint8_t* sf, const float* scale,
                             const int32_t* topk_ids, const float* topk_w, void* out_bf16,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* W4A16 forward ([MLM] How to extend: BF16 x NVFP4 'weight_only'; [FI] Tensor
 * and numerical contract, compute order): BF16 activations x_bf16 [T][H] meet
 * the same prepared weights, decoded on chip (E2M1 x E4M3 is exact in bf16);
 * fp32 accumulation; FC1 times alpha1, activation, bf16 handoff; FC2 times
 * alpha2, bf16 route rows; the same finalize.  Other arguments as
 * moe_nvfp4_forward; ws sized with w4a16 = 1. */
moe_status moe_nvfp4_forward_w4a16(const moe_dims* d, const moe_nvfp4_weights* w, int32_t T,
                                   int32_t K, const void* x_bf16, const int32_t* topk_ids,
                                   const float* topk_w, void* out_bf16, void* ws,
                                   size_t ws_bytes, moe_stream_t stream);

/* Per-tensor NVFP4 x NVFP4 recipe ([MLM] How to extend, "Per-tensor NVFP4 x
 * NVFP4": serving calibrated checkpoints).  a1_scale and a2_scale are the
 * static FC1 / FC2 input scales, DEVICE fp32 scalars (4-byte aligned) that stay
 * fixed across calls so graph replays need no host sync.  They are encode
 * scales, like w_scale: a row is quantized with enc = a (block scale
 * E4M3(fl(fl(amax_b/6)*a)), saturating), and a dequantized value is
 * code * block_scale / a.  They must be positive and finite.
 *
 * Weight prep of the recipe: the same codes and block scales as
 * moe_nvfp4_prepare_weights, with the input scales folded into the alphas:
 * fc1_alpha = 1 / (w_scale1 * a1_scale), fc2_alpha = 1 / (w_scale2 * a2_scale)
 * (each product and quotient one fp32 rounding; 0 for an all-zero expert). */
moe_status moe_nvfp4_prepare_weights_per_tensor(const moe_dims* d, const void* fc1_bf16,
                                                const void* fc2_bf16, const float* a1_scale,
                                                const float* a2_scale,
                                                const moe_nvfp4_weights* out,
                                                moe_stream_t stream);

/* Token quantization of the recipe: x_bf16 [T][H] -> codes [T][Hp/2] and
 * linear block scales sf [T][Hp/16] with the static encode scale a1_scale; no
 * per-token scale.  Alignment and padding as moe_nvfp4_quantize_tokens. */
moe_status moe_nvfp4_quantize_tokens_static(int32_t T, int32_t H, const void* x_bf16,
                                            const float* a1_scale, uint8_t* codes, uint8_t* sf,
                                            moe_stream_t stream);

/* W4A4 forward of the recipe: tokens from moe_nvfp4_quantize_tokens_static,
 * weights from moe_nvfp4_prepare_weights_per_tensor.  FC1 applies fc1_alpha
 * only (no per-token scale), the FC2 input is quantized with the static encode
 * scale a2_scale (fc2_input_scale = a2_scale), FC2 applies fc2_alpha only; the
 * finalize and every other argument as moe_nvfp4_forward (same workspace size). */
moe_status moe_nvfp4_forward_per_tensor(const moe_dims* d, const moe_nvfp4_weights* w, int32_t T,
                                        int32_t K, const uint8_t* codes, const uint8_t* sf,
                                        const float* a2_scale, const int32_t* topk_ids,
                                        const float* topk_w, void* out_bf16, void* ws,
                                        size_t ws_bytes, moe_stream_t stream);

/* The plain top-K router upstream of the layer ([MLM] Performance: "plain
 * top-8" routing, no group-limited routing; the router GEMM that produces the
 * logits is the caller's).  logits fp32 [T][E] -> topk_ids int32 [T][K]: the K
 * largest logits in descending order, equal logits to the lower expert id;
 * topk_w fp32 [T][K]: softmax over the K selected logits (shifted by the
 * largest, summed for k ascending), i.e. the full softmax renormalised over the
 * selected experts.  Logits must not be NaN.  1 <= E <= 1024,
 * 1 <= K <= min(32, E); pointers 4-byte aligned; T == 0 is a no-op.  Each
 * token's result depends only on its own row (batch invariant). */
moe_status moe_nvfp4_route_topk(int32_t T, int32_t E, int32_t K, const float* logits,
                                int32_t* topk_ids, float* topk_w, moe_stream_t stream);

/* Options of the *_ex forwards; a zero-initialised struct (or NULL) gives the
 * behaviour of the plain entry points. */
typedef struct {
  /* 1: topk_ids is int64 [T][K], 8-byte aligned ([FI] Tensor and numerical
   * contract: signed int32/int64 ids); a value outside the int32 range is an
   * invalid id (ignored and reported like one outside [-1, E)). */
  int32_t ids_int64;
  /* > 0 (SwiGLU only): clamped SwiGLU ([FI] Tensor and numerical contract:
   * "Clamp caps gate above the limit and clips up symmetrically"; the pages'
   * H200 run uses 10): gate = min(gate, L), up = min(max(up, -L), L), applied to
   * the scaled FC1 outputs before silu(gate) * up.  0: no clamp. */
  float swiglu_limit;
} moe_forward_opts;

/* moe_nvfp4_forward with options (topk_ids as described by opts). */
moe_status moe_nvfp4_forward_ex(const moe_dims* d, const moe_nvfp4_weights* w, int32_t T,
                                int32_t K, const uint8_t* codes, const uint8_t* sf,
                                const float* scale, const void* topk_ids, const float* topk_w,
                                void* out_bf16, void* ws, size_t ws_bytes,
                                const moe_forward_opts* opts, moe_stream_t stream);

/* moe_nvfp4_forward_w4a16 with options. */
moe_status moe_nvfp4_forward_w4a16_ex(const moe_dims* d, const moe_nvfp4_weights* w, int32_t T,
                                      int32_t K, const void* x_bf16, const void* topk_ids,
                                      const float* topk_w, void* out_bf16, void* ws,
                                      size_t ws_bytes, const moe_forward_opts* opts,
                                      moe_stream_t stream);

/* Test hook of the in-kernel failure detection: launches one thread that waits
 * on an mbarrier nothing arrives on and then on a flag nothing sets, with the
 * bounded waits of the GEMM kernels (2 s limit each, so the call's work takes
 * about 4 s).  Both waits give up and record a timeout, the kernel returns
 * normally and the context stays usable: moe_nvfp4_read_status(ws) then gives
 * MOE_ERR_DEVICE_TIMEOUT.  Uses (and zeroes) the first 68 bytes of ws; nothing
 * traps or faults. */
moe_status moe_nvfp4_selftest_wait_timeout(void* ws, size_t ws_bytes, moe_stream_t stream);

/* Device-reported status of the last forward that used `ws`: synchronises
 * `stream`, then returns MOE_ERR_BAD_EXPERT_ID, MOE_ERR_DEVICE_TIMEOUT or
 * MOE_OK.  The flags are rewritten by every forward.  Debug/test
 * helper; not capturable. */
moe_status moe_nvfp4_read_status(const void* ws, moe_stream_t stream);

/* Allocation-free W4A4 forward.  (The source pages have no counterpart: this
 * entry point exists for callers of this library.)  It is moe_nvfp4_forward
 * with the workspace taken from a scratch array that the library keeps in
 * device memory, so the caller passes only its inputs and outputs.  It is for
 * callers that may not allocate device memory themselves -- a plugin inside a
 * framework that owns all allocations, code running under a locked or budgeted
 * allocator, an embedded runtime with memory fixed at start-up.
 *   - The scratch is one array of 64 MiB per device, reserved on every device
 *     that loads the library and held until the process exits.  A (d, T, K)
 *     whose workspace (moe_nvfp4_workspace_bytes(d, T, K, 0)) exceeds 64 MiB
 *     is rejected with MOE_ERR_WORKSPACE_TOO_SMALL before anything runs.
 *   - The first call on each device looks up the array's device address (with
 *     that device current); make that first call outside any stream capture.
 *     The address is kept until the process exits: do not call cudaDeviceReset
 *     on a device where this entry point has been used (the array would move).
 *   - Shape errors are reported exactly as by moe_nvfp4_forward.
 *   - Nothing is allocated or freed, by the library or any routine it calls.
 *   - All calls on a device share the one array.  The forward clears the
 *     status words it needs zeroed; the rest is written before it is read, so
 *     the previous call's leftovers do no harm.  Calls whose execution overlaps
 *     on the GPU (different streams, no ordering between them) race on the
 *     array and give wrong results: order them on one stream or with events.
 *   - Device-reported status (bad ids) is not readable for this variant.
 * Arguments and outputs as moe_nvfp4_forward, without ws / ws_bytes. */
moe_status moe_nvfp4_forward_noalloc(const moe_dims* d, const moe_nvfp4_weights* w, int32_t T,
                                     int32_t K, const uint8_t* codes, const uint8_t* sf,
                                     const float* scale, const int32_t* topk_ids,
                                     const float* topk_w, void* out_bf16, moe_stream_t stream);

/* Profiling hook: register `n` cudaEvent_t handles (host pointer to an array of
 * event handles; n == 0 or events == NULL unregisters).  While registered,
 * every forward records events[0] before its first stage and events[i] after
 * stage i (1 routing, 2 FC1, 3 the FC2-input requant (W4A4) or the f16
 * conversion of the handoff rows (W4A16), 4 FC2, 5 finalize) on its stream,
 * for i < n.  Process-wide, not thread-safe; for benchmarks only.  The events
 * must stay alive while registered. */
moe_status moe_nvfp4_profile_events(void* const* events, int32_t n);

/* Profiling hook: register a device buffer of four uint64 (NULL unregisters;
 * 8-byte aligned, else MOE_ERR_MISALIGNED).  While registered, the grouped
 * GEMM launches of every forward fold the GPU's %globaltimer (ns) into it:
 * [0] / [1] the earliest CTA start / latest CTA end of the FC1 launch (or of
 * the one FC1 -> FC2 launch), [2] / [3] those of the FC2 launch, by atomic
 * min / max.  The caller sets [0], [2] to UINT64_MAX and [1], [3] to 0 before
 * a forward.  A launch's span excludes its launch latency, which event pairs
 * around it include.  Process-wide, not thread-safe; for benchmarks only. */
moe_status moe_nvfp4_profile_spans(void* device_spans);

#ifdef __cplusplus
}
#endif

#endif /* MOE_NVFP4_H_ */
