// router.cu -- the plain top-K router upstream of the expert layer
// (Megatron-LM PR #8262, "Performance": plain top-k routing, no group-limited
// routing).  Router logits [T][E] -> expert ids [T][K] and fp32 scores [T][K].
//
// One warp per token: the E logits sit in registers (expert lane + 32 i), K
// rounds of warp argmax pick the largest remaining logit (equal logits go to
// the lower expert id), then the scores are the softmax over the selected K
// logits (shift by the largest, exp, fixed-order sum), i.e. the full softmax
// renormalised over the selected experts.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

constexpr int kRouterMaxPerLane = 32;  // E <= 1024

__global__ void __launch_bounds__(256) route_topk_kernel(int T, int E, int K,
                                                         const float* __restrict__ logits,
                                                         int32_t* __restrict__ ids,
                                                         float* __restrict__ w) {
  pdl_wait();
  pdl_trigger();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* row = logits + (size_t)t * E;
  float v[kRouterMaxPerLane];
#pragma unroll
  for (int i = 0; i < kRouterMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldg(row + e) : 0.0f;  // one coalesced 128-byte load per i
  }
  uint32_t taken = 0;  // bit i: expert lane + 32 i already selected
  float sel_v = 0.0f;  // lane k keeps the k-th selected logit
  int sel_e = 0;
  for (int k = 0; k < K; ++k) {
    float bv = 0.0f;
    int be = INT_MAX;  // INT_MAX: no candidate yet (so that -inf logits can win)
#pragma unroll
    for (int i = 0; i < kRouterMaxPerLane; ++i) {
      if (32 * i >= E) break;  // warp-uniform: only the registers that hold experts
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (be == INT_MAX || v[i] > bv)) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, off);
      if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == k) {
      sel_v = bv;
      sel_e = be;
    }
  }
  // softmax over the selected logits: shift by the largest (the first), sum for k ascending
  const float m = __shfl_sync(0xFFFFFFFFu, sel_v, 0);
  const float ex = lane < K ? expf(__fsub_rn(sel_v, m)) : 0.0f;
  float sum = 0.0f;
  for (int k = 0; k < K; ++k) sum = __fadd_rn(sum, __shfl_sync(0xFFFFFFFFu, ex, k));
  if (lane < K) {
    ids[(size_t)t * K + lane] = sel_e;
    w[(size_t)t * K + lane] = __fdiv_rn(ex, sum);
  }
}

void launch_route_topk(int T, int E, int K, const float* logits, int32_t* ids, float* w,
                       cudaStream_t s) {
  const int warps = 8;
  launch_pdl(route_topk_kernel, dim3((T + warps - 1) / warps), dim3(warps * 32), 0, s, T, E, K,
             logits, ids, w);
}

}  // namespace moe
