// gemm_common.cuh -- pieces shared by the grouped GEMM kernels: the mbarrier
// ring accessor, the work-item map over token tiles and weight tiles, bounded
// waits that record an error and unwind, and named barriers.
#pragma once
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

struct Ring {
  uint8_t* base;  // 1024-aligned
  __device__ uint32_t bar(int i) const { return smem_u32(base + 8 * i); }
};

// A work item: token tile tt (rows valid rows of expert e) x weight tile mt.
// Items are numbered expert by expert, and within an expert weight-tile-major,
// so the token tiles that share a weight tile run on neighbouring CTAs at the
// same time and the weight tile comes from HBM once (then L2).  Loaded one item
// ahead of use.
struct TileInfo {
  int e, tt, mt, rows;
};
// The table entry of an item's token tile; split from tile_decode so that the
// load can be issued an item early and its fields computed only when used.
__device__ __forceinline__ int4 tile_raw(const GemmArgs& a, int item, int n_items) {
  if (item >= n_items) return make_int4(0, 0, 1, 0);
  return a.tiles[item / a.m_tiles];  // {expert, first tile, tiles, routes}
}
__device__ __forceinline__ TileInfo tile_decode(const GemmArgs& a, int item, int n_items,
                                                const int4& t) {
  if (item >= n_items) return TileInfo{0, 0, 0, 0};
  const int local = item - a.m_tiles * t.y;
  const int j = local % t.z;
  return TileInfo{t.x, t.y + j, local / t.z, min(kTileRows, t.w - kTileRows * j)};
}
__device__ __forceinline__ TileInfo tile_info(const GemmArgs& a, int item, int n_items) {
  return tile_decode(a, item, n_items, tile_raw(a, item, n_items));
}

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicOr(status + kStatusFlags, kFlagWaitTimeout);
      return false;
    }
  }
}

// After an abort: wait (one shared time limit) for the phases this thread armed
// on the stage `full` barriers, so that no copy still lands in shared memory
// once the CTA is gone.  A phase another thread never armed does not complete;
// the limit ends the wait, by which time this thread's own copies have landed.
__device__ __forceinline__ void drain_stages(const Ring& R, int bar0, const int* last_par, int n) {
  const uint64_t t0 = globaltimer();
  for (int s = 0; s < n; ++s) {
    if (last_par[s] < 0) continue;
    while (!mbar_try_wait_sleep(R.bar(bar0 + s), (uint32_t)last_par[s]))
      if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- dynamic work queue
// The producer claims work items from a per-launch global counter (the first
// one is blockIdx.x, later ones gridDim.x + atomicAdd) and publishes each
// item's TileInfo in a small shared-memory ring; the MMA thread, the
// scale/decode warps and the four epilogue warps pop them in the same order.
// A tile info with rows == 0 ends the stream.  Balances CTAs whose items
// differ in cost (token tiles of different sizes) or whose memory is slower.
constexpr int kItemSlots = 16;
// consumers of every item: the MMA thread, each scale/decode warp, 4 epilogue warps

struct ItemQueue {
  int4* ring;        // shared memory, kItemSlots entries
  uint32_t full0;    // kItemSlots mbarriers (count 1)
  uint32_t empty0;   // kItemSlots mbarriers (count = number of consumers)
  __device__ uint32_t full(int s) const { return full0 + 8 * s; }
  __device__ uint32_t empty(int s) const { return empty0 + 8 * s; }
};

struct QueuePos {
  int slot = 0;
  uint32_t phase = 0;
  __device__ void advance() {
    if (++slot == kItemSlots) {
      slot = 0;
      phase ^= 1;
    }
  }
};

// Producer side: publish `t` (rows == 0 ends the stream).  Single thread.
__device__ __forceinline__ bool queue_push(const ItemQueue& q, QueuePos& pos, const TileInfo& t,
                                           volatile int* abort_flag, int32_t* status) {
  if (!wait_or_abort(q.empty(pos.slot), pos.phase ^ 1, abort_flag, status)) return false;
  volatile int* dst = reinterpret_cast<volatile int*>(q.ring + pos.slot);
  dst[0] = t.e;
  dst[1] = t.tt;
  dst[2] = t.mt;
  dst[3] = t.rows;
  mbar_arrive(q.full(pos.slot));  // release: the entry is visible to every waiter
  pos.advance();
  return true;
}

// Consumer side for one thread: the next item, or rows == 0 at the end / on abort.
__device__ __forceinline__ TileInfo queue_pop_thread(const ItemQueue& q, QueuePos& pos,
                                                     volatile int* abort_flag, int32_t* status) {
  TileInfo t{0, 0, 0, 0};
  if (wait_or_abort(q.full(pos.slot), pos.phase, abort_flag, status)) {
    volatile int* src = reinterpret_cast<volatile int*>(q.ring + pos.slot);
    t = TileInfo{src[0], src[1], src[2], src[3]};
  }
  mbar_arrive(q.empty(pos.slot));
  pos.advance();
  return t;
}

// Consumer side for a whole warp: lane 0 waits and reads, the warp gets the
// same answer (warp-uniform, as the tcgen05 .sync.aligned ops need).
__device__ __forceinline__ TileInfo queue_pop_warp(const ItemQueue& q, QueuePos& pos,
                                                   volatile int* abort_flag, int32_t* status) {
  TileInfo t{0, 0, 0, 0};
  if ((threadIdx.x & 31) == 0) t = queue_pop_thread(q, pos, abort_flag, status);
  else pos.advance();
  t.e = __shfl_sync(0xFFFFFFFFu, t.e, 0);
  t.tt = __shfl_sync(0xFFFFFFFFu, t.tt, 0);
  t.mt = __shfl_sync(0xFFFFFFFFu, t.mt, 0);
  t.rows = __shfl_sync(0xFFFFFFFFu, t.rows, 0);
  return t;
}

}  // namespace moe
