// tg_streamk.cuh -- the partial sums of the stream-K tail (see tg_tile_scheduler.cuh) between
// the CTA pairs that share a tail tile.
//
// A worker that contributes to a tail tile (unit part 2) does not store it: each epilogue warp
// writes its 32 TMEM lanes of the fp32 accumulator to the worker's slot in a caller-supplied
// workspace and then publishes a flag of its own; the owner's warp with the same lane quadrant
// waits for that flag and adds the slot to its accumulator before converting and storing.  One
// flag per (worker, CTA of the pair, epilogue warp): nothing waits across warps.  A flag holds
// the launch's epoch, a value no earlier launch used, so the workspace needs no clearing.
//
// Slot layout (per worker and CTA, fp32): for 64-column chunk c, lane quadrant q, 4-column group
// g and lane i, the four values of row 32 q + i, columns 64 c + 4 g .. + 3 sit in float4
// ((c * 4 + q) * 16 + g) * 32 + i: one warp's part of a chunk is 8 KiB in one piece.  Both
// directions go through the bulk-copy engine: a contribution is staged in the epilogue warp's
// two 4 KiB buffers and bulk-stored; an owner bulk-loads each contribution into its share of
// the operand ring (idle by then: the owned tile is the worker's last unit) and adds it into
// its TMEM accumulator before the ordinary store.  Loads from registers, 16 per lane and chunk,
// kept too little in flight: measured, an owner spent about 2.4 us per chunk.
#pragma once

#include <cstdint>

#include "tg_config.h"
#include "tg_ptx.cuh"
#include "tg_tile_scheduler.cuh"

namespace tg {

__device__ __forceinline__ uint32_t sk_flag_index(uint32_t worker, uint32_t rank, uint32_t q) {
  return (worker * 2u + rank) * static_cast<uint32_t>(kEpiWarps) + q;
}

__device__ __forceinline__ float4* sk_slot(float4* partials, uint32_t slot_f4, uint32_t worker,
                                           uint32_t rank) {
  return partials + static_cast<uint64_t>(worker * 2u + rank) * slot_f4;
}

// float4 offset, within a slot, of chunk c's part for lane quadrant q (16 x 32 float4: 8 KiB)
__device__ __forceinline__ uint32_t sk_chunk_f4(uint32_t c, uint32_t q) {
  return (c * 4u + q) * 16u * 32u;
}

// After this warp's bulk stores of a contribution (issued by lane 0): wait until they have
// been performed, make them visible device-wide, then lane 0 sets the warp's flag to ``epoch``
// with release semantics.
__device__ __forceinline__ void sk_publish(uint32_t* flag, uint32_t epoch, uint32_t lane) {
  if (lane == 0) {
    bulk_wait_group<0>();
    fence_proxy_async_global();
    __threadfence();
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(epoch) : "memory");
  }
  __syncwarp();
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// The lowest worker whose tail range meets tail tile t (its first k-block is t * kb).  Workers
// lowest .. owner - 1 with a non-empty range are the tile's contributors.
__device__ __forceinline__ uint32_t sk_lowest_worker(uint32_t owner, uint32_t workers,
                                                     uint32_t tail, uint32_t kb, uint32_t t) {
  uint32_t c = owner;
  const uint64_t first = static_cast<uint64_t>(t) * kb;
  while (c > 0) {
    uint64_t lo, hi;
    PersistentTileScheduler::sk_range(c - 1, workers, tail, kb, lo, hi);
    if (hi <= first) break;
    --c;
  }
  return c;
}

__device__ __forceinline__ bool sk_has_range(uint32_t c, uint32_t workers, uint32_t tail,
                                             uint32_t kb) {
  uint64_t lo, hi;
  PersistentTileScheduler::sk_range(c, workers, tail, kb, lo, hi);
  return lo < hi;
}

}  // namespace tg
