// queue.cuh -- the work-item queue of the persistent kernels.
//
// One producer thread per CTA claims item ids from a global counter (zero at launch) and
// publishes them, in claim order, in a ring of ITEM_SLOTS shared-memory slots.  Slot s is guarded
// by two mbarriers: FULL(s) (count 1, the producer arrives after writing the id) and EMPTY(s)
// (count = number of consumers; each consumer arrives once it has read the id).  Every role of
// the CTA reads the same sequence of ids; an id >= the item count ends it.  CTAs that finish
// their items early claim more, so uneven items balance across the grid.
#pragma once

#include "ptx.cuh"
#include "vsa_internal.cuh"

namespace vsa {

constexpr int ITEM_SLOTS = 4;

// Producer: claim this CTA's k-th item into *w and publish it.  `full0` / `empty0` are the
// shared addresses of FULL(0) / EMPTY(0); the slots' barriers follow at 8-byte steps.  False on
// abort or when a wait runs past `limit_ns`.
__device__ __forceinline__ bool publish_item(uint32_t full0, uint32_t empty0, volatile int* queue,
                                             uint32_t k, int32_t* counter, volatile int* abort,
                                             uint64_t limit_ns, int* w) {
  const uint32_t slot = k % ITEM_SLOTS;
  if (!mbar_wait_bounded(empty0 + 8u * slot, ((k / ITEM_SLOTS) & 1u) ^ 1u, abort, limit_ns))
    return false;
  const int v = atomicAdd(counter, 1);
  queue[slot] = v;
  mbar_arrive(full0 + 8u * slot);  // release: the id is visible to whoever sees the phase
  *w = v;
  return true;
}

// Consumer (one thread): this CTA's k-th item; the slot is handed back at once.
__device__ __forceinline__ bool take_item(uint32_t full0, uint32_t empty0, volatile int* queue,
                                          uint32_t k, volatile int* abort, uint64_t limit_ns,
                                          int* w) {
  const uint32_t slot = k % ITEM_SLOTS;
  if (!mbar_wait_bounded(full0 + 8u * slot, (k / ITEM_SLOTS) & 1u, abort, limit_ns))
    return false;
  *w = queue[slot];
  mbar_arrive(empty0 + 8u * slot);
  return true;
}

// Consumer (a whole warp): lane 0 takes the item and broadcasts it; one arrival per warp.
__device__ __forceinline__ bool warp_take_item(uint32_t full0, uint32_t empty0,
                                               volatile int* queue, uint32_t k,
                                               volatile int* abort, uint64_t limit_ns, int lane,
                                               int* w) {
  int ok = 1, v = 0;
  if (lane == 0) ok = take_item(full0, empty0, queue, k, abort, limit_ns, &v) ? 1 : 0;
  *w = __shfl_sync(0xffffffffu, v, 0);
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

}  // namespace vsa
