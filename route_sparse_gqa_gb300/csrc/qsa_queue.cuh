// qsa_queue.cuh -- dynamic work queue of the tile kernels.
//
// An item is (KV head g, query tile).  Items are ranked heaviest first: rank r
// is the r-th tile of the work order (tiles sorted by chunk count,
// descending).  Two orders of (rank, head):
//   interleaved  idx = r * n_g + (g - g0): every head's heaviest tiles first;
//   head-major   idx = (g - g0) * (B * n_tiles) + r: head by head, heaviest
//                first within a head.
// Head-major keeps the K/V rows and fp32 dK/dV accumulators in use at any time
// to about one head's, which stays in L2 for long sequences where all heads'
// together would not; the launch chooses it when the heads' accumulators
// together exceed L2 (otherwise interleaving balances the tail better).  Each CTA's producer warp claims the next index with
// one atomic add on a global counter and publishes it in a small ring in shared
// memory; the CTA's other roles take the items from the ring in the same order.
// A CTA that finishes early therefore takes more items (list scheduling,
// longest first) instead of working through a fixed share.  The last CTA to
// finish resets the counter, so every launch starts from zero.
#pragma once

#include "qsa_tc_ptx.cuh"

namespace qsa {

constexpr int kQueueRing = 8;  // items published ahead of the slowest consumer

struct QueueItem {
    int64_t b, g, tile, t;
    int nch;
};

template <typename P>
__device__ __forceinline__ void queue_decode(const P &p, int32_t idx, QueueItem &it) {
    int64_t rank;
    if (p.head_major) {
        const int64_t per_head = p.B * p.n_tiles;
        rank = idx % per_head;
        it.g = p.g0 + idx / per_head;
    } else {
        rank = idx / p.n_g;
        it.g = p.g0 + idx % p.n_g;
    }
    it.tile = p.order[rank];
    it.b = it.tile / p.n_tiles;
    it.t = it.tile % p.n_tiles;
    it.nch = p.tile_nchunks[it.tile];
}

// One thread (the producer's lane 0): claims the item of ring position i, once
// every consumer has taken the slot's previous item, and publishes its index
// (-1 past the last item).  False if the wait for the slot ran out.
__device__ __forceinline__ bool queue_claim(int32_t *counter, int64_t n_items, volatile int32_t *ring, uint64_t *full,
                                            uint64_t *empty, int64_t i, const volatile int *abort, uint64_t limit_ns,
                                            int32_t &idx) {
    const int s = (int)(i % kQueueRing);
    // The slot's previous item is the one of position i - kQueueRing: parity of that round.
    if (i >= kQueueRing && !ptx::mbar_wait(empty + s, (uint32_t)((i / kQueueRing - 1) & 1), abort, limit_ns))
        return false;
    int32_t v = atomicAdd(counter, 1);
    if (v >= n_items) v = -1;
    ring[s] = v;
    ptx::mbar_arrive(full + s);  // release: the index is visible to every thread that sees the phase complete
    idx = v;
    return true;
}

// A consumer: the item index at ring position i.  Every consumer thread takes
// every position exactly once and in order (the slot's empty barrier counts
// them).  warp_wide: the whole warp calls it and gets one verdict.
__device__ __forceinline__ bool queue_take(const volatile int32_t *ring, uint64_t *full, uint64_t *empty, int64_t i,
                                           const volatile int *abort, uint64_t limit_ns, bool warp_wide,
                                           int32_t &idx) {
    const int s = (int)(i % kQueueRing);
    const uint32_t parity = (uint32_t)((i / kQueueRing) & 1);
    const bool ok = warp_wide ? ptx::mbar_wait_warp(full + s, parity, abort, limit_ns)
                              : ptx::mbar_wait(full + s, parity, abort, limit_ns);
    if (!ok) return false;
    idx = ring[s];
    ptx::mbar_arrive(empty + s);
    return true;
}

// One thread per CTA, after the CTA's last claim (successful or not): counts
// the CTA as finished; the last one resets the counter pair {next, done}.
__device__ __forceinline__ void queue_finish(int32_t *counter) {
    __threadfence();
    const int32_t prev = atomicAdd(counter + 1, 1);
    if (prev == (int32_t)gridDim.x - 1) {
        atomicExch(counter, 0);
        atomicExch(counter + 1, 0);
        __threadfence();
    }
}

}  // namespace qsa
