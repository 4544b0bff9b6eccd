// tiles.cuh -- the tile sequence each role of a persistent CTA walks.
//
// Static schedules (the host's zigzag / round-robin deal): the CTA's CSR
// slice [cta_ptr[blockIdx.x], cta_ptr[blockIdx.x + 1]).
//
// Dynamic schedules (the pages' dynamic balancing: "a finished SM claims the
// next queued tile"; yuxiaoba note, "Why both static and dynamic balancing
// help"): the schedule lists every tile once in claim order (longest first),
// the CTA takes tile blockIdx.x, then tiles P + atomicAdd(counter, 1) until
// T.  Only the claiming thread (the TMA producer) touches the counter; it
// hands each index to the CTA's other roles through a small shared-memory
// ring (full: one arrival after the index is written; empty: one arrival per
// consuming thread or warp after reading it).  -1 ends the sequence.  Every
// wait is the kernels' bounded wait; an abort ends the sequence too.
#pragma once
#include "sm103_ptx.cuh"

namespace jfa {

constexpr int kTileRing = 8;

struct TileRing {
  uint64_t full[kTileRing];
  uint64_t empty[kTileRing];
  int idx[kTileRing];
};

// TileSeq<false>: the static slice.  TileSeq<true>: the dynamic queue.  The
// kernels are instantiated for both, so the static path carries no trace of
// the dynamic one.  Role code calls claim (the producer), take (a thread) or
// take_warp (a warp); the counter, tile count and ring come from the
// kernel's parameters.
template <bool kDyn>
struct TileSeq;

template <>
struct TileSeq<false> {
  int i, end;
  __device__ TileSeq(const int32_t* cta_ptr, const int*)
      : i(cta_ptr[blockIdx.x]), end(cta_ptr[blockIdx.x + 1]) {}
  // slot: the schedule's CTA index (a pair of CTAs shares one)
  __device__ TileSeq(const int32_t* cta_ptr, const int*, int slot)
      : i(cta_ptr[slot]), end(cta_ptr[slot + 1]) {}
  __device__ int claim(int*, int, TileRing&, const Abort&) { return i < end ? i++ : -1; }
  __device__ int take(const int*, TileRing&, const Abort&) { return i < end ? i++ : -1; }
  __device__ int take_warp(const int*, TileRing&, const Abort&) { return i < end ? i++ : -1; }
};

template <>
struct TileSeq<true> {
  uint32_t k;  // ring entries handled
  __device__ TileSeq(const int32_t*, const int*) : k(0) {}
  __device__ TileSeq(const int32_t*, const int*, int) : k(0) {}

  // The claiming thread: claims the next tile and publishes it to the ring.
  __device__ int claim(int* counter, int T, TileRing& ring, const Abort& ab) {
    const uint32_t s = k % kTileRing, ph = (k / kTileRing) & 1;
    int idx = (k == 0) ? int(blockIdx.x) : int(gridDim.x) + atomicAdd(counter, 1);
    if (idx >= T) idx = -1;
    if (!mbar_wait(smem_u32(&ring.empty[s]), ph ^ 1, ab)) return -1;
    *reinterpret_cast<volatile int*>(&ring.idx[s]) = idx;
    mbar_arrive(smem_u32(&ring.full[s]));  // release: the index is visible to the waiters
    ++k;
    return idx;
  }

  // A consuming thread (one arrival per entry).
  __device__ int take(const int*, TileRing& ring, const Abort& ab) {
    const uint32_t s = k % kTileRing, ph = (k / kTileRing) & 1;
    if (!mbar_wait(smem_u32(&ring.full[s]), ph, ab)) return -1;
    const int idx = *reinterpret_cast<volatile int*>(&ring.idx[s]);
    mbar_arrive(smem_u32(&ring.empty[s]));
    ++k;
    return idx;
  }

  // A consuming warp: every lane gets the index, lane 0 arrives once.
  __device__ int take_warp(const int*, TileRing& ring, const Abort& ab) {
    const uint32_t s = k % kTileRing, ph = (k / kTileRing) & 1;
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ring.full[s]), ph, ab))) return -1;
    const int idx = *reinterpret_cast<volatile int*>(&ring.idx[s]);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&ring.empty[s]));
    ++k;
    return idx;
  }
};

// Initialise the ring's barriers (one thread, before the CTA-wide sync).
__device__ __forceinline__ void tile_ring_init(TileRing& r, uint32_t consumers) {
  for (int s = 0; s < kTileRing; ++s) {
    mbar_init(smem_u32(&r.full[s]), 1);
    mbar_init(smem_u32(&r.empty[s]), consumers);
  }
}

}  // namespace jfa
