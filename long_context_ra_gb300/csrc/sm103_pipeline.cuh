// Pieces shared by the sm_103a kernels: tile sizes, the bounded mbarrier
// waits of the watchdog, descriptor stepping, the ring walk over key tiles
// and the tile loader.
//
// Every wait is bounded.  A wait that runs out records a timeout in the
// device status word and raises a CTA-wide abort flag; the other waits of
// the CTA see the flag and give up too, so every role leaves its loop, the
// in-flight copies and MMAs are drained (again bounded) and TMEM is freed.
#pragma once

#include <cstdint>

#include "ra_internal.h"
#include "sm103_ptx.cuh"

namespace ra {
namespace sm103 {

using namespace ptx;

constexpr int kBM = 128;  // query rows per tile (TMEM lanes)
constexpr int kBN = 128;  // keys per K/V tile
// Default limit of a bounded wait, in SM cycles (about one second).  A
// launch may shorten it (FoldArgs / BackwardArgs wait_limit).  The drain
// after an abort always allows the full default, so that copies and MMAs
// still in flight land before the CTA leaves.
constexpr long long kWaitLimit = 1ll << 31;

struct Abort {
  volatile uint32_t* flag;
  int* status;
  long long limit;  // SM cycles a wait may take before it gives up
  __device__ void raise() const {
    *flag = 1u;
    atomicCAS(status, 0, kStatusTimeout);
  }
};

// Single-thread bounded wait.
__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, const Abort& ab) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*ab.flag) return false;
    if (clock64() - start > ab.limit) {
      ab.raise();
      return false;
    }
  }
}

// Bounded wait used while aborting (ignores the abort flag).
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const long long start = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - start > kWaitLimit) return;
  }
}

// Whole-warp bounded wait: every lane polls and the warp agrees on the
// outcome, so the warp stays converged for the .sync.aligned TMEM accesses.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const Abort& ab) {
  bool done = mbar_try_wait(bar, parity);
  if (__all_sync(0xffffffffu, done)) return true;
  const long long start = clock64();
  while (true) {
    done = done || mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    const bool timed_out = clock64() - start > ab.limit;
    const bool give_up = (*ab.flag != 0u) || timed_out;
    if (__any_sync(0xffffffffu, give_up)) {
      if (__any_sync(0xffffffffu, timed_out) && (threadIdx.x % 32) == 0) ab.raise();
      return false;
    }
  }
}

// The MMA thread builds each operand's shared-memory descriptor once and
// moves it by adding (byte offset >> 4) to its start-address field; every
// address here stays below 2^18 bytes, so the 14-bit field never carries.
__device__ __forceinline__ constexpr uint64_t desc_step(uint32_t bytes) { return bytes >> 4; }

// The K/V tiles one work unit visits, in order: ring steps t = t0 .. t1-1
// visit block j = (i - t) mod P ("Ring Attention: the math", "The ring
// schedule"), and within a block its 128-key tiles in local order.  Under the
// causal mask ("Ring attention, explained", "The causal-mask catch") only the
// tiles holding a key at or before the unit's last query take part; in every
// layout these are a prefix of the block's tiles, so fully masked tiles and
// blocks are skipped and every role walks the same sequence.
struct Walk {
  int64_t slice, N, c;  // slice index, tokens per slice, tokens per block
  int i, P, t0, t1, tiles, layout;
  bool causal;
  int64_t qlast;  // last query position of the unit (striped: last local row)
  int t, kt, nt;  // iteration state: step, tile within the block, tiles in it

  __device__ int block(int tt) const {
    int j = (i - tt) % P;
    return j < 0 ? j + P : j;
  }
  // Position of local row r of block j.
  __device__ int64_t pos(int j, int64_t r) const {
    if (layout == kZigzag) {
      const int64_t h = c / 2;
      return r < h ? j * h + r : (2 * static_cast<int64_t>(P) - 1 - j) * h + (r - h);
    }
    if (layout == kStriped) return j + static_cast<int64_t>(P) * r;
    return j * c + r;
  }
  // Tiles kt in [0, ntile) whose first key position first + kt*128 <= qlast.
  __device__ int prefix(int64_t first, int ntile) const {
    if (qlast < first) return 0;
    const int64_t n = (qlast - first) / kBN + 1;
    return n < ntile ? static_cast<int>(n) : ntile;
  }
  __device__ int count(int j) const {
    if (!causal) return tiles;
    if (layout == kStriped) {
      // key local row b is visible to query local row a iff b < a, or b == a and j <= i
      const int64_t lim = qlast - (j > i ? 1 : 0);
      if (lim < 0) return 0;
      const int64_t n = lim / kBN + 1;
      return n < tiles ? static_cast<int>(n) : tiles;
    }
    if (layout == kZigzag) {
      const int half = tiles / 2;
      const int a = prefix(j * (c / 2), half);
      return a < half ? a : half + prefix((2 * static_cast<int64_t>(P) - 1 - j) * (c / 2), half);
    }
    return prefix(j * c, tiles);
  }
  __device__ int total() const {
    int n = 0;
    for (int tt = t0; tt < t1; ++tt) n += count(block(tt));
    return n;
  }
  __device__ void skip() {
    while (t < t1 && kt >= nt) {
      ++t;
      kt = 0;
      nt = t < t1 ? count(block(t)) : 0;
    }
  }
  __device__ void start() {
    t = t0;
    kt = 0;
    nt = t < t1 ? count(block(t)) : 0;
    skip();
  }
  __device__ void next() {
    ++kt;
    skip();
  }
  // Current tile: first key position (contiguous, zigzag) or first local row.
  __device__ int64_t key_first() const {
    return layout == kStriped ? static_cast<int64_t>(kt) * kBN : pos(block(t), static_cast<int64_t>(kt) * kBN);
  }
};

// Issue the TMA loads of one 128-row tile (all its 64-column boxes): 2-D at
// row `row` of the [rows, d] view, or, for the striped layout, 3-D at
// (block j, local row) of the [slices * N / P, P, d] view.
template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* map, bool striped,
                                          int64_t row, int j, int64_t lrow, uint32_t bar) {
#pragma unroll
  for (int b = 0; b < D / 64; ++b) {
    if (striped)
      tma_load_3d(dst + b * kBM * 128, map, b * 64, j, static_cast<int32_t>(lrow), bar);
    else
      tma_load_2d(dst + b * kBM * 128, map, b * 64, static_cast<int32_t>(row), bar);
  }
}

}  // namespace sm103
}  // namespace ra
