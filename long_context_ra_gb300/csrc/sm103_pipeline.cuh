// Pieces shared by the sm_103a kernels: tile sizes, the bounded mbarrier
// waits of the watchdog, and descriptor stepping.
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
constexpr long long kWaitLimit = 1ll << 31;  // SM cycles, about one second

struct Abort {
  volatile uint32_t* flag;
  int* status;
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
    if (clock64() - start > kWaitLimit) {
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
    const bool timed_out = clock64() - start > kWaitLimit;
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

}  // namespace sm103
}  // namespace ra
