// Fork work from a caller's stream onto a library side stream and join it
// back, for launches that do not depend on one another (the backward's dQ
// and dK/dV kernels).  Under CUDA-graph capture the forked work becomes a
// parallel branch of the graph.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include "ra_internal.h"

namespace ra {

// A side stream per device (created on first use) and, per host thread and
// device, the two events that fork work onto it from a caller's stream and
// join it back.  An event re-recorded by a later call is safe: a wait binds
// to the record made before it was enqueued.
struct ForkJoin {
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;

  cudaError_t fork(cudaStream_t s, int dev) {
    static std::mutex mu;
    static cudaStream_t sides[kMaxDevices] = {};
    thread_local cudaEvent_t forks[kMaxDevices] = {}, joins[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    {
      std::lock_guard<std::mutex> lock(mu);
      if (!sides[dev]) {
        const cudaError_t e = cudaStreamCreateWithFlags(&sides[dev], cudaStreamNonBlocking);
        if (e != cudaSuccess) return e;
      }
      side = sides[dev];
    }
    for (cudaEvent_t* ev : {&forks[dev], &joins[dev]}) {
      if (*ev) continue;
      const cudaError_t e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
      if (e != cudaSuccess) return e;
    }
    ev_fork = forks[dev];
    ev_join = joins[dev];
    const cudaError_t e = cudaEventRecord(ev_fork, s);
    return e == cudaSuccess ? cudaStreamWaitEvent(side, ev_fork, 0) : e;
  }
  cudaError_t join(cudaStream_t s) {
    const cudaError_t e = cudaEventRecord(ev_join, side);
    return e == cudaSuccess ? cudaStreamWaitEvent(s, ev_join, 0) : e;
  }
};

}  // namespace ra
