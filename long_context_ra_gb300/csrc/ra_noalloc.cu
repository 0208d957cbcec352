// ra_forward_split_noalloc: the split forward for callers that cannot
// allocate device memory.
//
// Some callers may not call cudaMalloc once they are running: a plug-in
// living inside a host process whose memory pool already owns the whole
// device, or a latency-bound service loop where an allocation's implicit
// device synchronisation and unpredictable cost are not acceptable.  This
// entry point needs no workspace from them: its scratch (the G partial
// states of the split) lives in one file-scope device array that every GPU
// which loads the library holds until the process exits.
//
// The array is shared by every call on a device and keeps whatever the last
// call left in it.  Nothing in it needs to start at zero: the fold kernels
// write every row of every partial state before the merge reads it.  Calls
// that overlap on the GPU (different streams, or different host threads
// without ordering) race on the array and corrupt each other's results.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "ra.h"
#include "ra_internal.h"

namespace {

// Scratch of the allocation-free split forward (see RA_SPLIT_NOALLOC_SCRATCH_BYTES).
static __device__ __align__(256) unsigned char g_split_scratch[RA_SPLIT_NOALLOC_SCRATCH_BYTES];

using ra::kMaxDevices;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current, and cached.
ra_status scratch_address(void** out) {
  int dev = 0;
  const ra_status os = ra::current_ordinal(&dev);
  if (os != RA_OK) return os;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        major != 10 || minor != 3)
      return RA_ERR_ARCH;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_split_scratch) != cudaSuccess || !p) return RA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return RA_OK;
}

}  // namespace

extern "C" RA_API ra_status ra_forward_split_noalloc(const void* q, const void* k, const void* v,
                                                     void* out, float* lse, int32_t B, int32_t H,
                                                     int64_t N, int32_t d, int32_t P, int32_t G,
                                                     ra_dtype dtype, ra_stream_t stream) {
  // The arguments first, so that a bad one is reported as such whatever the
  // size; check_forward_args also bounds the row count.
  ra_status st = ra::check_forward_args(B, H, N, d, P, false, RA_LAYOUT_CONTIGUOUS, dtype);
  if (st != RA_OK) return st;
  if (G < 1 || G > RA_MAX_PARTIALS || G > P) return RA_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(B) * H * N;
  if (rows == 0) return RA_OK;
  if (!q || !k || !v || !out || !lse) return RA_ERR_INVALID_ARG;
  const uintptr_t al = dtype == RA_BF16 ? 16 : 4;
  for (const void* ptr : {q, k, v, static_cast<const void*>(out)})
    if (reinterpret_cast<uintptr_t>(ptr) % al != 0) return RA_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(lse) % 4 != 0) return RA_ERR_MISALIGNED;
  if (ra::split_workspace_bytes(rows, d, G) > RA_SPLIT_NOALLOC_SCRATCH_BYTES)
    return RA_ERR_UNSUPPORTED;  // the partial states do not fit the fixed scratch
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != RA_OK) return st;
  return ra::split_forward(q, k, v, out, lse, B, H, N, d, P, G, scratch,
                           RA_SPLIT_NOALLOC_SCRATCH_BYTES, dtype,
                           reinterpret_cast<cudaStream_t>(stream));
}
