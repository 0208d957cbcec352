// ra_forward_host: the forward for inputs and results in host memory, with
// the transfers overlapped with the compute.
//
// The (batch, head) slices are independent, so they are cut into chunks and
// run as a three-stage pipeline: upload (stream `up`), compute (the caller's
// stream and stream `comp`, alternating chunk by chunk so that one chunk's
// last wave of CTAs overlaps the next chunk's first), download (stream
// `down`).  Events order each chunk's stages; the caller's stream waits for
// the last download.  One cudaMemcpyAsync per tensor and chunk.

#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "ra.h"
#include "ra_internal.h"
#include "ra_trace.h"

namespace {

using ra::kMaxDevices;
// Up to this many chunks: enough that the first upload and the last download
// are small next to the compute.
constexpr int64_t kMaxChunks = 8;
// A chunk's q, k, v upload should carry at least this many bytes: below it
// the fixed cost of a chunk's copies, events and launch outweighs what
// pipelining hides (a problem of a few MB runs as one chunk).
constexpr int64_t kMinChunkBytes = 16ll << 20;

struct Streams {
  cudaStream_t up = nullptr, comp = nullptr, down = nullptr;
};

std::mutex g_mu;
Streams g_streams[kMaxDevices];

// The library's streams on the current device (an sm_103 GPU, else
// RA_ERR_ARCH), created on first use.
ra_status device_streams(Streams* out) {
  int dev = 0;
  const ra_status os = ra::current_ordinal(&dev);
  if (os != RA_OK) return os;
  std::lock_guard<std::mutex> lock(g_mu);
  Streams& s = g_streams[dev];
  if (!s.up) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        major != 10 || minor != 3)
      return RA_ERR_ARCH;
    Streams n;
    if (cudaStreamCreateWithFlags(&n.up, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&n.comp, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&n.down, cudaStreamNonBlocking) != cudaSuccess) {
      if (n.up) cudaStreamDestroy(n.up);
      if (n.comp) cudaStreamDestroy(n.comp);
      if (n.down) cudaStreamDestroy(n.down);
      return RA_ERR_CUDA;
    }
    s = n;
  }
  *out = s;
  return RA_OK;
}

constexpr int64_t round256(int64_t x) { return (x + 255) / 256 * 256; }

int64_t elem_bytes(ra_dtype dt) { return dt == RA_BF16 ? 2 : 4; }

// Events of one call, destroyed when the call returns (CUDA releases an
// event still pending once it completes).
struct Events {
  std::vector<cudaEvent_t> ev;
  ~Events() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
  cudaError_t make(cudaEvent_t* e) {
    const cudaError_t r = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
    if (r == cudaSuccess) ev.push_back(*e);
    return r;
  }
};

}  // namespace

extern "C" {

RA_API int64_t ra_forward_host_workspace_bytes(int32_t B, int32_t H, int64_t N, int32_t d,
                                               ra_dtype dtype) {
  if (B < 0 || H < 0 || N < 0 || d < 1 || (dtype != RA_F32 && dtype != RA_BF16)) return -1;
  const int64_t rows = static_cast<int64_t>(B) * H * N;
  return 4 * round256(rows * d * elem_bytes(dtype)) + round256(rows * 4);
}

RA_API ra_status ra_forward_host(const void* q, const void* k, const void* v, void* out,
                                 float* lse, int32_t B, int32_t H, int64_t N, int32_t d,
                                 int32_t P, int32_t causal, ra_layout layout, ra_dtype dtype,
                                 void* workspace, int64_t workspace_bytes, ra_stream_t stream) {
  RA_TRACE("ra_forward_host");
  if (causal != 0 && causal != 1) return RA_ERR_INVALID_ARG;
  ra_status st = ra::check_forward_args(B, H, N, d, P, causal != 0, layout, dtype);
  if (st != RA_OK) return st;
  const int64_t rows = static_cast<int64_t>(B) * H * N;
  if (rows == 0) return RA_OK;
  if (!q || !k || !v || !out || !lse || !workspace) return RA_ERR_INVALID_ARG;
  if (workspace_bytes < ra_forward_host_workspace_bytes(B, H, N, d, dtype))
    return RA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return RA_ERR_MISALIGNED;
  Streams ss;
  if ((st = device_streams(&ss)) != RA_OK) return st;
  cudaStream_t s0 = reinterpret_cast<cudaStream_t>(stream);

  // device copies: q | k | v | out | lse
  const int64_t tensor_bytes = rows * d * elem_bytes(dtype);
  char* base = static_cast<char*>(workspace);
  char* dev_t[4];
  for (int x = 0; x < 4; ++x) dev_t[x] = base + x * round256(tensor_bytes);
  float* dev_lse = reinterpret_cast<float*>(base + 4 * round256(tensor_bytes));
  const void* host_in[3] = {q, k, v};

  // chunks of whole slices
  const int64_t slices = static_cast<int64_t>(B) * H;
  const int64_t slice_bytes = N * d * elem_bytes(dtype);
  const int64_t by_size = 3 * slices * slice_bytes / kMinChunkBytes;
  int64_t n_chunks = slices < kMaxChunks ? slices : kMaxChunks;
  if (by_size < n_chunks) n_chunks = by_size < 1 ? 1 : by_size;

  Events evs;
  cudaEvent_t ev_start, ev_done;
  if (evs.make(&ev_start) != cudaSuccess || evs.make(&ev_done) != cudaSuccess)
    return RA_ERR_CUDA;
  std::vector<cudaEvent_t> ev_up(n_chunks), ev_comp(n_chunks);
  for (int64_t c = 0; c < n_chunks; ++c)
    if (evs.make(&ev_up[c]) != cudaSuccess || evs.make(&ev_comp[c]) != cudaSuccess)
      return RA_ERR_CUDA;

  // Nothing is queued before this point; from here on `s0` always ends up
  // waiting for whatever was queued, even on an error.
  cudaError_t e = cudaEventRecord(ev_start, s0);
  if (e != cudaSuccess) return RA_ERR_CUDA;
  e = cudaStreamWaitEvent(ss.up, ev_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ss.comp, ev_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ss.down, ev_start, 0);

  for (int64_t c = 0; c < n_chunks && e == cudaSuccess && st == RA_OK; ++c) {
    const int64_t s_lo = c * slices / n_chunks, s_hi = (c + 1) * slices / n_chunks;
    const int64_t off = s_lo * slice_bytes, bytes = (s_hi - s_lo) * slice_bytes;
    for (int x = 0; x < 3 && e == cudaSuccess; ++x)
      e = cudaMemcpyAsync(dev_t[x] + off, static_cast<const char*>(host_in[x]) + off, bytes,
                          cudaMemcpyHostToDevice, ss.up);
    if (e == cudaSuccess) e = cudaEventRecord(ev_up[c], ss.up);
    cudaStream_t sc = (c % 2 == 0) ? s0 : ss.comp;
    if (e == cudaSuccess) e = cudaStreamWaitEvent(sc, ev_up[c], 0);
    if (e != cudaSuccess) break;
    // one chunk = B' = 1, H' = slices of the chunk
    const int32_t hc = static_cast<int32_t>(s_hi - s_lo);
    float* lse_c = dev_lse + s_lo * N;
    const ra_stream_t rs = reinterpret_cast<ra_stream_t>(sc);
    st = causal ? ra_forward_causal(dev_t[0] + off, dev_t[1] + off, dev_t[2] + off,
                                    dev_t[3] + off, lse_c, 1, hc, N, d, P, layout, dtype, rs)
                : ra_forward(dev_t[0] + off, dev_t[1] + off, dev_t[2] + off, dev_t[3] + off,
                             lse_c, 1, hc, N, d, P, dtype, rs);
    if (st != RA_OK) break;
    e = cudaEventRecord(ev_comp[c], sc);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ss.down, ev_comp[c], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<char*>(out) + off, dev_t[3] + off, bytes,
                          cudaMemcpyDeviceToHost, ss.down);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(lse + s_lo * N, lse_c, (s_hi - s_lo) * N * sizeof(float),
                          cudaMemcpyDeviceToHost, ss.down);
  }

  // Join: the downloads follow every chunk's compute, which follows its
  // upload, so `s0` waiting for the download stream covers everything.
  // `comp` and `up` are joined too, for the work queued before an error.
  cudaError_t j = cudaEventRecord(ev_done, ss.down);
  if (j == cudaSuccess) j = cudaStreamWaitEvent(s0, ev_done, 0);
  cudaEvent_t ev_comp_end, ev_up_end;
  if (j == cudaSuccess) j = evs.make(&ev_comp_end);
  if (j == cudaSuccess) j = cudaEventRecord(ev_comp_end, ss.comp);
  if (j == cudaSuccess) j = cudaStreamWaitEvent(s0, ev_comp_end, 0);
  if (j == cudaSuccess) j = evs.make(&ev_up_end);
  if (j == cudaSuccess) j = cudaEventRecord(ev_up_end, ss.up);
  if (j == cudaSuccess) j = cudaStreamWaitEvent(s0, ev_up_end, 0);
  if (st != RA_OK) return st;
  return (e == cudaSuccess && j == cudaSuccess) ? RA_OK : RA_ERR_CUDA;
}

}  // extern "C"
