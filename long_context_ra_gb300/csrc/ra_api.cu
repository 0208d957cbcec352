// C ABI of the library: argument validation, TMA descriptor set-up and
// kernel dispatch.  Every check runs before anything is enqueued.

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "ra.h"
#include "ra_internal.h"
#include "ra_trace.h"

namespace ra {
namespace {

// Device-side watchdog word: kernels write a non-zero code when one of their
// bounded waits runs out.  One copy per device.
__device__ int g_status;

// Watchdog settings applied to every tensor-core launch (ra_watchdog_config).
constexpr int64_t kDefaultWaitCycles = int64_t{1} << 31;
std::atomic<int64_t> g_wait_limit{kDefaultWaitCycles};
std::atomic<int64_t> g_stall_cta{-1};

struct DeviceInfo {
  bool ready = false;
  bool is_sm103 = false;
  int sms = 0;
  int* status = nullptr;  // device address of g_status
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Looks up (once) the current device's properties and the address of its
// watchdog word.
ra_status current_device(DeviceInfo* out) {
  int dev = 0;
  const ra_status os = current_ordinal(&dev);
  if (os != RA_OK) return os;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return RA_ERR_ARCH;
    di.is_sm103 = prop.major == 10 && prop.minor == 3;
    di.sms = prop.multiProcessorCount;
    if (di.is_sm103) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return RA_ERR_CUDA;
      di.status = static_cast<int*>(p);
    }
    di.ready = true;
  }
  if (!di.is_sm103) return RA_ERR_ARCH;
  *out = di;
  return RA_OK;
}

ra_status get_encoder() {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_encode) return RA_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return RA_ERR_CUDA;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return RA_OK;
}

// 2-D bf16 view [rows, d] with a box of 128 rows x 64 columns (128 bytes) and
// the 128-byte swizzle the MMA descriptors expect.
ra_status make_map(CUtensorMap* map, const void* ptr, int64_t rows, int d) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? RA_OK : RA_ERR_CUDA;
}

// Strided (striped-layout) bf16 view of a [slices, N, d] tensor as
// [slices * N / P, P, d]: block j's local row r of slice s is (s*N/P + r, j).
// Box: 128 local rows x 1 block x 64 columns, 128-byte swizzle.
ra_status make_map_striped(CUtensorMap* map, const void* ptr, int64_t rows, int d, int P) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(P),
                              static_cast<cuuint64_t>(rows / P)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(d) * 2 * static_cast<cuuint64_t>(P)};
  const cuuint32_t box[3] = {64, 1, 128};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? RA_OK : RA_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

ra_status launched(cudaError_t e) { return e == cudaSuccess ? RA_OK : RA_ERR_CUDA; }

constexpr int64_t kMaxRows = (int64_t{1} << 31) - 1;  // TMA coordinates are int32

// Size rules of the attention-shaped calls (the arguments themselves are
// already known to be in range).
ra_status check_sizes(int64_t rows, int64_t N, int32_t d, int32_t P, ra_dtype dt) {
  if (N % P != 0) return RA_ERR_UNSUPPORTED;
  if (rows > kMaxRows) return RA_ERR_UNSUPPORTED;
  if (dt == RA_BF16) {
    if (d != 64 && d != 128) return RA_ERR_UNSUPPORTED;
    if ((N / P) % 128 != 0) return RA_ERR_UNSUPPORTED;
  } else if (d > 256) {
    return RA_ERR_UNSUPPORTED;
  }
  return RA_OK;
}

// Shared checks of the attention-shaped calls; fills the fold arguments.
ra_status check_attention(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                          int64_t N, int32_t d, int32_t P, ra_dtype dt, FoldArgs* a) {
  if (B < 0 || H < 0 || N < 0 || d < 1 || P < 1) return RA_ERR_INVALID_ARG;
  if (dt != RA_F32 && dt != RA_BF16) return RA_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(B) * H * N;
  if (rows != 0 && (!q || !k || !v)) return RA_ERR_INVALID_ARG;
  const ra_status sz = check_sizes(rows, N, d, P, dt);
  if (sz != RA_OK) return sz;
  const uintptr_t al = dt == RA_BF16 ? 16 : 4;
  if (!aligned(q, al) || !aligned(k, al) || !aligned(v, al)) return RA_ERR_MISALIGNED;
  *a = FoldArgs{};
  a->q = q;
  a->k = k;
  a->v = v;
  a->slices = static_cast<int64_t>(B) * H;
  a->nq = N;
  a->nk = N;
  a->d = d;
  a->P = P;
  a->G = 1;
  a->tau = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  a->scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  return RA_OK;
}

// Launch a fold of either precision.  The bf16 path builds the TMA maps over
// the [rows, d] views of q (slices * nq rows) and k, v (slices * nk rows).
ra_status run_fold(const FoldArgs& args, ra_dtype dt, cudaStream_t s) {
  if (dt == RA_F32) return launched(launch_fold_f32(args, s));
  FoldArgs a = args;
  a.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  a.stall_cta = g_stall_cta.load(std::memory_order_relaxed);
  ra_status st = get_encoder();
  if (st != RA_OK) return st;
  CUtensorMap tq, tk, tv;
  if (a.layout == kStriped) {
    if ((st = make_map_striped(&tq, a.q, a.slices * a.nq, a.d, a.P)) != RA_OK) return st;
    if ((st = make_map_striped(&tk, a.k, a.slices * a.nk, a.d, a.P)) != RA_OK) return st;
    if ((st = make_map_striped(&tv, a.v, a.slices * a.nk, a.d, a.P)) != RA_OK) return st;
  } else {
    if ((st = make_map(&tq, a.q, a.slices * a.nq, a.d)) != RA_OK) return st;
    if ((st = make_map(&tk, a.k, a.slices * a.nk, a.d)) != RA_OK) return st;
    if ((st = make_map(&tv, a.v, a.slices * a.nk, a.d)) != RA_OK) return st;
  }
  return launched(launch_fold_sm103(a, tq, tk, tv, s));
}

bool state_ok(const ra_state* st) {
  // An empty state (rows == 0) may carry NULL pointers.
  return st && st->rows >= 0 && st->d >= 1 && (st->rows == 0 || (st->m && st->l && st->o));
}

}  // namespace

ra_status current_ordinal(int* dev) {
  const cudaError_t e = cudaGetDevice(dev);
  if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver) return RA_ERR_ARCH;
  if (e != cudaSuccess) return RA_ERR_CUDA;
  if (*dev < 0 || *dev >= kMaxDevices) return RA_ERR_UNSUPPORTED;
  return RA_OK;
}

int device_sm_count() {
  DeviceInfo di;
  if (current_device(&di) != RA_OK) return 1;
  return di.sms;
}

}  // namespace ra

using namespace ra;

namespace ra {
namespace {

// Causal / layout checks shared by the causal entry points.
ra_status check_causal(int64_t N, int32_t P, ra_layout layout, ra_dtype dt, FoldArgs* a) {
  if (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_ZIGZAG && layout != RA_LAYOUT_STRIPED)
    return RA_ERR_INVALID_ARG;
  const int64_t c = P > 0 ? N / P : 0;
  if (layout == RA_LAYOUT_ZIGZAG && c % 2 != 0) return RA_ERR_UNSUPPORTED;
  if (dt == RA_BF16) {
    if (layout == RA_LAYOUT_ZIGZAG && c % 256 != 0) return RA_ERR_UNSUPPORTED;
    if (P > kMaxCausalSteps) return RA_ERR_UNSUPPORTED;
  }
  a->causal = 1;
  a->layout = static_cast<int32_t>(layout);
  return RA_OK;
}

}  // namespace

ra_status check_forward_args(int32_t B, int32_t H, int64_t N, int32_t d, int32_t P, bool causal,
                             ra_layout layout, ra_dtype dtype) {
  if (B < 0 || H < 0 || N < 0 || d < 1 || P < 1) return RA_ERR_INVALID_ARG;
  if (dtype != RA_F32 && dtype != RA_BF16) return RA_ERR_INVALID_ARG;
  const ra_status st = check_sizes(static_cast<int64_t>(B) * H * N, N, d, P, dtype);
  if (st != RA_OK) return st;
  FoldArgs a{};
  return causal ? check_causal(N, P, layout, dtype, &a) : RA_OK;
}

namespace {

ra_status forward_impl(const void* q, const void* k, const void* v, void* out, float* lse,
                       int32_t B, int32_t H, int64_t N, int32_t d, int32_t P, bool causal,
                       ra_layout layout, ra_dtype dtype, ra_stream_t stream) {
  FoldArgs a;
  ra_status st = check_attention(q, k, v, B, H, N, d, P, dtype, &a);
  if (st != RA_OK) return st;
  if (causal && (st = check_causal(N, P, layout, dtype, &a)) != RA_OK) return st;
  if (a.slices * a.nq == 0) return RA_OK;
  if (!out || !lse) return RA_ERR_INVALID_ARG;
  if (!aligned(out, dtype == RA_BF16 ? 16 : 4) || !aligned(lse, 4)) return RA_ERR_MISALIGNED;
  DeviceInfo di;
  if ((st = current_device(&di)) != RA_OK) return st;
  a.mode = kForward;
  a.out = out;
  a.lse = lse;
  a.status = di.status;
  return run_fold(a, dtype, reinterpret_cast<cudaStream_t>(stream));
}

ra_status partial_impl(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                       int64_t N, int32_t d, int32_t P, int32_t G, const ra_state* partials,
                       bool causal, ra_layout layout, ra_dtype dtype, ra_stream_t stream) {
  FoldArgs a;
  ra_status st = check_attention(q, k, v, B, H, N, d, P, dtype, &a);
  if (st != RA_OK) return st;
  if (causal && (st = check_causal(N, P, layout, dtype, &a)) != RA_OK) return st;
  if (!partials || G < 1 || G > RA_MAX_PARTIALS || G > P) return RA_ERR_INVALID_ARG;
  const int64_t rows = a.slices * a.nq;
  for (int g = 0; g < G; ++g) {
    const ra_state& p = partials[g];
    if (!state_ok(&p) || p.rows != rows || p.d != d) return RA_ERR_INVALID_ARG;
    if (!aligned(p.m, 4) || !aligned(p.l, 4) || !aligned(p.o, dtype == RA_BF16 ? 16 : 4))
      return RA_ERR_MISALIGNED;
    a.part.m[g] = p.m;
    a.part.l[g] = p.l;
    a.part.o[g] = p.o;
  }
  if (rows == 0) return RA_OK;
  DeviceInfo di;
  if ((st = current_device(&di)) != RA_OK) return st;
  a.mode = kPartial;
  a.G = G;
  a.status = di.status;
  return run_fold(a, dtype, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

int64_t split_workspace_bytes(int64_t rows, int32_t d, int32_t G) {
  auto up = [](int64_t x) { return (x + 255) / 256 * 256; };
  return static_cast<int64_t>(G) * (2 * up(rows * 4) + up(rows * static_cast<int64_t>(d) * 4));
}

ra_status split_forward(const void* q, const void* k, const void* v, void* out, float* lse,
                        int32_t B, int32_t H, int64_t N, int32_t d, int32_t P, int32_t G,
                        void* workspace, int64_t workspace_bytes, ra_dtype dtype,
                        cudaStream_t stream) {
  FoldArgs a;
  ra_status st = check_attention(q, k, v, B, H, N, d, P, dtype, &a);
  if (st != RA_OK) return st;
  if (G < 1 || G > RA_MAX_PARTIALS || G > P) return RA_ERR_INVALID_ARG;
  const int64_t rows = a.slices * a.nq;
  if (rows == 0) return RA_OK;
  if (!out || !lse || !workspace || workspace_bytes < 0) return RA_ERR_INVALID_ARG;
  if (!aligned(out, dtype == RA_BF16 ? 16 : 4) || !aligned(lse, 4) || !aligned(workspace, 256))
    return RA_ERR_MISALIGNED;
  if (workspace_bytes < split_workspace_bytes(rows, d, G)) return RA_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((st = current_device(&di)) != RA_OK) return st;
  // carve the G partial states out of the workspace
  auto up = [](int64_t x) { return (x + 255) / 256 * 256; };
  char* p = static_cast<char*>(workspace);
  MergeArgs mg{};
  for (int g = 0; g < G; ++g) {
    a.part.m[g] = reinterpret_cast<float*>(p);
    p += up(rows * 4);
    a.part.l[g] = reinterpret_cast<float*>(p);
    p += up(rows * 4);
    a.part.o[g] = reinterpret_cast<float*>(p);
    p += up(rows * static_cast<int64_t>(d) * 4);
  }
  mg.part = a.part;
  a.mode = kPartial;
  a.G = G;
  a.status = di.status;
  if ((st = run_fold(a, dtype, stream)) != RA_OK) return st;
  mg.G = G;
  mg.rows = rows;
  mg.d = d;
  mg.out = out;
  mg.lse = lse;
  mg.out_bf16 = dtype == RA_BF16 ? 1 : 0;
  mg.vec4 = (d % 4 == 0 && aligned(out, dtype == RA_BF16 ? 8 : 16)) ? 1 : 0;
  return launched(launch_merge(mg, stream));
}

}  // namespace ra

extern "C" {

RA_API ra_status ra_forward(const void* q, const void* k, const void* v, void* out, float* lse,
                            int32_t B, int32_t H, int64_t N, int32_t d, int32_t P, ra_dtype dtype,
                            ra_stream_t stream) {
  RA_TRACE("ra_forward");
  return forward_impl(q, k, v, out, lse, B, H, N, d, P, false, RA_LAYOUT_CONTIGUOUS, dtype,
                      stream);
}

RA_API ra_status ra_forward_causal(const void* q, const void* k, const void* v, void* out,
                                   float* lse, int32_t B, int32_t H, int64_t N, int32_t d,
                                   int32_t P, ra_layout layout, ra_dtype dtype,
                                   ra_stream_t stream) {
  RA_TRACE("ra_forward_causal");
  return forward_impl(q, k, v, out, lse, B, H, N, d, P, true, layout, dtype, stream);
}

RA_API ra_status ra_forward_partial(const void* q, const void* k, const void* v, int32_t B,
                                    int32_t H, int64_t N, int32_t d, int32_t P, int32_t G,
                                    const ra_state* partials, ra_dtype dtype,
                                    ra_stream_t stream) {
  RA_TRACE("ra_forward_partial");
  return partial_impl(q, k, v, B, H, N, d, P, G, partials, false, RA_LAYOUT_CONTIGUOUS, dtype,
                      stream);
}

RA_API ra_status ra_forward_partial_causal(const void* q, const void* k, const void* v,
                                           int32_t B, int32_t H, int64_t N, int32_t d, int32_t P,
                                           int32_t G, const ra_state* partials, ra_layout layout,
                                           ra_dtype dtype, ra_stream_t stream) {
  RA_TRACE("ra_forward_partial_causal");
  return partial_impl(q, k, v, B, H, N, d, P, G, partials, true, layout, dtype, stream);
}

RA_API int64_t ra_forward_split_workspace_bytes(int32_t B, int32_t H, int64_t N, int32_t d,
                                                int32_t G) {
  if (B < 0 || H < 0 || N < 0 || d < 1 || G < 1 || G > RA_MAX_PARTIALS) return -1;
  return split_workspace_bytes(static_cast<int64_t>(B) * H * N, d, G);
}

RA_API int32_t ra_forward_split_segments(int32_t B, int32_t H, int64_t N, int32_t d, int32_t P,
                                         ra_dtype dtype) {
  if (B < 1 || H < 1 || N < 1 || d < 1 || P < 1 || N % P != 0 || dtype != RA_BF16) return 1;
  const int64_t c = N / P;
  if (c % 128 != 0) return 1;
  const int64_t units = static_cast<int64_t>(B) * H * P * ((c / 128 + 1) / 2);
  const int64_t sms = device_sm_count();
  if (units >= sms) return 1;
  int64_t G = sms / units;  // the largest split that still runs in one wave
  // A segment needs enough K/V tiles to pay for its partial state and the
  // merge: at least 32 of them.
  const int64_t max_by_tiles = (N / 128) / 32;
  if (G > max_by_tiles) G = max_by_tiles;
  if (G > P) G = P;
  if (G > RA_MAX_PARTIALS) G = RA_MAX_PARTIALS;
  return static_cast<int32_t>(G < 1 ? 1 : G);
}

RA_API ra_status ra_forward_split(const void* q, const void* k, const void* v, void* out,
                                  float* lse, int32_t B, int32_t H, int64_t N, int32_t d,
                                  int32_t P, int32_t G, void* workspace, int64_t workspace_bytes,
                                  ra_dtype dtype, ra_stream_t stream) {
  RA_TRACE("ra_forward_split");
  return split_forward(q, k, v, out, lse, B, H, N, d, P, G, workspace, workspace_bytes, dtype,
                       reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace ra {
namespace {

ra_status backward_impl(const void* q, const void* k, const void* v, const void* out,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv,
                        float* workspace, int32_t B, int32_t H, int64_t N, int32_t d, int32_t P,
                        bool causal, ra_layout layout, ra_dtype dtype, ra_stream_t stream) {
  FoldArgs f;
  ra_status st = check_attention(q, k, v, B, H, N, d, P, dtype, &f);
  if (st != RA_OK) return st;
  if (causal && (st = check_causal(N, P, layout, dtype, &f)) != RA_OK) return st;
  const int64_t rows = f.slices * f.nq;
  if (rows == 0) return RA_OK;
  if (!out || !dout || !lse || !dq || !dk || !dv || !workspace) return RA_ERR_INVALID_ARG;
  const uintptr_t al = dtype == RA_BF16 ? 16 : 4;
  if (!aligned(out, al) || !aligned(dout, al) || !aligned(dq, al) || !aligned(dk, al) ||
      !aligned(dv, al) || !aligned(lse, 4) || !aligned(workspace, 16))
    return RA_ERR_MISALIGNED;
  DeviceInfo di;
  if ((st = current_device(&di)) != RA_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  BackwardArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.dout = dout;
  a.lse = lse;
  a.delta = workspace;
  a.nl = workspace + rows;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.slices = f.slices;
  a.N = N;
  a.d = d;
  a.P = P;
  a.causal = f.causal;
  a.layout = f.layout;
  a.tau = f.tau;
  a.scale_log2 = f.scale_log2;
  a.status = di.status;
  a.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  a.stall_cta = g_stall_cta.load(std::memory_order_relaxed);
  if ((st = launched(launch_delta(out, dout, lse, workspace, workspace + rows, rows, d, N, P,
                                  a.layout, dtype == RA_BF16, s))) != RA_OK)
    return st;
  if (dtype == RA_F32) return launched(launch_backward_f32(a, s));
  if ((st = get_encoder()) != RA_OK) return st;
  CUtensorMap tq, tk, tv, tdo;
  const void* src[4] = {q, k, v, dout};
  CUtensorMap* maps[4] = {&tq, &tk, &tv, &tdo};
  for (int x = 0; x < 4; ++x) {
    st = a.layout == kStriped ? make_map_striped(maps[x], src[x], rows, d, P)
                              : make_map(maps[x], src[x], rows, d);
    if (st != RA_OK) return st;
  }
  return launched(launch_backward_sm103(a, tq, tk, tv, tdo, s));
}

// One step of the ring backward: query block (q, dout, row terms) against
// one visiting block (k, v), adding into fp32 accumulators.  P = 1 over a
// block of c rows; `causal` masks later keys within the block (the diagonal
// block of a contiguous ring).
ra_status backward_block_impl(const void* q, const void* k, const void* v, const void* dout,
                              const float* lse, const float* rowterms, float* dq_acc,
                              float* dk_acc, float* dv_acc, int64_t batch, int64_t c, int32_t d,
                              int32_t causal, ra_dtype dtype, ra_stream_t stream) {
  if (batch < 0 || batch > INT32_MAX || causal < 0 || causal > 1) return RA_ERR_INVALID_ARG;
  FoldArgs f;
  ra_status st = check_attention(q, k, v, 1, static_cast<int32_t>(batch), c, d, 1, dtype, &f);
  if (st != RA_OK) return st;
  if (causal && (st = check_causal(c, 1, RA_LAYOUT_CONTIGUOUS, dtype, &f)) != RA_OK) return st;
  const int64_t rows = f.slices * f.nq;
  if (rows == 0) return RA_OK;
  if (!dout || !lse || !rowterms || !dq_acc || !dk_acc || !dv_acc) return RA_ERR_INVALID_ARG;
  const uintptr_t al = dtype == RA_BF16 ? 16 : 4;
  if (!aligned(dout, al) || !aligned(lse, 4) || !aligned(rowterms, 16) || !aligned(dq_acc, al) ||
      !aligned(dk_acc, al) || !aligned(dv_acc, al))
    return RA_ERR_MISALIGNED;
  DeviceInfo di;
  if ((st = current_device(&di)) != RA_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  BackwardArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.dout = dout;
  a.lse = lse;
  a.delta = rowterms;
  a.nl = rowterms + rows;
  a.dq = dq_acc;
  a.dk = dk_acc;
  a.dv = dv_acc;
  a.slices = f.slices;
  a.N = c;
  a.d = d;
  a.P = 1;
  a.causal = f.causal;
  a.layout = kContiguous;
  a.tau = f.tau;
  a.scale_log2 = f.scale_log2;
  a.status = di.status;
  a.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  a.stall_cta = g_stall_cta.load(std::memory_order_relaxed);
  a.accumulate = 1;
  if (dtype == RA_F32) return launched(launch_backward_f32(a, s));
  if ((st = get_encoder()) != RA_OK) return st;
  CUtensorMap tq, tk, tv, tdo;
  const void* src[4] = {q, k, v, dout};
  CUtensorMap* maps[4] = {&tq, &tk, &tv, &tdo};
  for (int x = 0; x < 4; ++x)
    if ((st = make_map(maps[x], src[x], rows, d)) != RA_OK) return st;
  return launched(launch_backward_sm103(a, tq, tk, tv, tdo, s));
}

}  // namespace
}  // namespace ra

extern "C" {

RA_API ra_status ra_backward_rowterms(const void* out, const void* dout, const float* lse,
                                      int64_t rows, int32_t d, ra_dtype dtype, float* workspace,
                                      ra_stream_t stream) {
  RA_TRACE("ra_backward_rowterms");
  if (rows < 0 || d < 1 || (dtype != RA_F32 && dtype != RA_BF16)) return RA_ERR_INVALID_ARG;
  if (rows > kMaxRows) return RA_ERR_UNSUPPORTED;
  if (rows == 0) return RA_OK;
  if (!out || !dout || !lse || !workspace) return RA_ERR_INVALID_ARG;
  const uintptr_t al = dtype == RA_BF16 ? 2 : 4;
  if (!aligned(out, al) || !aligned(dout, al) || !aligned(lse, 4) || !aligned(workspace, 16))
    return RA_ERR_MISALIGNED;
  DeviceInfo di;
  ra_status st = current_device(&di);
  if (st != RA_OK) return st;
  // one block of `rows` rows: block-major order is row order
  return launched(launch_delta(out, dout, lse, workspace, workspace + rows, rows, d, rows, 1,
                               kContiguous, dtype == RA_BF16,
                               reinterpret_cast<cudaStream_t>(stream)));
}

RA_API ra_status ra_backward_block(const void* q, const void* k, const void* v, const void* dout,
                                   const float* lse, const float* rowterms, float* dq_acc,
                                   float* dk_acc, float* dv_acc, int64_t batch, int64_t c,
                                   int32_t d, int32_t causal, ra_dtype dtype,
                                   ra_stream_t stream) {
  RA_TRACE("ra_backward_block");
  return backward_block_impl(q, k, v, dout, lse, rowterms, dq_acc, dk_acc, dv_acc, batch, c, d,
                             causal, dtype, stream);
}

RA_API ra_status ra_backward(const void* q, const void* k, const void* v, const void* out,
                             const void* dout, const float* lse, void* dq, void* dk, void* dv,
                             float* workspace, int32_t B, int32_t H, int64_t N, int32_t d,
                             int32_t P, ra_dtype dtype, ra_stream_t stream) {
  RA_TRACE("ra_backward");
  return backward_impl(q, k, v, out, dout, lse, dq, dk, dv, workspace, B, H, N, d, P, false,
                       RA_LAYOUT_CONTIGUOUS, dtype, stream);
}

RA_API ra_status ra_backward_causal(const void* q, const void* k, const void* v, const void* out,
                                    const void* dout, const float* lse, void* dq, void* dk,
                                    void* dv, float* workspace, int32_t B, int32_t H, int64_t N,
                                    int32_t d, int32_t P, ra_layout layout, ra_dtype dtype,
                                    ra_stream_t stream) {
  RA_TRACE("ra_backward_causal");
  return backward_impl(q, k, v, out, dout, lse, dq, dk, dv, workspace, B, H, N, d, P, true,
                       layout, dtype, stream);
}

RA_API ra_status ra_state_init(const ra_state* st, ra_stream_t stream) {
  RA_TRACE("ra_state_init");
  if (!state_ok(st)) return RA_ERR_INVALID_ARG;
  if (!aligned(st->m, 4) || !aligned(st->l, 4) || !aligned(st->o, 4)) return RA_ERR_MISALIGNED;
  if (st->rows == 0) return RA_OK;
  DeviceInfo di;
  ra_status s = current_device(&di);
  if (s != RA_OK) return s;
  return launched(launch_state_init(st->m, st->l, st->o, st->rows, st->d,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

RA_API ra_status ra_fold(const ra_state* st, const void* q, const void* kblk, const void* vblk,
                         int64_t batch, int64_t kv_rows, ra_dtype dtype, ra_stream_t stream) {
  RA_TRACE("ra_fold");
  if (!state_ok(st) || !q || !kblk || !vblk) return RA_ERR_INVALID_ARG;
  if (batch < 1 || kv_rows < 0) return RA_ERR_INVALID_ARG;
  if (dtype != RA_F32 && dtype != RA_BF16) return RA_ERR_INVALID_ARG;
  if (st->rows % batch != 0) return RA_ERR_UNSUPPORTED;
  const int32_t d = st->d;
  const int64_t rq = st->rows / batch;
  if (st->rows > kMaxRows || batch * kv_rows > kMaxRows) return RA_ERR_UNSUPPORTED;
  if (dtype == RA_BF16) {
    if (d != 64 && d != 128) return RA_ERR_UNSUPPORTED;
    if (rq % 128 != 0 || kv_rows % 128 != 0) return RA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(kblk, 16) || !aligned(vblk, 16) || !aligned(st->o, 16))
      return RA_ERR_MISALIGNED;
  } else {
    if (d > 256) return RA_ERR_UNSUPPORTED;
    if (!aligned(q, 4) || !aligned(kblk, 4) || !aligned(vblk, 4) || !aligned(st->o, 4))
      return RA_ERR_MISALIGNED;
  }
  if (!aligned(st->m, 4) || !aligned(st->l, 4)) return RA_ERR_MISALIGNED;
  if (st->rows == 0 || kv_rows == 0) return RA_OK;
  DeviceInfo di;
  ra_status s = current_device(&di);
  if (s != RA_OK) return s;
  FoldArgs a{};
  a.q = q;
  a.k = kblk;
  a.v = vblk;
  a.slices = batch;
  a.nq = rq;
  a.nk = kv_rows;
  a.d = d;
  a.P = 1;
  a.G = 1;
  a.mode = kFold;
  a.tau = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  a.st_m = st->m;
  a.st_l = st->l;
  a.st_o = st->o;
  a.status = di.status;
  return run_fold(a, dtype, reinterpret_cast<cudaStream_t>(stream));
}

RA_API ra_status ra_merge(const ra_state* partials, int32_t G, void* out, float* lse,
                          ra_dtype out_dtype, ra_stream_t stream) {
  RA_TRACE("ra_merge");
  if (!partials || G < 1 || G > RA_MAX_PARTIALS || !out || !lse) return RA_ERR_INVALID_ARG;
  if (out_dtype != RA_F32 && out_dtype != RA_BF16) return RA_ERR_INVALID_ARG;
  MergeArgs a{};
  const int64_t rows = partials[0].rows;
  const int32_t d = partials[0].d;
  bool vec = d % 4 == 0 && aligned(out, out_dtype == RA_BF16 ? 8 : 16);
  for (int g = 0; g < G; ++g) {
    const ra_state& p = partials[g];
    if (!state_ok(&p) || p.rows != rows || p.d != d) return RA_ERR_INVALID_ARG;
    if (!aligned(p.m, 4) || !aligned(p.l, 4) || !aligned(p.o, 4)) return RA_ERR_MISALIGNED;
    vec = vec && aligned(p.o, 16);
    a.part.m[g] = p.m;
    a.part.l[g] = p.l;
    a.part.o[g] = p.o;
  }
  if (!aligned(out, out_dtype == RA_BF16 ? 2 : 4) || !aligned(lse, 4)) return RA_ERR_MISALIGNED;
  if (rows == 0) return RA_OK;
  DeviceInfo di;
  ra_status s = current_device(&di);
  if (s != RA_OK) return s;
  a.G = G;
  a.rows = rows;
  a.d = d;
  a.out = out;
  a.lse = lse;
  a.out_bf16 = out_dtype == RA_BF16 ? 1 : 0;
  a.vec4 = vec ? 1 : 0;
  return launched(launch_merge(a, reinterpret_cast<cudaStream_t>(stream)));
}

RA_API ra_status ra_last_device_status(ra_stream_t stream) {
  RA_TRACE("ra_last_device_status");
  DeviceInfo di;
  ra_status s = current_device(&di);
  if (s != RA_OK) return s;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return RA_ERR_CUDA;
  int word = 0;
  const int zero = 0;
  if (cudaMemcpy(&word, di.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return RA_ERR_CUDA;
  if (cudaMemcpy(di.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return RA_ERR_CUDA;
  return word == 0 ? RA_OK : RA_ERR_TIMEOUT;
}

RA_API void ra_watchdog_config(int64_t wait_cycles, int64_t stall_cta) {
  g_wait_limit.store(wait_cycles > 0 ? wait_cycles : kDefaultWaitCycles,
                     std::memory_order_relaxed);
  g_stall_cta.store(stall_cta >= 0 ? stall_cta : -1, std::memory_order_relaxed);
}

RA_API const char* ra_status_string(ra_status s) {
  switch (s) {
    case RA_OK: return "RA_OK";
    case RA_ERR_INVALID_ARG: return "RA_ERR_INVALID_ARG: invalid argument";
    case RA_ERR_UNSUPPORTED: return "RA_ERR_UNSUPPORTED: shape or type not supported";
    case RA_ERR_MISALIGNED: return "RA_ERR_MISALIGNED: pointer alignment too small";
    case RA_ERR_ARCH: return "RA_ERR_ARCH: no compute capability 10.3 device";
    case RA_ERR_CUDA: return "RA_ERR_CUDA: CUDA call failed";
    case RA_ERR_TIMEOUT: return "RA_ERR_TIMEOUT: a kernel wait ran out (watchdog)";
  }
  return "unknown ra_status";
}

RA_API int32_t ra_version(void) { return 200; }  // 0.2.0

}  // extern "C"
