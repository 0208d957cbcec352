// Backward of ring attention: the row term D and the fp32 (FFMA) path.
//
// For the loss L = sum(dO * out) and P = softmax(tau Q K^T) per row:
//   D_r = sum_e dO_re out_re
//   dV = P^T dO;  dP = dO V^T;  dS = P * (dP - D);  dQ = tau dS K;  dK = tau dS^T Q
// with P recomputed from the forward's lse: P_rj = exp(tau q_r . k_j - lse_r)
// ("Ring attention, explained", step 6: the backward runs on the same ring,
// the key-value blocks carrying their gradient accumulators).
//
// The fp32 path has two kernels, neither with atomics:
//   dq: query rows walk the key blocks in ring order (i - t) mod P, as the
//       forward does;
//   dkv: key rows walk the query blocks their block visits on the ring,
//       (j + t) mod P, and accumulate dK and dV.
// For d <= 128 and grids of 128 CTAs or more both are tiled (64 stationary
// rows per CTA, 32-row tiles of the other side staged in shared memory);
// otherwise up to 8 warps share one row (each folds every S-th chunk of 32
// rows of the other side) and the lanes split the head dimension (lane e
// holds elements e, e + 32, ...).
// Causal ("Ring attention, explained", "The causal-mask catch"): a query at
// position n sees keys at positions <= n; `layout` says which positions form
// each block (contiguous, zigzag or striped), as in the forward.

#include <cuda_bf16.h>

#include <cmath>

#include <cooperative_groups.h>

#include "ra_fork.h"
#include "ra_internal.h"
#include "ra_layout.cuh"

namespace ra {
namespace {

// The per-query terms D and nl are stored block-major: (slice, block, local
// row), so that a query tile's 128 values are contiguous under every layout.
__device__ __forceinline__ int64_t bmajor(int layout, int64_t slice, int64_t N, int64_t n,
                                          int64_t P, int64_t c) {
  return slice * N + layout_block(layout, n, P, c) * c + layout_local(layout, n, P, c);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// D_r = sum_e dO_re * out_re and nl_r = -lse_r * log2(e) for every row, in
// block-major order; one warp per row.
template <bool kBf16>
__global__ void __launch_bounds__(256) delta_kernel(const void* out, const void* dout,
                                                    const float* lse, float* delta, float* nl,
                                                    int64_t rows, int d, int64_t N, int64_t P,
                                                    int layout) {
  const int lane = threadIdx.x % 32;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
       r < rows; r += stride) {
    float acc = 0.f;
    for (int e = lane; e < d; e += 32) {
      float o, g;
      if (kBf16) {
        o = __bfloat162float(static_cast<const __nv_bfloat16*>(out)[r * d + e]);
        g = __bfloat162float(static_cast<const __nv_bfloat16*>(dout)[r * d + e]);
      } else {
        o = static_cast<const float*>(out)[r * d + e];
        g = static_cast<const float*>(dout)[r * d + e];
      }
      acc = fmaf(o, g, acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) {
      const int64_t x = bmajor(layout, r / N, N, r % N, P, N / P);
      delta[x] = acc;
      nl[x] = -lse[r] * 1.4426950408889634f;
    }
  }
}

// Two dot products of length d at once, s = x.y and dp = u.w: 16-byte loads
// and two FMA chains each when every row starts on a 16-byte boundary (vec),
// a scalar tail otherwise.
__device__ __forceinline__ void dot2(const float* __restrict__ x, const float* __restrict__ y,
                                     const float* __restrict__ u, const float* __restrict__ w,
                                     int d, bool vec, float& s, float& dp) {
  float s0 = 0.f, s1 = 0.f, p0 = 0.f, p1 = 0.f;
  int e = 0;
  if (vec) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const float4* y4 = reinterpret_cast<const float4*>(y);
    const float4* u4 = reinterpret_cast<const float4*>(u);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    const int n4 = d / 4;
#pragma unroll 2
    for (int i = 0; i < n4; ++i) {
      const float4 a = x4[i], b = y4[i], c = u4[i], f = w4[i];
      s0 = fmaf(a.x, b.x, s0);
      s1 = fmaf(a.y, b.y, s1);
      s0 = fmaf(a.z, b.z, s0);
      s1 = fmaf(a.w, b.w, s1);
      p0 = fmaf(c.x, f.x, p0);
      p1 = fmaf(c.y, f.y, p1);
      p0 = fmaf(c.z, f.z, p0);
      p1 = fmaf(c.w, f.w, p1);
    }
    e = 4 * n4;
  }
  for (; e < d; ++e) {
    s0 = fmaf(x[e], y[e], s0);
    p0 = fmaf(u[e], w[e], p0);
  }
  s = s0 + s1;
  dp = p0 + p1;
}

// rows of every operand start on 16-byte boundaries
__device__ __forceinline__ bool rows_vec(const BackwardArgs& a) {
  const uintptr_t m = reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.k) |
                      reinterpret_cast<uintptr_t>(a.v) | reinterpret_cast<uintptr_t>(a.dout);
  return a.d % 4 == 0 && m % 16 == 0;
}

// Row kernels: one query row (dq) or key row (dkv) per S warps (1, 2, 4 or
// 8), the row's chunks of 32 rows of the other side dealt round robin to
// its warps; each warp accumulates its chunks, and the row's first warp
// adds the S partial sums in shared memory.  A CTA holds the S warps of
// each of its rows: max(4, S) warps, so that small grids still come in fine
// pieces.  The split kernels get 128 registers a thread (16 warps an SM),
// the unsplit ones 64.
template <int S>
struct RowCta {
  static constexpr int kWarps = S < 4 ? 4 : S;
  static constexpr int kRows = kWarps / S;
  static constexpr int kMinBlocks = S == 1 ? 8 : 16 / kWarps;
};
constexpr int kResidentWarps = 16;  // per SM, at 128 registers a thread

// Gradient of one query row over all key blocks in ring order.
template <int DV, int S>
__global__ void __launch_bounds__(RowCta<S>::kWarps * 32, RowCta<S>::kMinBlocks)
    dq_f32_kernel(const BackwardArgs a) {
  constexpr int kWarps = RowCta<S>::kWarps;
  constexpr int kRows = RowCta<S>::kRows;
  __shared__ __align__(16) float qs[kWarps][32 * DV];
  __shared__ __align__(16) float gs[kWarps][32 * DV];
  __shared__ float part[S > 1 ? kWarps : 1][32 * DV];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int sp = warp % S;
  const int d = a.d;
  const int64_t rid = static_cast<int64_t>(blockIdx.x) * kRows + warp / S;
  const bool live = rid < a.slices * a.N;
  const int64_t slice = live ? rid / a.N : 0, n = live ? rid % a.N : 0;
  const int64_t c = a.N / a.P;
  const int64_t nch = (c + 31) / 32;
  const int i = static_cast<int>(layout_block(a.layout, n, a.P, c));
  const float* q = static_cast<const float*>(a.q);
  const float* k = static_cast<const float*>(a.k);
  const float* v = static_cast<const float*>(a.v);
  const float* g = static_cast<const float*>(a.dout);
  float acc[DV];
#pragma unroll
  for (int x = 0; x < DV; ++x) acc[x] = 0.f;
  if (live) {
    for (int e = lane; e < d; e += 32) {
      qs[warp][e] = q[rid * d + e];
      gs[warp][e] = g[rid * d + e];
    }
    __syncwarp();
    const float lse = a.lse[rid], D = a.delta[bmajor(a.layout, slice, a.N, n, a.P, c)];
    const bool vec = rows_vec(a);
    const int64_t sb = slice * a.N;
    for (int t = 0; t < a.P; ++t) {
      int j = (i - t) % a.P;
      if (j < 0) j += a.P;
      // chunk ci of this block is the row's chunk t nch + ci
      for (int64_t ci = (sp - (static_cast<int64_t>(t) * nch) % S + S) % S; ci < nch; ci += S) {
        const int64_t c0 = ci * 32;
        if (a.causal && layout_pos(a.layout, j, c0, a.P, c) > n) break;  // rest of the block masked
        const int64_t key = c0 + lane;
        const int64_t kp = key < c ? layout_pos(a.layout, j, key, a.P, c) : 0;
        float ds = 0.f;
        if (key < c && (!a.causal || kp <= n)) {
          float s, dp;
          dot2(qs[warp], k + (sb + kp) * d, gs[warp], v + (sb + kp) * d, d, vec, s, dp);
          const float p = expf(s * a.tau - lse);
          ds = p * (dp - D);
        }
        // fixed trip count (ds = 0 for masked keys and keys past the block's
        // end, which read the slice's first row): several loads in flight
#pragma unroll 8
        for (int jj = 0; jj < 32; ++jj) {
          const float dsj = __shfl_sync(0xffffffffu, ds, jj);
          const int64_t kpj = __shfl_sync(0xffffffffu, kp, jj);
          const float* kr = k + (sb + kpj) * d;
#pragma unroll
          for (int x = 0; x < DV; ++x) {
            const int e = lane + 32 * x;
            if (e < d) acc[x] = fmaf(dsj, kr[e], acc[x]);
          }
        }
      }
    }
  }
  if (S > 1) {
#pragma unroll
    for (int x = 0; x < DV; ++x) part[warp][lane + 32 * x] = acc[x];
    __syncthreads();
    if (sp != 0 || !live) return;
#pragma unroll
    for (int x = 0; x < DV; ++x) {
      float sum = part[warp][lane + 32 * x];
#pragma unroll
      for (int y = 1; y < S; ++y) sum += part[warp + y][lane + 32 * x];
      acc[x] = sum;
    }
  } else if (!live) {
    return;
  }
  float* dq = static_cast<float*>(a.dq);
#pragma unroll
  for (int x = 0; x < DV; ++x) {
    const int e = lane + 32 * x;
    if (e < d) dq[rid * d + e] = (a.accumulate ? dq[rid * d + e] : 0.f) + acc[x] * a.tau;
  }
}

// Gradients of one key row over the query blocks its block visits.
template <int DV, int S>
__global__ void __launch_bounds__(RowCta<S>::kWarps * 32, RowCta<S>::kMinBlocks)
    dkv_f32_kernel(const BackwardArgs a) {
  constexpr int kWarps = RowCta<S>::kWarps;
  constexpr int kRows = RowCta<S>::kRows;
  __shared__ __align__(16) float ks[kWarps][32 * DV];
  __shared__ __align__(16) float vs[kWarps][32 * DV];
  __shared__ float part_k[S > 1 ? kWarps : 1][32 * DV];
  __shared__ float part_v[S > 1 ? kWarps : 1][32 * DV];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int sp = warp % S;
  const int d = a.d;
  const int64_t rid = static_cast<int64_t>(blockIdx.x) * kRows + warp / S;
  const bool live = rid < a.slices * a.N;
  const int64_t slice = live ? rid / a.N : 0, n = live ? rid % a.N : 0;
  const int64_t c = a.N / a.P;
  const int64_t nch = (c + 31) / 32;
  const int j = static_cast<int>(layout_block(a.layout, n, a.P, c));
  const float* q = static_cast<const float*>(a.q);
  const float* k = static_cast<const float*>(a.k);
  const float* v = static_cast<const float*>(a.v);
  const float* g = static_cast<const float*>(a.dout);
  float gk[DV], gv[DV];
#pragma unroll
  for (int x = 0; x < DV; ++x) gk[x] = gv[x] = 0.f;
  if (live) {
    for (int e = lane; e < d; e += 32) {
      ks[warp][e] = k[rid * d + e];
      vs[warp][e] = v[rid * d + e];
    }
    __syncwarp();
    const bool vec = rows_vec(a);
    const int64_t sb = slice * a.N;
    for (int t = 0; t < a.P; ++t) {
      const int i = (j + t) % a.P;  // the device holding this block at step t
      for (int64_t ci = (sp - (static_cast<int64_t>(t) * nch) % S + S) % S; ci < nch; ci += S) {
        const int64_t row = ci * 32 + lane;
        const int64_t qp = row < c ? layout_pos(a.layout, i, row, a.P, c) : 0;
        float p = 0.f, ds = 0.f;
        if (row < c && (!a.causal || qp >= n)) {
          float s, dp;
          dot2(q + (sb + qp) * d, ks[warp], g + (sb + qp) * d, vs[warp], d, vec, s, dp);
          p = expf(s * a.tau - a.lse[sb + qp]);
          ds = p * (dp - a.delta[sb + static_cast<int64_t>(i) * c + row]);
        }
        // fixed trip count (p = ds = 0 for masked rows and rows past the
        // block's end, which read the slice's first row): loads in flight
#pragma unroll 8
        for (int jj = 0; jj < 32; ++jj) {
          const float pj = __shfl_sync(0xffffffffu, p, jj);
          const float dsj = __shfl_sync(0xffffffffu, ds, jj);
          const int64_t qpj = __shfl_sync(0xffffffffu, qp, jj);
          const float* qr = q + (sb + qpj) * d;
          const float* gr = g + (sb + qpj) * d;
#pragma unroll
          for (int x = 0; x < DV; ++x) {
            const int e = lane + 32 * x;
            if (e < d) {
              gv[x] = fmaf(pj, gr[e], gv[x]);
              gk[x] = fmaf(dsj, qr[e], gk[x]);
            }
          }
        }
      }
    }
  }
  if (S > 1) {
#pragma unroll
    for (int x = 0; x < DV; ++x) {
      part_k[warp][lane + 32 * x] = gk[x];
      part_v[warp][lane + 32 * x] = gv[x];
    }
    __syncthreads();
    if (sp != 0 || !live) return;
#pragma unroll
    for (int x = 0; x < DV; ++x) {
      float sk = part_k[warp][lane + 32 * x], sv = part_v[warp][lane + 32 * x];
#pragma unroll
      for (int y = 1; y < S; ++y) {
        sk += part_k[warp + y][lane + 32 * x];
        sv += part_v[warp + y][lane + 32 * x];
      }
      gk[x] = sk;
      gv[x] = sv;
    }
  } else if (!live) {
    return;
  }
  float* dk = static_cast<float*>(a.dk);
  float* dv = static_cast<float*>(a.dv);
#pragma unroll
  for (int x = 0; x < DV; ++x) {
    const int e = lane + 32 * x;
    if (e < d) {
      dk[rid * d + e] = (a.accumulate ? dk[rid * d + e] : 0.f) + gk[x] * a.tau;
      dv[rid * d + e] = (a.accumulate ? dv[rid * d + e] : 0.f) + gv[x];
    }
  }
}

// Warps per row: at most 8, at most one per chunk of the row's walk, and
// only as many as stay resident at once.
int bwd_row_split(const BackwardArgs& a) {
  const int64_t rows = a.slices * a.N;
  const int64_t chunks = static_cast<int64_t>(a.P) * ((a.N / a.P + 31) / 32);
  const int64_t want = static_cast<int64_t>(device_sm_count()) * kResidentWarps;
  int S = 1;
  while (S < 8 && rows * S * 2 <= want && chunks >= S * 2) S *= 2;
  return S;
}

template <int DV, int S>
cudaError_t launch_bwd_rows(const BackwardArgs& a, cudaStream_t s) {
  const int64_t rows = a.slices * a.N;
  constexpr int kRows = RowCta<S>::kRows;
  const unsigned grid = static_cast<unsigned>((rows + kRows - 1) / kRows);
  // the two kernels are independent: dK/dV on a forked side stream
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  ForkJoin fj;
  if (e == cudaSuccess) e = fj.fork(s, dev);
  if (e != cudaSuccess) return e;
  dq_f32_kernel<DV, S><<<grid, RowCta<S>::kWarps * 32, 0, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dkv_f32_kernel<DV, S><<<grid, RowCta<S>::kWarps * 32, 0, fj.side>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return fj.join(s);
}

template <int DV>
cudaError_t launch_bwd_dv(const BackwardArgs& a, cudaStream_t s) {
  switch (bwd_row_split(a)) {
    case 8:
      return launch_bwd_rows<DV, 8>(a, s);
    case 4:
      return launch_bwd_rows<DV, 4>(a, s);
    case 2:
      return launch_bwd_rows<DV, 2>(a, s);
    default:
      return launch_bwd_rows<DV, 1>(a, s);
  }
}

// ---- tiled kernels (d <= 128, grids of 128 CTAs or more) ----
// As the tiled forward: a CTA of W = 4 or 8 warps keeps 64 rows stationary
// and streams 32-row tiles of the other side through shared memory.  With 8
// warps the two halves of the CTA (warps 0-3 and 4-7) take 16 streamed rows
// each, with 4 warps one takes all 32: lane (rg, kg) = (lane / 8, lane % 8)
// of warp w computes the 4 x NY blocks (NY = 2 or 4) of rows
// 16 (w % 4) + 4rg + 0..3 against streamed rows 16 (w / 4) + NY kg + ..,
// and accumulates its rows' gradients over its half's streamed rows in
// columns 4kg + 32m + 0..3; two halves' sums are added in shared memory at
// the end.  Eight warps on the same shared memory (one CTA an SM at d = 128)
// measured 30-47 % faster than four, and the launches use eight.  Tiles used
// as a product's reduction operand are stored transposed ([d][rows]) for
// 16-byte reads.
template <int W>
struct Warps {
  static constexpr int kThreads = 32 * W;
  static constexpr int kHalves = W / 4;
  static constexpr int kRows = 32 / kHalves;  // streamed rows per half of a tile
  static constexpr int kNY = kRows / 8;       // streamed rows per lane
};
constexpr int kTM = 64;         // stationary rows per CTA
constexpr int kTN = 32;         // streamed rows per tile
constexpr int kSS = kTM + 4;    // row stride of transposed stationary tiles, P^T, dS^T
constexpr int kNS = kTN + 4;    // row stride of transposed streamed tiles
// Each tiled CTA takes a whole SM (up to 158 KB of shared memory): the tiled
// kernels run when their CTAs, split over clusters where the tiles are too
// few for the SMs, number at least kTiledMinCtas; below that the row
// kernels, with many more warps, are faster.
constexpr int64_t kTiledMinCtas = 128;

template <int DT>
struct DqSmem {  // floats
  static constexpr int kQ = 0;                    // Q^T   [DT][kSS]
  static constexpr int kG = kQ + DT * kSS;        // dO^T  [DT][kSS]
  static constexpr int kK = kG + DT * kSS;        // K^T   [DT][kNS]
  static constexpr int kV = kK + DT * kNS;        // V^T   [DT][kNS]
  static constexpr int kKr = kV + DT * kNS;       // K     [kTN][DT + 4]
  static constexpr int kDS = kKr + kTN * (DT + 4);  // dS^T [kTN][kSS]
  static constexpr int kBytes = (kDS + kTN * kSS) * 4;
};

template <int DT>
struct DkvSmem {  // floats
  static constexpr int kK = 0;                    // K^T   [DT][kSS]
  static constexpr int kV = kK + DT * kSS;        // V^T   [DT][kSS]
  static constexpr int kQ = kV + DT * kSS;        // Q^T   [DT][kNS]
  static constexpr int kG = kQ + DT * kNS;        // dO^T  [DT][kNS]
  static constexpr int kQr = kG + DT * kNS;       // Q     [kTN][DT + 4]
  static constexpr int kGr = kQr + kTN * (DT + 4);  // dO  [kTN][DT + 4]
  static constexpr int kP = kGr + kTN * (DT + 4);   // P^T  [kTN][kSS]
  static constexpr int kDS = kP + kTN * kSS;        // dS^T [kTN][kSS]
  static constexpr int kBytes = (kDS + kTN * kSS) * 4;
};

// NY consecutive floats at p (8- or 16-byte aligned)
template <int NY>
__device__ __forceinline__ void load_ny(const float* p, float (&v)[NY]) {
  if constexpr (NY == 4) {
    const float4 x = *reinterpret_cast<const float4*>(p);
    v[0] = x.x;
    v[1] = x.y;
    v[2] = x.z;
    v[3] = x.w;
  } else {
    const float2 x = *reinterpret_cast<const float2*>(p);
    v[0] = x.x;
    v[1] = x.y;
  }
}

// s[x][y] += a[e][r0 + x] * b[e][c0 + y] and t[x][y] += c[e][r0 + x] * f[e][c0 + y]
// over e < d: the two 4 x NY score blocks of a lane from transposed tiles.
template <int NY>
__device__ __forceinline__ void two_blocks(const float* a, const float* b, const float* c,
                                           const float* f, int d, int sa, int sb, int r0,
                                           int c0, float (&s)[4][NY], float (&t)[4][NY]) {
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < NY; ++y) s[x][y] = t[x][y] = 0.f;
#pragma unroll 8
  for (int e = 0; e < d; ++e) {
    const float4 a4 = *reinterpret_cast<const float4*>(a + e * sa + r0);
    const float4 c4 = *reinterpret_cast<const float4*>(c + e * sa + r0);
    float bv[NY], fv[NY];
    load_ny<NY>(b + e * sb + c0, bv);
    load_ny<NY>(f + e * sb + c0, fv);
    const float av[4] = {a4.x, a4.y, a4.z, a4.w};
    const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < NY; ++y) {
        s[x][y] = fmaf(av[x], bv[y], s[x][y]);
        t[x][y] = fmaf(cv[x], fv[y], t[x][y]);
      }
  }
}

// acc[x][m][y] += sum over the half's streamed rows k = k0 .. k0 + KH - 1 of
// wT[k][r0 + x] * src[k][4 kg + 32 m + y]
template <int DT, int KH>
__device__ __forceinline__ void accumulate_rows(const float* wT, const float* src, int r0, int kg,
                                                int k0, float (&acc)[4][DT / 32][4]) {
#pragma unroll 8
  for (int k = k0; k < k0 + KH; ++k) {
    const float4 w4 = *reinterpret_cast<const float4*>(wT + k * kSS + r0);
    const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int m = 0; m < DT / 32; ++m) {
      const float4 v4 = *reinterpret_cast<const float4*>(src + k * (DT + 4) + 4 * kg + 32 * m);
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        acc[x][m][0] = fmaf(wv[x], v4.x, acc[x][m][0]);
        acc[x][m][1] = fmaf(wv[x], v4.y, acc[x][m][1]);
        acc[x][m][2] = fmaf(wv[x], v4.z, acc[x][m][2]);
        acc[x][m][3] = fmaf(wv[x], v4.w, acc[x][m][3]);
      }
    }
  }
}

// Stationary tile of 64 rows (block b, local rows r0 ..), transposed: the
// column e of row x at dst[e * kSS + x]; rows past the block and columns
// past d are zero.
template <int DT, int NT>
__device__ __forceinline__ void load_stationary(float* dst, const float* src, int layout, int b,
                                                int64_t r0, int64_t P, int64_t c, int d,
                                                int tid) {
  for (int x = tid; x < kTM * DT; x += NT) {
    const int row = x / DT, e = x % DT;
    const int64_t r = r0 + row;
    float val = 0.f;
    if (r < c && e < d) val = src[layout_pos(layout, b, r, P, c) * d + e];
    dst[e * kSS + row] = val;
  }
}


// The streamed tiles a tiled CTA visits, in order (this CTA's share: every
// split-th visible tile).  kDq: the query-stationary walk, key blocks
// (base - t) mod P, under the mask a block's tiles after the CTA's last query
// (lim) end it; else the key-stationary walk, query blocks (base + t) mod P,
// under the mask a tile whose last query precedes the CTA's first key (lim)
// is skipped.
template <bool kDq>
struct StreamWalk {
  int P, base, layout, split, cr;
  bool causal;
  int64_t c, lim;
  int t = 0, tix = 0;
  int64_t c0 = 0;
  __device__ int block() const {
    if (kDq) {
      const int j = (base - t) % P;
      return j < 0 ? j + P : j;
    }
    return (base + t) % P;
  }
  __device__ bool valid() const { return t < P; }
  // from (t, c0) to the first visible tile
  __device__ void visible() {
    while (t < P) {
      if (c0 >= c) {
        ++t;
        c0 = 0;
        continue;
      }
      if (causal) {
        const int b = block();
        if (kDq) {
          if (layout_pos(layout, b, c0, P, c) > lim) {  // rest of the block masked
            ++t;
            c0 = 0;
            continue;
          }
        } else {
          const int64_t qe = (c0 + kTN < c ? c0 + kTN : c) - 1;
          if (layout_pos(layout, b, qe, P, c) < lim) {
            c0 += kTN;
            continue;
          }
        }
      }
      return;
    }
  }
  // from (t, c0) to the first of this CTA's tiles
  __device__ void settle() {
    visible();
    while (t < P && tix % split != cr) {
      ++tix;
      c0 += kTN;
      visible();
    }
  }
  __device__ void advance() {
    ++tix;
    c0 += kTN;
    settle();
  }
};

// One streamed tile (block b, local rows c0 ..) of src, NT threads: the
// thread's kPre values, fetched into registers while the previous tile is
// computed and stored to shared memory (transposed into dT and, if dR,
// row-major into dR) when that one is done.
template <int DT, int NT>
struct Streamed {
  static constexpr int kPre = kTN * DT / NT;
  float r[kPre];
  __device__ void fetch(const float* src, int layout, int b, int64_t c0, int64_t P, int64_t c,
                        int d, int tid) {
#pragma unroll
    for (int it = 0; it < kPre; ++it) {
      const int x = tid + it * NT;
      const int row = x / DT, e = x % DT;
      const int64_t rr = c0 + row;
      r[it] = (rr < c && e < d) ? src[layout_pos(layout, b, rr, P, c) * d + e] : 0.f;
    }
  }
  __device__ void store(float* dT, float* dR, int tid) const {
#pragma unroll
    for (int it = 0; it < kPre; ++it) {
      const int x = tid + it * NT;
      const int row = x / DT, e = x % DT;
      dT[e * kNS + row] = r[it];
      if (dR) dR[row * (DT + 4) + e] = r[it];
    }
  }
};

// Sums of a split tile (split > 1: the CTAs of a cluster share one tile of
// 64 stationary rows, CTA r taking the streamed tiles r, r + split, ... of
// the walk): each CTA puts its nacc accumulators of the 64 rows into its
// shared memory ([acc][row][DT]); after a cluster barrier CTA r adds up rows
// r 64 / split .. over every CTA and writes them through put(row, e, sums);
// a second barrier keeps every CTA's shared memory until all have read it.
template <int DT>
__device__ __forceinline__ void put_rows(float* sm, int z, const float (&acc)[4][DT / 32][4],
                                         int lrow0, int kg) {
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int m = 0; m < DT / 32; ++m)
#pragma unroll
      for (int y = 0; y < 4; ++y)
        sm[(z * kTM + lrow0 + x) * DT + 4 * kg + 32 * m + y] = acc[x][m][y];
}

// acc += the sums put_rows wrote for the same thread's rows and columns.
template <int DT>
__device__ __forceinline__ void add_rows(const float* sm, int z, float (&acc)[4][DT / 32][4],
                                         int lrow0, int kg) {
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int m = 0; m < DT / 32; ++m)
#pragma unroll
      for (int y = 0; y < 4; ++y)
        acc[x][m][y] += sm[(z * kTM + lrow0 + x) * DT + 4 * kg + 32 * m + y];
}

// After put_rows of every accumulator (behind a __syncthreads).
template <int DT, int kAcc, int NT, typename Put>
__device__ __forceinline__ void split_sums(float* sm, int split, int cr, int tid, int d, Put put) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  const int rows_per = kTM / split;
  for (int idx = tid; idx < rows_per * d; idx += NT) {
    const int rr = cr * rows_per + idx / d, e = idx % d;
    float sums[kAcc];
#pragma unroll
    for (int z = 0; z < kAcc; ++z) sums[z] = 0.f;
    for (int p = 0; p < split; ++p) {
      const float* peer = cluster.map_shared_rank(sm, p);
#pragma unroll
      for (int z = 0; z < kAcc; ++z) sums[z] += peer[(z * kTM + rr) * DT + e];
    }
    put(rr, e, sums);
  }
  cluster.sync();
}

// dQ for 64 query rows of block i: the key blocks in ring order (i - t) mod P.
template <int DT, int W>
__global__ void __launch_bounds__(32 * W, DT == 64 && W == 8 ? 2 : 1)
    dq_f32_tiled(const BackwardArgs a, int split) {
  using S = DqSmem<DT>;
  using WW = Warps<W>;
  constexpr int kTT = WW::kThreads;
  constexpr int kTH = WW::kRows;
  constexpr int kNY = WW::kNY;
  extern __shared__ __align__(16) float sm[];
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int rg = lane / 8, kg = lane % 8;
  const int d = a.d;
  const int64_t c = a.N / a.P;
  const int64_t tiles = (c + kTM - 1) / kTM;
  const int cr = split > 1 ? static_cast<int>(blockIdx.x % split) : 0;  // rank in the cluster
  int64_t u = blockIdx.x / split;
  int qti = static_cast<int>(u % tiles);
  u /= tiles;
  int i = static_cast<int>(u % a.P);
  const int64_t slice = u / a.P;
  // under the mask the heaviest query tiles come first within each slice
  if (a.causal) causal_order(a.layout, a.P, static_cast<int>(tiles), true, i, qti);
  const int64_t qt = qti;
  const int64_t sb = slice * a.N;
  const float* q = static_cast<const float*>(a.q) + sb * d;
  const float* k = static_cast<const float*>(a.k) + sb * d;
  const float* v = static_cast<const float*>(a.v) + sb * d;
  const float* g = static_cast<const float*>(a.dout) + sb * d;
  const int64_t r0 = qt * kTM;
  load_stationary<DT, kTT>(sm + S::kQ, q, a.layout, i, r0, a.P, c, d, tid);
  load_stationary<DT, kTT>(sm + S::kG, g, a.layout, i, r0, a.P, c, d, tid);

  const int h = warp / 4;                // half: streamed rows kTH h ..
  const int lrow0 = 16 * (warp % 4) + 4 * rg;
  const int ccol = kTH * h + kNY * kg;   // this lane's kNY streamed rows in a tile
  int64_t qpos[4];
  bool rvalid[4];
  float lse[4], D[4];
  float acc[4][DT / 32][4];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int64_t r = r0 + lrow0 + x;
    rvalid[x] = r < c;
    qpos[x] = rvalid[x] ? layout_pos(a.layout, i, r, a.P, c) : 0;
    lse[x] = rvalid[x] ? a.lse[sb + qpos[x]] : 0.f;
    D[x] = rvalid[x] ? a.delta[sb + static_cast<int64_t>(i) * c + r] : 0.f;
#pragma unroll
    for (int m = 0; m < DT / 32; ++m)
#pragma unroll
      for (int y = 0; y < 4; ++y) acc[x][m][y] = 0.f;
  }
  const int64_t rlast = (r0 + kTM < c ? r0 + kTM : c) - 1;
  const int64_t qlast = layout_pos(a.layout, i, rlast, a.P, c);

  // K/V tiles in ring order, the next one fetched into registers while the
  // current one is computed
  StreamWalk<true> w{a.P, i, a.layout, split, cr, a.causal != 0, c, qlast};
  w.settle();
  Streamed<DT, kTT> nk, nv;
  if (w.valid()) {
    nk.fetch(k, a.layout, w.block(), w.c0, a.P, c, d, tid);
    nv.fetch(v, a.layout, w.block(), w.c0, a.P, c, d, tid);
  }
  while (w.valid()) {
    {
      const int j = w.block();
      const int64_t c0 = w.c0;
      __syncthreads();  // the previous tile's K, V and dS are no longer read
      nk.store(sm + S::kK, sm + S::kKr, tid);
      nv.store(sm + S::kV, nullptr, tid);
      __syncthreads();
      w.advance();
      if (w.valid()) {
        nk.fetch(k, a.layout, w.block(), w.c0, a.P, c, d, tid);
        nv.fetch(v, a.layout, w.block(), w.c0, a.P, c, d, tid);
      }
      float s[4][kNY], dp[4][kNY];
      two_blocks(sm + S::kQ, sm + S::kK, sm + S::kG, sm + S::kV, d, kSS, kNS, lrow0, ccol, s, dp);
      float ds[4][kNY];
#pragma unroll
      for (int y = 0; y < kNY; ++y) {
        const int64_t kk = c0 + ccol + y;
        const bool kvalid = kk < c;
        const int64_t kpos = kvalid ? layout_pos(a.layout, j, kk, a.P, c) : 0;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const bool vis = kvalid && rvalid[x] && (!a.causal || kpos <= qpos[x]);
          const float p = vis ? expf(s[x][y] * a.tau - lse[x]) : 0.f;
          ds[x][y] = p * (dp[x][y] - D[x]);
        }
      }
#pragma unroll
      for (int y = 0; y < kNY; ++y)
        *reinterpret_cast<float4*>(sm + S::kDS + (ccol + y) * kSS + lrow0) =
            make_float4(ds[0][y], ds[1][y], ds[2][y], ds[3][y]);
      __syncwarp();  // the warp reads back only the rows it wrote
      accumulate_rows<DT, kTH>(sm + S::kDS, sm + S::kKr, lrow0, kg, kTH * h, acc);
    }
  }
  float* dq = static_cast<float*>(a.dq);
  static_assert(kTM * DT <= DqSmem<DT>::kBytes / 4, "the sums fit the tiles' space");
  // the second half's sums into the first's
  __syncthreads();  // every warp is done with the tiles
  if (WW::kHalves == 2) {
    if (h == 1) put_rows<DT>(sm, 0, acc, lrow0, kg);
    __syncthreads();
    if (h == 0) add_rows<DT>(sm, 0, acc, lrow0, kg);
  }
  if (split > 1) {
    if (h == 0) put_rows<DT>(sm, 0, acc, lrow0, kg);  // each thread over what it read
    __syncthreads();
    split_sums<DT, 1, kTT>(sm, split, cr, tid, d, [&](int rr, int e, const float* sums) {
      const int64_t r = r0 + rr;
      if (r >= c) return;
      const int64_t row = (sb + layout_pos(a.layout, i, r, a.P, c)) * d;
      dq[row + e] = (a.accumulate ? dq[row + e] : 0.f) + sums[0] * a.tau;
    });
    return;
  }
  if (h == 1) return;
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    if (!rvalid[x]) continue;
    const int64_t row = (sb + qpos[x]) * d;
#pragma unroll
    for (int m = 0; m < DT / 32; ++m)
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int e = 4 * kg + 32 * m + y;
        if (e < d) dq[row + e] = (a.accumulate ? dq[row + e] : 0.f) + acc[x][m][y] * a.tau;
      }
  }
}

// dK, dV for 64 key rows of block j: the query blocks (j + t) mod P.
template <int DT, int W>
__global__ void __launch_bounds__(32 * W, DT == 64 && W == 8 ? 2 : 1)
    dkv_f32_tiled(const BackwardArgs a, int split) {
  using S = DkvSmem<DT>;
  using WW = Warps<W>;
  constexpr int kTT = WW::kThreads;
  constexpr int kTH = WW::kRows;
  constexpr int kNY = WW::kNY;
  extern __shared__ __align__(16) float sm[];
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int rg = lane / 8, kg = lane % 8;
  const int d = a.d;
  const int64_t c = a.N / a.P;
  const int64_t tiles = (c + kTM - 1) / kTM;
  const int cr = split > 1 ? static_cast<int>(blockIdx.x % split) : 0;  // rank in the cluster
  int64_t u = blockIdx.x / split;
  int kti = static_cast<int>(u % tiles);
  u /= tiles;
  int j = static_cast<int>(u % a.P);
  const int64_t slice = u / a.P;
  // under the mask the heaviest key tiles (the first rows) come first
  if (a.causal) causal_order(a.layout, a.P, static_cast<int>(tiles), false, j, kti);
  const int64_t kt = kti;
  const int64_t sb = slice * a.N;
  const float* q = static_cast<const float*>(a.q) + sb * d;
  const float* k = static_cast<const float*>(a.k) + sb * d;
  const float* v = static_cast<const float*>(a.v) + sb * d;
  const float* g = static_cast<const float*>(a.dout) + sb * d;
  const int64_t r0 = kt * kTM;
  load_stationary<DT, kTT>(sm + S::kK, k, a.layout, j, r0, a.P, c, d, tid);
  load_stationary<DT, kTT>(sm + S::kV, v, a.layout, j, r0, a.P, c, d, tid);

  const int h = warp / 4;                // half: streamed rows kTH h ..
  const int lrow0 = 16 * (warp % 4) + 4 * rg;
  const int ccol = kTH * h + kNY * kg;   // this lane's kNY streamed rows in a tile
  int64_t kpos[4];
  bool rvalid[4];
  float gk[4][DT / 32][4], gv[4][DT / 32][4];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int64_t r = r0 + lrow0 + x;
    rvalid[x] = r < c;
    kpos[x] = rvalid[x] ? layout_pos(a.layout, j, r, a.P, c) : 0;
#pragma unroll
    for (int m = 0; m < DT / 32; ++m)
#pragma unroll
      for (int y = 0; y < 4; ++y) gk[x][m][y] = gv[x][m][y] = 0.f;
  }
  const int64_t kfirst = layout_pos(a.layout, j, r0, a.P, c);  // the CTA's first key position

  // the query blocks (j + t) mod P this key block meets, tile by tile (under
  // the mask a query tile whose last query precedes every key here sees
  // none); the next Q/dO tile fetched into registers during the current one
  StreamWalk<false> w{a.P, j, a.layout, split, cr, a.causal != 0, c, kfirst};
  w.settle();
  Streamed<DT, kTT> nq, ng;
  if (w.valid()) {
    nq.fetch(q, a.layout, w.block(), w.c0, a.P, c, d, tid);
    ng.fetch(g, a.layout, w.block(), w.c0, a.P, c, d, tid);
  }
  while (w.valid()) {
    {
      const int i = w.block();  // the query block this key block meets
      const int64_t c0 = w.c0;
      __syncthreads();  // the previous tile's Q, dO, P and dS are no longer read
      nq.store(sm + S::kQ, sm + S::kQr, tid);
      ng.store(sm + S::kG, sm + S::kGr, tid);
      __syncthreads();
      w.advance();
      if (w.valid()) {
        nq.fetch(q, a.layout, w.block(), w.c0, a.P, c, d, tid);
        ng.fetch(g, a.layout, w.block(), w.c0, a.P, c, d, tid);
      }
      float s[4][kNY], dp[4][kNY];
      two_blocks(sm + S::kK, sm + S::kQ, sm + S::kV, sm + S::kG, d, kSS, kNS, lrow0, ccol, s, dp);
      float p[4][kNY], ds[4][kNY];
#pragma unroll
      for (int y = 0; y < kNY; ++y) {
        const int64_t qq = c0 + ccol + y;
        const bool qvalid = qq < c;
        const int64_t qpos = qvalid ? layout_pos(a.layout, i, qq, a.P, c) : 0;
        const float lse = qvalid ? a.lse[sb + qpos] : 0.f;
        const float D = qvalid ? a.delta[sb + static_cast<int64_t>(i) * c + qq] : 0.f;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const bool vis = qvalid && rvalid[x] && (!a.causal || qpos >= kpos[x]);
          p[x][y] = vis ? expf(s[x][y] * a.tau - lse) : 0.f;
          ds[x][y] = p[x][y] * (dp[x][y] - D);
        }
      }
#pragma unroll
      for (int y = 0; y < kNY; ++y) {
        *reinterpret_cast<float4*>(sm + S::kP + (ccol + y) * kSS + lrow0) =
            make_float4(p[0][y], p[1][y], p[2][y], p[3][y]);
        *reinterpret_cast<float4*>(sm + S::kDS + (ccol + y) * kSS + lrow0) =
            make_float4(ds[0][y], ds[1][y], ds[2][y], ds[3][y]);
      }
      __syncwarp();  // the warp reads back only the rows it wrote
      accumulate_rows<DT, kTH>(sm + S::kP, sm + S::kGr, lrow0, kg, kTH * h, gv);
      accumulate_rows<DT, kTH>(sm + S::kDS, sm + S::kQr, lrow0, kg, kTH * h, gk);
    }
  }
  float* dk = static_cast<float*>(a.dk);
  float* dv = static_cast<float*>(a.dv);
  static_assert(2 * kTM * DT <= DkvSmem<DT>::kBytes / 4, "the sums fit the tiles' space");
  // the second half's sums into the first's
  __syncthreads();  // every warp is done with the tiles
  if (WW::kHalves == 2) {
    if (h == 1) {
      put_rows<DT>(sm, 0, gk, lrow0, kg);
      put_rows<DT>(sm, 1, gv, lrow0, kg);
    }
    __syncthreads();
    if (h == 0) {
      add_rows<DT>(sm, 0, gk, lrow0, kg);
      add_rows<DT>(sm, 1, gv, lrow0, kg);
    }
  }
  if (split > 1) {
    if (h == 0) {  // each thread over what it read
      put_rows<DT>(sm, 0, gk, lrow0, kg);
      put_rows<DT>(sm, 1, gv, lrow0, kg);
    }
    __syncthreads();
    split_sums<DT, 2, kTT>(sm, split, cr, tid, d, [&](int rr, int e, const float* sums) {
      const int64_t r = r0 + rr;
      if (r >= c) return;
      const int64_t row = (sb + layout_pos(a.layout, j, r, a.P, c)) * d;
      dk[row + e] = (a.accumulate ? dk[row + e] : 0.f) + sums[0] * a.tau;
      dv[row + e] = (a.accumulate ? dv[row + e] : 0.f) + sums[1];
    });
    return;
  }
  if (h == 1) return;
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    if (!rvalid[x]) continue;
    const int64_t row = (sb + kpos[x]) * d;
#pragma unroll
    for (int m = 0; m < DT / 32; ++m)
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int e = 4 * kg + 32 * m + y;
        if (e < d) {
          dk[row + e] = (a.accumulate ? dk[row + e] : 0.f) + gk[x][m][y] * a.tau;
          dv[row + e] = (a.accumulate ? dv[row + e] : 0.f) + gv[x][m][y];
        }
      }
  }
}

// A tiled CTA takes a whole SM: when there are too few tiles of 64 rows for
// the SMs, each tile's walk is split over a cluster of 2, 4 or 8 CTAs, as
// long as every CTA keeps at least two streamed tiles.
int tiled_split(const BackwardArgs& a) {
  const int64_t ctas = a.slices * a.P * ((a.N / a.P + kTM - 1) / kTM);
  const int64_t walk = static_cast<int64_t>(a.P) * ((a.N / a.P + kTN - 1) / kTN);
  const int64_t sms = device_sm_count();
  int split = 1;
  while (split < 8 && ctas * split * 2 <= sms && walk >= 4 * split) split *= 2;
  return split;
}

template <int DT, int W>
cudaError_t launch_tiled_w(const BackwardArgs& a, cudaStream_t s) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(dq_f32_tiled<DT, W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DqSmem<DT>::kBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(dkv_f32_tiled<DT, W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               DkvSmem<DT>::kBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int split = tiled_split(a);
  const int64_t c = a.N / a.P;
  const unsigned grid = static_cast<unsigned>(a.slices * a.P * ((c + kTM - 1) / kTM) * split);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Warps<W>::kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(split);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = split > 1 ? 1 : 0;
  // the two kernels are independent: dK/dV on a forked side stream
  ForkJoin fj;
  e = fj.fork(s, dev);
  if (e != cudaSuccess) return e;
  cfg.dynamicSmemBytes = DqSmem<DT>::kBytes;
  e = cudaLaunchKernelEx(&cfg, dq_f32_tiled<DT, W>, a, split);
  if (e != cudaSuccess) return e;
  cfg.dynamicSmemBytes = DkvSmem<DT>::kBytes;
  cfg.stream = fj.side;
  e = cudaLaunchKernelEx(&cfg, dkv_f32_tiled<DT, W>, a, split);
  if (e != cudaSuccess) return e;
  return fj.join(s);
}

// Eight warps a CTA, with the next streamed tile prefetched (measured 14.7
// against 7.0 TFLOP/s for four warps without prefetch at d = 128, 17.3
// against 11.1 at d = 64; on one small d = 64 grid, H = 4, N = 1024, 8.4
// against 9.3).
template <int DT>
cudaError_t launch_tiled(const BackwardArgs& a, cudaStream_t s) {
  return launch_tiled_w<DT, 8>(a, s);
}
}  // namespace

cudaError_t launch_delta(const void* out, const void* dout, const float* lse, float* delta,
                         float* nl, int64_t rows, int32_t d, int64_t N, int32_t P,
                         int32_t layout, bool bf16, cudaStream_t s) {
  const int64_t need = (rows + 7) / 8;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
  const unsigned grid = static_cast<unsigned>(need < cap ? need : cap);
  if (bf16)
    delta_kernel<true><<<grid, 256, 0, s>>>(out, dout, lse, delta, nl, rows, d, N, P, layout);
  else
    delta_kernel<false><<<grid, 256, 0, s>>>(out, dout, lse, delta, nl, rows, d, N, P, layout);
  return cudaGetLastError();
}

cudaError_t launch_backward_f32(const BackwardArgs& a, cudaStream_t s) {
  const int64_t tiled_ctas = a.slices * a.P * ((a.N / a.P + kTM - 1) / kTM);
  if (a.d <= 128 && tiled_ctas * tiled_split(a) >= kTiledMinCtas) {
    if (a.d <= 64) return launch_tiled<64>(a, s);
    return launch_tiled<128>(a, s);
  }
  if (a.d <= 32) return launch_bwd_dv<1>(a, s);
  if (a.d <= 64) return launch_bwd_dv<2>(a, s);
  if (a.d <= 128) return launch_bwd_dv<4>(a, s);
  if (a.d <= 256) return launch_bwd_dv<8>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace ra
