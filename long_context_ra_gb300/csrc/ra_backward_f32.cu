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
//   dq: one warp per query row walks the key blocks in ring order
//       (i - t) mod P, as the forward does;
//   dkv: one warp per key row walks the query blocks its block visits on the
//       ring, (j + t) mod P, and accumulates dK and dV for its row.
// Lanes split the head dimension (lane e holds elements e, e + 32, ...).
// Causal ("Ring attention, explained", "The causal-mask catch"): a query at
// position n sees keys at positions <= n; `layout` says which positions form
// each block (contiguous, zigzag or striped), as in the forward.

#include <cuda_bf16.h>

#include <cmath>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kWarps = 4;

// Position of local row r of block j under `layout` (P blocks of c rows).
__device__ __forceinline__ int64_t bpos(int layout, int64_t j, int64_t r, int64_t P, int64_t c) {
  if (layout == kZigzag) {
    const int64_t h = c / 2;
    return r < h ? j * h + r : (2 * P - 1 - j) * h + (r - h);
  }
  if (layout == kStriped) return j + P * r;
  return j * c + r;
}

// Block holding position n.
__device__ __forceinline__ int64_t bblock(int layout, int64_t n, int64_t P, int64_t c) {
  if (layout == kZigzag) {
    const int64_t chunk = n / (c / 2);
    return chunk < P ? chunk : 2 * P - 1 - chunk;
  }
  if (layout == kStriped) return n % P;
  return n / c;
}

// Local row of position n inside its block.
__device__ __forceinline__ int64_t blocal(int layout, int64_t n, int64_t P, int64_t c) {
  if (layout == kZigzag) {
    const int64_t h = c / 2;
    return (n / h < P ? 0 : h) + n % h;
  }
  if (layout == kStriped) return n / P;
  return n % c;
}

// The per-query terms D and nl are stored block-major: (slice, block, local
// row), so that a query tile's 128 values are contiguous under every layout.
__device__ __forceinline__ int64_t bmajor(int layout, int64_t slice, int64_t N, int64_t n,
                                          int64_t P, int64_t c) {
  return slice * N + bblock(layout, n, P, c) * c + blocal(layout, n, P, c);
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

// Gradient of one query row (warp) over all key blocks in ring order.
template <int DV>
__global__ void __launch_bounds__(kWarps * 32) dq_f32_kernel(const BackwardArgs a) {
  __shared__ __align__(16) float qs[kWarps][32 * DV];
  __shared__ __align__(16) float gs[kWarps][32 * DV];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int d = a.d;
  const int64_t rid = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  if (rid >= a.slices * a.N) return;
  const int64_t slice = rid / a.N, n = rid % a.N;
  const int64_t c = a.N / a.P;
  const int i = static_cast<int>(bblock(a.layout, n, a.P, c));
  const float* q = static_cast<const float*>(a.q);
  const float* k = static_cast<const float*>(a.k);
  const float* v = static_cast<const float*>(a.v);
  const float* g = static_cast<const float*>(a.dout);
  for (int e = lane; e < d; e += 32) {
    qs[warp][e] = q[rid * d + e];
    gs[warp][e] = g[rid * d + e];
  }
  __syncwarp();
  const float lse = a.lse[rid], D = a.delta[bmajor(a.layout, slice, a.N, n, a.P, c)];
  const bool vec = rows_vec(a);
  float acc[DV];
#pragma unroll
  for (int x = 0; x < DV; ++x) acc[x] = 0.f;
  for (int t = 0; t < a.P; ++t) {
    int j = (i - t) % a.P;
    if (j < 0) j += a.P;
    const int64_t sb = slice * a.N;
    for (int64_t c0 = 0; c0 < c; c0 += 32) {
      if (a.causal && bpos(a.layout, j, c0, a.P, c) > n) break;  // rest of the block masked
      const int64_t key = c0 + lane;
      const int64_t kp = key < c ? bpos(a.layout, j, key, a.P, c) : 0;
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
  float* dq = static_cast<float*>(a.dq);
#pragma unroll
  for (int x = 0; x < DV; ++x) {
    const int e = lane + 32 * x;
    if (e < d) dq[rid * d + e] = (a.accumulate ? dq[rid * d + e] : 0.f) + acc[x] * a.tau;
  }
}

// Gradients of one key row (warp) over the query blocks its block visits.
template <int DV>
__global__ void __launch_bounds__(kWarps * 32) dkv_f32_kernel(const BackwardArgs a) {
  __shared__ __align__(16) float ks[kWarps][32 * DV];
  __shared__ __align__(16) float vs[kWarps][32 * DV];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int d = a.d;
  const int64_t rid = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  if (rid >= a.slices * a.N) return;
  const int64_t slice = rid / a.N, n = rid % a.N;
  const int64_t c = a.N / a.P;
  const int j = static_cast<int>(bblock(a.layout, n, a.P, c));
  const float* q = static_cast<const float*>(a.q);
  const float* k = static_cast<const float*>(a.k);
  const float* v = static_cast<const float*>(a.v);
  const float* g = static_cast<const float*>(a.dout);
  for (int e = lane; e < d; e += 32) {
    ks[warp][e] = k[rid * d + e];
    vs[warp][e] = v[rid * d + e];
  }
  __syncwarp();
  const bool vec = rows_vec(a);
  float gk[DV], gv[DV];
#pragma unroll
  for (int x = 0; x < DV; ++x) gk[x] = gv[x] = 0.f;
  for (int t = 0; t < a.P; ++t) {
    const int i = (j + t) % a.P;  // the device holding this block at step t
    const int64_t sb = slice * a.N;
    for (int64_t c0 = 0; c0 < c; c0 += 32) {
      const int64_t row = c0 + lane;
      const int64_t qp = row < c ? bpos(a.layout, i, row, a.P, c) : 0;
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

template <int DV>
cudaError_t launch_bwd_dv(const BackwardArgs& a, cudaStream_t s) {
  const int64_t rows = a.slices * a.N;
  const unsigned grid = static_cast<unsigned>((rows + kWarps - 1) / kWarps);
  dq_f32_kernel<DV><<<grid, kWarps * 32, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dkv_f32_kernel<DV><<<grid, kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
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
  if (a.d <= 32) return launch_bwd_dv<1>(a, s);
  if (a.d <= 64) return launch_bwd_dv<2>(a, s);
  if (a.d <= 128) return launch_bwd_dv<4>(a, s);
  if (a.d <= 256) return launch_bwd_dv<8>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace ra
