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

// Gradient of one query row (warp) over all key blocks in ring order.
template <int DV>
__global__ void __launch_bounds__(kWarps * 32) dq_f32_kernel(const BackwardArgs a) {
  __shared__ float qs[kWarps][32 * DV];
  __shared__ float gs[kWarps][32 * DV];
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
        const float* kr = k + (sb + kp) * d;
        const float* vr = v + (sb + kp) * d;
        float s = 0.f, dp = 0.f;
        for (int e = 0; e < d; ++e) {
          s = fmaf(qs[warp][e], kr[e], s);
          dp = fmaf(gs[warp][e], vr[e], dp);
        }
        const float p = expf(s * a.tau - lse);
        ds = p * (dp - D);
      }
      const int nk = c - c0 < 32 ? static_cast<int>(c - c0) : 32;
      for (int jj = 0; jj < nk; ++jj) {
        const float dsj = __shfl_sync(0xffffffffu, ds, jj);
        const int64_t kpj = __shfl_sync(0xffffffffu, kp, jj);
        if (dsj == 0.f) continue;
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
  __shared__ float ks[kWarps][32 * DV];
  __shared__ float vs[kWarps][32 * DV];
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
        const float* qr = q + (sb + qp) * d;
        const float* gr = g + (sb + qp) * d;
        float s = 0.f, dp = 0.f;
        for (int e = 0; e < d; ++e) {
          s = fmaf(qr[e], ks[warp][e], s);
          dp = fmaf(gr[e], vs[warp][e], dp);
        }
        p = expf(s * a.tau - a.lse[sb + qp]);
        ds = p * (dp - a.delta[sb + static_cast<int64_t>(i) * c + row]);
      }
      const int nq = c - c0 < 32 ? static_cast<int>(c - c0) : 32;
      for (int jj = 0; jj < nq; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
        const float dsj = __shfl_sync(0xffffffffu, ds, jj);
        const int64_t qpj = __shfl_sync(0xffffffffu, qp, jj);
        if (pj == 0.f && dsj == 0.f) continue;
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
