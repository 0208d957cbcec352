// Merge of G partial online-softmax states ("Ring Attention", bembew.net,
// "Global Integration"; exact by the shift invariance of "Ring Attention: the
// math", section "The online-softmax identity that makes streaming legal"):
//   m* = max_g m_g,  w_g = exp(m_g - m*),  l* = sum w_g l_g,
//   o* = sum w_g o_g,  out = o* / l*,  lse = m* + ln l*.
// Rows whose partials are all empty (m = -inf) give out = 0, lse = -inf.
//
// HBM-bound: one warp per row, lanes read consecutive 16-byte pieces of each
// partial's o row (fully coalesced), weights are computed once per row by the
// lanes in parallel and broadcast with shuffles.  For the common counts of
// partials (1, 2, 3, 4, 6, 8) and d <= 128 the count is a template argument,
// so that all of a row's loads are issued together, before the weights are
// ready.  The grid is a multiple of the SM count and strides over the rows.
//
// Also: the state initialiser m = -inf, l = 0, o = 0.

#include <cuda_bf16.h>

#include <cmath>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kMergeWarps = 8;

__device__ __forceinline__ float4 ld_stream(const float* p) {
  float4 r;
  asm("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
      : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
      : "l"(p));
  return r;
}

// Lane g (and g + 32) gets partial g's weight w_g = exp(m_g - m*); returns
// (m*, 1 / l*) with 1 / l* = 0 for a row whose partials are all empty.
__device__ __forceinline__ void row_weights(const MergeArgs& a, int64_t r, int lane, float& w0,
                                            float& w1, float& ms, float& inv) {
  float mg0 = -INFINITY, mg1 = -INFINITY, lg0 = 0.f, lg1 = 0.f;
  if (lane < a.G) {
    mg0 = a.part.m[lane][r];
    lg0 = a.part.l[lane][r];
  }
  if (lane + 32 < a.G) {
    mg1 = a.part.m[lane + 32][r];
    lg1 = a.part.l[lane + 32][r];
  }
  ms = fmaxf(mg0, mg1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ms = fmaxf(ms, __shfl_xor_sync(0xffffffffu, ms, o));
  const bool empty = ms == -INFINITY;
  w0 = (empty || lane >= a.G) ? 0.f : expf(mg0 - ms);
  w1 = (empty || lane + 32 >= a.G) ? 0.f : expf(mg1 - ms);
  float ls = w0 * lg0 + w1 * lg1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
  inv = ls > 0.f ? 1.f / ls : 0.f;
  if (lane == 0) a.lse[r] = empty ? -INFINITY : ms + logf(ls);
}

template <bool kOutBf16>
__device__ __forceinline__ void store4(const MergeArgs& a, int64_t off, float4 acc, float inv) {
  if (kOutBf16) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t*>(&lo);
    w.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + off) = w;
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(a.out) + off) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
}

// kG > 0: exactly kG partials and d <= 128 with 16-byte rows.  Each lane
// issues its kG 16-byte loads of the row before the weights are known, so
// every load of the row is in flight at once; the FMAs follow.
template <bool kOutBf16, int kG>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_fixed_kernel(const MergeArgs a) {
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int d = a.d;
  const int c = lane * 4;
  const bool active = c < d;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kMergeWarps;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kMergeWarps + warp; r < a.rows;
       r += stride) {
    float4 x[kG];
#pragma unroll
    for (int g = 0; g < kG; ++g)
      x[g] = active ? ld_stream(a.part.o[g] + r * d + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    float w0, w1, ms, inv;
    row_weights(a, r, lane, w0, w1, ms, inv);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      const float w = __shfl_sync(0xffffffffu, g < 32 ? w0 : w1, g & 31);
      acc.x = fmaf(w, x[g].x, acc.x);
      acc.y = fmaf(w, x[g].y, acc.y);
      acc.z = fmaf(w, x[g].z, acc.z);
      acc.w = fmaf(w, x[g].w, acc.w);
    }
    if (active) store4<kOutBf16>(a, r * d + c, acc, inv);
  }
}

// Any G and d: one warp per row, lanes stride over the columns.
template <bool kOutBf16>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const MergeArgs a) {
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int d = a.d;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kMergeWarps;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kMergeWarps + warp; r < a.rows;
       r += stride) {
    float w0, w1, ms, inv;
    row_weights(a, r, lane, w0, w1, ms, inv);
    if (a.vec4) {
      // Uniform trip count on every lane keeps the shuffles converged.
      for (int c0 = 0; c0 < d; c0 += 128) {
        const int c = c0 + lane * 4;
        const bool active = c < d;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int gi = 0; gi < a.G; ++gi) {
          const float w = __shfl_sync(0xffffffffu, gi < 32 ? w0 : w1, gi & 31);
          if (active) {
            const float4 x = ld_stream(a.part.o[gi] + r * d + c);
            acc.x = fmaf(w, x.x, acc.x);
            acc.y = fmaf(w, x.y, acc.y);
            acc.z = fmaf(w, x.z, acc.z);
            acc.w = fmaf(w, x.w, acc.w);
          }
        }
        if (active) store4<kOutBf16>(a, r * d + c, acc, inv);
      }
    } else {
      // The lane loop runs the same number of times on every lane so that the
      // shuffles below stay converged.
      for (int c0 = 0; c0 < d; c0 += 32) {
        const int c = c0 + lane;
        float acc = 0.f;
        for (int gi = 0; gi < a.G; ++gi) {
          const float w = __shfl_sync(0xffffffffu, gi < 32 ? w0 : w1, gi & 31);
          if (c < d) acc = fmaf(w, a.part.o[gi][r * d + c], acc);
        }
        if (c < d) {
          if (kOutBf16)
            static_cast<__nv_bfloat16*>(a.out)[r * d + c] = __float2bfloat16_rn(acc * inv);
          else
            static_cast<float*>(a.out)[r * d + c] = acc * inv;
        }
      }
    }
  }
}

__global__ void state_init_kernel(float* m, float* l, float* o, int64_t rows, int32_t d) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t n = rows * d;
  for (int64_t x = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; x < n;
       x += stride) {
    o[x] = 0.f;
    if (x < rows) {
      m[x] = -INFINITY;
      l[x] = 0.f;
    }
  }
}

}  // namespace

template <bool kOutBf16>
cudaError_t launch_merge_t(const MergeArgs& a, unsigned grid, cudaStream_t s) {
  constexpr unsigned kT = kMergeWarps * 32;
  if (a.vec4 && a.d <= 128) {
    switch (a.G) {
      case 1: merge_fixed_kernel<kOutBf16, 1><<<grid, kT, 0, s>>>(a); return cudaGetLastError();
      case 2: merge_fixed_kernel<kOutBf16, 2><<<grid, kT, 0, s>>>(a); return cudaGetLastError();
      case 3: merge_fixed_kernel<kOutBf16, 3><<<grid, kT, 0, s>>>(a); return cudaGetLastError();
      case 4: merge_fixed_kernel<kOutBf16, 4><<<grid, kT, 0, s>>>(a); return cudaGetLastError();
      case 6: merge_fixed_kernel<kOutBf16, 6><<<grid, kT, 0, s>>>(a); return cudaGetLastError();
      case 8: merge_fixed_kernel<kOutBf16, 8><<<grid, kT, 0, s>>>(a); return cudaGetLastError();
      default: break;
    }
  }
  merge_kernel<kOutBf16><<<grid, kT, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t s) {
  const int64_t need = (a.rows + kMergeWarps - 1) / kMergeWarps;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  const unsigned grid = static_cast<unsigned>(need < cap ? need : cap);
  return a.out_bf16 ? launch_merge_t<true>(a, grid, s) : launch_merge_t<false>(a, grid, s);
}

cudaError_t launch_state_init(float* m, float* l, float* o, int64_t rows, int32_t d,
                              cudaStream_t s) {
  const int64_t n = rows * d;
  const int64_t need = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  const unsigned grid = static_cast<unsigned>(need < cap ? need : cap);
  state_init_kernel<<<grid, 256, 0, s>>>(m, l, o, rows, d);
  return cudaGetLastError();
}

}  // namespace ra
