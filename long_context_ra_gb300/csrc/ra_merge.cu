// Merge of G partial online-softmax states ("Ring Attention", bembew.net,
// "Global Integration"; exact by the shift invariance of "Ring Attention: the
// math", section "The online-softmax identity that makes streaming legal"):
//   m* = max_g m_g,  w_g = exp(m_g - m*),  l* = sum w_g l_g,
//   o* = sum w_g o_g,  out = o* / l*,  lse = m* + ln l*.
// Rows whose partials are all empty (m = -inf) give out = 0, lse = -inf.
//
// HBM-bound: one warp per row, lanes read consecutive 16-byte pieces of each
// partial's o row (fully coalesced), weights are computed once per row by the
// lanes in parallel and broadcast with shuffles.  The grid is a multiple of
// the SM count and strides over the rows.
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
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}

template <bool kOutBf16>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const MergeArgs a) {
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int d = a.d;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kMergeWarps;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kMergeWarps + warp; r < a.rows;
       r += stride) {
    // Lane g (and g + 32) holds partial g's max and sum.
    float mg0 = -INFINITY, mg1 = -INFINITY, lg0 = 0.f, lg1 = 0.f;
    if (lane < a.G) {
      mg0 = a.part.m[lane][r];
      lg0 = a.part.l[lane][r];
    }
    if (lane + 32 < a.G) {
      mg1 = a.part.m[lane + 32][r];
      lg1 = a.part.l[lane + 32][r];
    }
    float ms = fmaxf(mg0, mg1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ms = fmaxf(ms, __shfl_xor_sync(0xffffffffu, ms, o));
    const bool empty = ms == -INFINITY;
    const float w0 = (empty || lane >= a.G) ? 0.f : expf(mg0 - ms);
    const float w1 = (empty || lane + 32 >= a.G) ? 0.f : expf(mg1 - ms);
    float ls = w0 * lg0 + w1 * lg1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    const float inv = ls > 0.f ? 1.f / ls : 0.f;

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
        if (!active) continue;
        if (kOutBf16) {
          __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
          __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
          uint2 w;
          w.x = *reinterpret_cast<uint32_t*>(&lo);
          w.y = *reinterpret_cast<uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + r * d + c) = w;
        } else {
          *reinterpret_cast<float4*>(static_cast<float*>(a.out) + r * d + c) =
              make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
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
    if (lane == 0) a.lse[r] = empty ? -INFINITY : ms + logf(ls);
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

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t s) {
  const int64_t need = (a.rows + kMergeWarps - 1) / kMergeWarps;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  const unsigned grid = static_cast<unsigned>(need < cap ? need : cap);
  if (a.out_bf16)
    merge_kernel<true><<<grid, kMergeWarps * 32, 0, s>>>(a);
  else
    merge_kernel<false><<<grid, kMergeWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
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
