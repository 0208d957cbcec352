// fp32 fold kernel (FFMA only, no TF32): the exact-precision path for any
// head dimension 1 <= d <= 256 and any block size.
//
// One warp owns one query row ("Ring Attention: the math", section "Sharding
// the sequence": queries stay home) and walks the key blocks in ring order
// j = (i - t) mod P (section "The ring schedule: passing K/V around").  Each
// block is folded 32 keys at a time -- one key per lane -- with the update of
// section "The online-softmax identity that makes streaming legal":
//   s = tau q.k;  m' = max(m, max s);  alpha = exp(m - m');
//   l' = alpha l + sum exp(s - m');  o' = alpha o + sum exp(s - m') v.
// Folding a block in chunks is exact by the same identity.  The lanes split
// o: lane e holds o[e], o[e + 32], ...
//
// Causal ("Ring attention, explained", "The causal-mask catch"): a query at
// position n sees key positions <= n.  Under every layout the positions of a
// block increase along its local order, so the visible keys of a block are a
// prefix and the walk over it stops at the first chunk that starts after n.

#include <cmath>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kWarps = 4;

// Position of local row r of block j under `layout` (P blocks of c rows).
__device__ __forceinline__ int64_t pos_of(int layout, int64_t j, int64_t r, int64_t P,
                                          int64_t c) {
  if (layout == kZigzag) {
    const int64_t h = c / 2;
    return r < h ? j * h + r : (2 * P - 1 - j) * h + (r - h);
  }
  if (layout == kStriped) return j + P * r;
  return j * c + r;
}

// Block holding position n.
__device__ __forceinline__ int64_t block_of(int layout, int64_t n, int64_t P, int64_t c) {
  if (layout == kZigzag) {
    const int64_t chunk = n / (c / 2);
    return chunk < P ? chunk : 2 * P - 1 - chunk;
  }
  if (layout == kStriped) return n % P;
  return n / c;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// tau q.k for one key row: four independent FMA chains, 16-byte loads when
// every row starts on a 16-byte boundary (vec), a scalar tail otherwise.
__device__ __forceinline__ float dot_row(const float* __restrict__ qrow,
                                         const float* __restrict__ kr, int d, bool vec) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  int e = 0;
  if (vec) {
    const float4* k4 = reinterpret_cast<const float4*>(kr);
    const float4* q4 = reinterpret_cast<const float4*>(qrow);
    const int n4 = d / 4;
#pragma unroll 4
    for (int x = 0; x < n4; ++x) {
      const float4 kk = k4[x];
      const float4 qq = q4[x];
      a0 = fmaf(qq.x, kk.x, a0);
      a1 = fmaf(qq.y, kk.y, a1);
      a2 = fmaf(qq.z, kk.z, a2);
      a3 = fmaf(qq.w, kk.w, a3);
    }
    e = 4 * n4;
  }
  for (; e < d; ++e) a0 = fmaf(qrow[e], kr[e], a0);
  return (a0 + a1) + (a2 + a3);
}

template <int DV>  // o values per lane: d <= 32 * DV
__global__ void __launch_bounds__(kWarps * 32) fold_f32_kernel(const FoldArgs a) {
  __shared__ __align__(16) float qs[kWarps][32 * DV];
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int d = a.d;
  const int64_t rid = static_cast<int64_t>(blockIdx.x) * kWarps + warp;  // query row
  const int g = blockIdx.y;                                              // segment
  if (rid >= a.slices * a.nq) return;  // whole warp leaves together
  const int64_t slice = rid / a.nq;
  const int64_t n = rid % a.nq;
  const int64_t cq = a.nq / a.P;
  const int64_t ck = a.nk / a.P;
  const int i = static_cast<int>(block_of(a.layout, n, a.P, cq));
  const int t0 = static_cast<int>(static_cast<int64_t>(g) * a.P / a.G);
  const int t1 = static_cast<int>(static_cast<int64_t>(g + 1) * a.P / a.G);

  // rows of k start on 16-byte boundaries when d is a multiple of 4 and k
  // itself is 16-byte aligned
  const bool vec = (d % 4 == 0) && (reinterpret_cast<uintptr_t>(a.k) % 16 == 0);
  const float* q = static_cast<const float*>(a.q) + rid * d;
  for (int e = lane; e < d; e += 32) qs[warp][e] = q[e];
  __syncwarp();

  float m = -INFINITY, l = 0.f;
  float o[DV];
#pragma unroll
  for (int v = 0; v < DV; ++v) o[v] = 0.f;
  if (a.mode == kFold) {
    m = a.st_m[rid];
    l = a.st_l[rid];
#pragma unroll
    for (int v = 0; v < DV; ++v) {
      const int e = lane + 32 * v;
      if (e < d) o[v] = a.st_o[rid * d + e];
    }
  }

  for (int t = t0; t < t1; ++t) {
    int j = (i - t) % a.P;
    if (j < 0) j += a.P;
    const float* kbase = static_cast<const float*>(a.k) + slice * a.nk * d;
    const float* vbase = static_cast<const float*>(a.v) + slice * a.nk * d;
    for (int64_t c0 = 0; c0 < ck; c0 += 32) {
      if (a.causal && pos_of(a.layout, j, c0, a.P, ck) > n) break;  // rest of block masked
      const int64_t key = c0 + lane;
      const int64_t kpos = key < ck ? pos_of(a.layout, j, key, a.P, ck) : 0;
      const bool valid = key < ck && (!a.causal || kpos <= n);
      float s = -INFINITY;
      if (valid) s = dot_row(qs[warp], kbase + kpos * d, d, vec) * a.tau;
      const float m_new = fmaxf(m, warp_max(s));
      const float alpha = m_new == -INFINITY ? 1.f : expf(m - m_new);
      const float p = valid ? expf(s - m_new) : 0.f;
      l = alpha * l + warp_sum(p);
#pragma unroll
      for (int v = 0; v < DV; ++v) o[v] *= alpha;
      // o += p V over the chunk's keys.  The loop has a fixed trip count
      // (masked keys and keys past the block's end have p = 0; the latter
      // read the slice's first row), so the V loads of several keys are in
      // flight at once.  As on the tensor-core path, a masked key's v is
      // multiplied by 0 rather than skipped.
#pragma unroll 8
      for (int jj = 0; jj < 32; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
        const float* vr = vbase + __shfl_sync(0xffffffffu, kpos, jj) * d;
#pragma unroll
        for (int v = 0; v < DV; ++v) {
          const int e = lane + 32 * v;
          if (e < d) o[v] = fmaf(pj, vr[e], o[v]);
        }
      }
      m = m_new;
    }
  }

  if (a.mode == kForward) {
    float* out = static_cast<float*>(a.out) + rid * d;
    const float inv = 1.f / l;
#pragma unroll
    for (int v = 0; v < DV; ++v) {
      const int e = lane + 32 * v;
      if (e < d) out[e] = o[v] * inv;
    }
    if (lane == 0) a.lse[rid] = m + logf(l);
  } else {
    float* mo = a.mode == kPartial ? a.part.m[g] : a.st_m;
    float* lo = a.mode == kPartial ? a.part.l[g] : a.st_l;
    float* oo = a.mode == kPartial ? a.part.o[g] : a.st_o;
#pragma unroll
    for (int v = 0; v < DV; ++v) {
      const int e = lane + 32 * v;
      if (e < d) oo[rid * d + e] = o[v];
    }
    if (lane == 0) {
      mo[rid] = m;
      lo[rid] = l;
    }
  }
}

template <int DV>
cudaError_t launch_dv(const FoldArgs& a, cudaStream_t s) {
  const int64_t rows = a.slices * a.nq;
  const dim3 grid(static_cast<unsigned>((rows + kWarps - 1) / kWarps), static_cast<unsigned>(a.G));
  fold_f32_kernel<DV><<<grid, kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fold_f32(const FoldArgs& a, cudaStream_t s) {
  if (a.d <= 32) return launch_dv<1>(a, s);
  if (a.d <= 64) return launch_dv<2>(a, s);
  if (a.d <= 128) return launch_dv<4>(a, s);
  if (a.d <= 256) return launch_dv<8>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace ra
