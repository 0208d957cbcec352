// fp32 fold kernel (FFMA only, no TF32): the exact-precision path for any
// head dimension 1 <= d <= 256 and any block size.
//
// One CTA (4 or 8 warps) owns 64 or 128 query rows of one query block i ("Ring
// Attention: the math", section "Sharding the sequence": queries stay home)
// and walks the key blocks in ring order j = (i - t) mod P (section "The ring
// schedule: passing K/V around").  Each block is folded 32 keys at a time
// with the update of section "The online-softmax identity that makes
// streaming legal":
//   s = tau q.k;  m' = max(m, max s);  alpha = exp(m - m');
//   l' = alpha l + sum exp(s - m');  o' = alpha o + sum exp(s - m') v.
// Folding a block in chunks is exact by the same identity.
//
// The query tile and each 32-key K/V tile are staged in shared memory and
// shared by the CTA's rows.  Warp w owns rows 16w .. 16w + 15; lane (rg, kg) =
// (lane / 8, lane % 8) computes the 4 x 4 block of scores of rows
// 16w + 4rg + 0..3 against keys 4kg + 0..3, and holds o of the same 4 rows
// in the columns 4kg + 32m + 0..3.  A row's max and sum are reduced over the
// 8 lanes of its group.  Q and K are stored transposed ([d][rows]) so that a
// lane reads 4 rows or 4 keys of one column as one 16-byte load.
//
// Causal ("Ring attention, explained", "The causal-mask catch"): a query at
// position n sees key positions <= n.  Under every layout the positions of a
// block increase along its local order, so the visible keys of a block are a
// prefix, and the walk over a block stops at the first tile that starts after
// the CTA's last query.

#include <cooperative_groups.h>

#include <cmath>

#include "ra_internal.h"
#include "ra_layout.cuh"

namespace ra {
namespace {

constexpr int kBN = 32;        // keys per K/V tile
constexpr int kKS = kBN + 4;   // row stride of the transposed K tile (floats)
// below this many CTAs of 64 rows (after the cluster split) the tiled
// kernel leaves most SMs idle, and the split-row kernel is faster
constexpr int64_t kSmallGrid = 128;

// Shared-memory footprint (floats) for head dimensions up to DT and BM
// query rows per CTA (2 BM threads: warp w owns rows 16w .. 16w + 15).
template <int DT, int BM>
struct Smem {
  static constexpr int kQS = BM + 4;              // row stride of Q^T and P^T
  static constexpr int kQ = 0;                    // Q^T  [DT][kQS]
  static constexpr int kK = kQ + DT * kQS;        // K^T  [DT][kKS]
  static constexpr int kV = kK + DT * kKS;        // V    [kBN][DT + 4]
  static constexpr int kP = kV + kBN * (DT + 4);  // P^T  [kBN][kQS]
  static constexpr int kFloats = kP + kBN * kQS;
  static constexpr int kBytes = kFloats * 4;
};

// The K/V tiles a CTA visits, in order: ring steps t = t0 .. t1 - 1 (block
// j = (i - t) mod P), each block's 32-key tiles in local order, under the
// causal mask only those starting at or before the CTA's last query.
struct TileCursor {
  int t, t1, i, j, P, layout;
  bool causal;
  int64_t c0, ck, qlast;
  __device__ void set_block() {
    j = (i - t) % P;
    if (j < 0) j += P;
  }
  __device__ bool valid() const { return t < t1; }
  // from (t, c0) forward to the first visible tile, or past the last step
  __device__ void settle() {
    while (t < t1) {
      if (c0 < ck && !(causal && layout_pos(layout, j, c0, P, ck) > qlast)) return;
      ++t;
      c0 = 0;
      if (t < t1) set_block();
    }
  }
  __device__ void advance() {
    c0 += kBN;
    settle();
  }
};

// max / sum over the 8 lanes of a row group (lanes 8g .. 8g + 7)
__device__ __forceinline__ float group_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
  return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
}
__device__ __forceinline__ float group_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x + __shfl_xor_sync(0xffffffffu, x, 4);
}

// split > 1: the CTAs of a cluster of `split` share one query tile, CTA r of
// the cluster folding the tiles r, r + split, ... of the tile's walk; their
// states are merged through distributed shared memory at the end.
template <int DT, int BM>  // d <= DT; DT in {64, 128, 256}; BM query rows per CTA (64, 128)
__global__ void __launch_bounds__(2 * BM) fold_f32_kernel(const FoldArgs a, int split) {
  constexpr int kBM = BM;
  constexpr int kThreads = 2 * BM;
  using S = Smem<DT, BM>;
  constexpr int kQS = S::kQS;
  constexpr int kCols = DT / 32;  // float4 column groups of o a lane holds
  extern __shared__ __align__(16) float sm[];
  float* qT = sm + S::kQ;
  float* kT = sm + S::kK;
  float* vs = sm + S::kV;
  float* pT = sm + S::kP;

  const int tid = threadIdx.x;
  const int warp = tid / 32, lane = tid % 32;
  const int rg = lane / 8, kg = lane % 8;
  const int d = a.d;
  const int64_t cq = a.nq / a.P;
  const int64_t ck = a.nk / a.P;
  const int64_t tiles_q = (cq + kBM - 1) / kBM;
  const int cr = split > 1 ? static_cast<int>(blockIdx.x % split) : 0;  // rank in the cluster
  int64_t u = blockIdx.x / split;
  int qti = static_cast<int>(u % tiles_q);
  u /= tiles_q;
  int i = static_cast<int>(u % a.P);
  const int64_t slice = u / a.P;
  // under the mask the heaviest query tiles come first within each slice
  if (a.causal) causal_order(a.layout, a.P, static_cast<int>(tiles_q), true, i, qti);
  const int64_t qt = qti;
  const int g = blockIdx.y;  // segment
  const int t0 = static_cast<int>(static_cast<int64_t>(g) * a.P / a.G);
  const int t1 = static_cast<int>(static_cast<int64_t>(g + 1) * a.P / a.G);
  const int64_t r0 = qt * kBM;  // first local query row of the CTA

  const float* q = static_cast<const float*>(a.q) + slice * a.nq * d;
  const float* kb = static_cast<const float*>(a.k) + slice * a.nk * d;
  const float* vb = static_cast<const float*>(a.v) + slice * a.nk * d;

  // Q^T tile: column e of row x at qT[e * kQS + x]; rows past the block and
  // columns past d are zero
  for (int x = tid; x < kBM * DT; x += kThreads) {
    const int row = x / DT, e = x % DT;
    const int64_t r = r0 + row;
    float val = 0.f;
    if (r < cq && e < d) val = q[layout_pos(a.layout, i, r, a.P, cq) * d + e];
    qT[e * kQS + row] = val;
  }

  // this lane's 4 rows: local rows, positions, state
  const int lrow0 = 16 * warp + 4 * rg;  // first of the 4 rows within the CTA
  int64_t qpos[4];
  bool rvalid[4];
  float m[4], l[4];
  float o[4][kCols][4];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int64_t r = r0 + lrow0 + x;
    rvalid[x] = r < cq;
    qpos[x] = rvalid[x] ? layout_pos(a.layout, i, r, a.P, cq) : 0;
    m[x] = -INFINITY;
    l[x] = 0.f;
#pragma unroll
    for (int c = 0; c < kCols; ++c)
#pragma unroll
      for (int y = 0; y < 4; ++y) o[x][c][y] = 0.f;
  }
  if (a.mode == kFold && cr == 0) {  // the incoming state joins the split once
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      if (!rvalid[x]) continue;
      const int64_t row = slice * a.nq + qpos[x];
      m[x] = a.st_m[row];
      l[x] = a.st_l[row];
#pragma unroll
      for (int c = 0; c < kCols; ++c)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int e = 4 * kg + 32 * c + y;
          if (e < d) o[x][c][y] = a.st_o[row * d + e];
        }
    }
  }
  // the CTA's last query position (positions grow along a block's rows)
  const int64_t rlast = (r0 + kBM < cq ? r0 + kBM : cq) - 1;
  const int64_t qlast = layout_pos(a.layout, i, rlast, a.P, cq);

  // K^T and V tiles; keys past the block and columns past d are zero.  In
  // the 128-wide class the next tile's values are fetched into registers
  // while the current tile is computed (kPre of K and of V a thread); at
  // DT = 64 the registers would cost a resident CTA per SM (measured slower),
  // and at DT = 256 there are none to spare.
  constexpr bool kPrefetch = DT == 128;
  constexpr int kPre = kPrefetch ? kBN * DT / kThreads : 1;
  float kr[kPre], vr[kPre];
  TileCursor cur{t0, t1, i, 0, a.P, a.layout, a.causal != 0, 0, ck, qlast};
  if (cur.valid()) cur.set_block();
  cur.settle();
  // this CTA's tiles: every split-th visible tile of the walk, from the cr-th
  int tix = 0;
  auto skip_others = [&]() {
    while (cur.valid() && tix % split != cr) {
      cur.advance();
      ++tix;
    }
  };
  auto advance_mine = [&]() {
    cur.advance();
    ++tix;
    skip_others();
  };
  skip_others();
  auto fetch = [&](const TileCursor& tc) {
#pragma unroll
    for (int it = 0; it < kPre; ++it) {
      const int x = tid + it * kThreads;
      const int key = x / DT, e = x % DT;
      const int64_t kk = tc.c0 + key;
      kr[it] = vr[it] = 0.f;
      if (kk < ck && e < d) {
        const int64_t row = layout_pos(a.layout, tc.j, kk, a.P, ck);
        kr[it] = kb[row * d + e];
        vr[it] = vb[row * d + e];
      }
    }
  };
  if (kPrefetch && cur.valid()) fetch(cur);
  while (cur.valid()) {
    const int j = cur.j;
    const int64_t c0 = cur.c0;
    __syncthreads();  // the previous tile's K, V and P are no longer read
    if (kPrefetch) {
#pragma unroll
      for (int it = 0; it < kPre; ++it) {
        const int x = tid + it * kThreads;
        const int key = x / DT, e = x % DT;
        kT[e * kKS + key] = kr[it];
        vs[key * (DT + 4) + e] = vr[it];
      }
    } else {
      for (int x = tid; x < kBN * DT; x += kThreads) {
        const int key = x / DT, e = x % DT;
        const int64_t kk = c0 + key;
        float kv = 0.f, vv = 0.f;
        if (kk < ck && e < d) {
          const int64_t row = layout_pos(a.layout, j, kk, a.P, ck);
          kv = kb[row * d + e];
          vv = vb[row * d + e];
        }
        kT[e * kKS + key] = kv;
        vs[key * (DT + 4) + e] = vv;
      }
    }
    __syncthreads();
    advance_mine();
    if (kPrefetch && cur.valid()) fetch(cur);  // in flight during this tile's math
    {

      // scores of the lane's 4 rows x 4 keys
      float s[4][4];
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) s[x][y] = 0.f;
#pragma unroll 16
      for (int e = 0; e < d; ++e) {
        const float4 qa = *reinterpret_cast<const float4*>(qT + e * kQS + lrow0);
        const float4 ka = *reinterpret_cast<const float4*>(kT + e * kKS + 4 * kg);
        const float qv[4] = {qa.x, qa.y, qa.z, qa.w};
        const float kv[4] = {ka.x, ka.y, ka.z, ka.w};
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
          for (int y = 0; y < 4; ++y) s[x][y] = fmaf(qv[x], kv[y], s[x][y]);
      }
      // masks: keys past the block, and (causal) keys after the query
      bool kvalid[4];
      int64_t kpos[4];
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int64_t kk = c0 + 4 * kg + y;
        kvalid[y] = kk < ck;
        kpos[y] = kvalid[y] ? layout_pos(a.layout, j, kk, a.P, ck) : 0;
      }
      float p[4][4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        float mx = -INFINITY;
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const bool vis = kvalid[y] && (!a.causal || kpos[y] <= qpos[x]);
          s[x][y] = vis ? s[x][y] * a.tau : -INFINITY;
          mx = fmaxf(mx, s[x][y]);
        }
        const float m_new = fmaxf(m[x], group_max(mx));
        const float alpha = m_new == -INFINITY ? 1.f : expf(m[x] - m_new);
        float sum = 0.f;
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          p[x][y] = s[x][y] == -INFINITY ? 0.f : expf(s[x][y] - m_new);
          sum += p[x][y];
        }
        l[x] = alpha * l[x] + group_sum(sum);
        m[x] = m_new;
#pragma unroll
        for (int c = 0; c < kCols; ++c)
#pragma unroll
          for (int y = 0; y < 4; ++y) o[x][c][y] *= alpha;
      }
      // P^T of the warp's rows, then o += p V over the tile's keys
#pragma unroll
      for (int y = 0; y < 4; ++y)
        *reinterpret_cast<float4*>(pT + (4 * kg + y) * kQS + lrow0) =
            make_float4(p[0][y], p[1][y], p[2][y], p[3][y]);
      __syncwarp();
#pragma unroll 16
      for (int key = 0; key < kBN; ++key) {
        const float4 pp = *reinterpret_cast<const float4*>(pT + key * kQS + lrow0);
        const float pv[4] = {pp.x, pp.y, pp.z, pp.w};
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          const float4 vv = *reinterpret_cast<const float4*>(vs + key * (DT + 4) + 4 * kg + 32 * c);
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            o[x][c][0] = fmaf(pv[x], vv.x, o[x][c][0]);
            o[x][c][1] = fmaf(pv[x], vv.y, o[x][c][1]);
            o[x][c][2] = fmaf(pv[x], vv.z, o[x][c][2]);
            o[x][c][3] = fmaf(pv[x], vv.w, o[x][c][3]);
          }
        }
      }
    }
  }

  float* mo = a.mode == kPartial ? a.part.m[g] : a.st_m;
  float* lo = a.mode == kPartial ? a.part.l[g] : a.st_l;
  float* oo = a.mode == kPartial ? a.part.o[g] : a.st_o;
  if (split > 1) {
    // Each CTA's state of the tile's kBM rows ([row][m, l, o]) into its shared
    // memory; CTA r then merges rows r kBM / split .. of every CTA's state
    // (the identity that merges partial states) and writes them.
    constexpr int kRS = DT + 2;
    static_assert(kBM * kRS <= S::kFloats, "merge rows fit the tiles' space");
    __syncthreads();  // every warp is done with the tiles
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      float* st = sm + (lrow0 + x) * kRS;
      if (kg == 0) {
        st[0] = m[x];
        st[1] = l[x];
      }
#pragma unroll
      for (int c = 0; c < kCols; ++c)
#pragma unroll
        for (int y = 0; y < 4; ++y) st[2 + 4 * kg + 32 * c + y] = o[x][c][y];
    }
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int rows_per = kBM / split;
    for (int idx = tid; idx < rows_per * (d + 1); idx += kThreads) {
      const int rr = cr * rows_per + idx / (d + 1);  // row of the tile
      const int e = idx % (d + 1) - 1;              // column, or -1: the row's m and l
      const int64_t r = r0 + rr;
      if (r >= cq) continue;
      float M = -INFINITY;
      for (int p = 0; p < split; ++p) M = fmaxf(M, cluster.map_shared_rank(sm, p)[rr * kRS]);
      float ls = 0.f, os = 0.f;
      for (int p = 0; p < split; ++p) {
        const float* st = cluster.map_shared_rank(sm, p) + rr * kRS;
        // an empty part (m = -inf) adds nothing, also when every part is empty
        const float w = st[0] == -INFINITY ? 0.f : expf(st[0] - M);
        ls = fmaf(w, st[1], ls);
        if (e >= 0) os = fmaf(w, st[2 + e], os);
      }
      const int64_t row = slice * a.nq + layout_pos(a.layout, i, r, a.P, cq);
      if (a.mode == kForward) {
        if (e >= 0)
          static_cast<float*>(a.out)[row * d + e] = os / ls;
        else
          a.lse[row] = M + logf(ls);
      } else if (e >= 0) {
        oo[row * d + e] = os;
      } else {
        mo[row] = M;
        lo[row] = ls;
      }
    }
    cluster.sync();  // every CTA's shared memory stays until all have read it
    return;
  }

  // write the rows: out = o / l and lse, or the state (m, l, o)
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    if (!rvalid[x]) continue;
    const int64_t row = slice * a.nq + qpos[x];
    if (a.mode == kForward) {
      float* out = static_cast<float*>(a.out) + row * d;
      const float inv = 1.f / l[x];
#pragma unroll
      for (int c = 0; c < kCols; ++c)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int e = 4 * kg + 32 * c + y;
          if (e < d) out[e] = o[x][c][y] * inv;
        }
      if (kg == 0) a.lse[row] = m[x] + logf(l[x]);
    } else {
#pragma unroll
      for (int c = 0; c < kCols; ++c)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int e = 4 * kg + 32 * c + y;
          if (e < d) oo[row * d + e] = o[x][c][y];
        }
      if (kg == 0) {
        mo[row] = m[x];
        lo[row] = l[x];
      }
    }
  }
}

// CTAs of the tiled kernel before the split: one per query tile of bm rows
int64_t tiled_units(const FoldArgs& a, int bm) {
  return a.slices * a.P * ((a.nq / a.P + bm - 1) / bm);
}

// CTAs of one tiled kernel resident on an SM, by registers and shared memory
int tiled_resident(int dt, int bm) {
  if (bm == 64) return dt == 256 ? 1 : 2;
  return dt == 64 ? 2 : 1;
}

// Too few CTAs for the SMs: each query tile's walk is split over a cluster
// of up to 8 CTAs, as long as every CTA keeps at least two K/V tiles.
int tiled_split(const FoldArgs& a, int dt, int bm) {
  const int64_t resident = static_cast<int64_t>(device_sm_count()) * tiled_resident(dt, bm);
  const int64_t tiles_kv = (a.P / a.G) * ((a.nk / a.P + kBN - 1) / kBN);  // per unit, at least
  const int64_t ctas = tiled_units(a, bm) * a.G;
  int split = 1;
  while (split < 8 && ctas * split * 2 <= resident && tiles_kv >= 4 * split) split *= 2;
  return split;
}

// 128-row tiles (8 warps) share the K/V staging between twice the rows:
// measured 10-14 % faster than 64-row tiles at d = 64 and 128 and 2x at 256
// on grids that fill the SMs, and faster on small grids too at d = 64, where
// two of them fit an SM (split over clusters like the 64-row ones).  At
// d = 128 and 256 one fits an SM, and on small grids 64-row tiles split
// over clusters measured faster (14.4 against 7.9 TFLOP/s at H = 1,
// N = 2048, P = 8).
int tiled_rows(const FoldArgs& a, int dt) {
  if (a.nq / a.P < 128) return 64;
  return dt == 64 || tiled_units(a, 128) * a.G >= device_sm_count() ? 128 : 64;
}

template <int DT, int BM>
cudaError_t launch_tiled(const FoldArgs& a, cudaStream_t s) {
  using S = Smem<DT, BM>;
  constexpr int kThreads = 2 * BM;
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(fold_f32_kernel<DT, BM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             S::kBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int64_t units = tiled_units(a, BM);
  const int split = tiled_split(a, DT, BM);
  if (split == 1) {
    const dim3 grid(static_cast<unsigned>(units), static_cast<unsigned>(a.G));
    fold_f32_kernel<DT, BM><<<grid, kThreads, S::kBytes, s>>>(a, 1);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units * split), static_cast<unsigned>(a.G));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = S::kBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(split);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fold_f32_kernel<DT, BM>, a, split);
}

template <int DT>
cudaError_t launch_dt(const FoldArgs& a, cudaStream_t s) {
  return tiled_rows(a, DT) == 128 ? launch_tiled<DT, 128>(a, s) : launch_tiled<DT, 64>(a, s);
}

// ---- small problems: a few warps per query row ----
// When the tiled kernel would launch only a few CTAs (a few hundred query
// rows), warps take rows instead, and each row's chunks of 32 keys (ring
// order: block j = (i - t) mod P, local order within it) are dealt round
// robin to S warps, so that the serial chain of a row is S times shorter.
// Each warp folds its chunks one key per lane (the lanes split o: lane e
// holds o[e], o[e + 32], ...) into its own (m, l, o); the S states of a row
// are then combined by the identity that merges partial states
//   m* = max m_s,  w_s = exp(m_s - m*),  l* = sum w_s l_s,  o* = sum w_s o_s
// (the same identity that lets the fold visit the keys in any order).

// A CTA holds the S warps of each of its rows: max(4, S) warps, so that
// small grids still come in fine pieces.  The split kernels get 128
// registers a thread (16 warps an SM), the unsplit one 64.
template <int S>
struct RowCta {
  static constexpr int kWarps = S < 4 ? 4 : S;
  static constexpr int kRows = kWarps / S;
  static constexpr int kMinBlocks = S == 1 ? 8 : 16 / kWarps;
};
constexpr int kResidentWarps = 16;  // per SM, at 128 registers a thread

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

// DV: o values per lane (d <= 32 DV); S: warps per row (1, 2, 4 or 8).
template <int DV, int S>
__global__ void __launch_bounds__(RowCta<S>::kWarps * 32, RowCta<S>::kMinBlocks)
    fold_f32_rows_kernel(const FoldArgs a) {
  constexpr int kWarps = RowCta<S>::kWarps;
  constexpr int kRows = RowCta<S>::kRows;  // query rows per CTA
  __shared__ __align__(16) float qs[kWarps][32 * DV];
  __shared__ float part_o[S > 1 ? kWarps : 1][32 * DV];
  __shared__ float part_ml[S > 1 ? kWarps : 1][2];
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int sp = warp % S;  // this warp's share of the row's chunks
  const int d = a.d;
  const int64_t rid = static_cast<int64_t>(blockIdx.x) * kRows + warp / S;  // query row
  const int g = blockIdx.y;                                                 // segment
  // a CTA's rows past the end do nothing, but still meet the merge's barrier
  const bool live = rid < a.slices * a.nq;
  const int64_t slice = live ? rid / a.nq : 0;
  const int64_t n = live ? rid % a.nq : 0;
  const int64_t cq = a.nq / a.P;
  const int64_t ck = a.nk / a.P;
  const int i = static_cast<int>(layout_block(a.layout, n, a.P, cq));
  const int t0 = static_cast<int>(static_cast<int64_t>(g) * a.P / a.G);
  const int t1 = static_cast<int>(static_cast<int64_t>(g + 1) * a.P / a.G);
  const int64_t nch = (ck + 31) / 32;  // chunks per block

  // rows of k start on 16-byte boundaries when d is a multiple of 4 and k
  // itself is 16-byte aligned
  const bool vec = (d % 4 == 0) && (reinterpret_cast<uintptr_t>(a.k) % 16 == 0);
  float m = -INFINITY, l = 0.f;
  float o[DV];
#pragma unroll
  for (int v = 0; v < DV; ++v) o[v] = 0.f;

  if (live) {
    const float* q = static_cast<const float*>(a.q) + rid * d;
    for (int e = lane; e < d; e += 32) qs[warp][e] = q[e];
    __syncwarp();
    if (a.mode == kFold && sp == 0) {  // the incoming state joins as one more part
      m = a.st_m[rid];
      l = a.st_l[rid];
#pragma unroll
      for (int v = 0; v < DV; ++v) {
        const int e = lane + 32 * v;
        if (e < d) o[v] = a.st_o[rid * d + e];
      }
    }
    const float* kbase = static_cast<const float*>(a.k) + slice * a.nk * d;
    const float* vbase = static_cast<const float*>(a.v) + slice * a.nk * d;
    for (int t = t0; t < t1; ++t) {
      int j = (i - t) % a.P;
      if (j < 0) j += a.P;
      // chunk ci of this block is the row's chunk (t - t0) nch + ci
      int64_t ci = (sp - (static_cast<int64_t>(t - t0) * nch) % S + S) % S;
      for (; ci < nch; ci += S) {
        const int64_t c0 = ci * 32;
        if (a.causal && layout_pos(a.layout, j, c0, a.P, ck) > n) break;  // rest of block masked
        const int64_t key = c0 + lane;
        const int64_t kpos = key < ck ? layout_pos(a.layout, j, key, a.P, ck) : 0;
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
        // read the slice's first row), so the V loads of several keys are
        // in flight at once.  As on the tensor-core path, a masked key's v
        // is multiplied by 0 rather than skipped.
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
  }

  if (S > 1) {
    // every part of the row into shared memory; the row's first warp merges
#pragma unroll
    for (int v = 0; v < DV; ++v) part_o[warp][lane + 32 * v] = o[v];
    if (lane == 0) {
      part_ml[warp][0] = m;
      part_ml[warp][1] = l;
    }
    __syncthreads();
    if (sp != 0 || !live) return;
    float mx = -INFINITY;
#pragma unroll
    for (int x = 0; x < S; ++x) mx = fmaxf(mx, part_ml[warp + x][0]);
    l = 0.f;
#pragma unroll
    for (int v = 0; v < DV; ++v) o[v] = 0.f;
#pragma unroll
    for (int x = 0; x < S; ++x) {
      const float mp = part_ml[warp + x][0];
      // an empty part (m = -inf) adds nothing, also when every part is empty
      const float w = mp == -INFINITY ? 0.f : expf(mp - mx);
      l = fmaf(w, part_ml[warp + x][1], l);
#pragma unroll
      for (int v = 0; v < DV; ++v) o[v] = fmaf(w, part_o[warp + x][lane + 32 * v], o[v]);
    }
    m = mx;
  } else if (!live) {
    return;
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

// Warps per row: at most 8, at most one per chunk of the row's segment, and
// only as many as stay resident at once.
int row_split(const FoldArgs& a) {
  const int64_t rows = a.slices * a.nq * a.G;
  const int64_t chunks = (a.P / a.G) * ((a.nk / a.P + 31) / 32);  // per row and segment, at least
  const int64_t want = static_cast<int64_t>(device_sm_count()) * kResidentWarps;
  int S = 1;
  while (S < 8 && rows * S * 2 <= want && chunks >= S * 2) S *= 2;
  return S;
}

template <int DV, int S>
cudaError_t launch_rows(const FoldArgs& a, cudaStream_t s) {
  const int64_t rows = a.slices * a.nq;
  constexpr int kRows = RowCta<S>::kRows;
  const dim3 grid(static_cast<unsigned>((rows + kRows - 1) / kRows), static_cast<unsigned>(a.G));
  fold_f32_rows_kernel<DV, S><<<grid, RowCta<S>::kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

template <int DV>
cudaError_t launch_dv(const FoldArgs& a, cudaStream_t s) {
  switch (row_split(a)) {
    case 8:
      return launch_rows<DV, 8>(a, s);
    case 4:
      return launch_rows<DV, 4>(a, s);
    case 2:
      return launch_rows<DV, 2>(a, s);
    default:
      return launch_rows<DV, 1>(a, s);
  }
}

}  // namespace

cudaError_t launch_fold_f32(const FoldArgs& a, cudaStream_t s) {
  if (a.slices * a.nq == 0) return cudaSuccess;
  const int dt = a.d <= 64 ? 64 : (a.d <= 128 ? 128 : 256);
  if (tiled_units(a, 64) * a.G * tiled_split(a, dt, 64) < kSmallGrid) {
    if (a.d <= 32) return launch_dv<1>(a, s);
    if (a.d <= 64) return launch_dv<2>(a, s);
    if (a.d <= 128) return launch_dv<4>(a, s);
    if (a.d <= 256) return launch_dv<8>(a, s);
    return cudaErrorInvalidValue;
  }
  if (a.d <= 64) return launch_dt<64>(a, s);
  if (a.d <= 128) return launch_dt<128>(a, s);
  if (a.d <= 256) return launch_dt<256>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace ra
