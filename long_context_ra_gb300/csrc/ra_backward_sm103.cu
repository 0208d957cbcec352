// Tensor-core backward kernels for bf16 inputs on sm_103a (GB300).
//
// The backward of ring attention runs on the same ring as the forward
// ("Ring attention, explained", step 6): the key-value blocks travel with
// their gradient accumulators.  For the loss L = sum(dO * out):
//   P = exp(tau Q K^T - lse)   (recomputed from the forward's lse)
//   dP = dO V^T;  dS = P * (dP - D),  D = rowsum(dO * out)
//   dV = P^T dO;  dK = tau dS^T Q;  dQ = tau dS K
// Two kernels, no atomics.  In both, the elementwise work runs in two
// passes: pass A makes p (needs S), pass B makes dS from the bf16 p (needs
// dP), and each overlaps a product on the tensor cores.
//   dkv_kernel  one 128-key tile of block j per CTA; at ring step t the block
//               is on device i = (j + t) mod P, so the CTA walks the query
//               tiles of those blocks.  TMEM: S^T [0,128), dP^T [128,256),
//               dV [256, 256+D), dK [256+D, 256+2D).  Pipe order per query
//               tile: dP^T = V dO^T (pass A runs meanwhile), dV += P^T dO
//               over pass A's parts (pass B runs meanwhile), dK += dS^T Q
//               over pass B's parts, then the next S^T = K Q^T.  P^T and
//               dS^T are bf16, the 16 values of each k-step packed over the
//               first 8 of their own 16 columns of S^T and dP^T (the A
//               operands of the dV and dK products).
//   dq_kernel   one 128-query tile per CTA walking the key tiles in the
//               forward's ring order (i - t) mod P.  TMEM: S in two buffers
//               [0,128) and [128,256), dP [256,384), dQ [384, 384+D).  S is
//               computed a tile ahead; pipe order per key tile: dQ += dS K
//               over pass B's parts, the next dP = dO V^T, then S = Q K^T two
//               tiles ahead.  K and V stream through separate rings.
// The row terms come precomputed per query row: D and nl = -lse * log2(e)
// (so that p = exp2(s * tau * log2(e) + nl)).
//
// Warp roles (G elementwise warpgroups; 128 G + 64 threads): warps 0 .. 4G-1
// elementwise (thread = tile row = TMEM lane), warp 4G TMA producer, warp
// 4G+1 TMEM allocator and MMA issuer.  G = 4 for the plain kernels and 2
// for the causal ones, each the faster of the two as measured (the causal
// kernels fit four warpgroups at 82-92 registers, but ran 6 % slower with
// them).  Every wait is bounded (see sm103_pipeline.cuh).

#include <cmath>

#include "ra_fork.h"
#include "ra_internal.h"
#include "ra_layout.cuh"
#include "sm103_pipeline.cuh"
#include "sm103_ptx.cuh"

namespace ra {
namespace {

using namespace ptx;
using namespace sm103;

template <int G>
struct Roles {
  static constexpr int kThreads = 128 * G + 64;
  static constexpr int kLoadWarp = 4 * G;
  static constexpr int kMmaWarp = 4 * G + 1;
  static constexpr int kParts = 2;               // parts of a tile's 128 columns
  static constexpr int kStepsPerPart = 8 / kParts;
  static constexpr int kStepsPerGroup = kStepsPerPart / G;  // k-steps of one warpgroup per part
  static constexpr int kPartThreads = 128 * G;  // arrivals per part: every warpgroup
};
template <bool kCausal>
constexpr int groups_for() { return kCausal ? 2 : 4; }

constexpr uint32_t kTmemCols = 512;
constexpr int kStages = 2;
// Each elementwise pass over a tile's 128 columns is done in two parts of 64
// columns, which are k-steps [4h, 4h + 4) of the TMEM-operand products;
// warpgroup g takes the k-steps 4h + g + G m, so every warpgroup works on
// every part.  The products that read part h start as soon as part h is
// done.  (Two parts measured faster than one, or than one per k-step pair.)
constexpr int kMaxParts = 4;

// 8 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::
                   "r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
               "r"(r[7])
               : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

template <int D>
struct Tiles {
  static constexpr int kBoxBytes = kBM * 128;  // 128 rows x 64 bf16
  static constexpr int kTileBytes = kBM * D * 2;
  static constexpr int kRowBytes = kBM * 4;  // one fp32 value per tile row
};

// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// D[tmem] = A B^T over d: 128 x 128 x D, both operands K-major in SMEM.
template <int D>
__device__ __forceinline__ void mma_nt(uint32_t d_tmem, uint64_t da, uint64_t db) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = desc_step((kk / 4) * Tiles<D>::kBoxBytes + (kk % 4) * 32);
    mma_bf16_ss(d_tmem, da + off, db + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// D[tmem] (+)= A[tmem] B over rows [16 k0, 16 k1) of B: A is 128 x 128 bf16
// in TMEM, the 16 values of k-step kk packed into the 8 columns at 16 kk; B
// an MN-major 128 x D tile in SMEM.  `accumulate` applies to the first
// product only.
template <int D, int k0, int k1>
__device__ __forceinline__ void mma_tn(uint32_t d_tmem, uint32_t a_tmem, uint64_t db,
                                       uint32_t accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, D, true);
#pragma unroll
  for (int kk = k0; kk < k1; ++kk)
    mma_bf16_ts(d_tmem, a_tmem + kk * 16, db + desc_step(kk * 16 * 128), idesc,
                kk == k0 ? accumulate : 1u);
}

// 8 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}

// The elementwise work of the dK/dV kernel in two passes, so that each
// overlaps a product on the tensor cores.  Pass A (needs only S^T) makes
//   p = exp2(s * sl2 + nl)        (nl per column, from SMEM)
// for the 16 columns [c, c + 16), masked to 0 outside [lo, hi), and stores p
// as bf16 pairs over the first 8 of these columns of tS (read by the dV
// product and by pass B).
// In the dQ kernel the row term is one scalar per thread (kPerColumn false:
// nl_row, and the mask keeps the columns below hi).
template <bool kPerColumn, bool kMask>
__device__ __forceinline__ void pass_p(int c, uint32_t tS, float sl2, const float* nl,
                                       float nl_row, int lo, int hi, uint32_t (&pk)[8]) {
  uint32_t s[16];
  tmem_ld16(tS + c, s);
  float ncol[16];
#pragma unroll
  for (int e = 0; e < 16; e += 4) {
    if (kPerColumn) {
      const float4 x = *reinterpret_cast<const float4*>(nl + c + e);
      ncol[e] = x.x, ncol[e + 1] = x.y, ncol[e + 2] = x.z, ncol[e + 3] = x.w;
    } else {
      ncol[e] = ncol[e + 1] = ncol[e + 2] = ncol[e + 3] = nl_row;
    }
  }
  tmem_ld_wait();
  reg_fence(s, 16);
  if (kMask) {
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if (c + e < lo || c + e >= hi) s[e] = 0xff800000u;  // -inf
  }
  const uint64_t sl2x2 = pack_f32x2(sl2, sl2);
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    const uint64_t x = fma_f32x2(pack_f32x2(__uint_as_float(s[e]), __uint_as_float(s[e + 1])),
                                 sl2x2, pack_f32x2(ncol[e], ncol[e + 1]));
    float x0, x1;
    unpack_f32x2(x, x0, x1);
    pk[e / 2] = pack_bf16x2(ex2(x0), ex2(x1));
  }
  tmem_st8(tS + c, pk);
}

// Pass B (needs dP^T and pass A): ds = p * (dp - Dr) on the same 16 columns,
// with p as the bf16 pairs pass A made (the same p the dV product uses):
// kept in registers (dK/dV kernel) or read back from tS (dQ kernel); ds is
// stored as bf16 pairs over the first 8 of these columns of tP.
template <bool kPerColumn, bool kPFromTmem>
__device__ __forceinline__ void pass_ds(int c, uint32_t tS, uint32_t tP, const float* dd,
                                        float d_row, uint32_t (&pk)[8]) {
  uint32_t g[16];
  tmem_ld16(tP + c, g);
  if (kPFromTmem) tmem_ld8(tS + c, pk);
  float dcol[16];
#pragma unroll
  for (int e = 0; e < 16; e += 4) {
    if (kPerColumn) {
      const float4 y = *reinterpret_cast<const float4*>(dd + c + e);
      dcol[e] = y.x, dcol[e + 1] = y.y, dcol[e + 2] = y.z, dcol[e + 3] = y.w;
    } else {
      dcol[e] = dcol[e + 1] = dcol[e + 2] = dcol[e + 3] = d_row;
    }
  }
  tmem_ld_wait();
  reg_fence(g, 16);
  if (kPFromTmem) reg_fence(pk, 8);
  uint32_t dk[8];
  const uint64_t minus1 = pack_f32x2(-1.f, -1.f);
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    const uint64_t p = pack_f32x2(__uint_as_float(pk[e / 2] << 16),
                                  __uint_as_float(pk[e / 2] & 0xffff0000u));
    // dp - Dr, then times p, two columns per instruction
    const uint64_t diff =
        fma_f32x2(pack_f32x2(dcol[e], dcol[e + 1]), minus1,
                  pack_f32x2(__uint_as_float(g[e]), __uint_as_float(g[e + 1])));
    float d0, d1;
    unpack_f32x2(mul_f32x2(p, diff), d0, d1);
    dk[e / 2] = pack_bf16x2(d0, d1);
  }
  tmem_st8(tP + c, dk);
}

// The query tiles a key tile visits in the dK/dV kernel: ring steps t = 0 ..
// P-1 bring query block i = (j + t) mod P (the key block is on device j + t
// at step t); under the causal mask only query tiles holding a query at or
// after the tile's first key take part, and in every layout these are a
// suffix of the block's tiles.
struct KWalk {
  int j, P, tiles, layout;
  int64_t c;
  bool causal;
  int64_t kfirst;  // first key position of the tile (striped: first local row)
  int t, qt, n0;   // iteration state: step, query tile, first visible tile of the block

  __device__ int block(int tt) const { return (j + tt) % P; }
  __device__ int64_t pos(int i, int64_t r) const {
    if (layout == kZigzag) {
      const int64_t h = c / 2;
      return r < h ? i * h + r : (2 * static_cast<int64_t>(P) - 1 - i) * h + (r - h);
    }
    if (layout == kStriped) return i + static_cast<int64_t>(P) * r;
    return i * c + r;
  }
  // Leading tiles (of ntile, the first starting at `first`) whose last query
  // comes before the tile's first key.
  __device__ int hidden(int64_t first, int ntile) const {
    const int64_t n = kfirst - first - (kBM - 1);  // tiles qt with first + qt*128 + 127 < kfirst
    if (n <= 0) return 0;
    const int64_t m = (n + kBM - 1) / kBM;
    return m < ntile ? static_cast<int>(m) : ntile;
  }
  __device__ int first_visible(int i) const {
    if (!causal) return 0;
    if (layout == kStriped) return hidden(-static_cast<int64_t>(j > i ? 1 : 0), tiles);
    if (layout == kZigzag) {
      const int half = tiles / 2;
      const int a = hidden(i * (c / 2), half);
      return a < half ? a : half + hidden((2 * static_cast<int64_t>(P) - 1 - i) * (c / 2), half);
    }
    return hidden(i * c, tiles);
  }
  __device__ int total() const {
    int n = 0;
    for (int tt = 0; tt < P; ++tt) n += tiles - first_visible(block(tt));
    return n;
  }
  __device__ void skip() {
    while (t < P && qt >= tiles) {
      ++t;
      if (t < P) qt = n0 = first_visible(block(t));
    }
  }
  __device__ void start() {
    t = 0;
    qt = n0 = first_visible(block(0));
    skip();
  }
  __device__ void next() {
    ++qt;
    skip();
  }
};

// The products over part h: k-steps [4h, 4h + 4) (16 rows of B each).
template <int D, int G>
__device__ __forceinline__ void mma_tn_part(uint32_t d_tmem, uint32_t a_tmem, uint64_t db, int h,
                                            uint32_t accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, D, true);
  constexpr int S = Roles<G>::kStepsPerPart;
#pragma unroll
  for (int e = 0; e < S; ++e) {
    const int kk = S * h + e;
    mma_bf16_ts(d_tmem, a_tmem + kk * 16, db + desc_step(kk * 16 * 128), idesc,
                e == 0 ? accumulate : 1u);
  }
}

// Store one TMEM row segment of 32 fp32 columns, times `scale`, as bf16.
__device__ __forceinline__ void store_row_bf16(uint32_t taddr, uint16_t* dst, float scale) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
  tmem_ld_wait();
  reg_fence(r, 32);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    uint4 w;
    w.x = pack_bf16x2(__uint_as_float(r[8 * e + 0]) * scale, __uint_as_float(r[8 * e + 1]) * scale);
    w.y = pack_bf16x2(__uint_as_float(r[8 * e + 2]) * scale, __uint_as_float(r[8 * e + 3]) * scale);
    w.z = pack_bf16x2(__uint_as_float(r[8 * e + 4]) * scale, __uint_as_float(r[8 * e + 5]) * scale);
    w.w = pack_bf16x2(__uint_as_float(r[8 * e + 6]) * scale, __uint_as_float(r[8 * e + 7]) * scale);
    d4[e] = w;
  }
}

// Add one TMEM row segment of 32 fp32 columns, times `scale`, into an fp32
// accumulator row in global memory (16-byte aligned).
__device__ __forceinline__ void add_row_f32(uint32_t taddr, float* dst, float scale) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
  float4* d4 = reinterpret_cast<float4*>(dst);
  float4 x[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) x[e] = d4[e];
  tmem_ld_wait();
  reg_fence(r, 32);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    x[e].x = fmaf(__uint_as_float(r[4 * e + 0]), scale, x[e].x);
    x[e].y = fmaf(__uint_as_float(r[4 * e + 1]), scale, x[e].y);
    x[e].z = fmaf(__uint_as_float(r[4 * e + 2]), scale, x[e].z);
    x[e].w = fmaf(__uint_as_float(r[4 * e + 3]), scale, x[e].w);
    d4[e] = x[e];
  }
}

// ---------------------------------------------------------------------------
// dK, dV: one key tile per CTA
// ---------------------------------------------------------------------------
template <int D>
struct DkvLayout {
  using T = Tiles<D>;
  static constexpr int kK = 0;
  static constexpr int kV = T::kTileBytes;
  static constexpr int kStage0 = 2 * T::kTileBytes;
  // stage: Q tile, dO tile, nl[128], D[128]
  static constexpr int kStageBytes = 2 * T::kTileBytes + 2 * T::kRowBytes;
  static constexpr int kBar = kStage0 + kStages * kStageBytes;
  // kv_full, stage_full[S], stage_empty[S], s_full, dp_full, pa[kMaxParts],
  // pb[kMaxParts], o_full, drain
  static constexpr int kNumBars = 1 + 2 * kStages + 4 + 2 * kMaxParts;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kSmem = kMisc + 16 + 1024;
  static_assert(kSmem <= 232448, "shared memory budget");
};

template <int D, bool kCausal, int G = groups_for<kCausal>()>
__global__ void __launch_bounds__(Roles<G>::kThreads, 1)
    dkv_kernel(const __grid_constant__ BackwardArgs a, const __grid_constant__ CUtensorMap tq,
               const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
               const __grid_constant__ CUtensorMap tdo) {
  using L = DkvLayout<D>;
  using T = Tiles<D>;
  // Where the next tile's S^T goes: it overwrites the p in tS, so it comes
  // after the dV products (pass B keeps p in registers).  With two
  // warpgroups (causal) it goes straight before dK; with four (plain) it
  // goes between dK's two parts, which measured 0.5-3 % faster there than
  // either straight before dK or after it.
  constexpr bool kSBetweenDk = !kCausal;
  constexpr int kLoadWarp = Roles<G>::kLoadWarp;
  constexpr int kMmaWarp = Roles<G>::kMmaWarp;
  constexpr int kParts = Roles<G>::kParts;
  constexpr int kPartThreads = Roles<G>::kPartThreads;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bar0 = base + L::kBar;
  auto kv_full = [&]() { return bar0; };
  auto st_full = [&](int s) { return bar0 + 8 * (1 + s); };
  auto st_empty = [&](int s) { return bar0 + 8 * (1 + kStages + s); };
  const uint32_t s_full = bar0 + 8 * (1 + 2 * kStages);  // S^T of the tile done
  const uint32_t dp_full = s_full + 8;                      // dP^T of the tile done
  auto pa = [&](int h) { return dp_full + 8 * (1 + h); };  // pass A, part h done
  auto pb = [&](int h) { return dp_full + 8 * (1 + kMaxParts + h); };  // pass B, part h done
  const uint32_t o_full = dp_full + 8 * (1 + 2 * kMaxParts);
  const uint32_t drain = o_full + 8;
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(gbase + L::kMisc);
  const Abort ab{tmem_holder + 1, a.status, a.wait_limit > 0 ? a.wait_limit : kWaitLimit};
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // unit: (slice, key block j, key tile kt); walk: the query tiles of the
  // blocks i = (j + t) mod P (see KWalk).  Under the mask the heaviest units
  // (the first key rows, seen by the most queries) come first within each
  // slice (causal_order).
  const int64_t c = a.N / a.P;
  const int tiles = static_cast<int>(c / kBN);
  int64_t u = blockIdx.x;
  int kt = static_cast<int>(u % tiles);
  u /= tiles;
  int j = static_cast<int>(u % a.P);
  const int64_t slice = u / a.P;
  if (kCausal) causal_order(a.layout, a.P, tiles, false, j, kt);
  const bool striped = a.layout == kStriped;
  KWalk walk;
  walk.j = j;
  walk.P = a.P;
  walk.tiles = tiles;
  walk.layout = a.layout;
  walk.c = c;
  walk.causal = kCausal;
  walk.kfirst = striped ? static_cast<int64_t>(kt) * kBM : walk.pos(j, static_cast<int64_t>(kt) * kBM);
  const int n_iter = walk.total();

  if (threadIdx.x == 0) {
    mbar_init(kv_full(), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(st_full(s), 1);
      mbar_init(st_empty(s), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    for (int h = 0; h < kParts; ++h) {
      mbar_init(pa(h), kPartThreads);
      mbar_init(pb(h), kPartThreads);
    }
    mbar_init(o_full, 1);
    mbar_init(drain, 1);
    *ab.flag = 0u;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(base + L::kMisc, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tS = tmem, tP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;

  if (warp == kLoadWarp) {
    if (lane == 0) {
      // A stalled CTA (a test aid) loads nothing: its consumers' waits run
      // out, raise the abort flag and return; nothing is in flight to drain.
      const bool stalled = static_cast<int64_t>(blockIdx.x) == a.stall_cta;
      const int64_t klr = static_cast<int64_t>(kt) * kBM;  // first local key row
      if (!stalled) {
        mbar_arrive_expect_tx(kv_full(), 2 * T::kTileBytes);
        load_tile<D>(base + L::kK, &tk, striped, slice * a.N + walk.pos(j, klr), j,
                     slice * c + klr, kv_full());
        load_tile<D>(base + L::kV, &tv, striped, slice * a.N + walk.pos(j, klr), j,
                     slice * c + klr, kv_full());
      }
      uint32_t issued = 0, last_parity = 0;
      bool ok = !stalled;
      KWalk w = walk;
      w.start();
      for (int it = 0; it < n_iter && ok; ++it, w.next()) {
        const int s = it % kStages;
        const uint32_t ph = static_cast<uint32_t>((it / kStages) & 1);
        if (!wait1(st_empty(s), ph ^ 1u, ab)) {
          ok = false;
          break;
        }
        const uint32_t sb = base + L::kStage0 + s * L::kStageBytes;
        const int i = w.block(w.t);
        const int64_t qlr = static_cast<int64_t>(w.qt) * kBM;  // first local query row
        const int64_t bm = slice * a.N + static_cast<int64_t>(i) * c + qlr;  // block-major
        mbar_arrive_expect_tx(st_full(s), 2 * T::kTileBytes + 2 * T::kRowBytes);
        load_tile<D>(sb, &tq, striped, slice * a.N + w.pos(i, qlr), i, slice * c + qlr,
                     st_full(s));
        load_tile<D>(sb + T::kTileBytes, &tdo, striped, slice * a.N + w.pos(i, qlr), i,
                     slice * c + qlr, st_full(s));
        bulk_load(sb + 2 * T::kTileBytes, a.nl + bm, T::kRowBytes, st_full(s));
        bulk_load(sb + 2 * T::kTileBytes + T::kRowBytes, a.delta + bm, T::kRowBytes, st_full(s));
        issued |= 1u << s;
        last_parity = (last_parity & ~(1u << s)) | (ph << s);
      }
      if (!ok) {
        if (!stalled) wait_drain(kv_full(), 0);
        for (int s = 0; s < kStages; ++s)
          if (issued & (1u << s)) wait_drain(st_full(s), (last_parity >> s) & 1u);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // Per tile, in pipe order: dP^T; dV over the parts of pass A as they
      // land; dK over the parts of pass B, with the next tile's S^T before
      // dK or between its parts (kSBetweenDk).  Pass A runs while dP^T is
      // on the tensor cores, pass B while dV is and the next pass A while
      // dK is.
      const uint64_t dK = desc_sw128(base + L::kK, 16, 1024);
      const uint64_t dV = desc_sw128(base + L::kV, 16, 1024);
      bool ok = wait1(kv_full(), 0, ab);
      if (ok && n_iter > 0) ok = wait1(st_full(0), 0, ab);
      if (ok && n_iter > 0) {
        tc_fence_after();
        mma_nt<D>(tS, dK, desc_sw128(base + L::kStage0, 16, 1024));  // S^T = K Q^T
        mma_commit(s_full);
      }
      for (int it = 0; it < n_iter && ok; ++it) {
        const int s = it % kStages;
        const uint32_t sb = base + L::kStage0 + s * L::kStageBytes;
        const uint32_t par = static_cast<uint32_t>(it & 1);
        mma_nt<D>(tP, dV, desc_sw128(sb + T::kTileBytes, 16, 1024));  // dP^T = V dO^T
        mma_commit(dp_full);
        const uint64_t dDOs = desc_sw128(sb + T::kTileBytes, T::kBoxBytes, 1024);
        const uint64_t dQs = desc_sw128(sb, T::kBoxBytes, 1024);
        const uint32_t acc = it > 0 ? 1u : 0u;
        for (int h = 0; h < kParts && ok; ++h) {
          if (!wait1(pa(h), par, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_tn_part<D, G>(tdV, tS, dDOs, h, h == 0 ? acc : 1u);  // dV += P^T dO, part h
        }
        // the next tile's S^T (K Q^T of the next stage), issued once the dV
        // products have read the p in tS: before dK, or after dK's part 0
        const int s1 = (it + 1) % kStages;
        const uint32_t s1_par = static_cast<uint32_t>(((it + 1) / kStages) & 1);
        const uint64_t dQ1 = desc_sw128(base + L::kStage0 + s1 * L::kStageBytes, 16, 1024);
        if (!kSBetweenDk && ok && it + 1 < n_iter) {
          if (!wait1(st_full(s1), s1_par, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_nt<D>(tS, dK, dQ1);
          mma_commit(s_full);
        }
        for (int h = 0; h < kParts && ok; ++h) {
          if (!wait1(pb(h), par, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_tn_part<D, G>(tdK, tP, dQs, h, h == 0 ? acc : 1u);  // dK += dS^T Q, part h
          if (kSBetweenDk && h == 0 && it + 1 < n_iter) {
            if (!wait1(st_full(s1), s1_par, ab)) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma_nt<D>(tS, dK, dQ1);
            mma_commit(s_full);
          }
        }
        if (!ok) break;
        mma_commit(st_empty(s));
      }
      if (ok) {
        mma_commit(o_full);
      } else {
        mma_commit(drain);
        wait_drain(drain, 0);
      }
    }
  } else if (warp < 4 * G) {
    const int wg = warp / 4;  // warpgroup: k-steps 4h + wg + G m of every part h
    const int row = (warp % 4) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp % 4) * 32) << 16;
    // this thread's key: position (striped: local row) for the mask
    const int64_t kref = walk.kfirst + row;
    KWalk w = walk;
    w.start();
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      if (kCausal && it > 0) w.next();
      const uint32_t par = static_cast<uint32_t>(it & 1);
      if (!wait_warp(s_full, par, ab)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int s = it % kStages;
      const float* rows = reinterpret_cast<const float*>(gbase + L::kStage0 +
                                                         s * L::kStageBytes + 2 * T::kTileBytes);
      int lo = 0;
      if (kCausal) {
        // query columns before this key are masked: positions qfirst + col
        const int i = w.block(w.t);
        const int64_t qlr = static_cast<int64_t>(w.qt) * kBM;
        const int64_t qref = striped ? qlr - (j > i ? 1 : 0) : w.pos(i, qlr);
        const int64_t m = kref - qref;
        lo = m < 0 ? 0 : (m > kBN ? kBN : static_cast<int>(m));
      }
      // pass A: p, feeding dV (warpgroup wg takes k-steps 4h + wg + G m of part h);
      // this thread's p stay in registers for pass B, since the next S^T
      // overwrites them in tS as soon as the dV products have read it
      uint32_t pkeep[kParts][Roles<G>::kStepsPerGroup][8];
#pragma unroll
      for (int h = 0; h < kParts; ++h) {
#pragma unroll
        for (int m = 0; m < Roles<G>::kStepsPerGroup; ++m)
          pass_p<true, kCausal>(16 * (Roles<G>::kStepsPerPart * h + wg + G * m), tS + lane_off,
                                a.scale_log2, rows, 0.f, lo, kBN, pkeep[h][m]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(pa(h));
      }
      // pass B: dS, feeding dK
      if (!wait_warp(dp_full, par, ab)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < kParts; ++h) {
#pragma unroll
        for (int m = 0; m < Roles<G>::kStepsPerGroup; ++m)
          pass_ds<true, false>(16 * (Roles<G>::kStepsPerPart * h + wg + G * m), tS + lane_off,
                               tP + lane_off, rows + kBM, 0.f, pkeep[h][m]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(pb(h));
      }
    }
    if (ok && wait_warp(o_full, 0, ab)) {
      tc_fence_after();
      const int64_t r = slice * a.N + walk.pos(j, static_cast<int64_t>(kt) * kBM + row);
      if (a.accumulate) {
        // block mode: add into the fp32 accumulators that travel with the block
        float* dv = static_cast<float*>(a.dv) + r * D;
        float* dk = static_cast<float*>(a.dk) + r * D;
#pragma unroll
        for (int cc = 32 * wg; cc < D; cc += 32 * G) {
          add_row_f32(tdV + lane_off + cc, dv + cc, 1.f);
          add_row_f32(tdK + lane_off + cc, dk + cc, a.tau);
        }
      } else {
        uint16_t* dv = static_cast<uint16_t*>(a.dv) + r * D;
        uint16_t* dk = static_cast<uint16_t*>(a.dk) + r * D;
#pragma unroll
        for (int cc = 32 * wg; cc < D; cc += 32 * G) {
          store_row_bf16(tdV + lane_off + cc, dv + cc, 1.f);
          store_row_bf16(tdK + lane_off + cc, dk + cc, a.tau);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// dQ: one query tile per CTA
// ---------------------------------------------------------------------------
template <int D>
struct DqLayout {
  using T = Tiles<D>;
  static constexpr int kKStages = 3;  // K is read by S (one tile ahead) and by dQ
  static constexpr int kVStages = 2;  // V only by dP
  static constexpr int kQ = 0;
  static constexpr int kDO = T::kTileBytes;
  static constexpr int kK0 = 2 * T::kTileBytes;
  static constexpr int kV0 = kK0 + kKStages * T::kTileBytes;
  static constexpr int kBar = kV0 + kVStages * T::kTileBytes;
  // q_full, k_full[3], k_empty[3], v_full[2], v_empty[2], s_full[2], dp_full,
  // pb[kMaxParts], o_full, drain
  static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 3 + kMaxParts + 2;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kSmem = kMisc + 16 + 1024;
  static_assert(kSmem <= 232448, "shared memory budget");
};

// dQ: one query tile per CTA.  TMEM: S in two buffers [0,128) and [128,256),
// dP [256,384), dQ [384, 384+D).  In pipe order, per key tile it: dQ(it) over
// the parts of pass B as they land, dP(it+1), then S(it+2) into the buffer
// S(it) used.  Pass A (p from S) of a tile runs while the tensor cores work
// on the previous tile's dQ and on its own dP; pass B (dS) while they work on
// the next S.
template <int D, bool kCausal, int G = groups_for<kCausal>()>
__global__ void __launch_bounds__(Roles<G>::kThreads, 1)
    dq_kernel(const __grid_constant__ BackwardArgs a, const __grid_constant__ CUtensorMap tq,
              const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
              const __grid_constant__ CUtensorMap tdo) {
  using L = DqLayout<D>;
  using T = Tiles<D>;
  constexpr int kLoadWarp = Roles<G>::kLoadWarp;
  constexpr int kMmaWarp = Roles<G>::kMmaWarp;
  constexpr int kParts = Roles<G>::kParts;
  constexpr int kPartThreads = Roles<G>::kPartThreads;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bar0 = base + L::kBar;
  const uint32_t q_full = bar0;
  auto k_full = [&](int s) { return bar0 + 8 * (1 + s); };
  auto k_empty = [&](int s) { return bar0 + 8 * (1 + L::kKStages + s); };
  auto v_full = [&](int s) { return bar0 + 8 * (1 + 2 * L::kKStages + s); };
  auto v_empty = [&](int s) { return bar0 + 8 * (1 + 2 * L::kKStages + L::kVStages + s); };
  const uint32_t bar_s = bar0 + 8 * (1 + 2 * L::kKStages + 2 * L::kVStages);
  auto s_full = [&](int b) { return bar_s + 8 * b; };  // S of the tile in buffer b done
  const uint32_t dp_full = bar_s + 16;
  auto pb = [&](int h) { return dp_full + 8 * (1 + h); };  // pass B, part h done
  const uint32_t o_full = dp_full + 8 * (1 + kMaxParts);
  const uint32_t drain = o_full + 8;
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(gbase + L::kMisc);
  const Abort ab{tmem_holder + 1, a.status, a.wait_limit > 0 ? a.wait_limit : kWaitLimit};
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // unit: (slice, query block i, query tile qt); walk: the forward's ring
  // order over key tiles (Walk).  Under the mask the heaviest units (the
  // last query rows) come first within each slice (causal_order).
  const int64_t c = a.N / a.P;
  const int tiles = static_cast<int>(c / kBN);
  int64_t u = blockIdx.x;
  int qt = static_cast<int>(u % tiles);
  u /= tiles;
  int i = static_cast<int>(u % a.P);
  const int64_t slice = u / a.P;
  if (kCausal) causal_order(a.layout, a.P, tiles, true, i, qt);
  const bool striped = a.layout == kStriped;
  const int64_t qlr0 = static_cast<int64_t>(qt) * kBM;  // first local query row
  Walk walk;
  walk.slice = slice;
  walk.N = a.N;
  walk.c = c;
  walk.i = i;
  walk.P = a.P;
  walk.t0 = 0;
  walk.t1 = a.P;
  walk.tiles = tiles;
  walk.layout = a.layout;
  walk.causal = kCausal;
  walk.qlast = striped ? qlr0 + kBM - 1 : walk.pos(i, qlr0 + kBM - 1);
  const int n_iter = walk.total();

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < L::kKStages; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < L::kVStages; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    mbar_init(s_full(0), 1);
    mbar_init(s_full(1), 1);
    mbar_init(dp_full, 1);
    for (int h = 0; h < kParts; ++h) mbar_init(pb(h), kPartThreads);
    mbar_init(o_full, 1);
    mbar_init(drain, 1);
    *ab.flag = 0u;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(base + L::kMisc, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tP = tmem + 256, tdQ = tmem + 384;
  auto tS = [&](int it) { return tmem + static_cast<uint32_t>((it & 1) * 128); };

  if (warp == kLoadWarp) {
    if (lane == 0) {
      // A stalled CTA (a test aid) loads nothing (see the dK/dV kernel).
      const bool stalled = static_cast<int64_t>(blockIdx.x) == a.stall_cta;
      if (!stalled) {
        mbar_arrive_expect_tx(q_full, 2 * T::kTileBytes);
        load_tile<D>(base + L::kQ, &tq, striped, slice * a.N + walk.pos(i, qlr0), i,
                     slice * c + qlr0, q_full);
        load_tile<D>(base + L::kDO, &tdo, striped, slice * a.N + walk.pos(i, qlr0), i,
                     slice * c + qlr0, q_full);
      }
      // per ring, the stages with a load in flight and their last parity
      uint32_t k_issued = 0, k_par = 0, v_issued = 0, v_par = 0;
      bool ok = !stalled;
      Walk w = walk;
      w.start();
      for (int it = 0; it < n_iter && ok; ++it, w.next()) {
        const int jb = w.block(w.t);
        const int64_t row = slice * a.N + w.key_first();
        const int64_t lrow = slice * c + static_cast<int64_t>(w.kt) * kBN;
        const int ks = it % L::kKStages;
        const uint32_t kph = static_cast<uint32_t>((it / L::kKStages) & 1);
        if (!wait1(k_empty(ks), kph ^ 1u, ab)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(k_full(ks), T::kTileBytes);
        load_tile<D>(base + L::kK0 + ks * T::kTileBytes, &tk, striped, row, jb, lrow, k_full(ks));
        k_issued |= 1u << ks;
        k_par = (k_par & ~(1u << ks)) | (kph << ks);
        const int vs = it % L::kVStages;
        const uint32_t vph = static_cast<uint32_t>((it / L::kVStages) & 1);
        if (!wait1(v_empty(vs), vph ^ 1u, ab)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(v_full(vs), T::kTileBytes);
        load_tile<D>(base + L::kV0 + vs * T::kTileBytes, &tv, striped, row, jb, lrow, v_full(vs));
        v_issued |= 1u << vs;
        v_par = (v_par & ~(1u << vs)) | (vph << vs);
      }
      if (!ok) {
        if (!stalled) wait_drain(q_full, 0);
        for (int s = 0; s < L::kKStages; ++s)
          if (k_issued & (1u << s)) wait_drain(k_full(s), (k_par >> s) & 1u);
        for (int s = 0; s < L::kVStages; ++s)
          if (v_issued & (1u << s)) wait_drain(v_full(s), (v_par >> s) & 1u);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint64_t dQ = desc_sw128(base + L::kQ, 16, 1024);
      const uint64_t dDO = desc_sw128(base + L::kDO, 16, 1024);
      const uint32_t k0 = base + L::kK0;  // K stage 0; stage s at + s * kTileBytes
      // Per key tile it: S(it) = Q K(it)^T into S buffer it % 2 (s_full),
      // dP(it) = dO V(it)^T (dp_full; frees V(it)), then dQ += dS K over the
      // parts of pass B.
      bool ok = wait1(q_full, 0, ab);
      if (ok && n_iter > 0) {
        ok = wait1(k_full(0), 0, ab);
        if (ok) {
          tc_fence_after();
          mma_nt<D>(tS(0), dQ, desc_sw128(k0, 16, 1024));
          mma_commit(s_full(0));
          ok = wait1(v_full(0), 0, ab);
        }
        if (ok) {
          tc_fence_after();
          mma_nt<D>(tP, dDO, desc_sw128(base + L::kV0, 16, 1024));
          mma_commit(dp_full);
          mma_commit(v_empty(0));
        }
        if (ok && n_iter > 1) {
          ok = wait1(k_full(1 % L::kKStages), static_cast<uint32_t>((1 / L::kKStages) & 1), ab);
          if (ok) {
            tc_fence_after();
            mma_nt<D>(tS(1), dQ, desc_sw128(k0 + (1 % L::kKStages) * T::kTileBytes, 16, 1024));
            mma_commit(s_full(1));
          }
        }
      }
      for (int it = 0; it < n_iter && ok; ++it) {
        const uint64_t dKs =
            desc_sw128(k0 + (it % L::kKStages) * T::kTileBytes, T::kBoxBytes, 1024);
        for (int h = 0; h < kParts && ok; ++h) {
          if (!wait1(pb(h), static_cast<uint32_t>(it & 1), ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_tn_part<D, G>(tdQ, tP, dKs, h, (it > 0 || h > 0) ? 1u : 0u);  // dQ += dS K, part h
        }
        if (!ok) break;
        mma_commit(k_empty(it % L::kKStages));
        // dP(it+1) overwrites dS(it) (read by the dQ products above, earlier
        // in the pipe) and dP(it) (read by pass B, complete); S(it+2) goes to
        // the buffer of S(it), whose p pass B has read too.
        if (it + 1 < n_iter) {
          const int vs = (it + 1) % L::kVStages;
          if (!wait1(v_full(vs), static_cast<uint32_t>(((it + 1) / L::kVStages) & 1), ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_nt<D>(tP, dDO, desc_sw128(base + L::kV0 + vs * T::kTileBytes, 16, 1024));
          mma_commit(dp_full);
          mma_commit(v_empty(vs));
        }
        if (it + 2 < n_iter) {
          const int ks = (it + 2) % L::kKStages;
          if (!wait1(k_full(ks), static_cast<uint32_t>(((it + 2) / L::kKStages) & 1), ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_nt<D>(tS(it + 2), dQ, desc_sw128(k0 + ks * T::kTileBytes, 16, 1024));
          mma_commit(s_full((it + 2) & 1));
        }
      }
      if (ok) {
        mma_commit(o_full);
      } else {
        mma_commit(drain);
        wait_drain(drain, 0);
      }
    }
  } else if (warp < 4 * G) {
    const int wg = warp / 4;  // warpgroup: k-steps 4h + wg + G m of every part h
    const int row = (warp % 4) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const int64_t lrow = qlr0 + row;
    const int64_t qpos = walk.pos(i, lrow);
    const int64_t r = slice * a.N + qpos;  // row of dq
    const int64_t bm = slice * a.N + static_cast<int64_t>(i) * c + lrow;  // block-major
    const float nl_row = a.nl[bm];  // the row terms were precomputed per query
    const float d_row = a.delta[bm];
    const int64_t qref = striped ? lrow : qpos;
    Walk w = walk;
    w.start();
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      if (kCausal && it > 0) w.next();
      // pass A: p into the S buffer of this tile
      if (!wait_warp(s_full(it & 1), static_cast<uint32_t>((it >> 1) & 1), ab)) {
        ok = false;
        break;
      }
      tc_fence_after();
      int hi = kBN;
      if (kCausal) {
        // keys after this query are masked: first key reference of the tile
        const int64_t first = w.key_first() + (striped && w.block(w.t) > i ? 1 : 0);
        const int64_t n = qref - first + 1;
        hi = n < 0 ? 0 : (n > kBN ? kBN : static_cast<int>(n));
      }
      const uint32_t tSt = tS(it) + lane_off;
#pragma unroll
      for (int h = 0; h < kParts; ++h)
#pragma unroll
        for (int m = 0; m < Roles<G>::kStepsPerGroup; ++m) {
          uint32_t pk[8];
          pass_p<false, kCausal>(16 * (Roles<G>::kStepsPerPart * h + wg + G * m), tSt,
                                 a.scale_log2, nullptr, nl_row, 0, hi, pk);
        }
      tmem_st_wait();  // pass B reads these p back
      // pass B: dS into dP's columns, feeding dQ
      if (!wait_warp(dp_full, static_cast<uint32_t>(it & 1), ab)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < kParts; ++h) {
#pragma unroll
        for (int m = 0; m < Roles<G>::kStepsPerGroup; ++m) {
          uint32_t pk[8];
          pass_ds<false, true>(16 * (Roles<G>::kStepsPerPart * h + wg + G * m), tSt,
                               tP + lane_off, nullptr, d_row, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(pb(h));
      }
    }
    if (ok && wait_warp(o_full, 0, ab)) {
      tc_fence_after();
      if (a.accumulate) {
        float* dq = static_cast<float*>(a.dq) + r * D;
#pragma unroll
        for (int cc = 32 * wg; cc < D; cc += 32 * G) add_row_f32(tdQ + lane_off + cc, dq + cc, a.tau);
      } else {
        uint16_t* dq = static_cast<uint16_t*>(a.dq) + r * D;
#pragma unroll
        for (int cc = 32 * wg; cc < D; cc += 32 * G)
          store_row_bf16(tdQ + lane_off + cc, dq + cc, a.tau);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool kCausal>
cudaError_t launch_d(const BackwardArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, const CUtensorMap& tdo, cudaStream_t s) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(dkv_kernel<D, kCausal>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DkvLayout<D>::kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(dq_kernel<D, kCausal>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, DqLayout<D>::kSmem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const unsigned grid = static_cast<unsigned>(a.slices * (a.N / kBM));
  constexpr int kThreads = Roles<groups_for<kCausal>()>::kThreads;
  // The two kernels are independent: dQ runs on a side stream, forked from
  // and joined back into `s` by events (so the pair also captures into a
  // CUDA graph as two branches), and its CTAs fill the SMs that the dK/dV
  // kernel's last wave leaves idle.
  ForkJoin fj;
  e = fj.fork(s, dev);
  if (e != cudaSuccess) return e;
  dkv_kernel<D, kCausal><<<grid, kThreads, DkvLayout<D>::kSmem, s>>>(a, tq, tk, tv, tdo);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dq_kernel<D, kCausal><<<grid, kThreads, DqLayout<D>::kSmem, fj.side>>>(a, tq, tk, tv, tdo);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return fj.join(s);
}

}  // namespace

cudaError_t launch_backward_sm103(const BackwardArgs& a, const CUtensorMap& tq,
                                  const CUtensorMap& tk, const CUtensorMap& tv,
                                  const CUtensorMap& tdo, cudaStream_t s) {
  if (a.causal) {
    if (a.d == 128) return launch_d<128, true>(a, tq, tk, tv, tdo, s);
    if (a.d == 64) return launch_d<64, true>(a, tq, tk, tv, tdo, s);
  } else {
    if (a.d == 128) return launch_d<128, false>(a, tq, tk, tv, tdo, s);
    if (a.d == 64) return launch_d<64, false>(a, tq, tk, tv, tdo, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ra
