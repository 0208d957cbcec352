// Tensor-core fold kernel for bf16 inputs on sm_103a (GB300).
//
// One CTA owns up to two 128-row query tiles of one query block i
// ("Ring Attention: the math", section "Sharding the sequence": queries stay
// home) and streams the key/value tiles of the blocks it visits in ring order
// j = (i - t) mod P (section "The ring schedule: passing K/V around").  Each
// 128-key tile is folded into the running per-row state with the update of
// section "The online-softmax identity that makes streaming legal":
//
//   S = tau * Q K^T             tcgen05.mma, bf16 -> fp32 in TMEM
//   m' = max(m, rowmax S)       softmax warps, registers
//   p  = exp(S - m'), l' = alpha l + sum p
//   O  = alpha O + p V          tcgen05.mma, p as bf16 from tensor memory
//
// The pages' send/recv of the next block while the current one is computed
// (section "Accumulation math, step by step") becomes a TMA prefetch of the
// next K/V tile into a free stage of a shared-memory ring.
//
// Warp roles (384 threads, launched at 168 registers a thread):
//   warps 0-3   softmax for query tile 0 (thread = row = TMEM lane)
//   warps 4-7   softmax for query tile 1
//   warp  8     TMA producer (one thread)
//   warp  9     TMEM allocator and MMA issuer (one thread)
//   warps 10-11 idle (they complete the third warpgroup)
// The third warpgroup gives registers back (setmaxnreg.dec to 88) and the two
// softmax warpgroups take them (setmaxnreg.inc to 208): 2 x 128 x 208 +
// 128 x 88 = 64512 = 384 x 168, the launch's register total.
//
// The two query tiles ping-pong: while one tile's softmax runs on the CUDA
// cores, the tensor cores work on the other tile's products.
//
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D),
// O1 [256+D, 256+2D).  The bf16 probabilities P_t overwrite the first 64
// columns of S_t once the softmax warps have read S_t, and feed the P V
// product straight from TMEM.  Shared memory (1024-byte aligned, 128-byte
// swizzle everywhere): Q0, Q1, kStages K/V tiles, mbarriers.
//
// The running max used for the exponentials is a per-row reference that is
// raised only when a tile's max exceeds it by more than kRescaleLog2 (log2
// units).  The identity holds for any reference, so l and o stay exact; most
// tiles then need no rescale of O in TMEM.  States leaving the kernel are
// re-expressed relative to the true running max.
//
// Every wait is bounded.  A wait that runs out records a timeout in the
// device status word, raises a CTA-wide abort flag, lets the in-flight TMA
// loads and MMAs finish (again bounded), frees TMEM and returns.

#include <cmath>

#include "ra_internal.h"
#include "ra_layout.cuh"
#include "sm103_pipeline.cuh"
#include "sm103_ptx.cuh"

namespace ra {
namespace {

using namespace ptx;
using namespace sm103;

constexpr int kThreads = 384;
constexpr uint32_t kRegsSoftmax = 208;
constexpr uint32_t kRegsOther = 88;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsOther == kThreads * 168,
              "register split must equal the launch's register total");
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
// Every p is >= 0, so a tile whose row sum of p is at most 2^kRescaleLog2
// has no p above 2^kRescaleLog2.
constexpr float kFastSumBound = 256.0f;
static_assert(kFastSumBound == (1 << static_cast<int>(kRescaleLog2)), "2^kRescaleLog2");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct Layout {
  static constexpr int kBoxBytes = kBM * 128;  // 128 rows x 128 bytes (64 bf16)
  static constexpr int kTileBytes = kBM * D * 2;
  static constexpr int kStages = D == 128 ? 4 : 6;
  static constexpr int kQ0 = 0;
  static constexpr int kQ1 = kTileBytes;
  static constexpr int kKV = 2 * kTileBytes;
  static constexpr int kBar = kKV + kStages * kTileBytes;
  // q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], o_full[2], drain
  static constexpr int kNumBars = 1 + 2 * kStages + 7;
  // TMEM base and abort flag, then the causal step table (int4 per step);
  // both start on a 16-byte boundary (the table is read as int4).
  static constexpr int kMisc = (kBar + kNumBars * 8 + 15) / 16 * 16;
  static constexpr int kSteps = kMisc + 16;
  static constexpr int kBytes = kSteps + kMaxCausalSteps * 16;
  static_assert(kSteps % 16 == 0, "the step table is read as int4");
  static constexpr int kSmem = kBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kSmem <= 232448, "shared memory budget");
};

template <int D>
struct Bars {
  uint32_t base;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t kv_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t kv_empty(int s) const { return base + 8 * (1 + Layout<D>::kStages + s); }
  __device__ uint32_t s_full(int t) const { return base + 8 * (1 + 2 * Layout<D>::kStages + t); }
  __device__ uint32_t p_full(int t) const { return base + 8 * (3 + 2 * Layout<D>::kStages + t); }
  __device__ uint32_t o_full(int t) const { return base + 8 * (5 + 2 * Layout<D>::kStages + t); }
  __device__ uint32_t drain() const { return base + 8 * (7 + 2 * Layout<D>::kStages); }
};

// Per ring step of a causal unit, as the softmax warps see it: the number of
// tiles visited and the offsets that give the first key of tile kt,
//   first(kt) = kt < tiles/2 ? a + kt*128 : b + (kt - tiles/2)*128,
// in the units of the query reference `qref` (the token position, or for the
// striped layout the local row, shifted by one when j > i).  The number of
// keys of the tile visible to the query is then qref - first(kt) + 1,
// clamped to [0, 128].
__device__ __forceinline__ int4 step_entry(const Walk& w, int tt) {
  const int j = w.block(tt);
  const int half = w.tiles / 2;
  int4 e;
  e.x = w.count(j);
  if (w.layout == kStriped) {
    e.y = j > w.i ? 1 : 0;
    e.z = e.y + half * kBN;
  } else {
    e.y = static_cast<int>(w.pos(j, 0));
    e.z = static_cast<int>(w.pos(j, static_cast<int64_t>(half) * kBN));
  }
  e.w = 0;
  return e;
}

// S[tmem] = Q K^T for one 128x128 tile: D/16 MMAs of K = 16 along d.  Q and K
// are K-major (d contiguous) in 128-byte-swizzled boxes of 64 columns; the
// k-th slice of 16 columns starts 32 bytes further inside its box.
// dq, dk: descriptors of the Q and K tiles (leading offset 16, stride 1024).
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t dq, uint64_t dk) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = desc_step((kk / 4) * Layout<D>::kBoxBytes + (kk % 4) * 32);
    mma_bf16_ss(d_tmem, dq + off, dk + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// O[tmem] (+)= P V for one tile: 8 MMAs of K = 16 keys.  P is read from TMEM
// (packed bf16 pairs, 8 columns per 16 keys); V is MN-major (d contiguous):
// 8 keys of one 64-column box form a 1024-byte swizzle atom (stride byte
// offset), the second box of 64 columns sits one box further (leading byte
// offset).
// dv: descriptor of the V tile (leading offset = one box, stride 1024).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t dv,
                                         uint32_t accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, D, true);
  mma_bf16_ts(d_tmem, p_tmem, dv, idesc, accumulate);
#pragma unroll
  for (int kk = 1; kk < kBN / 16; ++kk)
    mma_bf16_ts(d_tmem, p_tmem + kk * 8, dv + desc_step(kk * 16 * 128), idesc, 1u);
}

// p = exp2(s * sl2 + neg) for the 128 scores of this row, two per FMA; p is
// rounded to bf16 pairs and written over the first 64 columns of S (tS),
// where the P V product reads it.  Returns the row sum of p (four
// independent pair sums).
__device__ __forceinline__ float exp_store(const uint32_t (&s)[kBN], uint64_t scale2,
                                           uint64_t neg2, uint32_t tS) {
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t pk[32];
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const int j = half * 64 + 2 * jj;
      const uint64_t x =
          fma_f32x2(pack_f32x2(__uint_as_float(s[j]), __uint_as_float(s[j + 1])), scale2, neg2);
      float x0, x1;
      unpack_f32x2(x, x0, x1);
      const float p0 = ex2(x0), p1 = ex2(x1);
      acc[jj & 3] = add_f32x2(acc[jj & 3], pack_f32x2(p0, p1));
      pk[jj] = pack_bf16x2(p0, p1);
    }
    tmem_st32(tS + static_cast<uint32_t>(half * 32), pk);
  }
  float a0, a1, a2, a3, a4, a5, a6, a7;
  unpack_f32x2(acc[0], a0, a1);
  unpack_f32x2(acc[1], a2, a3);
  unpack_f32x2(acc[2], a4, a5);
  unpack_f32x2(acc[3], a6, a7);
  return ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
}

template <int D, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    fold_sm103_kernel(const __grid_constant__ FoldArgs a, const __grid_constant__ CUtensorMap tq,
                      const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const Bars<D> bars{base + L::kBar};
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(gbase + L::kMisc);
  const Abort ab{tmem_holder + 1, a.status, a.wait_limit > 0 ? a.wait_limit : kWaitLimit};

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // ---- work unit: (slice, query block i, segment g, tile pair pr) ----
  // Consecutive CTAs share (slice, i, g) and so walk the same K/V tiles in
  // the same order (L2 reuse).  Under the causal mask the heaviest units (the
  // last query rows) are numbered first within each slice (causal_order).
  const int64_t cq = a.nq / a.P;
  const int64_t ck = a.nk / a.P;
  const int tiles_q = static_cast<int>(cq / kBM);
  const int pairs = (tiles_q + 1) / 2;
  int64_t u = blockIdx.x;
  int pr = static_cast<int>(u % pairs);
  u /= pairs;
  const int g = static_cast<int>(u % a.G);
  u /= a.G;
  int i = static_cast<int>(u % a.P);
  const int64_t slice = u / a.P;
  if (kCausal) causal_order(a.layout, a.P, pairs, true, i, pr);
  const bool has_t1 = 2 * pr + 1 < tiles_q;
  const bool striped = a.layout == kStriped;
  Walk walk;
  walk.slice = slice;
  walk.N = a.nk;
  walk.c = ck;
  walk.i = i;
  walk.P = a.P;
  walk.t0 = static_cast<int>(static_cast<int64_t>(g) * a.P / a.G);
  walk.t1 = static_cast<int>(static_cast<int64_t>(g + 1) * a.P / a.G);
  walk.tiles = static_cast<int>(ck / kBN);
  walk.layout = a.layout;
  walk.causal = kCausal;
  const int64_t lr0 = static_cast<int64_t>(pr) * 2 * kBM;  // first local query row
  const int64_t lr_last = lr0 + (has_t1 ? 2 * kBM : kBM) - 1;
  walk.qlast = striped ? lr_last : walk.pos(i, lr_last);
  const int n_iter = walk.total();

  // ---- set-up ----
  if (threadIdx.x == 0) {
    mbar_init(bars.q_full(), 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bars.kv_full(s), 1);
      mbar_init(bars.kv_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bars.s_full(t), 1);
      mbar_init(bars.p_full(t), 128);
      mbar_init(bars.o_full(t), 1);
    }
    mbar_init(bars.drain(), 1);
    *ab.flag = 0u;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(base + L::kMisc, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kLoadWarp && lane == 0) {
    prefetch_tmap(&tq);
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == kLoadWarp) {
    // ================= TMA producer =================
    setmaxnreg_dec<kRegsOther>();
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_parity = 0;  // per-stage bit masks, for the drain
      // A stalled CTA (a test aid) loads nothing: its consumers' waits run
      // out, raise the abort flag and return; nothing is in flight to drain.
      bool ok = static_cast<int64_t>(blockIdx.x) != a.stall_cta;
      if (ok && n_iter > 0) {
        const uint32_t qbytes = (has_t1 ? 2u : 1u) * L::kTileBytes;
        mbar_arrive_expect_tx(bars.q_full(), qbytes);
        load_tile<D>(base + L::kQ0, &tq, striped, slice * a.nq + walk.pos(i, lr0), i,
                     slice * cq + lr0, bars.q_full());
        if (has_t1)
          load_tile<D>(base + L::kQ1, &tq, striped, slice * a.nq + walk.pos(i, lr0 + kBM), i,
                       slice * cq + lr0 + kBM, bars.q_full());
      }
      Walk kw = walk;
      kw.start();
      for (int it = 0; it < n_iter && ok; ++it, kw.next()) {
        const int j = kw.block(kw.t);
        const int64_t row = slice * a.nk + kw.key_first();         // 2-D row (not striped)
        const int64_t lrow = slice * ck + static_cast<int64_t>(kw.kt) * kBN;  // 3-D (striped)
        for (int kind = 0; kind < 2; ++kind) {
          if (!wait1(bars.kv_empty(stage), phase ^ 1u, ab)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bars.kv_full(stage), L::kTileBytes);
          load_tile<D>(base + L::kKV + stage * L::kTileBytes, kind == 0 ? &tk : &tv, striped, row, j,
                       lrow, bars.kv_full(stage));
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == L::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let every load already issued land before the CTA goes away.
        if (n_iter > 0 && static_cast<int64_t>(blockIdx.x) != a.stall_cta)
          wait_drain(bars.q_full(), 0);
        for (int s = 0; s < L::kStages; ++s)
          if (issued & (1u << s)) wait_drain(bars.kv_full(s), (last_parity >> s) & 1u);
      }
    }
  } else if (warp == kMmaWarp) {
    // ================= MMA issuer =================
    setmaxnreg_dec<kRegsOther>();
    if (lane == 0) {
      const uint32_t tS0 = tmem, tS1 = tmem + 128;
      const uint32_t tO0 = tmem + 256, tO1 = tmem + 256 + D;
      const uint64_t dQ0 = desc_sw128(base + L::kQ0, 16, 1024);
      const uint64_t dQ1 = desc_sw128(base + L::kQ1, 16, 1024);
      const uint64_t dK = desc_sw128(base + L::kKV, 16, 1024);  // stage 0, K-major
      const uint64_t dV = desc_sw128(base + L::kKV, L::kBoxBytes, 1024);  // stage 0, MN-major
      const bool from_state = a.mode == kFold;
      bool ok = n_iter > 0 && wait1(bars.q_full(), 0, ab);
      int cons = 0;  // K/V tiles consumed so far
      if (ok) ok = wait1(bars.kv_full(0), 0, ab);
      if (ok) {
        tc_fence_after();
        cons = 1;
        issue_qk<D>(tS0, dQ0, dK);
        mma_commit(bars.s_full(0));
        if (has_t1) {
          issue_qk<D>(tS1, dQ1, dK);
          mma_commit(bars.s_full(1));
        }
        mma_commit(bars.kv_empty(0));
      }
      for (int it = 0; it < n_iter && ok; ++it) {
        const uint32_t par = static_cast<uint32_t>(it & 1);
        const int sV = cons % L::kStages;
        if (!wait1(bars.kv_full(sV), static_cast<uint32_t>((cons / L::kStages) & 1), ab)) {
          ok = false;
          break;
        }
        ++cons;
        const uint64_t dVs = dV + desc_step(sV * L::kTileBytes);
        if (!wait1(bars.p_full(0), par, ab)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc = (it > 0 || from_state) ? 1u : 0u;
        issue_pv<D>(tO0, tS0, dVs, acc);
        const bool more = it + 1 < n_iter;
        uint64_t dKs = 0;
        int sK = 0;
        if (more) {
          sK = cons % L::kStages;
          if (!wait1(bars.kv_full(sK), static_cast<uint32_t>((cons / L::kStages) & 1), ab)) {
            ok = false;
            break;
          }
          ++cons;
          tc_fence_after();
          dKs = dK + desc_step(sK * L::kTileBytes);
          issue_qk<D>(tS0, dQ0, dKs);
          mma_commit(bars.s_full(0));
        }
        if (has_t1) {
          if (!wait1(bars.p_full(1), par, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv<D>(tO1, tS1, dVs, acc);
        }
        mma_commit(bars.kv_empty(sV));
        if (more) {
          if (has_t1) {
            issue_qk<D>(tS1, dQ1, dKs);
            mma_commit(bars.s_full(1));
          }
          mma_commit(bars.kv_empty(sK));
        }
      }
      if (ok) {
        mma_commit(bars.o_full(0));
        if (has_t1) mma_commit(bars.o_full(1));
      } else if (n_iter > 0) {
        // Wait for every MMA already issued before TMEM is released.
        mma_commit(bars.drain());
        wait_drain(bars.drain(), 0);
      }
    }
  } else if (warp < kLoadWarp) {
    // ================= softmax warps =================
    setmaxnreg_inc<kRegsSoftmax>();
    const int t = warp / 4;   // query tile
    const int wq = warp % 4;  // TMEM lane quarter of this warp
    if (kCausal) {
      // Step table for the mask, built by the 8 softmax warps together.
      const int nsteps = walk.t1 - walk.t0;
      int4* tab = reinterpret_cast<int4*>(gbase + L::kSteps);
      for (int x = threadIdx.x; x < nsteps; x += 256) tab[x] = step_entry(walk, walk.t0 + x);
      asm volatile("bar.sync 1, 256;" ::: "memory");
    }
    if (t == 0 || has_t1) {
      const int row = wq * 32 + lane;
      const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
      const uint32_t tS = tmem + lane_off + static_cast<uint32_t>(t * 128);
      const uint32_t tO = tmem + lane_off + 256u + static_cast<uint32_t>(t * D);
      const int64_t lrow = lr0 + t * kBM + row;  // local row in query block i
      const int64_t grow = slice * a.nq + walk.pos(i, lrow);  // row of q, out, lse, states
      const float sl2 = a.scale_log2;
      // causal: this thread's place in the step table (query reference,
      // current step and tile within it)
      const int4* steps = reinterpret_cast<const int4*>(gbase + L::kSteps);
      const int qref = kCausal ? static_cast<int>(striped ? lrow : walk.pos(i, lrow)) : 0;
      int ts = 0, tkt = 0;
      if (kCausal && n_iter > 0)
        while (tkt >= steps[ts].x) ++ts;

      float m_ref = -INFINITY;   // reference max of the exponentials (log2 units)
      float m_true = -INFINITY;  // true running max (log2 units)
      float l = 0.f;
      bool o_valid = false;
      if (a.mode == kFold) {
        m_ref = a.st_m[grow] * kLog2e;
        m_true = m_ref;
        l = a.st_l[grow];
        const float4* src = reinterpret_cast<const float4*>(a.st_o + grow * D);
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t r[32];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 x = src[c / 4 + e];
            r[4 * e + 0] = __float_as_uint(x.x);
            r[4 * e + 1] = __float_as_uint(x.y);
            r[4 * e + 2] = __float_as_uint(x.z);
            r[4 * e + 3] = __float_as_uint(x.w);
          }
          tmem_st32(tO + c, r);
        }
        tmem_st_wait();
        o_valid = true;
      }

      bool ok = true;
      for (int it = 0; it < n_iter; ++it) {
        if (kCausal && it > 0) {
          ++tkt;
          while (tkt >= steps[ts].x) {
            ++ts;
            tkt = 0;
          }
        }
        if (!wait_warp(bars.s_full(t), static_cast<uint32_t>(it & 1), ab)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t s[kBN];
#pragma unroll
        for (int c = 0; c < kBN; c += 32) tmem_ld32(tS + c, s + c);
        tmem_ld_wait();
        reg_fence(s, kBN);
        if (kCausal) {
          // keys after the query's own position take no part (score -inf)
          const int4 ent = steps[ts];
          const int half = walk.tiles / 2;
          const int first = tkt < half ? ent.y + tkt * kBN : ent.z + (tkt - half) * kBN;
          int nvis = qref - first + 1;
          nvis = nvis < 0 ? 0 : (nvis > kBN ? kBN : nvis);
          if (__any_sync(0xffffffffu, nvis < kBN)) {
#pragma unroll
            for (int c = 0; c < kBN; ++c)
              if (c >= nvis) s[c] = __float_as_uint(-INFINITY);
          }
        }

        const uint64_t scale2 = pack_f32x2(sl2, sl2);
        // Fast path (the forward, once the reference is set): the row max is
        // needed only to move the reference, which must move when some p
        // against it would exceed 2^kRescaleLog2.  A row sum of p at most
        // kFastSumBound rules that out (every p >= 0), so the exponentials
        // come first and the max is skipped.  If a row's sum is over the
        // bound (rarely: p is mostly well below 1), the warp redoes the tile
        // through the exact path below.  A unit's first tile goes there
        // directly.  Any reference gives the same l and o, so both paths are
        // exact.  The partial and fold modes always take the exact path,
        // since they report the true running max.
        bool redo = true;
        if (a.mode == kForward && __all_sync(0xffffffffu, m_ref != -INFINITY)) {
          const float lt = exp_store(s, scale2, pack_f32x2(-m_ref, -m_ref), tS);
          if (!__any_sync(0xffffffffu, lt > kFastSumBound)) {
            l += lt;
            redo = false;
          } else {
            tmem_st_wait();  // the redo's stores land after these
          }
        }
        if (redo) {
          // Row max: eight independent chains of three-input maxima.
          float mx[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) mx[e] = fmaxf(__uint_as_float(s[e]), __uint_as_float(s[e + 8]));
#pragma unroll
          for (int j = 16; j < kBN; j += 16) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              mx[e] = fmax3(mx[e], __uint_as_float(s[j + e]), __uint_as_float(s[j + 8 + e]));
          }
          const float rmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                   fmaxf(mx[6], mx[7]));
          const float m_new = rmax * sl2;
          m_true = fmaxf(m_true, m_new);
          const bool need = m_new > m_ref + kRescaleLog2;
          if (__any_sync(0xffffffffu, need)) {
            const float alpha = need ? ex2(m_ref - m_new) : 1.f;
            if (o_valid) {
#pragma unroll
              for (int c = 0; c < D; c += 32) {
                uint32_t r[32];
                tmem_ld32(tO + c, r);
                tmem_ld_wait();
                reg_fence(r, 32);
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                tmem_st32(tO + c, r);
              }
              tmem_st_wait();
            }
            if (need) {
              l *= alpha;
              m_ref = m_new;
            }
          }
          // a row that has seen no visible key yet keeps m_ref = -inf; its
          // masked scores must still give p = 0 rather than NaN
          const float neg = (kCausal && m_ref == -INFINITY) ? 0.f : -m_ref;
          l += exp_store(s, scale2, pack_f32x2(neg, neg), tS);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bars.p_full(t));
        o_valid = true;
      }

      if (n_iter == 0) {
        // Nothing of this unit is visible in its segment: an empty state.
        if (a.mode == kPartial) {
          float4* dst = reinterpret_cast<float4*>(a.part.o[g] + grow * D);
#pragma unroll
          for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
          a.part.m[g][grow] = -INFINITY;
          a.part.l[g][grow] = 0.f;
        }
      } else if (ok && wait_warp(bars.o_full(t), 0, ab)) {
        tc_fence_after();
        if (a.mode == kForward) {
          const float inv = 1.f / l;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + grow * D);
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t r[32];
            tmem_ld32(tO + c, r);
            tmem_ld_wait();
            reg_fence(r, 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(r[8 * e + 0]) * inv, __uint_as_float(r[8 * e + 1]) * inv);
              w.y = pack_bf16x2(__uint_as_float(r[8 * e + 2]) * inv, __uint_as_float(r[8 * e + 3]) * inv);
              w.z = pack_bf16x2(__uint_as_float(r[8 * e + 4]) * inv, __uint_as_float(r[8 * e + 5]) * inv);
              w.w = pack_bf16x2(__uint_as_float(r[8 * e + 6]) * inv, __uint_as_float(r[8 * e + 7]) * inv);
              dst[c / 8 + e] = w;
            }
          }
          a.lse[grow] = (m_ref + __log2f(l)) * kLn2;
        } else {
          // Re-express (l, o) relative to the true running max.
          const float fix = m_true == -INFINITY ? 1.f : ex2(m_ref - m_true);
          float* mo = a.mode == kPartial ? a.part.m[g] : a.st_m;
          float* lo = a.mode == kPartial ? a.part.l[g] : a.st_l;
          float* oo = a.mode == kPartial ? a.part.o[g] : a.st_o;
          float4* dst = reinterpret_cast<float4*>(oo + grow * D);
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t r[32];
            tmem_ld32(tO + c, r);
            tmem_ld_wait();
            reg_fence(r, 32);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[c / 4 + e] = make_float4(__uint_as_float(r[4 * e + 0]) * fix,
                                           __uint_as_float(r[4 * e + 1]) * fix,
                                           __uint_as_float(r[4 * e + 2]) * fix,
                                           __uint_as_float(r[4 * e + 3]) * fix);
          }
          mo[grow] = m_true * kLn2;
          lo[grow] = l * fix;
        }
      }
    }
  } else {
    setmaxnreg_dec<kRegsOther>();  // idle warps of the third warpgroup
  }

  // ---- teardown ----
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool kCausal>
cudaError_t launch_d(const FoldArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, cudaStream_t s) {
  using L = Layout<D>;
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(fold_sm103_kernel<D, kCausal>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int64_t cq = a.nq / a.P;
  const int64_t tiles_q = cq / kBM;
  const int64_t pairs = (tiles_q + 1) / 2;
  const int64_t grid = a.slices * a.P * a.G * pairs;
  fold_sm103_kernel<D, kCausal>
      <<<static_cast<unsigned>(grid), kThreads, L::kSmem, s>>>(a, tq, tk, tv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fold_sm103(const FoldArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, cudaStream_t s) {
  if (a.causal) {
    if (a.d == 128) return launch_d<128, true>(a, tq, tk, tv, s);
    if (a.d == 64) return launch_d<64, true>(a, tq, tk, tv, s);
  } else {
    if (a.d == 128) return launch_d<128, false>(a, tq, tk, tv, s);
    if (a.d == 64) return launch_d<64, false>(a, tq, tk, tv, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ra
