// Ring Attention oracle: plain, slow, fp64 CPU reference.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load this
// library; it is used by tests/, by the smoke check and by the CPU-baseline
// leg of the benchmark.  It shares no code, header or constant with the CUDA
// library.
//
// Sources followed (page title, section):
//   [A] "Ring Attention: the math" (aicassindra.com, transformer_math):
//       "The online-softmax identity that makes streaming legal" (running state
//       m, l, o and the per-block update), "The ring schedule: passing K/V
//       around" (block held at step t is (i - t) mod P), "Accumulation math,
//       step by step" (state init, final out = o / l), "A worked numeric
//       example" and "Sharding the sequence" (P contiguous blocks of b = N/P).
//   [B] "Ring Attention" (bembew.net): "Conceptual Algorithm" (the same update
//       per row; read per row, see reading R3 below) and "Global Integration"
//       (partial results merged into one output).
//   [C] "Ring attention, explained" (vibeengines.com): steps 1-4 (shard,
//       local block first, rotate, normalise; equals full attention up to
//       rounding) and "The causal-mask catch" (a query needs only keys at or
//       before it; striped and zigzag assignments of tokens to devices).
//
// Readings where the pages are silent (each also listed in the design notes):
//   R1  lse = m + ln l over the scaled scores tau*q.k (natural log).
//   R2  alpha = exp(m_old - m_new) is 0 when m_old = -inf and m_new is finite
//       (the worked example's first step); when both are -inf the state is
//       empty, alpha is taken as 1 and the block adds nothing.  A merge of
//       empty states gives out = 0, lse = -inf.
//   R3  [B]'s pseudocode writes the update without per-row broadcasting; it is
//       read per query row as in [A].
//   R4  N = tokens, P = devices/blocks, c = N / P ([A], [C]), not [B]'s use of
//       N for the block count.
//   R12 Causal: query at position n sees key positions <= n.  Layouts of the
//       tokens over the P blocks: contiguous (block j = positions j*c ..
//       j*c + c - 1), zigzag (block j = chunk j and chunk 2P-1-j of 2P chunks
//       of c/2 positions, each in increasing order) and striped (block j =
//       positions j, j + P, j + 2P, ...).  A block's keys are folded in this
//       local order; masked keys take no part (as a score of -inf would).
//   R13 Backward: the loss is L = sum(dO * out); P is recomputed from the
//       forward's lse; the row term D = sum(dO * out) ([C] step 6 names the
//       ring and the travelling accumulators, not the formulas, which are the
//       derivative of the forward written out).
//
// Every value is computed in double precision.  Inputs are converted exactly
// (f32 -> f64 and bf16 -> f64 are exact).  No blocking, fusion or reordering
// beyond what the recurrence states.
//
// Compile-time switch ORA_MUTANT (test use only, default 0): each non-zero
// value plants one deliberate mistake so that the tests can show that their
// pins catch it.  The correct build never defines it.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

#ifndef ORA_MUTANT
#define ORA_MUTANT 0
#endif

namespace {

enum { ORA_F64 = 0, ORA_F32 = 1, ORA_BF16 = 2 };
enum { ORA_CONTIGUOUS = 0, ORA_ZIGZAG = 1, ORA_STRIPED = 2 };

const double kNegInf = -std::numeric_limits<double>::infinity();

// bf16 is the upper half of an IEEE binary32; widening is exact.
inline double bf16_to_double(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// Read row `r` (d elements) of a [rows, d] array of the given element type
// into `dst` as doubles.
void load_row(const void* base, int dtype, int64_t r, int d, double* dst) {
  const int64_t off = r * static_cast<int64_t>(d);
  if (dtype == ORA_F64) {
    const double* p = static_cast<const double*>(base) + off;
    for (int e = 0; e < d; ++e) dst[e] = p[e];
  } else if (dtype == ORA_F32) {
    const float* p = static_cast<const float*>(base) + off;
    for (int e = 0; e < d; ++e) dst[e] = static_cast<double>(p[e]);
  } else {
    const uint16_t* p = static_cast<const uint16_t*>(base) + off;
    for (int e = 0; e < d; ++e) dst[e] = bf16_to_double(p[e]);
  }
}

// Run fn(i) for i in [0, n) on `threads` std::threads (contiguous chunks).
template <typename Fn>
void parallel_for(int64_t n, int threads, Fn fn) {
  if (threads < 1) threads = 1;
  if (n < threads) threads = static_cast<int>(n > 0 ? n : 1);
  if (threads == 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  std::vector<std::thread> pool;
  const int64_t chunk = (n + threads - 1) / threads;
  for (int t = 0; t < threads; ++t) {
    const int64_t lo = t * chunk, hi = std::min<int64_t>(n, lo + chunk);
    if (lo >= hi) break;
    pool.emplace_back([lo, hi, &fn]() {
      for (int64_t i = lo; i < hi; ++i) fn(i);
    });
  }
  for (auto& th : pool) th.join();
}

// Running online-softmax state of one query row ([A], "Keep three running
// quantities per query").
struct RowState {
  double m;               // running max of scores
  double l;               // running sum of exp(s - m)
  std::vector<double> o;  // running sum of exp(s - m) * v, length d
};

// One fold of the keys `rows[0..nb)` (row indices of a [*, d] K/V array)
// into `st` for query `q` (already converted to double).  This is the update
// of [A] "For each incoming K/V block":
//   s_j = q . k_j * tau;  m' = max(m, max_j s_j);  alpha = exp(m - m');
//   l' = alpha*l + sum_j exp(s_j - m');  o' = alpha*o + sum_j exp(s_j - m') v_j.
// Causal (R12): when `pos` is given, key j takes part only if pos[j] <= qpos.
void fold_keys(RowState& st, const double* q, int d, double tau,
               const void* k, const void* v, int dtype, const int64_t* rows, int64_t nb,
               const int64_t* pos, int64_t qpos, std::vector<double>& s,
               std::vector<double>& krow, std::vector<double>& vrow) {
  std::vector<int64_t> keep;
  keep.reserve(static_cast<size_t>(nb));
  for (int64_t j = 0; j < nb; ++j) {
#if ORA_MUTANT == 7
    if (!pos || pos[j] < qpos) keep.push_back(rows[j]);  // planted: strict mask
#else
    if (!pos || pos[j] <= qpos) keep.push_back(rows[j]);
#endif
  }
  nb = static_cast<int64_t>(keep.size());
  if (nb == 0) return;  // R2: a fully masked block adds nothing
  s.resize(static_cast<size_t>(nb));
  double bmax = kNegInf;
  for (int64_t j = 0; j < nb; ++j) {
    load_row(k, dtype, keep[j], d, krow.data());
    double dot = 0.0;
    for (int e = 0; e < d; ++e) dot += q[e] * krow[e];
#if ORA_MUTANT == 4
    s[j] = dot / static_cast<double>(d);  // planted: wrong scale 1/d
#else
    s[j] = dot * tau;
#endif
    if (s[j] > bmax) bmax = s[j];
  }
  const double m_new = st.m > bmax ? st.m : bmax;
  // R2: an empty state meeting a block of -inf scores stays empty
  // (alpha = 1, nothing added).
  if (m_new == kNegInf) return;
  const double alpha = std::exp(st.m - m_new);  // exp(-inf) = 0 on the first block
#if ORA_MUTANT == 1
  const double alpha_o = 1.0;  // planted: o not rescaled
#else
  const double alpha_o = alpha;
#endif
#if ORA_MUTANT == 2
  const double alpha_l = 1.0;  // planted: l not rescaled
#else
  const double alpha_l = alpha;
#endif
  double lsum = 0.0;
  for (int e = 0; e < d; ++e) st.o[e] *= alpha_o;
  for (int64_t j = 0; j < nb; ++j) {
#if ORA_MUTANT == 5
    const double p = std::exp(m_new - s[j]);  // planted: sign flip
#else
    const double p = std::exp(s[j] - m_new);
#endif
    lsum += p;
#if ORA_MUTANT == 6
    load_row(k, dtype, keep[j], d, vrow.data());  // planted: K used as V
#else
    load_row(v, dtype, keep[j], d, vrow.data());
#endif
    for (int e = 0; e < d; ++e) st.o[e] += p * vrow[e];
  }
  st.l = alpha_l * st.l + lsum;
  st.m = m_new;
}

// Block visited by query block i at ring step t: [A] "On step t, device i
// holds the K/V block from device (i - t) mod P".
inline int64_t ring_block(int64_t i, int64_t t, int64_t P) {
  int64_t j = (i - t) % P;
  if (j < 0) j += P;
  return j;
}

// Position of local row r of block j (R12; [A] "Sharding the sequence" for
// the contiguous split, [C] "The causal-mask catch" for zigzag and striped).
inline int64_t token_pos(int layout, int64_t j, int64_t r, int64_t P, int64_t c) {
  if (layout == ORA_ZIGZAG) {
    const int64_t h = c / 2;
    return r < h ? j * h + r : (2 * P - 1 - j) * h + (r - h);
  }
  if (layout == ORA_STRIPED) return j + P * r;
  return j * c + r;
}

// Block holding position n (inverse of token_pos).
inline int64_t block_of(int layout, int64_t n, int64_t P, int64_t c) {
  if (layout == ORA_ZIGZAG) {
    const int64_t chunk = n / (c / 2);
    return chunk < P ? chunk : 2 * P - 1 - chunk;
  }
  if (layout == ORA_STRIPED) return n % P;
  return n / c;
}

// Final normalisation out = o / l ([A] "After the final block") and R1.
void finish_row(const RowState& st, int d, double* out, double* lse) {
  for (int e = 0; e < d; ++e) out[e] = st.l > 0.0 ? st.o[e] / st.l : 0.0;
  *lse = st.l > 0.0 ? st.m + std::log(st.l) : kNegInf;
}

bool bad_dtype(int dtype) {
  return dtype != ORA_F64 && dtype != ORA_F32 && dtype != ORA_BF16;
}

}  // namespace

extern "C" {

// Visiting order of the ring: writes order[i*P + t] = block held by query
// block i at step t, for i, t in [0, P).
int ora_ring_order(int64_t P, int64_t* order) {
  if (P < 1 || !order) return 1;
  for (int64_t i = 0; i < P; ++i)
    for (int64_t t = 0; t < P; ++t) order[i * P + t] = ring_block(i, t, P);
  return 0;
}

// Dense softmax attention (the exact result the ring equals; [A] "Why one
// device runs out of room": S = QK^T / sqrt(d_k), and the softmax identity).
//   q, k, v: [BH, N, d] of `dtype`.
//   rows: R flat indices into [BH*N] (NULL means every row, R = BH*N).
//   causal != 0: the query at position n sees keys 0 .. n only (R12).
//   out: [R, d] doubles; lse: [R] doubles.
// For each row: s_j = tau q.k_j over its (b,h)'s visible keys; M = max s;
// L = sum exp(s - M); out = sum exp(s - M) v / L; lse = M + ln L.
int ora_dense(const void* q, const void* k, const void* v, int dtype, int64_t BH,
              int64_t N, int d, int causal, const int64_t* rows, int64_t R, double* out,
              double* lse, int threads) {
  if (!q || !k || !v || !out || !lse || BH < 0 || N < 0 || d < 1 || bad_dtype(dtype))
    return 1;
  if (!rows) R = BH * N;
  const double tau = 1.0 / std::sqrt(static_cast<double>(d));
  parallel_for(R, threads, [&](int64_t ri) {
    const int64_t r = rows ? rows[ri] : ri;
    const int64_t bh = r / N;
    const int64_t nk = causal ? r % N + 1 : N;  // visible keys 0 .. nk-1
    std::vector<double> qrow(d), krow(d), vrow(d), s(static_cast<size_t>(N));
    load_row(q, dtype, r, d, qrow.data());
    double M = kNegInf;
    for (int64_t j = 0; j < nk; ++j) {
      load_row(k, dtype, bh * N + j, d, krow.data());
      double dot = 0.0;
      for (int e = 0; e < d; ++e) dot += qrow[e] * krow[e];
      s[j] = dot * tau;
      if (s[j] > M) M = s[j];
    }
    double L = 0.0;
    std::vector<double> acc(d, 0.0);
    for (int64_t j = 0; j < nk; ++j) {
      const double p = std::exp(s[j] - M);
      L += p;
      load_row(v, dtype, bh * N + j, d, vrow.data());
      for (int e = 0; e < d; ++e) acc[e] += p * vrow[e];
    }
    for (int e = 0; e < d; ++e) out[ri * d + e] = acc[e] / L;
    lse[ri] = M + std::log(L);
  });
  return 0;
}

// Ring-order recurrence ([A] "Accumulation math, step by step").
//   P blocks of c = N / P rows; `layout` (R12) says which positions form a
//   block (0 contiguous, 1 zigzag, 2 striped); query position n lives in block
//   i = block_of(n).  Steps t in [t0, t1) are folded, visiting block
//   order[i*P + t] (NULL means the ring order (i - t) mod P).  t0 = 0, t1 = P
//   is the whole ring.
//   tile > 0 folds each visiting block in consecutive chunks of `tile` keys
//   (local order) instead of whole (exact by the same identity).
//   causal != 0 masks keys at positions after the query (R12).
//   The state starts at (m = -inf, l = 0, o = 0).
//   Outputs (any may be NULL): out [R, d] = o / l, lse [R] = m + ln l, and the
//   raw final state m_out [R], l_out [R], o_out [R, d].
int ora_ring(const void* q, const void* k, const void* v, int dtype, int64_t BH,
             int64_t N, int d, int64_t P, const int64_t* order, int64_t t0,
             int64_t t1, int64_t tile, int causal, int layout, const int64_t* rows,
             int64_t R, double* out, double* lse, double* m_out, double* l_out,
             double* o_out, int threads) {
  if (!q || !k || !v || BH < 0 || N < 0 || d < 1 || P < 1 || bad_dtype(dtype)) return 1;
  if (layout < ORA_CONTIGUOUS || layout > ORA_STRIPED) return 1;
  if (N % P != 0) return 2;
  if (layout == ORA_ZIGZAG && (N / P) % 2 != 0) return 2;
  if (t0 < 0 || t1 > P || t0 > t1 || tile < 0) return 1;
  if (!rows) R = BH * N;
  const int64_t c = N / P;
  const double tau = 1.0 / std::sqrt(static_cast<double>(d));
  parallel_for(R, threads, [&](int64_t ri) {
    const int64_t r = rows ? rows[ri] : ri;
    const int64_t bh = r / N, n = r % N, i = block_of(layout, n, P, c);
    std::vector<double> qrow(d), krow(d), vrow(d), s;
    std::vector<int64_t> krows(static_cast<size_t>(c)), kpos(static_cast<size_t>(c));
    load_row(q, dtype, r, d, qrow.data());
    RowState st{kNegInf, 0.0, std::vector<double>(d, 0.0)};
    const int64_t* mask = causal ? kpos.data() : nullptr;
#if ORA_MUTANT == 3
    // planted: [A]'s warning -- normalise each block, then average them.
    std::vector<double> avg(d, 0.0);
    int64_t nblk = 0;
#endif
    for (int64_t t = t0; t < t1; ++t) {
      const int64_t j = order ? order[i * P + t] : ring_block(i, t, P);
      for (int64_t x = 0; x < c; ++x) {
        kpos[x] = token_pos(layout, j, x, P, c);
        krows[x] = bh * N + kpos[x];
      }
#if ORA_MUTANT == 3
      RowState b{kNegInf, 0.0, std::vector<double>(d, 0.0)};
      fold_keys(b, qrow.data(), d, tau, k, v, dtype, krows.data(), c, mask, n, s, krow, vrow);
      if (b.l > 0.0) {
        for (int e = 0; e < d; ++e) avg[e] += b.o[e] / b.l;
        ++nblk;
      }
      fold_keys(st, qrow.data(), d, tau, k, v, dtype, krows.data(), c, mask, n, s, krow, vrow);
#else
      const int64_t step = tile == 0 ? c : tile;
      for (int64_t x0 = 0; x0 < c; x0 += step) {
        const int64_t nb = x0 + step < c ? step : c - x0;
        fold_keys(st, qrow.data(), d, tau, k, v, dtype, krows.data() + x0, nb,
                  mask ? mask + x0 : nullptr, n, s, krow, vrow);
      }
#endif
    }
#if ORA_MUTANT == 3
    if (nblk > 0) {
      for (int e = 0; e < d; ++e) st.o[e] = avg[e] / nblk * st.l;
    }
#endif
    if (out && lse) finish_row(st, d, out + ri * d, lse + ri);
    if (m_out) m_out[ri] = st.m;
    if (l_out) l_out[ri] = st.l;
    if (o_out)
      for (int e = 0; e < d; ++e) o_out[ri * d + e] = st.o[e];
  });
  return 0;
}

// Positions held by each block under a layout (R12): pos[j*c + r] = position
// of local row r of block j.
int ora_layout_positions(int layout, int64_t P, int64_t c, int64_t* pos) {
  if (!pos || P < 1 || c < 0 || layout < ORA_CONTIGUOUS || layout > ORA_STRIPED) return 1;
  if (layout == ORA_ZIGZAG && c % 2 != 0) return 2;
  for (int64_t j = 0; j < P; ++j)
    for (int64_t r = 0; r < c; ++r) pos[j * c + r] = token_pos(layout, j, r, P, c);
  return 0;
}

// One fold of a visiting block into a caller-held state, in place.
//   m, l: [R]; o: [R, d] (doubles).  R = batch * rows_per_batch.
//   q: [batch, R/batch, d]; kb, vb: [batch, Nk, d] of `dtype`.
// This is a single application of the update of [A] (one "incoming K/V
// block"), whole block at once.
int ora_fold(double* m, double* l, double* o, const void* q, const void* kb,
             const void* vb, int dtype, int64_t batch, int64_t R, int64_t Nk, int d,
             int threads) {
  if (!m || !l || !o || !q || !kb || !vb || batch < 1 || R < 0 || Nk < 0 || d < 1 ||
      bad_dtype(dtype))
    return 1;
  if (R % batch != 0) return 2;
  const int64_t rpb = R / batch;
  const double tau = 1.0 / std::sqrt(static_cast<double>(d));
  parallel_for(R, threads, [&](int64_t r) {
    const int64_t b = rpb > 0 ? r / rpb : 0;
    std::vector<double> qrow(d), krow(d), vrow(d), s;
    load_row(q, dtype, r, d, qrow.data());
    RowState st{m[r], l[r], std::vector<double>(o + r * d, o + (r + 1) * d)};
    std::vector<int64_t> krows(static_cast<size_t>(Nk));
    for (int64_t x = 0; x < Nk; ++x) krows[x] = b * Nk + x;
    fold_keys(st, qrow.data(), d, tau, kb, vb, dtype, krows.data(), Nk, nullptr, 0, s, krow,
              vrow);
    m[r] = st.m;
    l[r] = st.l;
    for (int e = 0; e < d; ++e) o[r * d + e] = st.o[e];
  });
  return 0;
}

// Merge of G partial states into one ([B] "Global Integration").  Each partial
// g holds (m_g, l_g, o_g) with l_g = sum exp(s - m_g) and o_g = sum exp(s -
// m_g) v over its own keys; by the shift invariance of [A]'s identity:
//   m* = max_g m_g;  w_g = exp(m_g - m*);  l* = sum w_g l_g;  o* = sum w_g o_g;
//   out = o* / l*;  lse = m* + ln l*.
//   m, l: [G, R]; o: [G, R, d].  Outputs out [R, d], lse [R] and optionally the
//   merged state (m_out, l_out, o_out; any may be NULL).
int ora_merge(const double* m, const double* l, const double* o, int64_t G, int64_t R,
              int d, double* out, double* lse, double* m_out, double* l_out,
              double* o_out) {
  if (!m || !l || !o || G < 1 || R < 0 || d < 1) return 1;
  for (int64_t r = 0; r < R; ++r) {
    double ms = kNegInf;
    for (int64_t g = 0; g < G; ++g)
      if (m[g * R + r] > ms) ms = m[g * R + r];
    RowState st{ms, 0.0, std::vector<double>(d, 0.0)};
    if (ms != kNegInf) {
      for (int64_t g = 0; g < G; ++g) {
        const double w = std::exp(m[g * R + r] - ms);  // 0 for an empty partial
        st.l += w * l[g * R + r];
        for (int e = 0; e < d; ++e) st.o[e] += w * o[(g * R + r) * d + e];
      }
    }
    if (out && lse) finish_row(st, d, out + r * d, lse + r);
    if (m_out) m_out[r] = st.m;
    if (l_out) l_out[r] = st.l;
    if (o_out)
      for (int e = 0; e < d; ++e) o_out[r * d + e] = st.o[e];
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Backward pass ([C] step 6: "Run the backward pass on the same ring": the
// key-value blocks travel with their gradient accumulators).  For the loss
// L = sum(dO * out), with P = softmax(tau Q K^T) per row:
//   dV = P^T dO;  dP = dO V^T;  D_r = sum_e dO_re * out_re (= sum_j P_rj dP_rj);
//   dS = P * (dP - D);  dQ = tau dS K;  dK = tau dS^T Q.
// P is recomputed from the forward's lse: P_rj = exp(tau q_r . k_j - lse_r).
// ---------------------------------------------------------------------------

// Ring-order backward of one (b, h) slice, fp64.  Query block i (device i)
// keeps Q_i, dO_i, out_i, lse_i and its dQ_i; at step t it holds key block
// j = (i - t) mod P together with that block's dK_j, dV_j accumulators and
// adds the contributions of the pair (i, j).  Inputs are converted to fp64;
// lse and out are the forward's (any precision, given as doubles).
static void backward_slice(const std::vector<double>& q, const std::vector<double>& k,
                           const std::vector<double>& v, const std::vector<double>& out,
                           const std::vector<double>& dout, const std::vector<double>& lse,
                           int64_t N, int d, int64_t P, int causal, int layout,
                           std::vector<double>& dq, std::vector<double>& dk,
                           std::vector<double>& dv) {
  const double tau = 1.0 / std::sqrt(static_cast<double>(d));
  const int64_t c = N / P;
  std::vector<double> D(static_cast<size_t>(N));
  for (int64_t r = 0; r < N; ++r) {
    double acc = 0.0;
    for (int e = 0; e < d; ++e) acc += dout[r * d + e] * out[r * d + e];
    D[r] = acc;
  }
  for (int64_t i = 0; i < P; ++i) {
    for (int64_t t = 0; t < P; ++t) {
      const int64_t j = ring_block(i, t, P);
      for (int64_t x = 0; x < c; ++x) {
        const int64_t r = token_pos(layout, i, x, P, c);  // query position
        for (int64_t y = 0; y < c; ++y) {
          const int64_t n = token_pos(layout, j, y, P, c);  // key position
#if ORA_MUTANT == 7
          if (causal && n >= r) continue;
#else
          if (causal && n > r) continue;
#endif
          double s = 0.0;
          for (int e = 0; e < d; ++e) s += q[r * d + e] * k[n * d + e];
          const double p = std::exp(s * tau - lse[r]);
          double dp = 0.0;
          for (int e = 0; e < d; ++e) dp += dout[r * d + e] * v[n * d + e];
#if ORA_MUTANT == 8
          const double ds = p * dp;  // planted: the row term D dropped
#else
          const double ds = p * (dp - D[r]);
#endif
          for (int e = 0; e < d; ++e) {
            dq[r * d + e] += tau * ds * k[n * d + e];
            dk[n * d + e] += tau * ds * q[r * d + e];
            dv[n * d + e] += p * dout[r * d + e];
          }
        }
      }
    }
  }
}

// Backward of ring attention for every (b, h) slice (threads over slices).
//   q, k, v: [BH, N, d] of `dtype`; out, dout: [BH, N, d] doubles; lse: [BH*N]
//   doubles (the forward's outputs and the incoming gradient).
//   dq, dk, dv: [BH, N, d] doubles (written).
int ora_backward(const void* q, const void* k, const void* v, int dtype, const double* out,
                 const double* dout, const double* lse, int64_t BH, int64_t N, int d, int64_t P,
                 int causal, int layout, double* dq, double* dk, double* dv, int threads) {
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) return 1;
  if (BH < 0 || N < 0 || d < 1 || P < 1 || bad_dtype(dtype)) return 1;
  if (layout < ORA_CONTIGUOUS || layout > ORA_STRIPED) return 1;
  if (N % P != 0 || (layout == ORA_ZIGZAG && (N / P) % 2 != 0)) return 2;
  parallel_for(BH, threads, [&](int64_t bh) {
    const size_t sz = static_cast<size_t>(N) * d;
    std::vector<double> qs(sz), ks(sz), vs(sz), os(sz), dos(sz), ls(static_cast<size_t>(N));
    std::vector<double> gq(sz, 0.0), gk(sz, 0.0), gv(sz, 0.0);
    for (int64_t r = 0; r < N; ++r) {
      load_row(q, dtype, bh * N + r, d, qs.data() + r * d);
      load_row(k, dtype, bh * N + r, d, ks.data() + r * d);
      load_row(v, dtype, bh * N + r, d, vs.data() + r * d);
      ls[r] = lse[bh * N + r];
    }
    for (size_t x = 0; x < sz; ++x) {
      os[x] = out[bh * sz + x];
      dos[x] = dout[bh * sz + x];
    }
    backward_slice(qs, ks, vs, os, dos, ls, N, d, P, causal, layout, gq, gk, gv);
    for (size_t x = 0; x < sz; ++x) {
      dq[bh * sz + x] = gq[x];
      dk[bh * sz + x] = gk[x];
      dv[bh * sz + x] = gv[x];
    }
  });
  return 0;
}

// Gradient rows of the backward, for sampled rows of large problems: the same
// formulas as ora_backward, organised per output row (causal: R12 mask).
//   qrows[Rq]: flat rows whose dQ is wanted (dq [Rq, d]);
//   krows[Rk]: flat rows whose dK and dV are wanted (dk, dv [Rk, d]).
//   out, dout: [BH, N, d] of `dtype` (the forward's output and the incoming
//   gradient); lse: [BH*N] doubles.
int ora_backward_rows(const void* q, const void* k, const void* v, int dtype, const void* out,
                      const void* dout, const double* lse, int64_t BH, int64_t N, int d,
                      int causal, const int64_t* qrows, int64_t Rq, double* dq,
                      const int64_t* krows, int64_t Rk, double* dk, double* dv, int threads) {
  if (!q || !k || !v || !out || !dout || !lse || BH < 0 || N < 1 || d < 1 || bad_dtype(dtype))
    return 1;
  if ((Rq > 0 && (!qrows || !dq)) || (Rk > 0 && (!krows || !dk || !dv))) return 1;
  const double tau = 1.0 / std::sqrt(static_cast<double>(d));
  auto row_D = [&](int64_t r, std::vector<double>& a, std::vector<double>& b) {
    load_row(out, dtype, r, d, a.data());
    load_row(dout, dtype, r, d, b.data());
    double acc = 0.0;
    for (int e = 0; e < d; ++e) acc += a[e] * b[e];
    return acc;
  };
  parallel_for(Rq + Rk, threads, [&](int64_t x) {
    std::vector<double> qa(d), ga(d), ka(d), va(d), oa(d), acc1(d, 0.0), acc2(d, 0.0);
    if (x < Rq) {
      const int64_t r = qrows[x], bh = r / N;
      const double D = row_D(r, oa, ga);  // ga = dout_r
      load_row(q, dtype, r, d, qa.data());
      const int64_t nk = causal ? r - bh * N + 1 : N;  // keys at or before the query (R12)
      for (int64_t j = 0; j < nk; ++j) {
        load_row(k, dtype, bh * N + j, d, ka.data());
        load_row(v, dtype, bh * N + j, d, va.data());
        double s = 0.0, dp = 0.0;
        for (int e = 0; e < d; ++e) {
          s += qa[e] * ka[e];
          dp += ga[e] * va[e];
        }
        const double ds = std::exp(s * tau - lse[r]) * (dp - D);
        for (int e = 0; e < d; ++e) acc1[e] += tau * ds * ka[e];
      }
      for (int e = 0; e < d; ++e) dq[x * d + e] = acc1[e];
    } else {
      const int64_t xi = x - Rq, n = krows[xi], bh = n / N;
      load_row(k, dtype, n, d, ka.data());
      load_row(v, dtype, n, d, va.data());
      for (int64_t r = causal ? n : bh * N; r < (bh + 1) * N; ++r) {  // queries that see n
        const double D = row_D(r, oa, ga);  // ga = dout_r
        load_row(q, dtype, r, d, qa.data());
        double s = 0.0, dp = 0.0;
        for (int e = 0; e < d; ++e) {
          s += qa[e] * ka[e];
          dp += ga[e] * va[e];
        }
        const double p = std::exp(s * tau - lse[r]);
        const double ds = p * (dp - D);
        for (int e = 0; e < d; ++e) {
          acc1[e] += tau * ds * qa[e];
          acc2[e] += p * ga[e];
        }
      }
      for (int e = 0; e < d; ++e) {
        dk[xi * d + e] = acc1[e];
        dv[xi * d + e] = acc2[e];
      }
    }
  });
  return 0;
}

// Build marker: lets a test confirm which variant it loaded.
int ora_mutant(void) { return ORA_MUTANT; }

}  // extern "C"
