// Internal interface between the C ABI layer (ra_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ra.h"

namespace ra {

// What a fold launch does with its state.
enum Mode : int32_t {
  kForward = 0,  // empty state, all P ring steps, write out = o / l and lse
  kPartial = 1,  // empty state, one segment of ring steps, write (m, l, o)
  kFold = 2,     // load (m, l, o), fold one block, write (m, l, o) back
};

// How the tokens of a slice are dealt to the P blocks (causal load balance).
enum Layout : int32_t {
  kContiguous = 0,  // block j = positions j*c .. j*c + c - 1
  kZigzag = 1,      // block j = chunks j and 2P-1-j of 2P chunks of c/2 positions
  kStriped = 2,     // block j = positions j, j + P, j + 2P, ...
};

// Per-segment partial-state pointers (device).
struct PartialPtrs {
  float* m[RA_MAX_PARTIALS];
  float* l[RA_MAX_PARTIALS];
  float* o[RA_MAX_PARTIALS];
};

// Everything a fold kernel needs besides the TMA descriptors.
//
// The work is `slices` independent problems (B*H heads, or the batch of a
// fold call).  Slice s has nq query rows and nk key rows, each cut into P
// contiguous blocks (cq = nq / P, ck = nk / P).  Query block i visits key
// block (i - t) mod P at ring step t.  In partial mode the P steps are split
// into G contiguous segments; in fold mode P = G = 1.  Tensors are in token
// order; `layout` says which positions form block j (the rows a query block
// holds and the key rows a ring step brings), `causal` masks later keys.
struct FoldArgs {
  const void* q;  // [slices, nq, d]
  const void* k;  // [slices, nk, d]
  const void* v;  // [slices, nk, d]
  int64_t slices;
  int64_t nq;
  int64_t nk;
  int32_t d;
  int32_t P;
  int32_t G;
  int32_t mode;
  int32_t causal;    // 1: a query sees key positions <= its own
  int32_t layout;    // Layout of the tokens over the blocks
  float tau;         // 1 / sqrt(d)
  float scale_log2;  // tau * log2(e)
  void* out;         // forward: [slices, nq, d] (input dtype)
  float* lse;        // forward: [slices, nq]
  float* st_m;       // fold: state in/out
  float* st_l;
  float* st_o;
  int* status;       // device watchdog word (0 = fine)
  int64_t wait_limit;  // SM cycles a bounded wait may take (tensor path)
  int64_t stall_cta;   // test aid: this CTA of the tensor path loads nothing (-1: none)
  PartialPtrs part;  // partial mode
};

// Everything a backward launch needs besides the TMA descriptors.  Tensors
// are [slices, N, d] in token order; lse and delta are [slices * N].
struct BackwardArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* dout;
  const float* lse;    // the forward's log-sum-exp (natural log, scaled scores)
  const float* nl;     // -lse * log2(e) (tensor path)
  const float* delta;  // D = rowsum(dout * out)
  void* dq;
  void* dk;
  void* dv;
  int64_t slices;
  int64_t N;
  int32_t d;
  int32_t P;
  int32_t causal;    // 1: a query sees key positions <= its own
  int32_t layout;    // Layout of the tokens over the blocks
  float tau;         // 1 / sqrt(d)
  float scale_log2;  // tau * log2(e)
  int* status;       // device watchdog word
  int64_t wait_limit;  // SM cycles a bounded wait may take
  int64_t stall_cta;   // test aid: this CTA of each tensor-core kernel loads nothing (-1: none)
  int32_t accumulate;  // 1: dq, dk, dv are fp32 accumulators; add instead of store
};

struct MergeArgs {
  PartialPtrs part;
  int32_t G;
  int64_t rows;
  int32_t d;
  void* out;
  float* lse;
  int32_t out_bf16;
  int32_t vec4;  // o rows and out allow 16-byte (f32) / 8-byte (bf16) vector access
};

// Launchers (each returns the launch's cudaError_t).
cudaError_t launch_fold_sm103(const FoldArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, cudaStream_t s);
cudaError_t launch_fold_f32(const FoldArgs& a, cudaStream_t s);
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t s);
// D = rowsum(dout * out) and nl = -lse * log2(e) per query row, stored
// block-major: (slice, block, local row) under `layout` (P blocks).
cudaError_t launch_delta(const void* out, const void* dout, const float* lse, float* delta,
                         float* nl, int64_t rows, int32_t d, int64_t N, int32_t P,
                         int32_t layout, bool bf16, cudaStream_t s);
cudaError_t launch_backward_f32(const BackwardArgs& a, cudaStream_t s);
cudaError_t launch_backward_sm103(const BackwardArgs& a, const CUtensorMap& tq,
                                  const CUtensorMap& tk, const CUtensorMap& tv,
                                  const CUtensorMap& tdo, cudaStream_t s);
cudaError_t launch_state_init(float* m, float* l, float* o, int64_t rows, int32_t d,
                              cudaStream_t s);

// Largest P of the causal tensor-core path: the softmax warps keep one
// 16-byte entry per ring step of a work unit in shared memory.
constexpr int kMaxCausalSteps = 1024;

// Watchdog codes written to FoldArgs::status.
constexpr int kStatusTimeout = 1;

// Number of SMs of the current device (cached).
int device_sm_count();

// Devices the library keeps per-device state for (ordinals 0 .. kMaxDevices-1).
constexpr int kMaxDevices = 64;

// Ordinal of the current device: RA_ERR_ARCH when there is no usable device
// or driver, RA_ERR_CUDA for another failure of the lookup,
// RA_ERR_UNSUPPORTED for an ordinal of kMaxDevices or more.
ra_status current_ordinal(int* dev);

// The argument and size checks of ra_forward / ra_forward_causal, without
// the buffers: the status those calls would return for a valid set of
// buffers.
ra_status check_forward_args(int32_t B, int32_t H, int64_t N, int32_t d, int32_t P, bool causal,
                             ra_layout layout, ra_dtype dtype);

// Bytes of scratch for G partial states of `rows` rows of width d: per
// segment m [rows], l [rows], o [rows, d] fp32, each 256-byte aligned.
int64_t split_workspace_bytes(int64_t rows, int32_t d, int32_t G);

// The split forward: fold G segments of the ring into partial states held in
// `workspace`, then merge them into out and lse (all on `stream`).
ra_status split_forward(const void* q, const void* k, const void* v, void* out, float* lse,
                        int32_t B, int32_t H, int64_t N, int32_t d, int32_t P, int32_t G,
                        void* workspace, int64_t workspace_bytes, ra_dtype dtype,
                        cudaStream_t stream);

}  // namespace ra
