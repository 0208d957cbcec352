/*
 * ra.h -- C ABI of the GB300 (sm_103a) Ring Attention fold library.
 *
 * The library computes exact softmax attention the way Ring Attention does:
 * the sequence of N tokens is cut into P contiguous blocks of c = N / P tokens
 * ("Ring Attention: the math", section "Sharding the sequence"); query block i
 * visits the K/V blocks in ring order j = (i - t) mod P for t = 0 .. P-1
 * (section "The ring schedule: passing K/V around") and folds each visiting
 * block into a running per-row state (m, l, o) (section "The online-softmax
 * identity that makes streaming legal"):
 *
 *     s_j = tau * q . k_j,   tau = 1 / sqrt(d)
 *     m'  = max(m, max_j s_j)
 *     l'  = exp(m - m') * l + sum_j exp(s_j - m')
 *     o'  = exp(m - m') * o + sum_j exp(s_j - m') * v_j
 *
 * and finishes with out = o / l (section "Accumulation math, step by step").
 * lse = m + ln l is also returned (natural log, scaled scores).
 *
 * The ring is virtual: one GPU holds every block and the neighbour exchange of
 * the pages becomes double-buffered on-chip staging.
 *
 * Conventions shared by every call
 *   - All data pointers are DEVICE pointers owned by the caller.  The library
 *     allocates no device memory; it never frees caller memory.
 *   - Tensors are dense and row-major.  Attention tensors use [B, H, N, d]
 *     with d contiguous (the element at (b, h, n, e) is at ((b*H + h)*N + n)*d
 *     + e).
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream).  A
 *     returned RA_OK means the work was validated and enqueued.  Kernel
 *     faults surface through the CUDA runtime as usual; a bounded-wait
 *     watchdog inside the kernels is reported by ra_last_device_status().
 *     The backward calls run their two independent kernels side by side:
 *     one on `stream`, one on a library-owned stream forked from `stream`
 *     by an event and joined back into it by another before the call
 *     returns, so work enqueued on `stream` afterwards sees both (and
 *     under CUDA-graph capture the pair becomes two branches).
 *   - Arguments are validated before anything is enqueued; on any error the
 *     call returns the status and launches nothing.  No call throws.
 *   - Calls whose total row count is zero return RA_OK and launch nothing;
 *     their data pointers may then be NULL (an empty tensor's address).
 *   - Element types: RA_BF16 inputs run on the tensor cores (tcgen05, fp32
 *     accumulation) and need d in {64, 128}, c % 128 == 0 and 16-byte aligned
 *     q, k, v and out.  RA_F32 inputs run on the fp32 FFMA path (no TF32) for
 *     any 1 <= d <= 256 and any c >= 1; pointers must be 4-byte aligned.
 *   - The device must be compute capability 10.3 (GB300); others give
 *     RA_ERR_ARCH.
 */
#ifndef RA_H_
#define RA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define RA_API __attribute__((visibility("default")))
#else
#define RA_API
#endif

/* cudaStream_t without including the CUDA headers (same type). */
typedef struct CUstream_st* ra_stream_t;

typedef enum ra_status {
  RA_OK = 0,
  RA_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum          */
  RA_ERR_UNSUPPORTED = 2, /* valid but not handled: P does not divide N, ... */
  RA_ERR_MISALIGNED = 3,  /* pointer alignment below what the path needs    */
  RA_ERR_ARCH = 4,        /* no CUDA device, or not compute capability 10.3  */
  RA_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed               */
  RA_ERR_TIMEOUT = 6      /* a kernel's bounded wait ran out (watchdog)      */
} ra_status;

typedef enum ra_dtype { RA_F32 = 0, RA_BF16 = 1 } ra_dtype;

/*
 * How the N tokens of a (b, h) slice are dealt to the P ring blocks ("Ring
 * attention, explained", section "The causal-mask catch"; the contiguous
 * split is "Ring Attention: the math", section "Sharding the sequence").
 * Tensors stay in token order; the layout only decides which positions form
 * block j, hence which keys each ring step brings and how the causal work is
 * spread over the blocks:
 *   RA_LAYOUT_CONTIGUOUS  block j = positions j*c .. j*c + c - 1
 *   RA_LAYOUT_ZIGZAG      block j = chunks j and 2P-1-j of 2P chunks of c/2
 *                         positions (equal causal work per block)
 *   RA_LAYOUT_STRIPED     block j = positions j, j + P, j + 2P, ...
 */
typedef enum ra_layout {
  RA_LAYOUT_CONTIGUOUS = 0,
  RA_LAYOUT_ZIGZAG = 1,
  RA_LAYOUT_STRIPED = 2
} ra_layout;

/* Largest number of partial states ra_forward_partial / ra_merge accept. */
#define RA_MAX_PARTIALS 64

/*
 * Running online-softmax state of `rows` query rows (section "The
 * online-softmax identity that makes streaming legal": "Keep three running
 * quantities per query").  Device pointers, fp32, caller-owned:
 *   m[rows]     running max of the scaled scores (-inf when empty)
 *   l[rows]     running sum of exp(s - m)
 *   o[rows, d]  running sum of exp(s - m) * v, unnormalised
 * m is always the true running max of the scores folded so far, so a state
 * written by the library is exactly the pages' (m, l, o).
 */
typedef struct ra_state {
  float* m;
  float* l;
  float* o;
  int64_t rows;
  int32_t d;
} ra_state;

/*
 * ra_forward -- full ring attention forward.
 * Pages: "Ring Attention: the math", section "Accumulation math, step by step"
 * (per-device loop over t, out = o / l) run for every query block i; ring
 * order from section "The ring schedule: passing K/V around".
 *   q, k, v  [B, H, N, d] of `dtype`.
 *   out      [B, H, N, d] of `dtype` (bf16 rounded to nearest even).
 *   lse      [B, H, N] fp32, natural log over scaled scores; may not be NULL.
 *   P        ring blocks; must divide N (else RA_ERR_UNSUPPORTED).
 * Errors: RA_ERR_INVALID_ARG (null pointer, B/H/N < 0, d < 1, P < 1, bad
 * dtype), RA_ERR_UNSUPPORTED (N % P != 0; bf16 with d not in {64, 128} or
 * c % 128 != 0; f32 with d > 256), RA_ERR_MISALIGNED, RA_ERR_ARCH, RA_ERR_CUDA.
 */
RA_API ra_status ra_forward(const void* q, const void* k, const void* v, void* out,
                            float* lse, int32_t B, int32_t H, int64_t N, int32_t d,
                            int32_t P, ra_dtype dtype, ra_stream_t stream);

/*
 * ra_forward_causal -- ring attention forward under the causal mask: the
 * query at position n attends to key positions 0 .. n only ("Ring Attention:
 * the math", section "Causal masking, load balance, and other wrinkles";
 * "Ring attention, explained", section "The causal-mask catch").  Query block
 * i visits the blocks in ring order (i - t) mod P as ra_forward does; K/V
 * tiles that hold no visible key are skipped, the others are masked per key.
 *   layout   which positions form each block (see ra_layout).
 * Other arguments as ra_forward.  Extra rules: zigzag needs c even (bf16:
 * c % 256 == 0); the bf16 path needs P <= 1024.
 * Errors: as ra_forward, and RA_ERR_INVALID_ARG for an unknown layout.
 */
RA_API ra_status ra_forward_causal(const void* q, const void* k, const void* v, void* out,
                                   float* lse, int32_t B, int32_t H, int64_t N, int32_t d,
                                   int32_t P, ra_layout layout, ra_dtype dtype,
                                   ra_stream_t stream);

/*
 * ra_forward_partial -- the ring split into G contiguous segments of steps.
 * Partial g folds steps t in [floor(g*P/G), floor((g+1)*P/G)) of every query
 * block's ring order from an empty state and writes its (m, l, o) to
 * partials[g] (no normalisation).  ra_merge of the G partials gives the same
 * out/lse as ra_forward.  This is the "Global Integration" of partial results
 * in "Ring Attention" (bembew.net), section "The Step-by-Step Process".
 *   partials  host array of G ra_state, each with rows = B*H*N and d = d;
 *             their m/l/o are device buffers (o must be 16-byte aligned on
 *             the bf16 path).
 *   1 <= G <= min(P, RA_MAX_PARTIALS).
 * Other arguments and errors as ra_forward.
 */
RA_API ra_status ra_forward_partial(const void* q, const void* k, const void* v,
                                    int32_t B, int32_t H, int64_t N, int32_t d, int32_t P,
                                    int32_t G, const ra_state* partials, ra_dtype dtype,
                                    ra_stream_t stream);

/*
 * ra_forward_partial_causal -- ra_forward_partial under the causal mask and
 * a layout (see ra_forward_causal).  A row that sees no visible key in a
 * segment gets an empty partial (m = -inf, l = 0, o = 0), which ra_merge
 * ignores.
 */
RA_API ra_status ra_forward_partial_causal(const void* q, const void* k, const void* v,
                                           int32_t B, int32_t H, int64_t N, int32_t d, int32_t P,
                                           int32_t G, const ra_state* partials, ra_layout layout,
                                           ra_dtype dtype, ra_stream_t stream);

/*
 * ra_forward_split -- ra_forward for problems too small to fill the GPU: the
 * ring of every query block is split into G contiguous segments of steps
 * that are folded in parallel into partial states, which are then merged
 * ("Ring Attention" (bembew.net), "Global Integration"; exact by the
 * shift invariance of "Ring Attention: the math", section "The online-softmax
 * identity").  Same result as ra_forward up to rounding.
 *   G          1 <= G <= min(P, RA_MAX_PARTIALS); ra_forward_split_segments
 *              gives a choice for the current device.
 *   workspace  caller-owned device scratch of at least
 *              ra_forward_split_workspace_bytes(B, H, N, d, G) bytes,
 *              256-byte aligned; overwritten (no initial value needed).
 * Other arguments as ra_forward.  Errors: as ra_forward; RA_ERR_INVALID_ARG
 * for a bad G, a NULL or too small workspace; RA_ERR_MISALIGNED if the
 * workspace is not 256-byte aligned.
 */
RA_API ra_status ra_forward_split(const void* q, const void* k, const void* v, void* out,
                                  float* lse, int32_t B, int32_t H, int64_t N, int32_t d,
                                  int32_t P, int32_t G, void* workspace, int64_t workspace_bytes,
                                  ra_dtype dtype, ra_stream_t stream);

/* Scratch bytes ra_forward_split needs (-1 for invalid sizes). */
RA_API int64_t ra_forward_split_workspace_bytes(int32_t B, int32_t H, int64_t N, int32_t d,
                                                int32_t G);

/*
 * Segments for ra_forward_split on the current device: 1 when the plain
 * forward already gives every SM work, else the largest G whose G x (CTAs
 * of the plain forward) still fit in one wave of the SMs, keeping
 * at least 32 K/V tiles (4096 keys) per segment and at most
 * min(P, RA_MAX_PARTIALS).  bf16 only (returns 1 otherwise).
 */
RA_API int32_t ra_forward_split_segments(int32_t B, int32_t H, int64_t N, int32_t d, int32_t P,
                                         ra_dtype dtype);

/* Size of the fixed device scratch of ra_forward_split_noalloc: 32 MiB. */
#define RA_SPLIT_NOALLOC_SCRATCH_BYTES (32ll * 1024 * 1024)

/*
 * ra_forward_split_noalloc -- ra_forward_split for callers that cannot
 * allocate device memory.  The pages have no counterpart; this is a service
 * of the library.  Some callers may not call cudaMalloc once they run: a
 * plug-in inside a host whose memory pool already owns the device, or a
 * latency-bound loop that cannot accept an allocation's implicit device
 * synchronisation.  They pass only inputs and outputs; the G partial states
 * live in one library-owned device array of RA_SPLIT_NOALLOC_SCRATCH_BYTES
 * that every GPU which loads the library holds until the process exits.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The array is part of the library's device code: every process that
 *     loads the library's kernels on a GPU holds its 32 MiB there (at module
 *     load under CUDA_MODULE_LOADING=EAGER, else when the module is first
 *     used), whether or not this entry point is ever called.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.  A cudaDeviceReset invalidates the cached address:
 *     call no entry point of this library after resetting a device it used.
 *   - Every call on a device shares the array: calls that overlap on the GPU
 *     (other streams, unordered host threads) race and corrupt each other.
 *     Nothing in it needs to start at zero; each call writes all it reads.
 * Arguments as ra_forward_split, without the workspace.
 * Errors: as ra_forward_split (the arguments are checked first, so a bad
 * argument gives RA_ERR_INVALID_ARG or RA_ERR_MISALIGNED whatever the
 * size); then RA_ERR_UNSUPPORTED when the partial states
 * (ra_forward_split_workspace_bytes(B, H, N, d, G)) exceed
 * RA_SPLIT_NOALLOC_SCRATCH_BYTES -- nothing is launched then; use
 * ra_forward_split with a caller workspace, or a smaller G.
 */
RA_API ra_status ra_forward_split_noalloc(const void* q, const void* k, const void* v,
                                          void* out, float* lse, int32_t B, int32_t H, int64_t N,
                                          int32_t d, int32_t P, int32_t G, ra_dtype dtype,
                                          ra_stream_t stream);

/*
 * ra_forward_host -- ra_forward (causal = 0) or ra_forward_causal
 * (causal = 1, with `layout`) for inputs and results in HOST memory.  The
 * pages have no counterpart: it is the same computation with the transfers
 * folded in.  The B*H independent (batch, head) slices are cut into up to 8
 * chunks of whole slices, each carrying at least 16 MiB of q, k, v (a
 * smaller problem is one chunk).
 * Chunk c's q, k, v are copied to the device while earlier chunks compute,
 * and its out, lse are copied back while later chunks compute, so only the
 * first chunk's upload and the last chunk's download are not hidden.
 *   q, k, v    HOST [B, H, N, d] of `dtype`.  Page-locked (pinned) memory
 *              lets the copies overlap the compute; pageable memory gives the
 *              same results with the copies serialised.
 *   out, lse   HOST [B, H, N, d] of `dtype` and [B, H, N] fp32 (written).
 *   workspace  DEVICE scratch of at least ra_forward_host_workspace_bytes
 *              bytes, 256-byte aligned, owned by the caller; it holds the
 *              device copies of q, k, v, out and lse.
 * The call is asynchronous on `stream` like the others: the host buffers
 * must stay valid, and out/lse are complete, only once `stream` has reached
 * the point of the call (e.g. after cudaStreamSynchronize).  The copies and
 * half of the chunks run on streams the library creates once per device;
 * `stream` waits for all of them before any later work.  Calls that may
 * overlap on the GPU need workspaces of their own.
 * Errors: as ra_forward / ra_forward_causal (checked before anything is
 * queued); RA_ERR_INVALID_ARG for a NULL buffer or a workspace that is too
 * small; RA_ERR_MISALIGNED for a workspace not 256-byte aligned.  A CUDA
 * error after the first copy was queued returns RA_ERR_CUDA; `stream` still
 * waits for the work already queued.
 */
RA_API ra_status ra_forward_host(const void* q, const void* k, const void* v, void* out,
                                 float* lse, int32_t B, int32_t H, int64_t N, int32_t d,
                                 int32_t P, int32_t causal, ra_layout layout, ra_dtype dtype,
                                 void* workspace, int64_t workspace_bytes, ra_stream_t stream);

/* Device scratch bytes ra_forward_host needs (-1 for invalid sizes). */
RA_API int64_t ra_forward_host_workspace_bytes(int32_t B, int32_t H, int64_t N, int32_t d,
                                               ra_dtype dtype);

/*
 * ra_backward -- gradients of ring attention ("Ring attention, explained",
 * step 6: the backward runs on the same ring, the key-value blocks carrying
 * their gradient accumulators).  For the loss L = sum(dout * out):
 *     P = exp(tau q.k - lse)  (recomputed from the forward's lse)
 *     dV = P^T dout;  dP = dout V^T;  dS = P * (dP - D),  D = rowsum(dout * out)
 *     dQ = tau dS K;  dK = tau dS^T Q
 * dK and dV of block j are accumulated while the block visits the query
 * blocks (j + t) mod P; dQ of block i while it meets the key blocks
 * (i - t) mod P.  No atomics: every gradient row is written once.
 *   q, k, v, out, dout  [B, H, N, d] of `dtype` (out and lse from ra_forward).
 *   lse         [B, H, N] fp32.
 *   dq, dk, dv  [B, H, N, d] of `dtype` (written).
 *   workspace   caller-owned fp32 scratch of 2 * B * H * N floats, 16-byte
 *               aligned; receives D and -lse * log2(e).
 * Size and alignment rules as ra_forward (bf16: d in {64, 128}, c % 128 == 0,
 * 16-byte aligned tensors).
 * Errors: as ra_forward; RA_ERR_INVALID_ARG for a NULL buffer.
 */
RA_API ra_status ra_backward(const void* q, const void* k, const void* v, const void* out,
                             const void* dout, const float* lse, void* dq, void* dk, void* dv,
                             float* workspace, int32_t B, int32_t H, int64_t N, int32_t d,
                             int32_t P, ra_dtype dtype, ra_stream_t stream);

/*
 * ra_backward_causal -- ra_backward for ra_forward_causal: the mask and the
 * layout as there (a query at position n sees key positions <= n).  Under the
 * mask the key block j meets only the query tiles at or after its keys, the
 * query block i only the key tiles at or before its queries.  Size rules as
 * ra_forward_causal.
 */
RA_API ra_status ra_backward_causal(const void* q, const void* k, const void* v, const void* out,
                                    const void* dout, const float* lse, void* dq, void* dk,
                                    void* dv, float* workspace, int32_t B, int32_t H, int64_t N,
                                    int32_t d, int32_t P, ra_layout layout, ra_dtype dtype,
                                    ra_stream_t stream);

/*
 * ra_backward_rowterms -- the per-query terms of the backward for `rows`
 * query rows: D = rowsum(dout * out) and -lse * log2(e), written to
 * workspace[0 .. rows) and workspace[rows .. 2 rows).  The first step of the
 * ring backward on a device ("Ring attention, explained", step 6), before
 * its query block meets the visiting blocks with ra_backward_block.
 *   out, dout  [rows, d] of `dtype` (out from the forward);  lse [rows] fp32.
 *   workspace  caller-owned fp32 [2 * rows], 16-byte aligned.
 * Errors: RA_ERR_INVALID_ARG (NULL pointer, rows < 0, d < 1, bad dtype),
 * RA_ERR_UNSUPPORTED (rows >= 2^31), RA_ERR_MISALIGNED, RA_ERR_ARCH,
 * RA_ERR_CUDA.
 */
RA_API ra_status ra_backward_rowterms(const void* out, const void* dout, const float* lse,
                                      int64_t rows, int32_t d, ra_dtype dtype, float* workspace,
                                      ra_stream_t stream);

/*
 * ra_backward_block -- one step of the ring backward across devices ("Ring
 * attention, explained", step 6: the backward runs on the same ring, the
 * key-value blocks carrying their gradient accumulators).  The query block
 * (q, dout, its lse and row terms) meets one visiting K/V block and adds
 *     dq_acc += tau dS K,   dk_acc += tau dS^T Q,   dv_acc += P^T dout
 * with P = exp(tau q.k - lse) and dS = P * (dout V^T - D).  dk_acc and
 * dv_acc belong to the visiting block and travel with it; dq_acc stays.
 *   q, dout       [batch, c, d] of `dtype` (the query block).
 *   k, v          [batch, c, d] of `dtype` (the visiting block).
 *   lse           [batch, c] fp32 (the forward's, natural log).
 *   rowterms      [2 * batch * c] fp32 from ra_backward_rowterms.
 *   dq_acc        [batch, c, d] fp32, accumulated; dk_acc, dv_acc likewise.
 *   causal        0: every key visible; 1: the block is the query block's
 *                 own (key r visible to query r' iff r <= r', the diagonal
 *                 block of a contiguous causal ring).
 * Size rules as ra_backward with N = c and P = 1 (bf16: d in {64, 128},
 * c % 128 == 0, 16-byte aligned tensors and accumulators).  Accumulators
 * are read and written in place: calls that overlap on the GPU and share an
 * accumulator race.
 * Errors: as ra_backward; RA_ERR_INVALID_ARG for a NULL pointer or causal
 * not 0 or 1.
 */
RA_API ra_status ra_backward_block(const void* q, const void* k, const void* v, const void* dout,
                                   const float* lse, const float* rowterms, float* dq_acc,
                                   float* dk_acc, float* dv_acc, int64_t batch, int64_t c,
                                   int32_t d, int32_t causal, ra_dtype dtype,
                                   ra_stream_t stream);

/*
 * ra_state_init -- set a state to empty: m = -inf, l = 0, o = 0 ("Ring
 * Attention: the math", section "Accumulation math, step by step": "state = (m
 * = -inf, l = 0, o = 0)").
 * Errors: RA_ERR_INVALID_ARG (null state or pointers, rows < 0, d < 1),
 * RA_ERR_ARCH, RA_ERR_CUDA.
 */
RA_API ra_status ra_state_init(const ra_state* st, ra_stream_t stream);

/*
 * ra_fold -- fold ONE visiting K/V block into a caller-held state, in place
 * ("Ring Attention: the math", section "The online-softmax identity that
 * makes streaming legal": "For each incoming K/V block").  This is the
 * operation a ring device performs at every step; chaining it over the blocks
 * in ring order reproduces ra_forward's state.
 *   st       state of st->rows = batch * rq rows (rq query rows per batch
 *            entry), d = st->d.
 *   q        [batch, rq, d] queries of `dtype`.
 *   kblk,    [batch, kv_rows, d] keys and values of the visiting block.
 *   vblk
 * kv_rows == 0 leaves the state unchanged.  The bf16 path needs rq % 128 == 0
 * and kv_rows % 128 == 0; the f32 path takes any sizes.
 * Errors: as ra_forward; RA_ERR_UNSUPPORTED when rows is not a multiple of
 * batch or a bf16 size rule is broken.
 */
RA_API ra_status ra_fold(const ra_state* st, const void* q, const void* kblk,
                         const void* vblk, int64_t batch, int64_t kv_rows,
                         ra_dtype dtype, ra_stream_t stream);

/*
 * ra_merge -- combine G partial states of the same rows into out and lse
 * ("Ring Attention" (bembew.net), "Global Integration"; exact by the shift
 * invariance in "Ring Attention: the math", section "The online-softmax
 * identity"):
 *     m* = max_g m_g,  w_g = exp(m_g - m*),  l* = sum_g w_g l_g,
 *     o* = sum_g w_g o_g,  out = o* / l*,  lse = m* + ln l*.
 * Empty partials (m = -inf, l = 0) contribute nothing; rows whose partials
 * are all empty give out = 0 and lse = -inf.  With G = 1 this is the final
 * normalisation out = o / l of a single state.
 *   partials  host array of G states with equal rows and d.
 *   out       [rows, d] of out_dtype; lse [rows] fp32.
 * Errors: RA_ERR_INVALID_ARG (null pointers, G < 1 or > RA_MAX_PARTIALS,
 * mismatched rows/d), RA_ERR_MISALIGNED (out or o not 4-byte aligned),
 * RA_ERR_ARCH, RA_ERR_CUDA.
 */
RA_API ra_status ra_merge(const ra_state* partials, int32_t G, void* out, float* lse,
                          ra_dtype out_dtype, ra_stream_t stream);

/*
 * ra_watchdog_config -- settings of the bounded waits in the tensor-core
 * kernels (bf16 forward, fold, partial, split and backward calls).  The
 * pages have no counterpart: it belongs to the library's failure detection.
 *   wait_cycles  SM clock cycles one wait of a kernel may take before the
 *                kernel gives up: it records RA_ERR_TIMEOUT (read by
 *                ra_last_device_status), lets the copies and products it
 *                has in flight finish, frees its tensor memory and returns.
 *                <= 0 restores the default, 2^31 cycles (about a second).
 *   stall_cta    a test aid: >= 0 makes the CTA with this index of every
 *                later tensor-core launch (the fold kernel of the forward,
 *                causal, partial, fold and split calls; the dK/dV and dQ
 *                kernels of the backward calls) load no input, so that its
 *                waits run out and the call reports RA_ERR_TIMEOUT; the rows
 *                of that CTA are then not written.  -1 (the default) turns
 *                it off.
 * The settings are process-wide and apply to calls made after this one, on
 * every device and thread.  Never fails.
 */
RA_API void ra_watchdog_config(int64_t wait_cycles, int64_t stall_cta);

/*
 * ra_last_device_status -- synchronise `stream`, then read and clear the
 * device-side watchdog word of the current device.  Returns RA_ERR_TIMEOUT if
 * any kernel since the last call gave up a bounded wait (its results are then
 * invalid), RA_ERR_CUDA if the synchronisation failed, else RA_OK.
 */
RA_API ra_status ra_last_device_status(ra_stream_t stream);

/* Static, human-readable name of a status code. */
RA_API const char* ra_status_string(ra_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
RA_API int32_t ra_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RA_H_ */
