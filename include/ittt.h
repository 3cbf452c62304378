/*
 * ittt.h -- C-ABI of libittt.so, the In-Place Test-Time Training fast-weight
 * layer for NVIDIA GB300 (sm_103a).
 *
 * The layer (pages: "[논문리뷰] In-Place Test-Time Training", Method §1 eq.
 * (2)-(4), Method §2 eq. (5)-(6), Method §3 "Implementation Details"):
 *
 *   Z     = SiLU(H W_gate^T) (.) (H W_up^T)                  (eq. 2)
 *   Vhat  = Conv1D(X0) W_target^T                             (eq. 5)
 *   W_0   = W_down0          (reset per sequence / document, Method §3)
 *   for each chunk i of C tokens, in order:
 *     O_[i]   = Z_[i] W_i^T                                   (eq. 3, apply)
 *     W_{i+1} = W_i + eta * Vhat_[i]^T Z_[i]                  (eq. 6, update)
 *
 * Conv1D is a depthwise three-tap convolution with taps ordered
 * (t-1, t, t+1), conv_w[c, k] multiplying X0[t-1+k, c], no bias.  Taps that
 * reach outside the current chunk read zero (ITTT_PAD_CHUNK, the default: the
 * pages' "causal padding" that keeps each chunk's update delta isolated to
 * that chunk) or, with ITTT_PAD_SEQUENCE, only taps outside the sequence read
 * zero.
 *
 * Conventions for every entry point:
 *   - Tensors are described by ittt_tensor: a DEVICE pointer, a dtype, and
 *     row-major shapes with element strides.  The last dimension must be
 *     contiguous (stride 1) and every tensor must be densely packed
 *     row-major; the data pointer must be 16-byte aligned.
 *   - Shapes: H, X0 [B,T,d] bf16; W_gate, W_up [f,d] bf16; W_down0 [d,f]
 *     bf16 or fp32; W_target [d,d] bf16; conv_w [d,3] fp32; out [B,T,d]
 *     bf16 or fp32.  Weights use the [out_features, in_features] layout.
 *     H, X0, W_gate, W_up and W_target may instead all be fp32
 *     (ITTT_FLAG_FP32_INPUTS).
 *   - Supported sizes: d and f multiples of 8 (16-byte rows), any chunk
 *     >= 1, any T >= 1, B*T < 2^31.  When chunk does not divide T the last
 *     chunk is the shorter remainder (a stream that ends mid-chunk).  Chunks
 *     that are multiples of 64 tokens run at full speed; other lengths are
 *     exact but pay for masking at every chunk end.  (ITTT_FLAG_FUSED_CONV
 *     and ITTT_FLAG_DUAL have narrower limits, stated with each.)  Anything
 *     else returns ITTT_ERR_UNSUPPORTED or ITTT_ERR_INVALID_ARG before any
 *     launch.
 *   - Ownership: the caller owns every buffer; the library keeps no pointer
 *     after a call returns.  `out` must not overlap any input.
 *   - Asynchrony: work is enqueued on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and the call returns without synchronising.
 *     Scratch memory comes from cudaMallocAsync/cudaFreeAsync on the same
 *     stream unless the caller passes a workspace.
 *   - Errors: a status code is returned, no exception crosses the ABI, and
 *     ittt_last_error() describes the most recent failure on this thread.
 *     Argument errors are detected before anything is enqueued.  Device-side
 *     failures (a bounded wait that ran out) are reported by
 *     ittt_stream_status().
 *   - Per-device state: the first call on a device looks up device addresses
 *     (the status word, the fixed scratch of ittt_forward_noalloc) and
 *     creates a memory pool; they are kept for the life of the process.
 *     Resetting the device (cudaDeviceReset) or destroying its primary
 *     context after that first call is not supported: later calls would use
 *     addresses of the destroyed context.
 */
#ifndef ITTT_H_
#define ITTT_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ITTT_API __attribute__((visibility("default")))
#else
#define ITTT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* ittt_stream_t; /* same type as cudaStream_t */

typedef enum {
  ITTT_OK = 0,
  ITTT_ERR_INVALID_ARG = 1, /* bad pointer, dtype, shape, stride or alias */
  ITTT_ERR_UNSUPPORTED = 2, /* valid, but outside the supported sizes */
  ITTT_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  ITTT_ERR_OOM = 4,         /* scratch allocation failed */
  ITTT_ERR_TIMEOUT = 5      /* a kernel's bounded wait ran out */
} ittt_status;

typedef enum { ITTT_BF16 = 0, ITTT_FP32 = 1 } ittt_dtype;

typedef enum {
  ITTT_PAD_CHUNK = 0,    /* conv taps outside the current chunk read 0 */
  ITTT_PAD_SEQUENCE = 1  /* conv taps outside the sequence read 0 */
} ittt_pad_mode;

/* A dense row-major device tensor.  `stride` is in elements. */
typedef struct {
  void* data;
  int32_t dtype; /* ittt_dtype */
  int32_t ndim;  /* 1..4 */
  int64_t shape[4];
  int64_t stride[4];
} ittt_tensor;

/*
 * Options for ittt_forward_ex.  Zero-initialise and set what you need; every
 * pointer may be NULL.
 *
 *   pad_mode   ittt_pad_mode for the convolution boundary.
 *   cu_seqlens HOST array of num_docs + 1 token offsets: packed documents.
 *              H, X0, out (and eta_tok, z_buf, vhat_buf) then hold B = 1
 *              row of T tokens in which document k is the token range
 *              [cu_seqlens[k], cu_seqlens[k+1]); cu_seqlens[0] = 0,
 *              cu_seqlens[num_docs] = T, and every document has at least one
 *              token.  Each document runs like a sequence of its own: its
 *              fast weight starts from W_0 (or its state_in) -- the state is
 *              reset at document boundaries (Method §3, causality and
 *              boundary handling) -- its chunks start at its first token,
 *              its last chunk may be shorter, and no convolution tap crosses
 *              into another document.  Read during the call only: the
 *              derived tables are written to a pinned, device-mapped host
 *              buffer that one extra kernel copies into device scratch, so
 *              such a call cannot be captured into a CUDA graph.  Not
 *              combinable with ITTT_FLAG_FUSED_CONV or ITTT_FLAG_DUAL.
 *   num_docs   number of packed documents (0 when cu_seqlens is NULL).
 *   state_in   fp32 [S,d,f]: per-sequence (S = B) or per-document
 *              (S = num_docs) initial fast weight.  Replaces W_down0 (which
 *              may then be NULL) -- continues a stream of chunks from a
 *              state returned by an earlier call, or starts a span of a
 *              sequence from the prefix of the spans before it
 *              (ittt_state_prefix).
 *   state_out  fp32 [S,d,f]: receives each sequence's or document's fast
 *              weight after its LAST chunk's update (an update the output
 *              itself never needs).  May be state_in itself (the same
 *              buffer, updated in place); any other overlap with an input
 *              is rejected.
 *   z_buf      bf16 [B,T,f]: caller buffer used as the Z scratch; after the
 *              call it holds Z.  Lets tests inspect the intermediate.
 *   vhat_buf   bf16 [B,T,d]: same for the update's left operand, which the
 *              library stores with eta folded in: it holds eta * Vhat.
 *   snap_buf   bf16 [B,n,d,f] (n = ceil(T/chunk)): same for the bf16
 *              snapshots W_0 .. W_{n-1} that the apply step reads.  Packed
 *              documents: [1,N,d,f] with N the chunks of all documents,
 *              document k's W_0 at slot sum_{j<k} ceil(len_j / chunk).
 *   workspace  device scratch of workspace_bytes >= ittt_workspace_bytes_ex
 *              (...) for the same options (256-byte aligned); when given,
 *              nothing is allocated.
 *   eta_tok    fp32 [B,T]: per-token learning-rate weights; token t's term
 *              of the chunk update is scaled by eta * eta_tok[b,t] (the
 *              large-chunk update with a rate per token of "Test-Time
 *              Training Done Right").  NULL: every weight is 1.  The update
 *              averaged over its chunk (eta times the chunk's mean of
 *              Vhat_t^T Z_t) is eta_tok[b,t] = 1 / (length of t's chunk).
 *   events     profiling: NULL, or 2 * ITTT_NUM_PHASES cudaEvent_t handles.
 *              events[2k] and events[2k+1] are recorded right before and
 *              right after phase k (ittt_phase order) on `stream`, so each
 *              pair brackets one phase on the device timeline.  A phase with
 *              nothing to do records both.  A NULL entry is not recorded
 *              (time only the phases you need: an event between two kernels
 *              costs a little and keeps the second from starting its set-up
 *              early).
 *   flags      ITTT_FLAG_* bits.
 */
typedef struct {
  int32_t pad_mode;
  int32_t flags;
  const ittt_tensor* state_in;
  ittt_tensor* state_out;
  ittt_tensor* z_buf;
  ittt_tensor* vhat_buf;
  ittt_tensor* snap_buf;
  void* workspace;
  size_t workspace_bytes;
  void* const* events;
  const ittt_tensor* eta_tok;
  const int64_t* cu_seqlens;
  int64_t num_docs;
} ittt_opts;

/* ittt_opts.flags */
/* Compute the convolution inside the W_target GEMM (extra warps build each
 * A tile from raw X0 rows in shared memory) instead of in its own kernel.
 * Same results; slower on GB300, where the fused convolution is repeated for
 * every 256-column output tile.  Needs chunk and T multiples of 64. */
#define ITTT_FLAG_FUSED_CONV 1
/* Compute O with the dual form O_[i] = Z_[i] W_0^T + eta sum_{j<i}
 * (Z_[i] Z_[j]^T) Vhat_[j] instead of walking the fast-weight state: a
 * scores kernel writes the block-lower part of Z Z^T (bf16, B*T*T*2 bytes of
 * scratch) and one GEMM accumulates both terms.  Same layer, different
 * rounding.  Forces the form a call would otherwise choose by sequence
 * length (see "Form choice" below).  Not combinable with state_out or
 * snap_buf; chunk must be a multiple of 64 that divides T. */
#define ITTT_FLAG_DUAL 2
/* Normalise the fast weight after every update, row by row over its d_ff
 * inputs: W_{i+1} = L2-Normalize(W_i + eta Vhat_[i]^T Z_[i]) with
 * L2-Normalize(W)[m,:] = W[m,:] / max(||W[m,:]||_2, 1e-12) (the normalised
 * update rule of "[논문리뷰] Test-Time Training Done Right", Non-Linear
 * Update of Fast-Weight; W_down0 is applied as given).  The update is then
 * not additive: the walk runs one launch per chunk with the fp32 state in
 * device scratch ([S,d,f] fp32 more scratch).  Snapshots and state_out hold
 * normalised states.  Not combinable with ITTT_FLAG_DUAL. */
#define ITTT_FLAG_L2_NORM 4
/* Run every GEMM on single CTAs (128-row tiles) instead of CTA pairs
 * (tcgen05 cta_group::2 on 2-CTA clusters, the default wherever a pair can be
 * resident).  Same results; for systems where 2-CTA clusters cannot be
 * scheduled and for comparing the two. */
#define ITTT_FLAG_SINGLE_CTA 8
/* Fold the call's chunks into the fast weight without applying it:
 * state_out (required) receives W_start + eta sum_i Vhat_[i]^T Z_[i] over
 * every chunk of each sequence or document, W_start being state_in, else
 * W_down0, else (both NULL) zero -- with a zero start it is the sum of the
 * call's per-chunk deltas, the quantity the parallel form of Method §3 sums
 * ahead of the apply ("Implementation Details", context parallelism).  The
 * update is additive, so the whole sequence is one contraction over its
 * tokens: no snapshots are formed and nothing is applied (out may be NULL;
 * snap_buf must be NULL).  Not combinable with ITTT_FLAG_DUAL or
 * ITTT_FLAG_L2_NORM. */
#define ITTT_FLAG_UPDATE_ONLY 16
/* z_buf and vhat_buf are INPUTS: they already hold Z and eta * Vhat for
 * these tokens (from an earlier call with the same H, X0, weights, eta,
 * eta_tok, chunk and pad mode, e.g. an ITTT_FLAG_UPDATE_ONLY call), so the
 * conv, target and gate/up phases are skipped.  H, X0, W_gate, W_up,
 * W_target and conv_w are checked for shape but not read. */
#define ITTT_FLAG_REUSE_ZV 32
/* Never use the dual form (see "Form choice" below). */
#define ITTT_FLAG_PRIMAL 64
/* fp32 inputs.  A call whose H is fp32 takes H, X0, W_gate, W_up and
 * W_target as fp32 (all five; W_down0, state_in and conv_w as usual).  The
 * inputs are not rounded to bf16: each fp32 value x is split into two bf16
 * parts, hi = bf16(x) and lo = bf16(x - hi), and the gate/up and target
 * products are formed as hi*hi + hi*lo + lo*hi on the same tensor-core
 * kernels by contracting over a concatenated K of 3 d; the dropped lo*lo
 * term is below 2^-16 relative.  The convolution Xc of X0 is computed in
 * fp32 and split the same way.  Z and eta*Vhat are then the fp32 products
 * rounded once to bf16; the fast-weight walk and the apply are as for bf16
 * inputs.  The gate/up and target phases cost 3x the FLOPs of bf16 inputs;
 * the scratch gains the split copies (H and Xc M x 3d, W_gate and W_up
 * f x 3d, W_target d x 3d, all bf16) in place of the bf16 Xc.  Not with
 * ITTT_FLAG_FUSED_CONV.  ittt_forward / ittt_forward_ex infer the mode from
 * H's dtype (setting this flag with bf16 H is an error);
 * ittt_workspace_bytes_ex and ittt_plan_form size and plan for it when the
 * flag is set. */
#define ITTT_FLAG_FP32_INPUTS 128

/*
 * Form choice.  Without ITTT_FLAG_DUAL or ITTT_FLAG_PRIMAL a call uses the
 * dual form when it can (regular sequences, chunk a multiple of 64 dividing
 * T, at least two chunks, no state_out, snap_buf, packed documents,
 * ITTT_FLAG_L2_NORM or ITTT_FLAG_FUSED_CONV) and its sequences are short:
 * T < 2.5 d f / (d + f) tokens.  The dual form's extra FLOPs grow with T^2
 * and equal the walk's update FLOPs at T = 2 d f / (d + f); the primal walk
 * also writes and re-reads one d x f weight snapshot per chunk whatever the
 * chunk's length, which moves the measured crossover on GB300 to 1.25-1.3
 * times that length (d 2560, f 9728: the dual form 5.6x faster at 64 x 256
 * tokens, 1.06x at 4 x 4096, 0.82x at 2 x 8192, 0.3x at 2 x 32768).  Both
 * forms compute the same layer; they round differently.  ittt_plan_form
 * says which form a call would use.
 */

/* Kernel phases of one forward call, in launch order. */
typedef enum {
  ITTT_PHASE_CONV = 0,      /* Xc = depthwise 3-tap conv of X0 (CUDA cores; empty
                               when fused into the target GEMM) */
  ITTT_PHASE_TARGET = 1,    /* eta*Vhat = eta * Xc W_target^T (tensor cores) */
  ITTT_PHASE_GATEUP = 2,    /* Z = SiLU(H W_gate^T) * (H W_up^T) (tensor cores) */
  ITTT_PHASE_SNAPSHOT0 = 3, /* bf16 copy of the initial fast weight */
  ITTT_PHASE_UPDATE = 4,    /* prefix walk of Vhat^T Z, snapshots W_1..W_{n-1}
                               (dual form: the scores Z Z^T) */
  ITTT_PHASE_APPLY = 5      /* O_[i] = Z_[i] W_i^T (tensor cores; dual form:
                               Z_[i] W_0^T + S_[i] eta Vhat) */
} ittt_phase;
#define ITTT_NUM_PHASES 6

/*
 * One forward pass of the layer over a batch of B independent sequences,
 * each starting from W_down0 (pages: Method §1 eq. (1)-(4), §2 eq. (5)-(6),
 * §3 three-stage parallel form).  eta is the fast-weight learning rate;
 * chunk is C.  out [B,T,d] receives O in its own dtype (bf16 or fp32).
 * Arithmetic: bf16 operands, fp32 accumulation, fp32 fast-weight state;
 * Z, Vhat and the per-chunk weight snapshots are rounded to bf16 (nearest
 * even) before they enter a tensor-core contraction.
 */
ITTT_API ittt_status ittt_forward(const ittt_tensor* H, const ittt_tensor* X0,
                         const ittt_tensor* W_gate, const ittt_tensor* W_up,
                         const ittt_tensor* W_down0,
                         const ittt_tensor* W_target,
                         const ittt_tensor* conv_w, float eta, int64_t chunk,
                         ittt_tensor* out, ittt_stream_t stream);

/* ittt_forward with options (see ittt_opts).  opts may be NULL. */
ITTT_API ittt_status ittt_forward_ex(const ittt_tensor* H, const ittt_tensor* X0,
                            const ittt_tensor* W_gate,
                            const ittt_tensor* W_up,
                            const ittt_tensor* W_down0,
                            const ittt_tensor* W_target,
                            const ittt_tensor* conv_w, float eta,
                            int64_t chunk, ittt_tensor* out,
                            ittt_stream_t stream, const ittt_opts* opts);

/*
 * ittt_forward for callers that cannot allocate device memory while they
 * run: a serving loop with a fixed, fully partitioned memory budget, a
 * process whose device memory belongs to another framework's caching
 * allocator, a real-time path that forbids allocation after start-up.
 * The pages have no counterpart: this is a deployment variant of
 * ittt_forward with the same arguments and kernels, always in the primal form
 * (ittt_forward picks the dual form for short sequences; the two round
 * differently).
 *
 * It calls no allocating routine.  Its scratch lives in one library-wide
 * device array of ITTT_NOALLOC_SCRATCH_BYTES (64 MiB) that every GPU which
 * loads the library holds until the process exits; a call that needs more
 * (B*T*(f + 2d)*2 + B*n*d*f*2 bytes with n = ceil(T/chunk), each part
 * rounded up to 256) returns
 * ITTT_ERR_UNSUPPORTED before anything is enqueued.  All calls share that
 * array, so calls that overlap on the GPU (other streams, other threads)
 * race: serialise them on one stream.  The first call on a device does a
 * one-time set-up (it looks up the array's device address); make that first
 * call before any stream capture.  Pad mode is ITTT_PAD_CHUNK; sizes as for
 * ittt_forward; inputs bf16 only (an fp32 H, X0, W_gate, W_up or W_target
 * returns ITTT_ERR_INVALID_ARG).  Device-side failures are reported by
 * ittt_stream_status().
 */
#define ITTT_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
ITTT_API ittt_status ittt_forward_noalloc(const ittt_tensor* H, const ittt_tensor* X0,
                                          const ittt_tensor* W_gate, const ittt_tensor* W_up,
                                          const ittt_tensor* W_down0,
                                          const ittt_tensor* W_target,
                                          const ittt_tensor* conv_w, float eta, int64_t chunk,
                                          ittt_tensor* out, ittt_stream_t stream);

/*
 * state[s] = W_start[s] + sum_{k < count} deltas[k, s] for each of the S
 * fast-weight states, summed in fp32 in that order (W_start first, then
 * deltas[0], deltas[1], ...).  This is the exclusive prefix of the parallel
 * form ("[논문리뷰] In-Place Test-Time Training", Method §3 "Implementation
 * Details": per-chunk deltas computed in parallel, one prefix sum, then the
 * apply): when span k of a sequence has folded its chunks into deltas[k]
 * (ITTT_FLAG_UPDATE_ONLY from a zero start), span r starts from the prefix
 * with count = r.
 *   W_start  W_down0 [d,f] bf16 or fp32 (shared by every state), an fp32
 *            [S,d,f] per-state start, or NULL (zero).
 *   deltas   fp32 [R,S,d,f] device tensor; count in 0..R.
 *   state    fp32 [S,d,f] device tensor; must not overlap the inputs.
 * Enqueued on `stream` like ittt_forward; argument errors are reported
 * before anything is enqueued.
 */
ITTT_API ittt_status ittt_state_prefix(const ittt_tensor* W_start, const ittt_tensor* deltas,
                                       int32_t count, ittt_tensor* state, ittt_stream_t stream);

/*
 * Bytes of device scratch one call needs for these sizes with default flags
 * when the caller supplies no z_buf / vhat_buf / snap_buf (0 if the sizes
 * are unsupported).
 */
ITTT_API size_t ittt_workspace_bytes(int64_t B, int64_t T, int64_t d, int64_t f,
                            int64_t chunk);

/*
 * Bytes of device scratch an ittt_forward_ex call with these options needs
 * (0 if the call would be rejected).  Reads opts->flags, pad_mode,
 * cu_seqlens / num_docs, and which of state_in, state_out, z_buf, vhat_buf
 * and snap_buf are non-NULL (not their contents).  opts may be NULL.
 */
ITTT_API size_t ittt_workspace_bytes_ex(int64_t B, int64_t T, int64_t d, int64_t f,
                                        int64_t chunk, const ittt_opts* opts);

/* Form a call with these sizes and options would run: ITTT_FORM_PRIMAL or
 * ITTT_FORM_DUAL, or -1 if the call would be rejected.  opts may be NULL. */
#define ITTT_FORM_PRIMAL 0
#define ITTT_FORM_DUAL 1
ITTT_API int32_t ittt_plan_form(int64_t B, int64_t T, int64_t d, int64_t f, int64_t chunk,
                                const ittt_opts* opts);

/*
 * Caps the device scratch one call may allocate (bytes; 0, the default,
 * means no cap) for every later call in this process: a call that would
 * allocate more returns ITTT_ERR_OOM before anything is enqueued.  Calls
 * given a caller workspace allocate nothing and are not affected.  Lets a
 * process keep the library inside a memory budget, and lets tests take the
 * out-of-memory path without exhausting the device.
 */
ITTT_API void ittt_set_scratch_limit(size_t bytes);

/*
 * Exercises the failure path of the kernels' bounded waits without a fault:
 * enqueues on `stream` one small kernel whose threads wait on a barrier that
 * nothing completes.  One warp gives up after `limit_ns` (1e3 .. 1e9 ns),
 * records the timeout in the device status word and raises its block's
 * abort flag; the other warp, allowed four times as long, unwinds on the
 * flag, so the kernel ends after about `limit_ns` and the context stays
 * usable.  The next ittt_stream_status() on that stream then returns
 * ITTT_ERR_TIMEOUT (and clears the record).  Returns ITTT_ERR_INVALID_ARG
 * for a limit outside the range (nothing enqueued), ITTT_ERR_CUDA if the
 * launch fails, else ITTT_OK.
 */
ITTT_API ittt_status ittt_check_wait_timeout(uint64_t limit_ns, ittt_stream_t stream);

/*
 * Synchronises `stream`, then reports any device-side failure recorded by
 * this library's kernels on the current device since the previous call
 * (ITTT_ERR_TIMEOUT when a bounded wait ran out) or a pending CUDA error
 * (ITTT_ERR_CUDA).  Clears the recorded failure.
 */
ITTT_API ittt_status ittt_stream_status(ittt_stream_t stream);

/* Message for the last failure on the calling thread ("" if none).  Valid
 * until the next call into this library on the same thread. */
ITTT_API const char* ittt_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
ITTT_API int32_t ittt_version(void);

/*
 * Kernel launches one ittt_forward / ittt_forward_ex call makes for these
 * sizes with default options and a bf16 W_down0 (for launch accounting; 0
 * if unsupported): conv, target, gate/up, the update walk when a chunk
 * updates, apply (the dual form's scores and dual apply in their place when
 * the call chooses it: the same count).  An fp32 W_down0, state_in or snap_buf adds the snapshot-0
 * copy; packed documents add the table staging kernel; ITTT_FLAG_L2_NORM
 * launches the walk once per updating chunk plus a finalising launch.
 */
ITTT_API int32_t ittt_launch_count(int64_t B, int64_t T, int64_t d, int64_t f,
                          int64_t chunk);

#ifdef __cplusplus
}
#endif

#endif /* ITTT_H_ */
