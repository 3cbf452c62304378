// kernels.h -- internal launchers of libittt.so (host side, C++).  The C-ABI
// in ittt_api.cu validates arguments, builds the TMA tensor maps and calls
// these in data-flow order: conv -> target -> gate/up -> snapshot 0 ->
// update -> apply (or, in the dual form, scores -> dual apply).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

namespace ittt {

// Launches `kernel` with programmatic stream serialization: its CTAs may start
// (set-up only -- every kernel of this library waits in griddep_wait() before
// it touches global memory) while the previous grid on the stream finishes,
// which hides the launch latency and set-up between back-to-back kernels.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

struct LaunchEnv {
  cudaStream_t stream;
  int num_sms;
  unsigned int* status;  // device status word (kStatusTimeout bits)
  // kNumTickets counters in device memory, zero before the call's first
  // kernel: the apply's unit counter (it takes its units dynamically) and
  // the arrival counters of its split last round.
  unsigned int* tickets = nullptr;
  // kApplyPartBytes of fp32 scratch for the partial sums of the apply's
  // split last round, or nullptr (the round is then not split).
  float* apply_part = nullptr;
};
// The apply's partial last round of t units on P CTA pairs (2t <= P) may run
// each unit as up to four pieces over disjoint K ranges; a piece's CTA writes
// its 128 x 256 fp32 partial, and the last of the pieces adds them.
constexpr int kMaxApplyTailPieces = 76;  // t x pieces <= P <= 76 pairs (152 SMs)
constexpr size_t kApplyPieceBytes = size_t(2) * 128 * 256 * 4;  // both CTAs' partials
constexpr size_t kApplyPartBytes = size_t(kMaxApplyTailPieces) * kApplyPieceBytes;
enum TicketSlot : int {
  kTicketApply = 0,
  kTicketApplyTail = 4,  // one counter per (tail unit, CTA of the pair)
  kNumTickets = kTicketApplyTail + 2 * kMaxApplyTailPieces
};

// The documents along the packed token axis, each with its own fast-weight
// state that starts from W_0 (the state is reset at document boundaries:
// "[논문리뷰] In-Place Test-Time Training", Method §3, causality and boundary
// handling).  Either B sequences of T tokens (starts == nullptr), or a table
// uploaded by the host: document k covers tokens [starts[k], starts[k+1])
// and owns snapshot slots [chunk_base[k], chunk_base[k+1]), one per chunk;
// chunk_doc[g] is the document of slot g.  Chunks start at each document's
// first token; a document's last chunk may be shorter than C.
struct DocMap {
  const int* starts;      // [ndocs + 1] device, or nullptr
  const int* chunk_base;  // [ndocs + 1] device, or nullptr
  const int* chunk_doc;   // [nchunks] device, or nullptr
  const int* tile_base;   // [nchunks + 1] device: 128-row tiles before slot g, or nullptr
  const int* tile_base2;  // [nchunks + 1] device: 256-row tiles before slot g, or nullptr
  int ndocs;              // documents (B when regular)
  int nchunks;            // snapshot slots over all documents
  int ntiles;             // 128-row tiles over all chunks
  int ntiles2;            // 256-row tiles over all chunks
  int T;                  // tokens per sequence (regular) / in the pack
  int n;                  // chunks per sequence (regular)
  int C;
  int mtc;                // 128-row tiles of a full chunk (regular)
  int tiles_per_seq;      // 128-row tiles of a sequence (regular)
  int mtc2;               // 256-row tiles of a full chunk (regular)
  int tiles_per_seq2;     // 256-row tiles of a sequence (regular)

  __host__ __device__ bool packed() const { return starts != nullptr; }
#ifdef __CUDACC__
  __device__ __forceinline__ int start(int k) const { return starts ? __ldg(starts + k) : k * T; }
  __device__ __forceinline__ int len(int k) const {
    return starts ? __ldg(starts + k + 1) - __ldg(starts + k) : T;
  }
  __device__ __forceinline__ int first_chunk(int k) const {
    return chunk_base ? __ldg(chunk_base + k) : k * n;
  }
  __device__ __forceinline__ int num_chunks(int k) const {
    return chunk_base ? __ldg(chunk_base + k + 1) - __ldg(chunk_base + k) : n;
  }
  __device__ __forceinline__ int doc_of_chunk(int g) const {
    return chunk_doc ? __ldg(chunk_doc + g) : g / n;
  }
  // Snapshot slot g and row tile mt (of 128 rows, or 256 with `wide`, within
  // the chunk) of the t-th non-empty row tile, over all chunks in slot order.
  __device__ __forceinline__ int slot_of_tile(int t, int* mt, bool wide = false) const {
    const int* base = wide ? tile_base2 : tile_base;
    if (!base) {
      const int per = wide ? tiles_per_seq2 : tiles_per_seq;
      const int m = wide ? mtc2 : mtc;
      const int b = t / per;
      const int r = t - b * per;
      const int i = min(r / m, n - 1);
      *mt = r - i * m;
      return b * n + i;
    }
    int lo = 0, hi = nchunks;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(base + mid) <= t) lo = mid; else hi = mid;
    }
    *mt = t - __ldg(base + lo);
    return lo;
  }
  // Document holding token row r (binary search over the starts).
  __device__ __forceinline__ int doc_of_token(int r) const {
    if (!starts) return r / T;
    int lo = 0, hi = ndocs;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(starts + mid) <= r) lo = mid; else hi = mid;
    }
    return lo;
  }
#endif
};

// state[s] = W_start[s] + sum_{k < count} deltas[k, s] over S states of
// df = d * f fp32 elements (df a multiple of 64), added in that order.
// w0_kind: 0 zero start, 1 shared bf16 [d, f], 2 shared fp32 [d, f],
// 3 fp32 [S, d, f].  deltas: [count.., S, d, f] fp32.
cudaError_t launch_state_prefix(const LaunchEnv& env, const void* w0, int w0_kind,
                                const float* deltas, int count, float* state, int64_t S,
                                int64_t df);

// Z[M, f] = SiLU(H W_gate^T) * (H W_up^T) on single CTAs (fallback).  Tensor
// maps: H [M, K] box {64,128}; W_gate, W_up [f, K] box {64,128}; Z [M, f] box
// {64,128} for the TMA stores.  All bf16, K = d_model.
cudaError_t launch_gateup(const LaunchEnv& env, const CUtensorMap& tm_h,
                          const CUtensorMap& tm_wg, const CUtensorMap& tm_wu,
                          const CUtensorMap& tm_zs, int M, int f, int K);

// The same on CTA pairs (256-row tiles); cudaErrorNotSupported when no pair
// can be resident (nothing launched).
cudaError_t launch_gateup_pair(const LaunchEnv& env, const CUtensorMap& tm_h,
                               const CUtensorMap& tm_wg, const CUtensorMap& tm_wu,
                               const CUtensorMap& tm_zs, int M, int f, int K);

// Xc = three-tap depthwise conv of X0 (zero padding at chunk edges, or only
// at document edges when pad_mode = 1), rounded to bf16.  tm_x0 maps X0
// [rows, d] bf16 with box {kConvMapBoxCols, kConvMapBoxRows} and no
// swizzle; xc: [rows, d].
cudaError_t launch_conv(const LaunchEnv& env, const CUtensorMap& tm_x0, const float* conv_w,
                        __nv_bfloat16* xc, int64_t rows, const DocMap& docs, int d,
                        int pad_mode);
// fp32 inputs (k_fp32_inputs.cu): dst[r, k*cols + c] = part k of src[r, c]
// for k < nseg, the bf16 rounding hi = bf16(x) or, where bit k of lo_mask is
// set, the remainder lo = bf16(x - hi).  src [rows, cols] fp32, cols a
// multiple of 8; dst [rows, nseg*cols] bf16.
cudaError_t launch_split_bf16(const LaunchEnv& env, const float* src, int64_t rows, int cols,
                              __nv_bfloat16* dst, int nseg, unsigned lo_mask);
// The convolution of an fp32 X0 [rows, d] (as launch_conv, in fp32), split
// into xc3 [rows, 3d] bf16 as [Xc_hi | Xc_hi | Xc_lo].
cudaError_t launch_conv_fp32(const LaunchEnv& env, const float* x0, const float* conv_w,
                             __nv_bfloat16* xc3, int64_t rows, const DocMap& docs, int d,
                             int pad_mode);

// The box launch_conv's X0 map must have: {channels, rows}.
constexpr uint32_t kConvMapBoxCols = 256, kConvMapBoxRows = 66;

// vhat[M, d] = eta * eta_tok[row] * (Conv1D(X0) W_target^T), rounded once to
// bf16 (eta_tok may be null: weight 1).
// Split (fused = false): tm_a maps Xc [M, d] with box {64,128} and the
// output goes out through tm_vs (vhat [M, d], box {64,128}).
// Fused: tm_a maps X0 [M, d] with box {64,130}, the kernel computes the conv
// itself and stores vhat directly.  tm_wt: W_target [d, d] box {64,256}.
// K: the split variant's contraction length (0: d; 2d for fp32 inputs, whose
// A operand is [Xc | Xc] and B [W_target hi | lo]); the fused variant has K = d.
cudaError_t launch_target(const LaunchEnv& env, const CUtensorMap& tm_a,
                          const CUtensorMap& tm_wt, const CUtensorMap& tm_vs,
                          const float* conv_w, const float* eta_tok, __nv_bfloat16* vhat,
                          float eta, int M, int T, int d, int C, int pad_mode, bool fused,
                          int K = 0);

// The split variant on CTA pairs (256-row tiles): tm_xc maps Xc [M, d] box
// {64,128}, tm_wt maps W_target [d, d] box {64,128}, tm_vs as above.
// cudaErrorNotSupported when no pair can be resident (nothing launched).
cudaError_t launch_target_pair(const LaunchEnv& env, const CUtensorMap& tm_xc,
                               const CUtensorMap& tm_wt, const CUtensorMap& tm_vs,
                               const float* eta_tok, __nv_bfloat16* vhat, float eta, int M,
                               int d, int K = 0);

// Slot docs.first_chunk(k) of snap = bf16(W_0 of document k) for every k.
// w0 is bf16 or fp32, [d, f] shared (w0_bstride = 0) or one per document.
cudaError_t launch_snapshot0(const LaunchEnv& env, const void* w0, bool w0_fp32,
                             int64_t w0_bstride, __nv_bfloat16* snap, const DocMap& docs, int d,
                             int f);

struct UpdateArgs {
  DocMap docs;
  const int* upd_docs;  // device list of the documents that update, or nullptr (all)
  int n_udocs;          // documents that update (0: no launch)
  bool final_update;    // also the last chunk's update (the caller wants the state)
  int d, f;
  const void* w0;       // bf16 or fp32 initial state
  bool w0_fp32;
  int64_t w0_bstride;
  float* state_out;     // [documents, d, f] fp32 or nullptr
  bool allow_pairs;     // every updated chunk is a multiple of 64 tokens
};

// Fast-weight update walk: for each (document, 128 x 512 state tile) the
// fp32 state starts at W_0 in TMEM and the per-chunk deltas
// (eta Vhat_[i])^T Z_[i] accumulate onto it; after chunk i the epilogue
// writes bf16(W_{i+1}) into the document's snapshot slot i+1.  Tensor maps:
// eta*Vhat [M, d] box {64,64}; Z [M, f] box {64,64} (both read MN-major);
// snapshots as [slots][d][f] with box {64,128,1} for the TMA stores.
cudaError_t launch_update(const LaunchEnv& env, const CUtensorMap& tm_vhat,
                          const CUtensorMap& tm_z, const CUtensorMap& tm_snap_store,
                          const UpdateArgs& a);

struct NormUpdateArgs {
  DocMap docs;
  const int* upd_docs;  // updating documents, most updates first (nullptr: all)
  int n_udocs;          // updating documents (0: no launch)
  int n_steps;          // launches: the largest number of updates of a document
  const int* active;    // host [n_steps]: documents still updating at chunk i
  int d, f;
  const void* w0;
  bool w0_fp32;
  int64_t w0_bstride;
  float* state;         // scratch: documents x ceil(d/128) x ceil(f/32) tiles of 16 KB
  float* partial;       // scratch [2][documents][2 * ceil(f/512)][d] fp32
  __nv_bfloat16* snap;  // [slots, d, f]: slots 1..n-1 of each document written
  float* state_out;     // [documents, d, f] fp32 or nullptr
  bool allow_pairs;     // every updated chunk a multiple of 64 tokens and d of 256
  // Scratch of the walk with the state resident in TMEM (regular batches on
  // CTA pairs; nullptr: not available): row sums of squares for up to
  // walk_pairs CTA pairs, and 2 x walk_pairs arrival counters.
  float* walk_part;
  unsigned int* walk_arrive;
  int walk_pairs;
};

// Bytes of that scratch for d_ff = f and up to `pairs` CTA pairs.
size_t norm_walk_part_bytes(int f, int pairs);
size_t norm_walk_arrive_bytes(int pairs);
constexpr int kNormWalkMaxPairs = 128;

// The fast-weight walk with L2 normalisation of every updated state, rows
// over d_ff.  Regular batches on CTA pairs keep the fp32 state in TMEM for
// the whole walk (one launch; the pairs holding a row block exchange row sums
// of squares at every chunk boundary); otherwise one launch per chunk with
// the state in HBM, then one finalising launch.  Tensor maps:
// eta*Vhat and Z as for launch_update; the snapshots as [slots][d][f] with
// box {64,128,1} for TMA stores.  Runs on CTA pairs when allowed and two can
// be resident, else on single CTAs.
cudaError_t launch_norm_update(const LaunchEnv& env, const CUtensorMap& tm_vhat,
                               const CUtensorMap& tm_z, const CUtensorMap& tm_snap_store,
                               const NormUpdateArgs& a);

// O_[i] = Z_[i] snap[slot of chunk i]^T for every chunk of every document,
// one CTA per 128-row tile (fallback when no CTA pair can be resident).
// Tensor maps: Z [M, f] box {64,128}; snapshots [slots*d, f] box {64,256};
// bf16 O [M, d] with box {64,64} for the TMA stores (unused for fp32 O).
// Chunks of any length; a document's last chunk may be shorter than C.
// tm_w0 (nullptr, or bf16 W_0 [d, f] with tm_snap's box): read instead of a
// document's first snapshot slot, which is then never read.
cudaError_t launch_apply(const LaunchEnv& env, const CUtensorMap& tm_z,
                         const CUtensorMap& tm_snap, const CUtensorMap* tm_w0,
                         const CUtensorMap& tm_os, void* out, bool out_fp32,
                         const DocMap& docs, int d, int f);

// The same on CTA pairs (256-row tiles, tcgen05 cta_group::2): tm_snap and
// tm_w0 have box {64,128} (each CTA loads its 128 of the tile's 256
// columns).  Returns cudaErrorNotSupported when no pair can be resident
// (nothing launched).
cudaError_t launch_apply_pair(const LaunchEnv& env, const CUtensorMap& tm_z,
                              const CUtensorMap& tm_snap, const CUtensorMap* tm_w0,
                              const CUtensorMap& tm_os, void* out, bool out_fp32,
                              const DocMap& docs, int d, int f);

// Dual form, scores: S[b, t, s] = Z_t . Z_s (bf16) for every token t of chunk
// i >= 1 and every token s < i*C of the same sequence (and zeros for the
// other tokens s before the first token of the last chunk of t's 256-row
// group).  Tensor maps: Z [B*T, f] with box {64,128} (tm_zq) and box
// {64,256} (tm_zk).  With allow_pairs it runs on CTA pairs when a pair can
// be resident, else on single CTAs; both write the same entries.
cudaError_t launch_scores(const LaunchEnv& env, const CUtensorMap& tm_zq,
                          const CUtensorMap& tm_zk, __nv_bfloat16* s, int B, int T, int f,
                          int C, bool allow_pairs);

// Dual form, apply: O_[i] = Z_[i] W_0^T + S_[i, <iC] (eta Vhat)_[<iC].  Tensor
// maps: Z [B*T, f] box {64,128}; bf16 W_0 [Bw*d, f] box {64,256} (tm_w0) and
// {64,128} (tm_w0_pair) (Bw = B when w0_per_seq, else 1); S [B*T, T] box
// {64,128}; eta*Vhat [B*T, d] box {64,64}.  With allow_pairs it runs on CTA
// pairs (256-row tiles) when a pair can be resident, else on single CTAs;
// both read the same scores entries and give the same result.
cudaError_t launch_dual_apply(const LaunchEnv& env, const CUtensorMap& tm_z,
                              const CUtensorMap& tm_w0, const CUtensorMap& tm_w0_pair,
                              const CUtensorMap& tm_s, const CUtensorMap& tm_v, bool w0_per_seq,
                              void* out, bool out_fp32, int B, int T, int d, int f, int C,
                              bool allow_pairs);

// Defined in ittt_api.cu, for entry points in other translation units.
cudaError_t status_word_address(unsigned int** out);
void set_last_error(const char* msg);

}  // namespace ittt
