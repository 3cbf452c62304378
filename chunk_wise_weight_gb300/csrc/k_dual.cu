// k_dual.cu -- the dual (attention-like) form of the chunk-wise apply:
//   O_[i] = Z_[i] W_0^T + eta * sum_{j<i} (Z_[i] Z_[j]^T) Vhat_[j]
// i.e. the apply step with W_i = W_0 + eta * sum_{j<i} Vhat_[j]^T Z_[j]
// ("[논문리뷰] In-Place Test-Time Training", Method §1 eq. (3), §2 eq. (6);
// the block-causal mask view of apply/update orderings in "[논문리뷰]
// Test-Time Training Done Right", "Apply 연산과 Update 연산의 실행 순서").
//
// Both kernels tile the token axis in tiles that may span chunk edges
// (chunks are multiples of 64 tokens).  The rows of a 256-row group read the
// scores of every token before the first token of the group's LAST row's
// chunk, s_end:
//   scores: S[t, s] = Z_t . Z_s for s < s_end of t's group, where s lies in
//           an earlier chunk than t, and 0 where it does not (t's own chunk
//           inside the group's range), in a 128 x 256 tile per unit (K =
//           d_ff), rounded once to bf16 into a [B, T, T] buffer of which
//           only those entries are ever written or read;
//   apply:  one accumulator per 256 x 256 output tile on a CTA pair (each
//           CTA 128 rows; 128 x 256 tiles on single CTAs where no pair fits)
//           takes first Z W_0^T (K = d_ff, both operands K-major) and then
//           S (eta Vhat) over the tokens s < s_end (S K-major, eta*Vhat read
//           MN-major), so the instruction and shared-memory descriptors
//           change inside the accumulation; the zero scores add nothing to
//           a row whose chunk starts before s_end, so both tilings give the
//           same sums.
// The dual form does no state update at all, and its work grows with the
// square of the context: per chunk i it costs 2*C*d*f + i*2*C^2*(d + f)
// FLOPs against 4*C*d*f for the primal apply and update -- but it writes no
// d x f snapshot per chunk, so it wins on short sequences (the planner picks
// it below T = 2.5 d f / (d + f)).
#include "kernels.h"
#include "pipeline.cuh"
#include "pipeline_pair.cuh"

namespace ittt {
namespace {

constexpr uint32_t kMnBox = 64 * 64 * 2;  // one {64 cols, 64 tokens} box

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int k) {
  return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
}
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int k) {
  return sdesc_sw128(base + uint32_t(k) * 2048u, kMnBox, 1024u);
}

struct ScoresParams {
  CUtensorMap tm_zq;    // Z [B*T, f] box {64, 128}  (rows t)
  CUtensorMap tm_zk;    // Z [B*T, f] box {64, 256}  (rows s)
  __nv_bfloat16* s;     // [B, T, T]
  int B, T, C, n, mts, mts2, kblocks;  // mts, mts2: 128- and 256-row tiles of a sequence
  int live1, live2;  // units with work per sequence: 128-row and 256-row tiles
};

// First token of the chunk of the last row of the `rows`-row tile at t0:
// the scores the tile's rows read are those of tokens s < that.
__host__ __device__ __forceinline__ int tile_s_end(int t0, int rows, int T, int C) {
  const int last = (t0 + rows < T ? t0 + rows : T) - 1;
  return (last / C) * C;
}

// The scores kernel fills, for every row, the range its 256-row group reads
// (the CTA-pair apply's tile; a 128-row tile of the single-CTA apply reads a
// part of it).
__host__ __device__ __forceinline__ int group_s_end(int t0, int T, int C) {
  return tile_s_end(t0 - t0 % (2 * kBM), 2 * kBM, T, C);
}

// Score tiles (kBN tokens s each) the rows of the `rows`-row tile m read.
__host__ __device__ __forceinline__ int score_tiles(int m, int rows, int T, int C) {
  return (group_s_end(m * rows, T, C) + kBN - 1) / kBN;
}

// Only tiles with work are units: the k-th of a sequence is row tile *m and
// score tile *nt, counting score_tiles(m) units per row tile (a short scan:
// a sequence has at most a few hundred row tiles).
__device__ __forceinline__ void live_unit(int k, int rows, int ntiles, int T, int C, int* m,
                                          int* nt) {
  int mm = 0;
  for (; mm < ntiles - 1; ++mm) {
    const int L = score_tiles(mm, rows, T, C);
    if (k < L) break;
    k -= L;
  }
  *m = mm;
  *nt = k;
}

// Row t (tile row `row` at t0) keeps the scores of tokens before its own
// chunk; the rest of the tile's range (t's chunk, when a later chunk's row
// shares the group) is written as zeros.  Chunks are multiples of 64 tokens,
// so an 8-column group lies wholly on one side.
__device__ __forceinline__ void scores_epilogue(const ScoresParams& p, int b, int t0, int s0,
                                              int rows_valid, int cols_valid, int row,
                                              uint32_t trow) {
  const bool row_ok = row < rows_valid;
  const int t = t0 + (row_ok ? row : 0);
  const int own = (t / p.C) * p.C;  // first token of t's chunk
  __nv_bfloat16* srow = p.s + (size_t(b) * p.T + size_t(t)) * size_t(p.T);
#pragma unroll 1
  for (int c = 0; c < kBN; c += 32) {
    uint32_t v[32];
    tmem_ld_32cols(trow + uint32_t(c), v);
    tmem_wait_ld();
    pin_regs(v);
    if (!row_ok) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int cc = c + 8 * q;
      if (cc < cols_valid) {
        const uint4 val =
            (s0 + cc < own)
                ? make_uint4(
                      pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                      pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                      pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                      pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])))
                : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(srow + s0 + cc) = val;
      }
    }
  }
  }

struct ScoresSched : SchedDefaults {
  using Params = ScoresParams;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN, false, false);

  const Params& p;
  int arow0 = 0, brow0 = 0, rows_valid = 0, cols_valid = 0, acc = 0, b = 0, t0 = 0, s0 = 0;
  bool live = false;

  __device__ explicit ScoresSched(const Params& pp) : p(pp) {}
  __device__ int num_units() const { return p.B * p.live1; }
  __device__ void begin_unit(int u, int local) {
    int mt = 0, nt = 0;
    b = u / p.live1;
    live_unit(u - b * p.live1, kBM, p.mts, p.T, p.C, &mt, &nt);
    t0 = mt * kBM;
    s0 = nt * kBN;
    const int s_end = group_s_end(t0, p.T, p.C);
    live = s0 < s_end;  // only tokens before the 256-row group's last chunk
    arow0 = b * p.T + t0;
    brow0 = b * p.T + s0;
    rows_valid = min(kBM, p.T - t0);
    cols_valid = min(kBN, s_end - s0);
    acc = local & 1;
  }
  __device__ int num_segments() const { return live ? 1 : 0; }
  __device__ int seg_acc(int) const { return acc; }
  __device__ int seg_kblocks(int) const { return p.kblocks; }
  __device__ bool seg_fresh(int) const { return true; }
  __device__ void load(int, int kb, uint8_t* stage, uint64_t* bar) const {
    const int k = kb * kBK;
    tma_load_2d(stage, &p.tm_zq, bar, k, arow0);
    tma_load_2d(stage + kATileBytes, &p.tm_zk, bar, k, brow0);
  }
  static __device__ uint64_t a_desc(uint32_t base, int k) { return kmajor_desc(base, k); }
  static __device__ uint64_t b_desc(uint32_t base, int k) { return kmajor_desc(base, k); }

  __device__ void epilogue(int, int row, uint32_t trow) const {
    scores_epilogue(p, b, t0, s0, rows_valid, cols_valid, row, trow);
  }
};

// The scores on CTA pairs: 256 x 256 tiles, each CTA 128 rows t and 128 of
// the tokens s (both operands Z rows, box {64, 128}).
struct ScoresPairSched : PairDefaults {
  using Params = ScoresParams;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(2 * kBM, kBN, false, false);

  const Params& p;
  const int rank;
  int arow0 = 0, brow0 = 0, rows_valid = 0, cols_valid = 0, acc = 0, b = 0, t0 = 0, s0 = 0;
  bool live = false;

  __device__ ScoresPairSched(const Params& pp, uint32_t r) : p(pp), rank(int(r)) {}
  __device__ int num_units() const { return p.B * p.live2; }
  __device__ void begin_unit(int u, int local) {
    int mt = 0, nt = 0;
    b = u / p.live2;
    live_unit(u - b * p.live2, 2 * kBM, p.mts2, p.T, p.C, &mt, &nt);
    const int g0 = mt * (2 * kBM);
    t0 = g0 + rank * kBM;
    s0 = nt * kBN;
    const int s_end = tile_s_end(g0, 2 * kBM, p.T, p.C);  // the same for both CTAs
    live = s0 < s_end;
    arow0 = b * p.T + t0;
    brow0 = b * p.T + s0 + rank * kBM;
    rows_valid = min(kBM, p.T - t0);  // <= 0: the group ends in the other half
    cols_valid = min(kBN, s_end - s0);
    acc = local & 1;
  }
  __device__ int num_segments() const { return live ? 1 : 0; }
  __device__ int seg_acc(int) const { return acc; }
  __device__ int seg_kblocks(int) const { return p.kblocks; }
  __device__ bool seg_fresh(int) const { return true; }
  __device__ void load(int, int kb, uint8_t* stage, uint32_t bar) const {
    const int k = kb * kBK;
    tma_load_2d_pair(stage, &p.tm_zq, bar, k, arow0);
    tma_load_2d_pair(stage + kPairATileBytes, &p.tm_zq, bar, k, brow0);
  }
  static __device__ uint64_t a_desc(uint32_t base, int k) { return kmajor_desc(base, k); }
  static __device__ uint64_t b_desc(uint32_t base, int k) { return kmajor_desc(base, k); }
  __device__ void epilogue(int, int row, uint32_t trow) const {
    scores_epilogue(p, b, t0, s0, rows_valid, cols_valid, row, trow);
  }
};

struct DualParams {
  CUtensorMap tm_z;   // Z        [B*T, f]   box {64, 128}
  CUtensorMap tm_w0;  // bf16 W_0 [Bw*d, f]  box {64, 256} (CTA pairs: {64, 128})
  CUtensorMap tm_s;   // scores   [B*T, T]   box {64, 128}
  CUtensorMap tm_v;   // eta*Vhat [B*T, d]   box {64, 64} (read MN-major)
  void* out;
  int out_fp32;
  int w0_per_seq;
  int B, T, d, C, n, mts, mts2, nt, kf;  // mts, mts2: 128- and 256-row tiles of a sequence
};

// 256 output columns of row `row` of a tile at token row arow0 (rows past
// rows_valid and columns past d are not written).
__device__ __forceinline__ void dual_epilogue(const DualParams& p, int arow0, int rows_valid,
                                              int n0, int row, uint32_t trow) {
  const bool row_ok = row < rows_valid;
  const size_t grow = size_t(arow0 + (row_ok ? row : 0));
#pragma unroll 1
  for (int c = 0; c < kBN; c += 32) {
    uint32_t v[32];
    tmem_ld_32cols(trow + uint32_t(c), v);
    tmem_wait_ld();
    pin_regs(v);
    if (!row_ok) continue;
    if (p.out_fp32) {
      float* orow = static_cast<float*>(p.out) + grow * size_t(p.d);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int col = n0 + c + 4 * q;
        if (col < p.d)
          *reinterpret_cast<uint4*>(orow + col) =
              make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    } else {
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + grow * size_t(p.d);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int col = n0 + c + 8 * q;
        if (col < p.d)
          *reinterpret_cast<uint4*>(orow + col) = make_uint4(
              pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
              pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
              pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
              pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
      }
    }
  }
}

struct DualSched : SchedDefaults {
  using Params = DualParams;
  static constexpr bool kMixedOperands = true;
  static constexpr uint32_t kIdescKK = idesc_bf16_f32(kBM, kBN, false, false);
  static constexpr uint32_t kIdescKM = idesc_bf16_f32(kBM, kBN, false, true);
  static constexpr uint32_t kIdesc = kIdescKK;

  const Params& p;
  int b = 0, s_end = 0, arow0 = 0, n0 = 0, rows_valid = 0, acc = 0, wrow0 = 0;

  __device__ explicit DualSched(const Params& pp) : p(pp) {}
  __device__ int num_units() const { return p.B * p.mts * p.nt; }
  // Latest tiles (longest K) first.
  __device__ void begin_unit(int u, int local) {
    const int nt = u % p.nt;
    const int r = u / p.nt;
    const int mt = p.mts - 1 - (r % p.mts);
    b = r / p.mts;
    const int t0 = mt * kBM;
    s_end = tile_s_end(t0, kBM, p.T, p.C);
    arow0 = b * p.T + t0;
    n0 = nt * kBN;
    rows_valid = min(kBM, p.T - t0);
    wrow0 = (p.w0_per_seq ? b * p.d : 0) + n0;
    acc = local & 1;
  }
  __device__ int num_segments() const { return 1; }
  __device__ int seg_acc(int) const { return acc; }
  __device__ int seg_kblocks(int) const { return p.kf + s_end / kBK; }
  __device__ bool seg_fresh(int) const { return true; }

  __device__ void load(int, int kb, uint8_t* stage, uint64_t* bar) const {
    if (kb < p.kf) {
      const int k = kb * kBK;
      tma_load_2d(stage, &p.tm_z, bar, k, arow0);
      tma_load_2d(stage + kATileBytes, &p.tm_w0, bar, k, wrow0);
    } else {
      const int s0 = (kb - p.kf) * kBK;  // token of an earlier chunk
      tma_load_2d(stage, &p.tm_s, bar, s0, arow0);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        tma_load_2d(stage + kATileBytes + q * kMnBox, &p.tm_v, bar, n0 + 64 * q, b * p.T + s0);
    }
  }
  __device__ uint32_t idesc(int, int kb) const { return kb < p.kf ? kIdescKK : kIdescKM; }
  __device__ uint64_t a_desc(int, int, uint32_t base, int k) const { return kmajor_desc(base, k); }
  __device__ uint64_t b_desc(int, int kb, uint32_t base, int k) const {
    return kb < p.kf ? kmajor_desc(base, k) : mnmajor_desc(base, k);
  }

  __device__ void epilogue(int, int row, uint32_t trow) const {
    dual_epilogue(p, arow0, rows_valid, n0, row, trow);
  }
};

// The same on CTA pairs: 256-row tiles (each CTA its 128 rows of Z or of the
// scores, and 128 of the 256 output columns' W_0 rows or eta*Vhat columns),
// both CTAs' rows sharing one scores range.
struct DualPairSched : PairDefaults {
  using Params = DualParams;
  static constexpr bool kMixedOperands = true;
  static constexpr uint32_t kIdescKK = idesc_bf16_f32(2 * kBM, kBN, false, false);
  static constexpr uint32_t kIdescKM = idesc_bf16_f32(2 * kBM, kBN, false, true);
  static constexpr uint32_t kIdesc = kIdescKK;

  const Params& p;
  const int rank;
  int b = 0, s_end = 0, arow0 = 0, n0 = 0, rows_valid = 0, acc = 0, wrow0 = 0;

  __device__ DualPairSched(const Params& pp, uint32_t r) : p(pp), rank(int(r)) {}
  __device__ int num_units() const { return p.B * p.mts2 * p.nt; }
  // Latest tiles (longest K) first.
  __device__ void begin_unit(int u, int local) {
    const int nt = u % p.nt;
    const int r = u / p.nt;
    const int mt = p.mts2 - 1 - (r % p.mts2);
    b = r / p.mts2;
    const int t0 = mt * (2 * kBM);
    s_end = tile_s_end(t0, 2 * kBM, p.T, p.C);
    const int r0 = t0 + rank * kBM;  // this CTA's first row in the sequence
    arow0 = b * p.T + r0;
    n0 = nt * kBN;
    rows_valid = min(kBM, p.T - r0);  // <= 0: the tile ends in the other half
    wrow0 = (p.w0_per_seq ? b * p.d : 0) + n0 + rank * kBM;
    acc = local & 1;
  }
  __device__ int num_segments() const { return 1; }
  __device__ int seg_acc(int) const { return acc; }
  __device__ int seg_kblocks(int) const { return p.kf + s_end / kBK; }
  __device__ bool seg_fresh(int) const { return true; }
  __device__ void load(int, int kb, uint8_t* stage, uint32_t bar) const {
    if (kb < p.kf) {
      const int k = kb * kBK;
      tma_load_2d_pair(stage, &p.tm_z, bar, k, arow0);
      tma_load_2d_pair(stage + kPairATileBytes, &p.tm_w0, bar, k, wrow0);
    } else {
      const int s0 = (kb - p.kf) * kBK;  // token of an earlier chunk
      tma_load_2d_pair(stage, &p.tm_s, bar, s0, arow0);
#pragma unroll
      for (int q = 0; q < 2; ++q)
        tma_load_2d_pair(stage + kPairATileBytes + q * kMnBox, &p.tm_v, bar,
                         n0 + rank * kBM + 64 * q, b * p.T + s0);
    }
  }
  __device__ uint32_t idesc(int, int kb) const { return kb < p.kf ? kIdescKK : kIdescKM; }
  __device__ uint64_t a_desc(int, int, uint32_t base, int k) const { return kmajor_desc(base, k); }
  __device__ uint64_t b_desc(int, int kb, uint32_t base, int k) const {
    return kb < p.kf ? kmajor_desc(base, k) : mnmajor_desc(base, k);
  }
  __device__ void epilogue(int, int row, uint32_t trow) const {
    dual_epilogue(p, arow0, rows_valid, n0, row, trow);
  }
};

__global__ void __launch_bounds__(PipeShape<ScoresSched>::kThreads, 1)
    scores_kernel(const __grid_constant__ ScoresParams p, unsigned int* status) {
  run_pipeline<ScoresSched>(p, status);
}

__global__ void __launch_bounds__(kBaseThreads, 1)
    scores_pair_kernel(const __grid_constant__ ScoresParams p, unsigned int* status) {
  run_pipeline_pair<ScoresPairSched>(p, status);
}

__global__ void __launch_bounds__(PipeShape<DualSched>::kThreads, 1)
    dual_apply_kernel(const __grid_constant__ DualParams p, unsigned int* status) {
  run_pipeline<DualSched>(p, status);
}

__global__ void __launch_bounds__(kBaseThreads, 1)
    dual_apply_pair_kernel(const __grid_constant__ DualParams p, unsigned int* status) {
  run_pipeline_pair<DualPairSched>(p, status);
}

}  // namespace

cudaError_t launch_scores(const LaunchEnv& env, const CUtensorMap& tm_zq, const CUtensorMap& tm_zk,
                          __nv_bfloat16* s, int B, int T, int f, int C, bool allow_pairs) {
  ScoresParams p;
  p.tm_zq = tm_zq;
  p.tm_zk = tm_zk;
  p.s = s;
  p.B = B;
  p.T = T;
  p.C = C;
  p.n = T / C;
  p.mts = (T + kBM - 1) / kBM;
  p.mts2 = (T + 2 * kBM - 1) / (2 * kBM);
  p.kblocks = (f + kBK - 1) / kBK;
  p.live1 = p.live2 = 0;
  for (int m = 0; m < p.mts; ++m) p.live1 += score_tiles(m, kBM, T, C);
  for (int m = 0; m < p.mts2; ++m) p.live2 += score_tiles(m, 2 * kBM, T, C);
  if (p.n < 2 || p.live1 == 0) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  if (allow_pairs) {
    const size_t smem = pair_smem_bytes<ScoresPairSched>();
    if ((e = cudaFuncSetAttribute(scores_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(smem))) != cudaSuccess)
      return e;
    static std::atomic<int> resident{-1};
    int pairs = 0;
    if ((e = max_pairs(reinterpret_cast<const void*>(scores_pair_kernel), smem, env, &pairs,
                       &resident)) != cudaSuccess)
      return e;
    if (pairs >= 1) {
      const int64_t units = int64_t(B) * p.live2;
      return launch_on_pairs(reinterpret_cast<const void*>(scores_pair_kernel),
                             int(units < pairs ? units : pairs), smem, env, &p);
    }
  }
  const int64_t units = int64_t(B) * p.live1;
  e = cudaFuncSetAttribute(scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(pipe_smem_bytes<ScoresSched>()));
  if (e != cudaSuccess) return e;
  const int grid = units < env.num_sms ? int(units) : env.num_sms;
  return launch_pdl(scores_kernel, dim3(grid), dim3(PipeShape<ScoresSched>::kThreads),
                    pipe_smem_bytes<ScoresSched>(), env.stream, p, env.status);
}

cudaError_t launch_dual_apply(const LaunchEnv& env, const CUtensorMap& tm_z,
                              const CUtensorMap& tm_w0, const CUtensorMap& tm_w0_pair,
                              const CUtensorMap& tm_s, const CUtensorMap& tm_v, bool w0_per_seq,
                              void* out, bool out_fp32, int B, int T, int d, int f, int C,
                              bool allow_pairs) {
  DualParams p;
  p.tm_z = tm_z;
  p.tm_w0 = tm_w0;
  p.tm_s = tm_s;
  p.tm_v = tm_v;
  p.out = out;
  p.out_fp32 = out_fp32 ? 1 : 0;
  p.w0_per_seq = w0_per_seq ? 1 : 0;
  p.B = B;
  p.T = T;
  p.d = d;
  p.C = C;
  p.n = T / C;
  p.mts = (T + kBM - 1) / kBM;
  p.mts2 = (T + 2 * kBM - 1) / (2 * kBM);
  p.nt = (d + kBN - 1) / kBN;
  p.kf = (f + kBK - 1) / kBK;
  cudaError_t e = cudaSuccess;
  if (allow_pairs) {
    // CTA pairs where two can be resident: 256-row tiles.
    DualParams q = p;
    q.tm_w0 = tm_w0_pair;
    const size_t smem = pair_smem_bytes<DualPairSched>();
    if ((e = cudaFuncSetAttribute(dual_apply_pair_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) !=
        cudaSuccess)
      return e;
    static std::atomic<int> resident{-1};
    int pairs = 0;
    if ((e = max_pairs(reinterpret_cast<const void*>(dual_apply_pair_kernel), smem, env, &pairs,
                       &resident)) != cudaSuccess)
      return e;
    if (pairs >= 1) {
      const int64_t units = int64_t(B) * q.mts2 * q.nt;
      return launch_on_pairs(reinterpret_cast<const void*>(dual_apply_pair_kernel),
                             int(units < pairs ? units : pairs), smem, env, &q);
    }
  }
  const int64_t units = int64_t(B) * p.mts * p.nt;
  e = cudaFuncSetAttribute(dual_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(pipe_smem_bytes<DualSched>()));
  if (e != cudaSuccess) return e;
  const int grid = units < env.num_sms ? int(units) : env.num_sms;
  return launch_pdl(dual_apply_kernel, dim3(grid), dim3(PipeShape<DualSched>::kThreads),
                    pipe_smem_bytes<DualSched>(), env.stream, p, env.status);
}

}  // namespace ittt
