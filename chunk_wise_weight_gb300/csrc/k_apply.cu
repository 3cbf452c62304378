// k_apply.cu -- apply step for every chunk of every document in one launch:
//   O_[i] = Z_[i] W_i^T
// ("[논문리뷰] In-Place Test-Time Training", Method §1 eq. (3); all chunks in
// parallel as in Method §3 stage 3).
//
// W_i is the bf16 snapshot the update kernel wrote into the chunk's slot
// (a document's first slot holds W_0; when W_0 is one shared bf16 matrix
// and no caller snapshot buffer is given, first chunks read W_0 itself and
// that slot is never written).  A work unit is (128-row tile of a
// chunk, 256-column tile of d_model); only tiles that hold rows of their
// chunk are enumerated (slot order), so short chunks leave no idle units in
// the persistent schedule.  Rows past the chunk's end belong to another
// chunk: they are computed but not stored.
// Full tiles and 64-row halves leave through TMA stores; a tile that ends
// elsewhere (a chunk or document length that is not a multiple of 64) is
// written row by row with masked 16-byte stores.
#include "kernels.h"
#include "pipeline.cuh"
#include "pipeline_pair.cuh"

namespace ittt {
namespace {

struct ApplyParams {
  CUtensorMap tm_z;     // Z          [M, f]        box {64, 128}
  CUtensorMap tm_snap;  // snapshots  [slots*d, f]  box {64, 256} (pairs: {64, 128})
  CUtensorMap tm_w0;    // bf16 W_0   [d, f], same box; read for first chunks when w0_direct
  CUtensorMap tm_os;    // bf16 O     [M, d]        box {64, 64} (store)
  void* out;            // O [M, d], bf16 or fp32
  int out_fp32;
  DocMap docs;
  int w0_direct;        // a document's first chunk reads W_0 itself, not its snapshot slot
  int d, f;
  int nt, kblocks;
  unsigned int* ticket;  // the pair kernel's unit counter (LaunchEnv::tickets)
  // CTA pairs: units [0, nfull) whole; each later unit (the partial last
  // round) as ksplit pieces over consecutive K ranges, whose fp32 partials
  // go to part and whose arrivals count in tail_ctr.
  int nfull, ksplit;
  float* part;
  unsigned int* tail_ctr;
};

// bf16 O in whole 64-row halves: 64-column TMA stores (columns >= d are
// clipped).  Otherwise (fp32 O, or a tile that ends inside a 64-row half):
// direct 16-byte stores of the valid rows.
__device__ __forceinline__ void apply_epilogue(const ApplyParams& p, int arow0, int rows_valid,
                                               int n0, int row, uint32_t trow, EpiStager& st) {
  if (!p.out_fp32 && (rows_valid == kBM || rows_valid == 64)) {
#pragma unroll 1
    for (int g = 0; g < kBN / 64; ++g) {
      uint8_t* buf = st.acquire();
#pragma unroll 1
      for (int hc = 0; hc < 2; ++hc) {
        uint32_t v[32];
        tmem_ld_32cols(trow + uint32_t(g * 64 + hc * 32), v);
        tmem_wait_ld();
        pin_regs(v);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st.put(buf, hc * 4 + q,
                 make_uint4(
                     pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                     pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                     pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                     pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]))));
      }
      st.commit(buf, [&](uint8_t* src) {
        tma_store_2d(&p.tm_os, src, n0 + g * 64, arow0);
        if (rows_valid > 64) tma_store_2d(&p.tm_os, src + 64 * 128, n0 + g * 64, arow0 + 64);
      });
    }
    return;
  }
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
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int col = n0 + c + 8 * q;
        if (col < p.d)
          *reinterpret_cast<uint4*>(orow + col) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
    }
  }
}

struct ApplySched : SchedDefaults {
  using Params = ApplyParams;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN, false, false);
  static constexpr bool kStagedStores = true;

  const Params& p;
  int arow0 = 0, brow0 = 0, rows_valid = 0, n0 = 0, acc = 0;
  const CUtensorMap* bmap = nullptr;

  __device__ explicit ApplySched(const Params& pp) : p(pp) {}
  __device__ int num_units() const { return p.docs.ntiles * p.nt; }
  __device__ void begin_unit(int u, int local) {
    const int nt = u % p.nt;
    int mt = 0;
    const int g = p.docs.slot_of_tile(u / p.nt, &mt);
    const int k = p.docs.doc_of_chunk(g);
    const int i = g - p.docs.first_chunk(k);
    const int len = p.docs.len(k);
    arow0 = p.docs.start(k) + i * p.docs.C + mt * kBM;
    const bool first = i == 0 && p.w0_direct;
    bmap = first ? &p.tm_w0 : &p.tm_snap;
    brow0 = (first ? 0 : g * p.d) + nt * kBN;
    rows_valid = min(kBM, min(p.docs.C, len - i * p.docs.C) - mt * kBM);
    n0 = nt * kBN;
    acc = local & 1;
  }
  __device__ int num_segments() const { return rows_valid > 0 ? 1 : 0; }
  __device__ int seg_acc(int) const { return acc; }
  __device__ int seg_kblocks(int) const { return p.kblocks; }
  __device__ bool seg_fresh(int) const { return true; }

  __device__ void load(int, int kb, uint8_t* stage, uint64_t* bar) const {
    const int k = kb * kBK;
    tma_load_2d(stage, &p.tm_z, bar, k, arow0);
    tma_load_2d(stage + kATileBytes, bmap, bar, k, brow0);
  }
  static __device__ uint64_t a_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }
  static __device__ uint64_t b_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }

  __device__ void epilogue(int, int row, uint32_t trow, EpiStager& st) const {
    apply_epilogue(p, arow0, rows_valid, n0, row, trow, st);
  }
};

__global__ void __launch_bounds__(PipeShape<ApplySched>::kThreads, 1)
    apply_kernel(const __grid_constant__ ApplyParams p, unsigned int* status) {
  run_pipeline<ApplySched>(p, status);
}

// CTA pairs: a unit is (256-row tile of a chunk, 256-column tile of d);
// this CTA holds rows [128 rank, 128 rank + 128) of the tile and loads the
// snapshot rows of its 128 columns.
struct ApplyPairSched : PairDefaults {
  using Params = ApplyParams;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(2 * kBM, kBN, false, false);
  static constexpr bool kStagedStores = true;
  static constexpr bool kDynamicUnits = true;

  const Params& p;
  const int rank;
  int arow0 = 0, brow0 = 0, rows_valid = 0, n0 = 0, acc = 0;
  int kb0 = 0, nkb = 0, piece = -1, tail = 0;  // K range; piece of a tail unit (-1: whole)
  const CUtensorMap* bmap = nullptr;

  __device__ ApplyPairSched(const Params& pp, uint32_t r) : p(pp), rank(int(r)) {}
  __device__ unsigned int* unit_ticket() const { return p.ticket; }
  __device__ int num_units() const {
    return p.nfull + (p.docs.ntiles2 * p.nt - p.nfull) * p.ksplit;
  }
  __device__ void begin_unit(int u, int local) {
    int w = u;
    piece = -1;
    kb0 = 0;
    nkb = p.kblocks;
    if (u >= p.nfull) {
      const int q = u - p.nfull;
      tail = q / p.ksplit;
      piece = q - tail * p.ksplit;
      w = p.nfull + tail;
      kb0 = piece * p.kblocks / p.ksplit;
      nkb = (piece + 1) * p.kblocks / p.ksplit - kb0;
    }
    const int nt = w % p.nt;
    int mt = 0;
    const int g = p.docs.slot_of_tile(w / p.nt, &mt, true);
    const int k = p.docs.doc_of_chunk(g);
    const int i = g - p.docs.first_chunk(k);
    const int len = p.docs.len(k);
    const int r0 = mt * (2 * kBM) + rank * kBM;  // first row of this CTA's half in the chunk
    arow0 = p.docs.start(k) + i * p.docs.C + r0;
    const bool first = i == 0 && p.w0_direct;
    bmap = first ? &p.tm_w0 : &p.tm_snap;
    brow0 = (first ? 0 : g * p.d) + nt * kBN + rank * kBM;
    rows_valid = min(kBM, min(p.docs.C, len - i * p.docs.C) - r0);
    n0 = nt * kBN;
    acc = local & 1;
  }
  __device__ int num_segments() const { return 1; }
  __device__ int seg_acc(int) const { return acc; }
  __device__ int seg_kblocks(int) const { return nkb; }
  __device__ bool seg_fresh(int) const { return true; }
  __device__ void load(int, int kb, uint8_t* stage, uint32_t bar) const {
    const int k = (kb0 + kb) * kBK;
    tma_load_2d_pair(stage, &p.tm_z, bar, k, arow0);
    tma_load_2d_pair(stage + kPairATileBytes, bmap, bar, k, brow0);
  }
  static __device__ uint64_t a_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }
  static __device__ uint64_t b_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }
  // The second half of a tile may lie past its chunk (rows_valid <= 0):
  // computed, nothing stored.
  __device__ void epilogue(int, int row, uint32_t trow, EpiStager& st) const {
    if (piece >= 0 && !sum_pieces(row, trow, st)) return;
    apply_epilogue(p, arow0, rows_valid, n0, row, trow, st);
  }

  // A piece of a split unit: publish this CTA's fp32 partial (its 128 rows),
  // count the arrival, and -- in the CTA that completes the count -- add the
  // pieces' partials in piece order into TMEM (true: the caller stores the
  // sum as the unit's output).  Nobody waits for another CTA here.
  __device__ bool sum_pieces(int row, uint32_t trow, EpiStager& st) const {
    // A piece's partial (both CTAs, 2 x 128 rows x 256 columns) is stored
    // column-group-major: [64 groups of 4 columns][128 rows][4], so a warp's
    // 16-byte accesses to one group cover 512 contiguous bytes.
    const size_t tile = size_t(2 * kBM) * kBN;
    float4* base = reinterpret_cast<float4*>(p.part + size_t(tail) * p.ksplit * tile +
                                             size_t(rank) * kBM * kBN) + row;
    float4* mine = base + size_t(piece) * (tile / 4);
#pragma unroll 1
    for (int c = 0; c < kBN; c += 32) {
      uint32_t v[32];
      tmem_ld_32cols(trow + uint32_t(c), v);
      tmem_wait_ld();
      pin_regs(v);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        __stcg(mine + size_t(c / 4 + q) * kBM,
               make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                           __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])));
    }
    __threadfence();  // this row's partial before the arrival below
    // A staging buffer (not stored from) carries the verdict to every row.
    volatile int* flag = reinterpret_cast<volatile int*>(st.acquire());
    if (row == 0)
      *flag = atomicAdd(p.tail_ctr + 2 * tail + rank, 1u) == unsigned(p.ksplit - 1) ? 1 : 0;
    epilogue_group_bar(st.group);
    const bool last = *flag != 0;
    epilogue_group_bar(st.group);
    if (!last) return false;
    __threadfence();  // the other pieces' partials after their arrivals
    // 32 columns per step: every other piece's loads are issued before the
    // sum, which then adds the pieces in order.
#pragma unroll 1
    for (int c = 0; c < kBN; c += 32) {
      float4 x[4][8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q < p.ksplit && q != piece) {
          const float4* src = base + size_t(q) * (tile / 4) + size_t(c / 4) * kBM;
#pragma unroll
          for (int j = 0; j < 8; ++j) x[q][j] = __ldcg(src + size_t(j) * kBM);
        }
      }
      uint32_t v[32];
      tmem_ld_32cols(trow + uint32_t(c), v);
      tmem_wait_ld();
      pin_regs(v);
      float sum[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) sum[j] = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q < p.ksplit) {
          if (q == piece) {
#pragma unroll
            for (int j = 0; j < 32; ++j) sum[j] += __uint_as_float(v[j]);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              sum[4 * j] += x[q][j].x;
              sum[4 * j + 1] += x[q][j].y;
              sum[4 * j + 2] += x[q][j].z;
              sum[4 * j + 3] += x[q][j].w;
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(sum[j]);
      tmem_st_32cols(trow + uint32_t(c), v);
    }
    tmem_wait_st();
    return true;
  }
};

__global__ void __launch_bounds__(kBaseThreads, 1)
    apply_pair_kernel(const __grid_constant__ ApplyParams p, unsigned int* status) {
  run_pipeline_pair<ApplyPairSched>(p, status);
}

}  // namespace

cudaError_t launch_apply_pair(const LaunchEnv& env, const CUtensorMap& tm_z,
                              const CUtensorMap& tm_snap, const CUtensorMap* tm_w0,
                              const CUtensorMap& tm_os, void* out, bool out_fp32,
                              const DocMap& docs, int d, int f) {
  ApplyParams p;
  p.tm_z = tm_z;
  p.tm_snap = tm_snap;
  p.w0_direct = tm_w0 != nullptr ? 1 : 0;
  p.tm_w0 = tm_w0 != nullptr ? *tm_w0 : tm_snap;
  p.tm_os = tm_os;
  p.out = out;
  p.out_fp32 = out_fp32 ? 1 : 0;
  p.docs = docs;
  p.d = d;
  p.f = f;
  p.nt = (d + kBN - 1) / kBN;
  p.kblocks = (f + kBK - 1) / kBK;
  p.ticket = env.tickets != nullptr ? env.tickets + kTicketApply : nullptr;
  if (p.ticket == nullptr) return cudaErrorInvalidValue;
  const int64_t units = int64_t(docs.ntiles2) * p.nt;
  if (units == 0) return cudaSuccess;
  const size_t smem = pair_smem_bytes<ApplyPairSched>();
  cudaError_t e = cudaFuncSetAttribute(apply_pair_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  static std::atomic<int> resident{-1};
  int pairs = 0;
  if ((e = max_pairs(reinterpret_cast<const void*>(apply_pair_kernel), smem, env, &pairs,
                     &resident)) != cudaSuccess)
    return e;
  if (pairs < 1) return cudaErrorNotSupported;
  // A partial last round of t units (after at least two full rounds) runs
  // each unit as S pieces over disjoint K ranges, S <= 4 and t S <= pairs,
  // so that round takes about 1/S of a unit's MMAs plus the partials' round
  // trip (1 x 8192 tokens: 320 units on 76 pairs, t = 16, S = 4; the apply
  // 247.6 -> 228.4 us in a per-unit trace).
  p.nfull = int(units);
  p.ksplit = 1;
  p.part = nullptr;
  p.tail_ctr = nullptr;
  const int64_t t = units % pairs;
  if (env.apply_part != nullptr && units >= 2 * int64_t(pairs) && t > 0 && 2 * t <= pairs) {
    int S = int(pairs / t);
    S = S < 4 ? S : 4;
    S = S < p.kblocks ? S : p.kblocks;
    if (S >= 2 && t * S <= kMaxApplyTailPieces) {
      p.nfull = int(units - t);
      p.ksplit = S;
      p.part = env.apply_part;
      p.tail_ctr = env.tickets + kTicketApplyTail;
    }
  }
  const int64_t total = p.nfull + (units - p.nfull) * p.ksplit;
  if (total < pairs) pairs = int(total);
  return launch_on_pairs(reinterpret_cast<const void*>(apply_pair_kernel), pairs, smem, env, &p);
}

cudaError_t launch_apply(const LaunchEnv& env, const CUtensorMap& tm_z, const CUtensorMap& tm_snap,
                         const CUtensorMap* tm_w0, const CUtensorMap& tm_os, void* out,
                         bool out_fp32, const DocMap& docs, int d, int f) {
  ApplyParams p;
  p.ticket = nullptr;  // one CTA per SM: fixed stride, no split round
  p.nfull = 0;
  p.ksplit = 1;
  p.part = nullptr;
  p.tail_ctr = nullptr;
  p.tm_z = tm_z;
  p.tm_snap = tm_snap;
  p.w0_direct = tm_w0 != nullptr ? 1 : 0;
  p.tm_w0 = tm_w0 != nullptr ? *tm_w0 : tm_snap;
  p.tm_os = tm_os;
  p.out = out;
  p.out_fp32 = out_fp32 ? 1 : 0;
  p.docs = docs;
  p.d = d;
  p.f = f;
  p.nt = (d + kBN - 1) / kBN;
  p.kblocks = (f + kBK - 1) / kBK;
  const int64_t units = int64_t(docs.ntiles) * p.nt;
  if (units == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(pipe_smem_bytes<ApplySched>()));
  if (e != cudaSuccess) return e;
  const int grid = units < env.num_sms ? int(units) : env.num_sms;
  return launch_pdl(apply_kernel, dim3(grid), dim3(PipeShape<ApplySched>::kThreads),
                    pipe_smem_bytes<ApplySched>(), env.stream, p, env.status);
}

}  // namespace ittt
