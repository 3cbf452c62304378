// k_update.cu -- the fast-weight update, walked chunk by chunk:
//   W_{i+1} = W_i + eta * Vhat_[i]^T Z_[i]
// ("[논문리뷰] In-Place Test-Time Training", Method §2 eq. (6); the prefix
// sum of Method §3 stage 2, "In-Place TTT" reading notes 实现细节).
//
// The per-chunk deltas do not depend on W (the loss is linear in it), so
// the state after chunk i is W_0 plus one long contraction over the tokens
// of chunks 0..i.  A work unit owns two 128 (d_model) x 256 (d_ff) blocks
// ("halves") of the state.  Each half's fp32 state lives in one TMEM
// accumulator for the whole walk: the epilogue warps load W_0 into it
// (tcgen05.st) and the MMAs accumulate (eta Vhat_[i])^T Z_[i] on top, eta
// having been folded into Vhat by the target kernel.  The MMAs alternate
// halves chunk by chunk: while the tensor core accumulates chunk i of one
// half, the epilogue reads the other half's state at its chunk boundary and
// writes the bf16 snapshot W_{i+1} that the apply kernel reads.  The fp32 state reaches HBM only when the caller asks
// for the final state.
//
// Both operands are read MN-major: the contraction index (token) is the row
// index of Vhat [T, d] and of Z [T, f].  A 64-token stage holds, per operand,
// 64-column TMA boxes of 64 token lines x 128 bytes each.  A chunk whose
// length is not a multiple of 64 ends inside a stage: the MMA thread zeroes
// the token lines past its end (within the last 16-token slice it issues)
// and skips the slices after them.
#include <type_traits>

#include "kernels.h"
#include "pipeline.cuh"
#include "pipeline_pair.cuh"

namespace ittt {
namespace {

constexpr uint32_t kMnBoxBytes = 64 * 64 * 2;  // one {64 cols, 64 tokens} box

// One 64-token stage of the update: eta*Vhat^T rows m0..m0+127 (A, two
// boxes) and Z columns n0..n0+255 (B, four boxes) of tokens tok..tok+63.
__device__ __forceinline__ void load_update_stage(const CUtensorMap& tm_v, const CUtensorMap& tm_z,
                                                  uint8_t* stage, uint64_t* bar, int m0, int n0,
                                                  int tok) {
  uint8_t* sb = stage + kATileBytes;
  tma_load_2d(stage, &tm_v, bar, m0, tok);
  tma_load_2d(stage + kMnBoxBytes, &tm_v, bar, m0 + 64, tok);
#pragma unroll
  for (int q = 0; q < 4; ++q) tma_load_2d(sb + q * kMnBoxBytes, &tm_z, bar, n0 + 64 * q, tok);
}

// Token lines [from, to) of both operands' boxes read zero: tokens past the
// chunk's end (another chunk's) must not enter its sum.  A whole 128-byte
// line is one token, so the swizzle does not matter here.
__device__ __forceinline__ void clear_token_lines(uint8_t* stage, int from, int to) {
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
  for (int box = 0; box < 6; ++box) {
    uint4* line = reinterpret_cast<uint4*>(stage + box * kMnBoxBytes);
#pragma unroll 1
    for (int t = from; t < to; ++t)
#pragma unroll
      for (int c = 0; c < 8; ++c) line[t * 8 + c] = zero;
  }
}

// MN-major, 128-byte swizzle: a 16-token slice is 16 lines of 128 B; the
// 64-column groups of the tile are one box (lbo) apart.
__device__ __forceinline__ uint64_t mn_desc(uint32_t base, int k) {
  return sdesc_sw128(base + uint32_t(k) * 2048u, kMnBoxBytes, 1024u);
}

// Eight fp32 values of the initial state W_0 (bf16 or fp32 source; zeros
// outside the [d, f] state, and everywhere when w0 is null: a zero start).
__device__ __forceinline__ void load_w0_8(const void* w0, bool fp32, size_t off, bool ok,
                                          float* w) {
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = 0.f;
  if (!ok || w0 == nullptr) return;
  if (fp32) {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(w0) + off);
    const float4 lo = __ldg(src), hi = __ldg(src + 1);
    w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
    w[4] = hi.x; w[5] = hi.y; w[6] = hi.z; w[7] = hi.w;
  } else {
    const uint4 raw =
        __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(w0) + off));
    const uint32_t r4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f2 = unpack_bf16x2(r4[j]);
      w[2 * j] = f2.x;
      w[2 * j + 1] = f2.y;
    }
  }
}

struct UpdateParams {
  CUtensorMap tm_v;  // eta*Vhat [M, d]  box {64, 64}
  CUtensorMap tm_z;  // Z        [M, f]  box {64, 64}
  CUtensorMap tm_ss; // snapshots as [slots][d rows][f cols], box {64, 128, 1} (store)
  const void* w0;
  int w0_fp32;
  int64_t w0_bstride;   // elements between documents' initial states (0: shared)
  float* state_out;     // [documents, d, f] or nullptr
  DocMap docs;
  const int* upd_docs;  // documents that update, longest first; nullptr: all
  int n_udocs;
  int final_update;     // also update with the last chunk (for state_out)
  int d, f;
  int MT, NH, NP;       // row blocks of d_model (128 rows, 256 on CTA pairs);
                        // 256- and 512-column blocks of d_ff
  int P;                // pairs of halves: documents x MT x NP
  int RG;               // pairs walked whole: full rounds over the grid
  int split;            // the last partial round walks its halves one by one
};

// A unit is a pair of 128 (d_model) x 256 (d_ff) state blocks, (document,
// 512-column block, 128-row block) listed d_model block fastest: the CTAs
// of one round over the grid share the same document's chunks and Z column
// blocks, so those stream from DRAM about once.  The MMAs of a pair
// alternate chunk by chunk, so each chunk-boundary epilogue of one half
// overlaps the other half's MMAs.  When the pairs do not fill the last round
// (Q pairs left, 2Q <= CTAs) those pairs are walked as 2Q single halves on
// as many CTAs, which shortens the longest CTA by one half-walk.
//
// On CTA pairs (kPair; every chunk a multiple of 64 tokens) a block is 256
// d_model rows: each CTA keeps its 128 rows of eta*Vhat^T and 128 of the
// half's 256 Z columns in shared memory, and its 128 state rows of both
// halves in its own TMEM.
// W_0 (bf16 or fp32, rows of f elements, the document's at doc_off) rows
// [m0, m0 + 128) x columns [n0, n0 + 256) into this epilogue group's TMEM
// rows (zeros outside [d, f], or everywhere without W_0).  The rows are
// read coalesced: per pass the group's 128 threads load the block's 128
// rows x 128 bytes (four rows per warp instruction) into a staging tile,
// then each thread takes its own row from shared memory into TMEM.  (One
// thread per row, each warp load touching 32 rows, took ~11 us and held up
// the first chunks of every unit.)
__device__ __forceinline__ void preload_w0_staged(const void* w0v, bool f32, size_t doc_off,
                                                  int m0, int n0, int d, int f, int row,
                                                  uint32_t trow, EpiStager& st) {
  const size_t es = f32 ? 4 : 2;
  const int cols = int(128 / es);  // columns per pass: 64 bf16 or 32 fp32
  const char* w0 = static_cast<const char*>(w0v);
#pragma unroll 1
  for (int c0 = 0; c0 < kBN; c0 += cols) {
    uint8_t* buf = st.acquire();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int idx = i * kEpilogueThreads + row;  // 16-byte piece of the tile
      const int r = idx >> 3, ch = idx & 7;
      const int m = m0 + r;
      const int col = n0 + c0 + ch * int(16 / es);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (w0 != nullptr && m < d && col < f)
        v = __ldg(reinterpret_cast<const uint4*>(w0 + (doc_off + size_t(m) * f + col) * es));
      *reinterpret_cast<uint4*>(buf + r * 128 + ((ch ^ (r & 7)) << 4)) = v;
    }
    epilogue_group_bar(st.group);
    const uint8_t* mine = buf + row * 128;
    if (f32) {
      uint32_t v[32];
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint4 x = *reinterpret_cast<const uint4*>(mine + ((ch ^ (row & 7)) << 4));
        v[4 * ch] = x.x;
        v[4 * ch + 1] = x.y;
        v[4 * ch + 2] = x.z;
        v[4 * ch + 3] = x.w;
      }
      tmem_st_32cols(trow + uint32_t(c0), v);
    } else {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t v[32];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int ch = 4 * half + k;
          const uint4 x = *reinterpret_cast<const uint4*>(mine + ((ch ^ (row & 7)) << 4));
          const uint32_t r4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f2 = unpack_bf16x2(r4[j]);
            v[8 * k + 2 * j] = __float_as_uint(f2.x);
            v[8 * k + 2 * j + 1] = __float_as_uint(f2.y);
          }
        }
        tmem_st_32cols(trow + uint32_t(c0 + 32 * half), v);
      }
    }
    epilogue_group_bar(st.group);  // every row taken before the next pass refills the tile
  }
}

template <bool kPair>
struct UpdateSchedT : std::conditional_t<kPair, PairDefaults, SchedDefaults> {
  using Params = UpdateParams;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(kPair ? 2 * kBM : kBM, kBN, true, true);
  static constexpr bool kPreload = true;
  static constexpr bool kStagedStores = true;
  static constexpr bool kRaggedK = !kPair;
  static constexpr bool kStagedPreload = true;  // W_0 read coalesced through a staging tile
  static constexpr bool kEarlyRelease = kPair;
  static constexpr bool kPrefetchPreload = kPair;

  const Params& p;
  const int rank;
  int nh = 0;                 // halves in this unit (0, 1 or 2)
  int doc = 0, m0 = 0, tok0 = 0, slot0 = 0;
  int hn0[2] = {0, 0};        // first d_ff column of each half
  int len = 0, nch = 0, nupd = 0;

  __device__ explicit UpdateSchedT(const Params& pp, uint32_t r = 0) : p(pp), rank(int(r)) {}
  __device__ int num_units() const {
    return p.split ? p.RG + 2 * (p.P - p.RG) : p.P;
  }
  __device__ void begin_unit(int u, int) {
    int pi = u, first = 0, want = 2;
    if (p.split && u >= p.RG) {
      pi = p.RG + (u - p.RG) / 2;
      first = (u - p.RG) % 2;
      want = 1;
    }
    const int q = pi / (p.MT * p.NP);
    const int r = pi - q * p.MT * p.NP;
    const int np = r / p.MT;
    const int hb0 = 2 * np + first;
    nh = min(want, p.NH - hb0);
    if (nh < 0) nh = 0;
    doc = p.upd_docs ? __ldg(p.upd_docs + q) : q;
    m0 = kPair ? (r % p.MT) * (2 * kBM) + rank * kBM : (r % p.MT) * kBM;
    hn0[0] = hb0 * kBN;
    hn0[1] = (hb0 + 1) * kBN;
    tok0 = p.docs.start(doc);
    slot0 = p.docs.first_chunk(doc);
    len = p.docs.len(doc);
    nch = p.docs.num_chunks(doc);
    nupd = nh > 0 ? (p.final_update ? nch : nch - 1) : 0;
  }
  __device__ int num_segments() const { return nupd * nh; }
  __device__ int unit_accs() const { return nupd > 0 ? nh : 0; }
  __device__ int seg_acc(int s) const { return nh == 2 ? (s & 1) : 0; }
  __device__ int seg_chunk(int s) const { return nh == 2 ? (s >> 1) : s; }
  // Tokens of chunk i of the document (the last chunk may be shorter).
  __device__ int chunk_len(int i) const { return min(p.docs.C, len - i * p.docs.C); }
  __device__ int seg_kblocks(int s) const { return (chunk_len(seg_chunk(s)) + kBK - 1) / kBK; }
  __device__ int k_valid(int s, int kb) const {
    return min(kBK, chunk_len(seg_chunk(s)) - kb * kBK);
  }
  __device__ bool seg_fresh(int) const { return false; }  // starts from the preloaded W_0

  __device__ void load(int s, int kb, uint8_t* stage, uint64_t* bar) const {
    const int i = seg_chunk(s);
    const int h = s - i * nh;
    load_update_stage(p.tm_v, p.tm_z, stage, bar, m0, h ? hn0[1] : hn0[0],
                      tok0 + i * p.docs.C + kb * kBK);
  }
  // CTA pairs: this CTA's 128 rows of eta*Vhat^T (two boxes) and its 128 of
  // the half's Z columns (two boxes).
  __device__ void load(int s, int kb, uint8_t* stage, uint32_t bar) const {
    const int i = seg_chunk(s);
    const int h = s - i * nh;
    const int tok = tok0 + i * p.docs.C + kb * kBK;
    const int n0 = (h ? hn0[1] : hn0[0]) + rank * kBM;
    tma_load_2d_pair(stage, &p.tm_v, bar, m0, tok);
    tma_load_2d_pair(stage + kMnBoxBytes, &p.tm_v, bar, m0 + 64, tok);
    tma_load_2d_pair(stage + kPairATileBytes, &p.tm_z, bar, n0, tok);
    tma_load_2d_pair(stage + kPairATileBytes + kMnBoxBytes, &p.tm_z, bar, n0 + 64, tok);
  }
  __device__ void clear_k(uint8_t* stage, int from, int to) const {
    clear_token_lines(stage, from, to);
  }
  static __device__ uint64_t a_desc(uint32_t base, int k) { return mn_desc(base, k); }
  static __device__ uint64_t b_desc(uint32_t base, int k) { return mn_desc(base, k); }

  // This unit's W_0 rows (what preload reads) into L2, a unit ahead: the
  // preload at the unit boundary then reads from L2, not DRAM.
  __device__ void prefetch_preload(int row) const {
    const int m = m0 + row;
    if (p.w0 == nullptr || m >= p.d) return;
    const size_t es = p.w0_fp32 ? 4 : 2;
    const char* base = static_cast<const char*>(p.w0) +
                       (size_t(doc) * size_t(p.w0_bstride) + size_t(m) * size_t(p.f)) * es;
    for (int h = 0; h < nh; ++h) {
      const int ncols = min(kBN, p.f - hn0[h]);
      for (size_t b = 0; b < size_t(ncols) * es; b += 128) prefetch_l2(base + size_t(hn0[h]) * es + b);
    }
  }

  // W_0 rows of half h into its accumulator (zeros outside the state): a
  // unit's first chunk waits for this (see preload_w0_staged).
  __device__ void preload(int h, int row, uint32_t trow, EpiStager& st) const {
    preload_w0_staged(p.w0, p.w0_fp32 != 0, size_t(doc) * size_t(p.w0_bstride), m0,
                      h ? hn0[1] : hn0[0], p.d, p.f, row, trow, st);
  }

  // State after chunk i of this half: snapshot W_{i+1} (bf16, four 64-column
  // TMA stores through the slot-bounded 3-D map, so rows >= d and columns
  // >= f are not written) and, after the last update, the fp32 state when
  // the caller wants it (direct stores).
  __device__ void epilogue(int s, int row, uint32_t trow, EpiStager& stg) const {
    epilogue(s, row, trow, stg, [] {});
  }
  // On CTA pairs the epilogue hands the accumulator on itself: a snapshot
  // row is read whole from TMEM into registers (as bf16 pairs) first, then
  // `handoff` releases the accumulator -- or, after a unit's last chunk,
  // preloads the next unit's W_0 into it and releases it -- so the next MMAs
  // into it start while the snapshot is staged and stored.  (Behind the
  // other half's MMAs that wait was hidden between chunks; a unit walking a
  // single half waited for the whole epilogue at every chunk, and every
  // unit's first chunks for the last snapshot's stores and the preload.)
  template <class Handoff>
  __device__ void epilogue(int s, int row, uint32_t trow, EpiStager& stg,
                           Handoff&& handoff) const {
    const int i = seg_chunk(s);
    const int h = s - i * nh;
    const int m = m0 + row;
    const bool row_ok = m < p.d;
    const int n0 = h ? hn0[1] : hn0[0];
    const bool write_snap = (i + 1) < nch;
    float* st = (p.state_out != nullptr && (i + 1) == nupd)
                    ? p.state_out + (size_t(doc) * p.d + size_t(row_ok ? m : 0)) * size_t(p.f)
                    : nullptr;
    const int slot = slot0 + i + 1;
    if (write_snap && st == nullptr) {
      uint32_t pk[kBN / 2];  // the row's 256 columns as bf16 pairs
#pragma unroll
      for (int c = 0; c < kBN; c += 64) {  // two loads per wait: the hand-off waits on this
        uint32_t v[32], w[32];
        tmem_ld_32cols(trow + uint32_t(c), v);
        tmem_ld_32cols(trow + uint32_t(c + 32), w);
        tmem_wait_ld();
        pin_regs(v);
        pin_regs(w);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          pk[c / 2 + j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
          pk[c / 2 + 16 + j] =
              pack_bf16x2(__uint_as_float(w[2 * j]), __uint_as_float(w[2 * j + 1]));
        }
      }
      handoff();
#pragma unroll
      for (int g = 0; g < kBN / 64; ++g) {
        uint8_t* buf = stg.acquire();
#pragma unroll
        for (int q = 0; q < 8; ++q)
          stg.put(buf, q,
                  make_uint4(pk[g * 32 + 4 * q], pk[g * 32 + 4 * q + 1], pk[g * 32 + 4 * q + 2],
                             pk[g * 32 + 4 * q + 3]));
        stg.commit(buf, [&](uint8_t* src) { tma_store_3d(&p.tm_ss, src, n0 + g * 64, m0, slot); });
      }
      return;
    }
#pragma unroll 1
    for (int g = 0; g < kBN / 64; ++g) {
      uint8_t* buf = write_snap ? stg.acquire() : nullptr;
#pragma unroll 1
      for (int hc = 0; hc < 2; ++hc) {
        const int c = g * 64 + hc * 32;
        uint32_t v[32];
        tmem_ld_32cols(trow + uint32_t(c), v);
        tmem_wait_ld();
        pin_regs(v);
        if (write_snap) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            stg.put(buf, hc * 4 + q,
                    make_uint4(
                        pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                        pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                        pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                        pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]))));
        }
        if (st != nullptr && row_ok) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int col = n0 + c + 8 * q;
            if (col < p.f) {
              uint4* dst = reinterpret_cast<uint4*>(st + col);
              dst[0] = make_uint4(v[8 * q], v[8 * q + 1], v[8 * q + 2], v[8 * q + 3]);
              dst[1] = make_uint4(v[8 * q + 4], v[8 * q + 5], v[8 * q + 6], v[8 * q + 7]);
            }
          }
        }
      }
      if (write_snap)
        stg.commit(buf, [&](uint8_t* src) { tma_store_3d(&p.tm_ss, src, n0 + g * 64, m0, slot); });
    }
    handoff();
  }
};

using UpdateSched = UpdateSchedT<false>;
using UpdatePairSched = UpdateSchedT<true>;

__global__ void __launch_bounds__(PipeShape<UpdateSched>::kThreads, 1)
    update_kernel(const __grid_constant__ UpdateParams p, unsigned int* status) {
  run_pipeline<UpdateSched>(p, status);
}

__global__ void __launch_bounds__(kBaseThreads, 1)
    update_pair_kernel(const __grid_constant__ UpdateParams p, unsigned int* status) {
  run_pipeline_pair<UpdatePairSched>(p, status);
}

// ----------------------------------------------------------------------------
// Fast-weight L2 normalisation ("[논문리뷰] Test-Time Training Done Right",
// Non-Linear Update of Fast-Weight): W_{i+1} = L2-Normalize(W_i + eta dW_i),
// each row of the state divided by its norm over the d_ff inputs.  The row
// norm couples every column block of a row, which live in different CTAs,
// so the walk runs one launch per chunk i:
//   preload  W_i = c_i S_i into TMEM (i = 0: W_0 as given), where S_i is the
//            unnormalised fp32 state in HBM and c_i = 1 / ||row of S_i||
//            from the previous launch's per-block partial sums; the bf16
//            snapshot W_i goes out from the same registers;
//   MMA      accumulate (eta Vhat_[i])^T Z_[i];
//   epilogue store S_{i+1} in place of S_i (a unit reads its block before it
//            writes it, and no other unit touches that block) and its row
//            sums of squares per 512-column unit into partial[(i+1) & 1].
// S is kept tiled: 16 KB tiles of 128 rows x 32 fp32 columns, chunk-major:
// 16-byte chunk c (columns 4c..4c+3) of row r at byte (c * 128 + r) * 16.
// The epilogue writes a tile with one contiguous bulk copy from a staging
// buffer of the same layout (a warp's 32 rows of one chunk are 512
// consecutive bytes, so its shared-memory stores are conflict-free), and a
// warp of the preload reads one chunk of its 32 rows as 512 consecutive
// bytes of the tile (coalesced), so the state's round trip through HBM runs
// in long contiguous bursts.
// A final kernel normalises the last state into the last snapshot or into
// state_out.
// ----------------------------------------------------------------------------

// Sum of a row's partial sums of squares (two 128-column parts per
// 256-column block), four independent accumulators (the loads overlap).
// The update kernel's preload and the finalising kernel both call it, so
// they agree bit for bit.
__device__ __forceinline__ float sum_partials(const float* base, size_t stride, int nparts) {
  // One term per 256-column block, its two 128-column parts added first;
  // the block terms go round four accumulators in block order.
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  const int nblk = nparts >> 1;
  auto blk = [&](int b) {
    return __ldcg(base + size_t(2 * b) * stride) + __ldcg(base + size_t(2 * b + 1) * stride);
  };
  int b = 0;
  for (; b + 4 <= nblk; b += 4) {
    a0 += blk(b);
    a1 += blk(b + 1);
    a2 += blk(b + 2);
    a3 += blk(b + 3);
  }
  for (; b < nblk; ++b) a0 += blk(b);
  return (a0 + a1) + (a2 + a3);
}

__device__ __forceinline__ float row_scale_of(float ss) { return 1.0f / fmaxf(sqrtf(ss), 1e-12f); }

struct NormUpdateParams {
  CUtensorMap tm_v;      // eta*Vhat [M, d]  box {64, 64}
  CUtensorMap tm_z;      // Z        [M, f]  box {64, 64}
  CUtensorMap tm_ss;     // snapshots as [slots][d rows][f cols] bf16, box {64, 128, 1} (store)
  const void* w0;
  int w0_fp32;
  int64_t w0_bstride;
  float* state;          // S, tiled: [documents][ceil(d/128)][ceil(f/32)] tiles of 4096 fp32
  float* partial;        // [2][documents][nparts][d] row sums of squares per 256-column
                         // block of the state, in two 128-column parts
  __nv_bfloat16* snap;   // [slots, d, f]
  DocMap docs;
  const int* upd_docs;   // updating documents, most updates first; nullptr: all
  int n_active;          // documents with an update at chunk i
  int i;                 // the chunk this launch updates with
  int d, f, mt, np, ncb;  // mt: row blocks of a unit (128 rows, 256 on CTA pairs);
                          // ncb: 32-column tiles per 128-row block
  int mtb;                // 128-row blocks of the state (its tile layout)
  int nparts;             // partial sums per row: 2 per 256-column block
};

// First fp32 of S's tile (document, 128-row block, 32-column block).
// Chunk c of row r of a tile: float4 index c * kBM + r.
__device__ __forceinline__ float* state_tile(float* state, int ncb, int mt_all, int doc, int mt,
                                             int cb) {
  return state + ((size_t(doc) * mt_all + mt) * ncb + cb) * size_t(kBM * 32);
}

// On CTA pairs (kPair; every chunk a multiple of 64 tokens and d a multiple
// of 256) a unit's row block is 256 rows: each CTA loads its 128 rows of
// eta*Vhat^T and 128 of each half's Z columns, and preloads, stores and sums
// the state of its own 128 rows.  There two groups of four epilogue warps
// share the work, each on 128 of every half's 256 columns (five operand
// stages leave room for the second group's staging buffers): the preloads and
// epilogues, not the MMAs, bound this walk.
template <bool kPair>
struct NormUpdateSchedT : std::conditional_t<kPair, PairDefaults, SchedDefaults> {
  using Params = NormUpdateParams;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(kPair ? 2 * kBM : kBM, kBN, true, true);
  static constexpr bool kPreload = true;
  static constexpr bool kRaggedK = !kPair;
  static constexpr bool kStagedStores = true;
  static constexpr bool kStagedPreload = true;
  static constexpr int kEpilogueGroups = kPair ? 2 : 1;
  static constexpr int kNumStages = kPair ? 5 : 4;
  static constexpr int kGroupCols = kBN / kEpilogueGroups;  // columns of a half per group
  // A row's sum of squares is kept per 256-column block of the state (one
  // half) in two parts, columns 0-127 and 128-255: the two epilogue groups
  // on pairs each own one part, a single CTA sums both in the same order,
  // so both walks round alike.
  static constexpr int kPartCols = 128;

  const Params& p;
  const int rank;
  int doc = 0, tok = 0, clen = 0, slot = 0, m0 = 0, nbase = 0, npi = 0, halves = 1;

  __device__ explicit NormUpdateSchedT(const Params& pp, uint32_t r = 0) : p(pp), rank(int(r)) {}
  __device__ int num_units() const { return p.n_active * p.mt * p.np; }
  __device__ void begin_unit(int u, int) {
    const int mt = u % p.mt;
    const int r = u / p.mt;
    const int np = r % p.np;
    const int q = r / p.np;
    doc = p.upd_docs ? __ldg(p.upd_docs + q) : q;
    tok = p.docs.start(doc) + p.i * p.docs.C;
    clen = min(p.docs.C, p.docs.len(doc) - p.i * p.docs.C);
    slot = p.docs.first_chunk(doc) + p.i;
    m0 = kPair ? mt * (2 * kBM) + rank * kBM : mt * kBM;
    npi = np;
    nbase = np * (2 * kBN);
    halves = (nbase + kBN < p.f) ? 2 : 1;
  }
  __device__ int num_segments() const { return halves; }
  __device__ int unit_accs() const { return halves; }
  __device__ int seg_acc(int s) const { return s; }
  __device__ int seg_kblocks(int) const { return (clen + kBK - 1) / kBK; }
  __device__ int k_valid(int, int kb) const { return min(kBK, clen - kb * kBK); }
  __device__ bool seg_fresh(int) const { return false; }
  __device__ void load(int s, int kb, uint8_t* stage, uint64_t* bar) const {
    load_update_stage(p.tm_v, p.tm_z, stage, bar, m0, nbase + s * kBN, tok + kb * kBK);
  }
  // CTA pairs: this CTA's 128 rows of eta*Vhat^T and its 128 of the half's
  // Z columns (two 64-wide boxes each).
  __device__ void load(int s, int kb, uint8_t* stage, uint32_t bar) const {
    const int t = tok + kb * kBK;
    const int n0 = nbase + s * kBN + rank * kBM;
    tma_load_2d_pair(stage, &p.tm_v, bar, m0, t);
    tma_load_2d_pair(stage + kMnBoxBytes, &p.tm_v, bar, m0 + 64, t);
    tma_load_2d_pair(stage + kPairATileBytes, &p.tm_z, bar, n0, t);
    tma_load_2d_pair(stage + kPairATileBytes + kMnBoxBytes, &p.tm_z, bar, n0 + 64, t);
  }
  __device__ void clear_k(uint8_t* stage, int from, int to) const {
    clear_token_lines(stage, from, to);
  }
  static __device__ uint64_t a_desc(uint32_t base, int k) { return mn_desc(base, k); }
  static __device__ uint64_t b_desc(uint32_t base, int k) { return mn_desc(base, k); }

  __device__ size_t partial_at(int par, int blk, int m) const {
    return ((size_t(par) * p.docs.ndocs + doc) * p.nparts + blk) * size_t(p.d) + m;
  }

  // W_i of this half into its accumulator, and out as snapshot slot i
  // (bf16 64-column tiles through the staging buffers, TMA stores clipped at
  // d and f).
  __device__ void preload(int h, int row, uint32_t trow, EpiStager& st) const {
    const int m = m0 + row;
    const bool row_ok = m < p.d;
    const int n0 = nbase + h * kBN;
    const int c_begin = st.group * kGroupCols, c_end = c_begin + kGroupCols;
    if (p.i == 0) {
      const size_t off =
          size_t(doc) * size_t(p.w0_bstride) + size_t(row_ok ? m : 0) * size_t(p.f);
#pragma unroll 1
      for (int c = c_begin; c < c_end; c += 32) {
        uint32_t v[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int col = n0 + c + 8 * q;
          float w[8];
          load_w0_8(p.w0, p.w0_fp32 != 0, off + col, row_ok && col < p.f, w);
#pragma unroll
          for (int j = 0; j < 8; ++j) v[8 * q + j] = __float_as_uint(w[j]);
        }
        tmem_st_32cols(trow + uint32_t(c), v);
      }
      return;
    }
    const float scale =
        row_ok ? row_scale_of(sum_partials(p.partial + partial_at(p.i & 1, 0, m), p.d, p.nparts))
               : 0.f;
    // 64 columns (two tiles) per step: sixteen independent 16-byte loads of
    // this row's two 128-byte tile rows.
#pragma unroll 1
    for (int c = c_begin; c < c_end; c += 64) {
      float w[64];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int col0 = n0 + c + 32 * t;
        const bool tile_ok = col0 < p.f;
        const float4* tile = reinterpret_cast<const float4*>(
            state_tile(p.state, p.ncb, p.mtb, doc, m0 / kBM, tile_ok ? col0 / 32 : 0));
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (tile_ok) v = __ldcg(tile + q * kBM + row);
          w[32 * t + 4 * q] = v.x;
          w[32 * t + 4 * q + 1] = v.y;
          w[32 * t + 4 * q + 2] = v.z;
          w[32 * t + 4 * q + 3] = v.w;
        }
      }
#pragma unroll
      for (int j = 0; j < 64; ++j) w[j] *= scale;
      uint8_t* buf = st.acquire();
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st.put(buf, q,
               make_uint4(pack_bf16x2(w[8 * q], w[8 * q + 1]), pack_bf16x2(w[8 * q + 2], w[8 * q + 3]),
                          pack_bf16x2(w[8 * q + 4], w[8 * q + 5]),
                          pack_bf16x2(w[8 * q + 6], w[8 * q + 7])));
      st.commit(buf, [&](uint8_t* src) { tma_store_3d(&p.tm_ss, src, n0 + c, m0, slot); });
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        uint32_t v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(w[32 * hc + j]);
        tmem_st_32cols(trow + uint32_t(c + 32 * hc), v);
      }
    }
  }

  // S_{i+1} of this half back to HBM (its 32-column tiles through the
  // staging buffers, one bulk copy each), and its row sum of squares.
  __device__ void epilogue(int s, int row, uint32_t trow, EpiStager& st) const {
    const int m = m0 + row;
    const bool row_ok = m < p.d;
    const int n0 = nbase + s * kBN;
    const int c_begin = st.group * kGroupCols, c_end = c_begin + kGroupCols;
    float ss0 = 0.f, ss1 = 0.f;
#pragma unroll 1
    for (int c = c_begin; c < c_end; c += 32) {
      uint32_t v[32];
      tmem_ld_32cols(trow + uint32_t(c), v);
      tmem_wait_ld();
      pin_regs(v);
      if (n0 + c < p.f) {  // the same for every epilogue thread
        uint8_t* buf = st.acquire();
#pragma unroll
        for (int q = 0; q < 8; ++q)  // chunk-major, as the tile is in HBM
          *reinterpret_cast<uint4*>(buf + (q * kBM + row) * 16) =
              make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        st.commit(buf, [&](uint8_t* src) {
          bulk_store(state_tile(p.state, p.ncb, p.mtb, doc, m0 / kBM, (n0 + c) / 32), src,
                     kStagingTileBytes);
        });
      }
      if (row_ok) {
        const bool first = c < kPartCols;
        float a = first ? ss0 : ss1;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (n0 + c + j < p.f) {
            const float x = __uint_as_float(v[j]);
            a = fmaf(x, x, a);
          }
        }
        if (first) ss0 = a; else ss1 = a;
      }
    }
    if (row_ok) {
      const int blk = 2 * (2 * npi + s);  // this half's 256-column block, part 0
      if (c_begin < kPartCols) __stcg(p.partial + partial_at((p.i + 1) & 1, blk, m), ss0);
      if (c_end > kPartCols) __stcg(p.partial + partial_at((p.i + 1) & 1, blk + 1, m), ss1);
    }
  }
};

using NormUpdateSched = NormUpdateSchedT<false>;
using NormUpdatePairSched = NormUpdateSchedT<true>;

__global__ void __launch_bounds__(PipeShape<NormUpdateSched>::kThreads, 1)
    norm_update_kernel(const __grid_constant__ NormUpdateParams p, unsigned int* status) {
  run_pipeline<NormUpdateSched>(p, status);
}

__global__ void __launch_bounds__(pair_threads<NormUpdatePairSched>(), 1)
    norm_update_pair_kernel(const __grid_constant__ NormUpdateParams p, unsigned int* status) {
  run_pipeline_pair<NormUpdatePairSched>(p, status);
}

// ----------------------------------------------------------------------------
// The normalised walk with the fp32 state resident in TMEM (regular batches on
// CTA pairs; "[논문리뷰] Test-Time Training Done Right", Non-Linear Update of
// Fast-Weight, rows normalised over d_ff after every update).
//
// The row norm couples every column block of a row, so the CTA pairs that
// hold one row block's column blocks form a group that exchanges row sums of
// squares at every chunk boundary; the fp32 state itself never leaves the
// chip.  With nf = ceil(f / 256) column blocks, G = floor(pairs / nf) groups
// of nf pairs run at once (f = 9728: 38 blocks, two groups filling 76 pairs).
// A row task is (sequence b, 256-row block m); round r gives group g's
// accumulator h the task 2Gr + Gh + g, and pair j of the group its column
// block j.  Each pair so walks two independent 256 x 256 blocks of the state
// (one per TMEM accumulator, rows of different tasks), alternating chunk by
// chunk: while the tensor core adds chunk i's delta to one block, the
// epilogue normalises the other.
//
// At a boundary the epilogue of accumulator h (state S_{i+1} = W_i + eta
// dW_i in TMEM):
//   1. sums the squares of its row over each 128-column half of its block
//      (the per-launch walk's two parts) and publishes the two parts' sum;
//   2. arrives on its (accumulator, group) counter and waits until every CTA
//      of the group has published (a bounded spin on the counter);
//   3. adds the nf block sums of its row in block order, forms
//      W_{i+1} = S_{i+1} / ||row||, writes it back into TMEM for the next
//      chunk and out as the bf16 snapshot (or, after the last update, the
//      fp32 state_out).
// The arithmetic (partial sums per 256-column block and 128-column part,
// their order, the scale, the chunk's delta added onto W_i by the tensor
// core) is the per-launch walk's, so both give the same bits.  Every CTA of
// the grid must be resident at once: the launch is exactly G nf pairs, no
// more than can be resident.
// ----------------------------------------------------------------------------
struct NormWalkParams {
  CUtensorMap tm_v;      // eta*Vhat [M, d]  box {64, 64}
  CUtensorMap tm_z;      // Z        [M, f]  box {64, 64}
  CUtensorMap tm_ss;     // snapshots as [slots][d rows][f cols] bf16, box {64, 128, 1} (store)
  const void* w0;
  int w0_fp32;
  int64_t w0_bstride;
  float* state_out;      // [B, d, f] fp32, or nullptr
  float* part;           // [2][G][2][nparts][256] row sums of squares, one per 256-column block
  unsigned int* arrive;  // [2][G] arrival counters, zero at launch
  int B, T, C, n, nupd;  // sequences, tokens each, chunk, chunks, updates per sequence
  int d, f, nd, nf, G, nparts, rounds;
};

// sum_partials' sum of one row's `n` block terms, `stride` floats apart
// (each already the sum of its block's two 128-column parts): the same four
// accumulators in the same order, fed by loads issued 64 at a time.
__device__ __forceinline__ float sum_partials_batched(const float* base, size_t stride, int n) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  const int full = n & ~3;
#pragma unroll 1
  for (int b0 = 0; b0 < full; b0 += 64) {
    float v[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) v[j] = b0 + j < full ? __ldcg(base + size_t(b0 + j) * stride) : 0.f;
#pragma unroll
    for (int j = 0; j < 64; j += 4) {
      if (b0 + j < full) {
        a0 += v[j];
        a1 += v[j + 1];
        a2 += v[j + 2];
        a3 += v[j + 3];
      }
    }
  }
  for (int b = full; b < n; ++b) a0 += __ldcg(base + size_t(b) * stride);
  return (a0 + a1) + (a2 + a3);
}

struct NormWalkSched : PairDefaults {
  using Params = NormWalkParams;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(2 * kBM, kBN, true, true);
  static constexpr bool kPreload = true;
  static constexpr bool kStagedStores = true;
  static constexpr bool kStagedPreload = true;
  static constexpr bool kBindsSync = true;
  static constexpr bool kAccTeams = true;   // epilogue group h owns accumulator h
  static constexpr int kEpilogueGroups = 2;
  static constexpr int kNumStages = 5;
  static constexpr int kPartCols = 128;     // a row's sum of squares in two parts

  const Params& p;
  const int rank;
  int nh = 0, g = 0, fb = 0, rnd = 0;
  int doc0 = 0, doc1 = 0, m00 = 0, m01 = 0;  // per accumulator: sequence, first row
  volatile int* abort_flag = nullptr;
  unsigned int* status = nullptr;
  mutable bool broken = false;  // a group wait ran out: do not wait again

  __device__ NormWalkSched(const Params& pp, uint32_t r) : p(pp), rank(int(r)) {}
  __device__ void bind_sync(volatile int* a, unsigned int* st) {
    abort_flag = a;
    status = st;
  }
  __device__ int num_units() const { return p.rounds * p.G * p.nf; }
  __device__ void begin_unit(int u, int) {
    const int per = p.G * p.nf;
    rnd = u / per;
    const int pr = u - rnd * per;
    g = pr / p.nf;
    fb = pr - g * p.nf;
    const int t0 = rnd * 2 * p.G + g, t1 = t0 + p.G;
    const int tasks = p.B * p.nd;
    nh = t1 < tasks ? 2 : (t0 < tasks ? 1 : 0);
    doc0 = t0 / p.nd;
    doc1 = t1 / p.nd;
    m00 = (t0 - doc0 * p.nd) * (2 * kBM) + rank * kBM;
    m01 = (t1 - doc1 * p.nd) * (2 * kBM) + rank * kBM;
  }
  __device__ int doc_of(int h) const { return h ? doc1 : doc0; }
  __device__ int row0_of(int h) const { return h ? m01 : m00; }
  __device__ int num_segments() const { return p.nupd * nh; }
  __device__ int unit_accs() const { return nh; }
  __device__ int seg_acc(int s) const { return nh == 2 ? (s & 1) : 0; }
  __device__ int seg_chunk(int s) const { return nh == 2 ? (s >> 1) : s; }
  __device__ int seg_kblocks(int s) const {
    return (min(p.C, p.T - seg_chunk(s) * p.C) + kBK - 1) / kBK;
  }
  __device__ bool seg_fresh(int) const { return false; }  // onto W_i in TMEM
  // This CTA's 128 rows of eta*Vhat^T and its 128 of the block's 256 Z
  // columns, two 64-wide boxes each.
  __device__ void load(int s, int kb, uint8_t* stage, uint32_t bar) const {
    const int h = seg_acc(s);
    const int tok = doc_of(h) * p.T + seg_chunk(s) * p.C + kb * kBK;
    const int n0 = fb * kBN + rank * kBM;
    tma_load_2d_pair(stage, &p.tm_v, bar, row0_of(h), tok);
    tma_load_2d_pair(stage + kMnBoxBytes, &p.tm_v, bar, row0_of(h) + 64, tok);
    tma_load_2d_pair(stage + kPairATileBytes, &p.tm_z, bar, n0, tok);
    tma_load_2d_pair(stage + kPairATileBytes + kMnBoxBytes, &p.tm_z, bar, n0 + 64, tok);
  }
  static __device__ uint64_t a_desc(uint32_t base, int k) { return mn_desc(base, k); }
  static __device__ uint64_t b_desc(uint32_t base, int k) { return mn_desc(base, k); }

  // W_0 (as given, not normalised) into accumulator h: these rows' 256
  // columns (the group that owns the accumulator; see preload_w0_staged).
  __device__ void preload(int h, int row, uint32_t trow, EpiStager& st) const {
    preload_w0_staged(p.w0, p.w0_fp32 != 0, size_t(doc_of(h)) * size_t(p.w0_bstride),
                      row0_of(h), fb * kBN, p.d, p.f, row, trow, st);
  }

  // Publish, exchange within the group, normalise (see above); run by the
  // epilogue group that owns accumulator h, on all 256 columns of its rows.
  __device__ void epilogue(int s, int row, uint32_t trow, EpiStager& st) const {
    const int h = seg_acc(s);
    const int i = seg_chunk(s);
    const int k = rnd * p.nupd + i;  // boundaries this (accumulator, group) passed before
    const int m = row0_of(h) + row;
    const int n0 = fb * kBN;
    const int prow = rank * kBM + row;  // this row within the 256-row block
    const float* pbase =
        p.part + ((size_t(h) * p.G + g) * 2 + (k & 1)) * size_t(p.nparts) * (2 * kBM) + prow;
    // 1. the two parts' sums of squares of S_{i+1} (columns 0-127, 128-255)
    float ss[2] = {0.f, 0.f};
#pragma unroll 1
    for (int c = 0; c < kBN; c += 32) {
      uint32_t v[32];
      tmem_ld_32cols(trow + uint32_t(c), v);
      tmem_wait_ld();
      pin_regs(v);
      float a = c < kPartCols ? ss[0] : ss[1];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (n0 + c + j < p.f) {
          const float x = __uint_as_float(v[j]);
          a = fmaf(x, x, a);
        }
      }
      if (c < kPartCols) ss[0] = a; else ss[1] = a;
    }
    // published as one term per block, the two parts added as the HBM
    // walks' readers add them
    __stcg(const_cast<float*>(pbase) + size_t(fb) * (2 * kBM), ss[0] + ss[1]);
    // 2. every CTA of the group has published
    epilogue_group_bar(st.group);
    if (row == 0) {
      unsigned int* ctr = p.arrive + h * p.G + g;
      __threadfence();
      atomicAdd(ctr, 1u);
      if (!broken) {
        const unsigned int want = 2u * unsigned(p.nf) * unsigned(k + 1);
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(ctr) < want) {
          if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
            broken = true;
            atomicOr(status, kStatusTimeout);
            break;
          }
          __nanosleep(128);
        }
      }
    }
    epilogue_group_bar(st.group);
    // 3. W_{i+1} = S_{i+1} / ||row||: into TMEM, out as snapshot or state_out
    const float scale = row_scale_of(sum_partials_batched(pbase, 2 * kBM, p.nparts));
    const bool last = (i + 1) == p.nupd;
    const bool write_snap = (i + 1) < p.n;
    float* so = (p.state_out != nullptr && last)
                    ? p.state_out + (size_t(doc_of(h)) * p.d + m) * size_t(p.f)
                    : nullptr;
    const int slot = doc_of(h) * p.n + i + 1;
#pragma unroll 1
    for (int c = 0; c < kBN; c += 64) {
      uint8_t* buf = write_snap ? st.acquire() : nullptr;
#pragma unroll 1
      for (int hc = 0; hc < 2; ++hc) {
        const int cc = c + 32 * hc;
        uint32_t v[32];
        tmem_ld_32cols(trow + uint32_t(cc), v);
        tmem_wait_ld();
        pin_regs(v);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * scale);
        if (!last) tmem_st_32cols(trow + uint32_t(cc), v);
        if (write_snap) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            st.put(buf, hc * 4 + q,
                   make_uint4(
                       pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                       pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                       pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                       pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]))));
        }
        if (so != nullptr) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int col = n0 + cc + 8 * q;
            if (col < p.f) {
              uint4* dst = reinterpret_cast<uint4*>(so + col);
              dst[0] = make_uint4(v[8 * q], v[8 * q + 1], v[8 * q + 2], v[8 * q + 3]);
              dst[1] = make_uint4(v[8 * q + 4], v[8 * q + 5], v[8 * q + 6], v[8 * q + 7]);
            }
          }
        }
      }
      if (write_snap)
        st.commit(buf, [&](uint8_t* src) { tma_store_3d(&p.tm_ss, src, n0 + c, row0_of(h), slot); });
    }
    if (!last) tmem_wait_st();  // the next chunk's MMAs add onto W_{i+1}
  }
};

__global__ void __launch_bounds__(pair_threads<NormWalkSched>(), 1)
    norm_walk_pair_kernel(const __grid_constant__ NormWalkParams p, unsigned int* status) {
  run_pipeline_pair<NormWalkSched>(p, status);
}

// The last state of each updating document, normalised: into state_out
// (fp32, when the last chunk also updated) or into the document's last
// snapshot slot (bf16).  One block per (row m, document).
__global__ void __launch_bounds__(256)
    norm_finalize_kernel(const float* __restrict__ state, const float* __restrict__ partial,
                         __nv_bfloat16* __restrict__ snap, float* __restrict__ state_out,
                         DocMap docs, const int* __restrict__ upd_docs, int final_update, int d,
                         int f, int nparts) {
  griddep_wait();  // programmatic launch: the previous grid is done
  griddep_launch_dependents();
  __shared__ float row_scale;
  const int m = blockIdx.x;
  const int doc = upd_docs ? __ldg(upd_docs + blockIdx.y) : int(blockIdx.y);
  const int nch = docs.num_chunks(doc);
  const int j = final_update ? nch : nch - 1;  // state index after the last update
  if (threadIdx.x == 0)
    row_scale = row_scale_of(
        sum_partials(partial + (size_t(j & 1) * docs.ndocs + doc) * nparts * size_t(d) + m, d,
                     nparts));
  __syncthreads();
  const float scale = row_scale;
  const size_t row = (size_t(doc) * d + m) * size_t(f);
  const int mt_all = (d + kBM - 1) / kBM;
  const int ncb = (f + 31) / 32;
  const int r = m % kBM;
  for (int c = threadIdx.x * 8; c < f; c += blockDim.x * 8) {
    // chunks c/4 and c/4 + 1 of row r in the tile of column block c / 32
    const float4* tile = reinterpret_cast<const float4*>(
        state_tile(const_cast<float*>(state), ncb, mt_all, doc, m / kBM, c / 32));
    const int q = (c % 32) / 4;
    const float4 lo = tile[q * kBM + r];
    const float4 hi = tile[(q + 1) * kBM + r];
    const float w[8] = {lo.x * scale, lo.y * scale, lo.z * scale, lo.w * scale,
                        hi.x * scale, hi.y * scale, hi.z * scale, hi.w * scale};
    if (final_update) {
      float4* dst = reinterpret_cast<float4*>(state_out + row + c);
      dst[0] = make_float4(w[0], w[1], w[2], w[3]);
      dst[1] = make_float4(w[4], w[5], w[6], w[7]);
    } else {
      const size_t at = (size_t(docs.first_chunk(doc) + nch - 1) * d + m) * size_t(f) + c;
      *reinterpret_cast<uint4*>(snap + at) =
          make_uint4(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]), pack_bf16x2(w[4], w[5]),
                     pack_bf16x2(w[6], w[7]));
    }
  }
}

// Snapshot slot of each document's first chunk = bf16(W_0 of that document).
__global__ void __launch_bounds__(256)
    snapshot0_kernel(const void* __restrict__ w0, int w0_fp32, int64_t w0_bstride,
                     __nv_bfloat16* __restrict__ snap, DocMap docs, int64_t df) {
  griddep_wait();  // programmatic launch: the previous grid is done
  griddep_launch_dependents();
  const int64_t per = df >> 3;
  const int64_t total = int64_t(docs.ndocs) * per;
  for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t b = idx / per;
    const int64_t e = (idx - b * per) * 8;
    uint4 out;
    if (w0_fp32) {
      const float4* src =
          reinterpret_cast<const float4*>(static_cast<const float*>(w0) + b * w0_bstride + e);
      const float4 lo = __ldg(src), hi = __ldg(src + 1);
      out = make_uint4(pack_bf16x2(lo.x, lo.y), pack_bf16x2(lo.z, lo.w), pack_bf16x2(hi.x, hi.y),
                       pack_bf16x2(hi.z, hi.w));
    } else {
      out = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(w0) +
                                                 b * w0_bstride + e));
    }
    *reinterpret_cast<uint4*>(snap + int64_t(docs.first_chunk(int(b))) * df + e) = out;
  }
  fence_proxy_async_global();  // the apply reads the snapshots through TMA
}

}  // namespace

cudaError_t launch_snapshot0(const LaunchEnv& env, const void* w0, bool w0_fp32,
                             int64_t w0_bstride, __nv_bfloat16* snap, const DocMap& docs, int d,
                             int f) {
  const int64_t df = int64_t(d) * f;
  const int64_t total = int64_t(docs.ndocs) * (df / 8);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = int64_t(env.num_sms) * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(snapshot0_kernel, dim3(unsigned(blocks)), dim3(256), 0, env.stream, w0,
                    w0_fp32 ? 1 : 0, w0_bstride, snap, docs, df);
}

// state[s] = W_start[s] + deltas[0, s] + ... + deltas[count-1, s], four fp32
// elements a thread-step, added in that order.  w0_kind: 0 zero start, 1 a
// shared bf16 [d, f], 2 a shared fp32 [d, f], 3 fp32 [S, d, f].  df = d * f
// is a multiple of 64, so a group of four never straddles two states.
__global__ void __launch_bounds__(256)
    state_prefix_kernel(const void* __restrict__ w0, int w0_kind, const float* __restrict__ deltas,
                        int64_t per_delta, int count, float* __restrict__ state, int64_t df,
                        int64_t groups) {
  griddep_wait();  // programmatic launch: the previous grid is done
  griddep_launch_dependents();
  for (int64_t g = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
       g += int64_t(gridDim.x) * blockDim.x) {
    const int64_t e = g * 4;
    const int64_t r = e % df;  // element within its state
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (w0_kind == 1) {
      const uint2 raw = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(w0) + r));
      const float2 lo = unpack_bf16x2(raw.x), hi = unpack_bf16x2(raw.y);
      acc = make_float4(lo.x, lo.y, hi.x, hi.y);
    } else if (w0_kind == 2 || w0_kind == 3) {
      acc = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(w0) +
                                                  (w0_kind == 3 ? e : r)));
    }
#pragma unroll 1
    for (int k = 0; k < count; ++k) {
      const float4 v = __ldcs(reinterpret_cast<const float4*>(deltas + int64_t(k) * per_delta + e));
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    *reinterpret_cast<float4*>(state + e) = acc;
  }
  fence_proxy_async_global();  // a later walk may read the state with bulk copies
}

cudaError_t launch_state_prefix(const LaunchEnv& env, const void* w0, int w0_kind,
                                const float* deltas, int count, float* state, int64_t S,
                                int64_t df) {
  const int64_t groups = S * df / 4;
  if (groups == 0) return cudaSuccess;
  // Grid-stride over a few blocks per SM: the kernel streams HBM.
  const int64_t want = (groups + 255) / 256;
  const int64_t cap = int64_t(env.num_sms) * 8;
  const int grid = int(want < cap ? want : cap);
  return launch_pdl(state_prefix_kernel, dim3(grid), dim3(256), 0, env.stream, w0, w0_kind, deltas,
                    S * df, count, state, df, groups);
}

cudaError_t launch_update(const LaunchEnv& env, const CUtensorMap& tm_vhat, const CUtensorMap& tm_z,
                          const CUtensorMap& tm_snap_store, const UpdateArgs& a) {
  if (a.n_udocs <= 0) return cudaSuccess;
  UpdateParams p;
  p.tm_v = tm_vhat;
  p.tm_z = tm_z;
  p.tm_ss = tm_snap_store;
  p.w0 = a.w0;
  p.w0_fp32 = a.w0_fp32 ? 1 : 0;
  p.w0_bstride = a.w0_bstride;
  p.state_out = a.state_out;
  p.docs = a.docs;
  p.upd_docs = a.upd_docs;
  p.n_udocs = a.n_udocs;
  p.final_update = a.final_update ? 1 : 0;
  p.d = a.d;
  p.f = a.f;
  p.NH = (a.f + kBN - 1) / kBN;
  p.NP = (a.f + 2 * kBN - 1) / (2 * kBN);
  // The grid's width in units: CTA pairs when every updated chunk is a
  // multiple of 64 tokens and pairs can be resident, else single CTAs.
  static std::atomic<int> resident{-1};
  const size_t psmem = pair_smem_bytes<UpdatePairSched>();
  int pairs = 0;
  cudaError_t e = cudaSuccess;
  if (a.allow_pairs) {
    if ((e = cudaFuncSetAttribute(update_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(psmem))) != cudaSuccess)
      return e;
    if ((e = max_pairs(reinterpret_cast<const void*>(update_pair_kernel), psmem, env, &pairs,
                       &resident)) != cudaSuccess)
      return e;
  }
  const bool use_pairs = pairs >= 1;
  const int width = use_pairs ? pairs : env.num_sms;
  p.MT = use_pairs ? (a.d + 2 * kBM - 1) / (2 * kBM) : (a.d + kBM - 1) / kBM;
  const int64_t P = int64_t(p.n_udocs) * p.MT * p.NP;
  const int64_t Q = P % width;
  p.P = int(P);
  p.RG = int(P - Q);
  p.split = (Q > 0 && 2 * Q <= width) ? 1 : 0;
  const int64_t units = p.split ? p.RG + 2 * Q : P;
  const int grid = int(units < width ? units : width);
  if (use_pairs)
    return launch_on_pairs(reinterpret_cast<const void*>(update_pair_kernel), grid, psmem, env, &p);
  e = cudaFuncSetAttribute(update_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(pipe_smem_bytes<UpdateSched>()));
  if (e != cudaSuccess) return e;
  return launch_pdl(update_kernel, dim3(grid), dim3(PipeShape<UpdateSched>::kThreads),
                    pipe_smem_bytes<UpdateSched>(), env.stream, p, env.status);
}

size_t norm_walk_part_bytes(int f, int pairs) {
  const int nf = (f + kBN - 1) / kBN;
  const int groups = pairs / nf > 0 ? pairs / nf : 1;
  return size_t(2) * groups * 2 * size_t(nf) * (2 * kBM) * sizeof(float);
}

size_t norm_walk_arrive_bytes(int pairs) { return size_t(2) * pairs * sizeof(unsigned int); }

namespace {

// The walk with the state in TMEM, when the batch is regular, CTA pairs are
// allowed and at least one group of pairs (one per 256-column block) can be
// resident.  Returns cudaErrorNotSupported (nothing enqueued) otherwise.
cudaError_t launch_norm_walk(const LaunchEnv& env, const CUtensorMap& tm_vhat,
                             const CUtensorMap& tm_z, const CUtensorMap& tm_snap_store,
                             const NormUpdateArgs& a) {
  if (!a.allow_pairs || a.docs.packed() || a.walk_part == nullptr || a.walk_arrive == nullptr ||
      a.upd_docs != nullptr || a.n_udocs != a.docs.ndocs)
    return cudaErrorNotSupported;
  const int nf = (a.f + kBN - 1) / kBN;
  static std::atomic<int> resident{-1};
  const size_t smem = pair_smem_bytes<NormWalkSched>();
  cudaError_t e = cudaFuncSetAttribute(norm_walk_pair_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  int pairs = 0;
  if ((e = max_pairs(reinterpret_cast<const void*>(norm_walk_pair_kernel), smem, env, &pairs,
                     &resident, pair_threads<NormWalkSched>())) != cudaSuccess)
    return e;
  if (pairs > a.walk_pairs) pairs = a.walk_pairs;
  const int G = pairs / nf;
  if (G < 1) return cudaErrorNotSupported;
  NormWalkParams p;
  memset(&p, 0, sizeof(p));
  p.tm_v = tm_vhat;
  p.tm_z = tm_z;
  p.tm_ss = tm_snap_store;
  p.w0 = a.w0;
  p.w0_fp32 = a.w0_fp32 ? 1 : 0;
  p.w0_bstride = a.w0_bstride;
  p.state_out = a.state_out;
  p.part = a.walk_part;
  p.arrive = a.walk_arrive;
  p.B = a.docs.ndocs;
  p.T = a.docs.T;
  p.C = a.docs.C;
  p.n = a.docs.n;
  p.nupd = a.n_steps;
  p.d = a.d;
  p.f = a.f;
  p.nd = a.d / (2 * kBM);
  p.nf = nf;
  p.G = G;
  p.nparts = nf;
  const int tasks = p.B * p.nd;
  p.rounds = (tasks + 2 * G - 1) / (2 * G);
  if ((e = cudaMemsetAsync(a.walk_arrive, 0, norm_walk_arrive_bytes(G), env.stream)) !=
      cudaSuccess)
    return e;
  return launch_on_pairs(reinterpret_cast<const void*>(norm_walk_pair_kernel), G * nf, smem, env,
                         &p, pair_threads<NormWalkSched>());
}

}  // namespace

cudaError_t launch_norm_update(const LaunchEnv& env, const CUtensorMap& tm_vhat,
                               const CUtensorMap& tm_z, const CUtensorMap& tm_snap_store,
                               const NormUpdateArgs& a) {
  if (a.n_udocs <= 0) return cudaSuccess;
  {
    const cudaError_t e = launch_norm_walk(env, tm_vhat, tm_z, tm_snap_store, a);
    if (e != cudaErrorNotSupported) return e;
    cudaGetLastError();
  }
  NormUpdateParams p;
  p.tm_v = tm_vhat;
  p.tm_z = tm_z;
  p.tm_ss = tm_snap_store;
  p.w0 = a.w0;
  p.w0_fp32 = a.w0_fp32 ? 1 : 0;
  p.w0_bstride = a.w0_bstride;
  p.state = a.state;
  p.partial = a.partial;
  p.snap = a.snap;
  p.docs = a.docs;
  p.upd_docs = a.upd_docs;
  p.d = a.d;
  p.f = a.f;
  p.mtb = (a.d + kBM - 1) / kBM;
  p.np = (a.f + 2 * kBN - 1) / (2 * kBN);
  p.ncb = (a.f + 31) / 32;
  // CTA pairs where allowed and two can be resident: each SM then reads a
  // third less operand data per FLOP.
  static std::atomic<int> resident{-1};
  const size_t psmem = pair_smem_bytes<NormUpdatePairSched>();
  int pairs = 0;
  cudaError_t e = cudaSuccess;
  if (a.allow_pairs) {
    if ((e = cudaFuncSetAttribute(norm_update_pair_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, int(psmem))) !=
        cudaSuccess)
      return e;
    if ((e = max_pairs(reinterpret_cast<const void*>(norm_update_pair_kernel), psmem, env, &pairs,
                       &resident, pair_threads<NormUpdatePairSched>())) != cudaSuccess)
      return e;
  }
  const bool use_pairs = pairs >= 1;
  p.mt = use_pairs ? (a.d + 2 * kBM - 1) / (2 * kBM) : p.mtb;
  p.nparts = 2 * ((a.f + kBN - 1) / kBN);
  if (!use_pairs &&
      (e = cudaFuncSetAttribute(norm_update_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(pipe_smem_bytes<NormUpdateSched>()))) != cudaSuccess)
    return e;
  for (int i = 0; i < a.n_steps; ++i) {
    p.i = i;
    p.n_active = a.active[i];
    const int64_t units = int64_t(p.n_active) * p.mt * p.np;
    if (units == 0) continue;
    if (use_pairs) {
      e = launch_on_pairs(reinterpret_cast<const void*>(norm_update_pair_kernel),
                          int(units < pairs ? units : pairs), psmem, env, &p,
                          pair_threads<NormUpdatePairSched>());
    } else {
      const int grid = units < env.num_sms ? int(units) : env.num_sms;
      e = launch_pdl(norm_update_kernel, dim3(grid), dim3(PipeShape<NormUpdateSched>::kThreads),
                     pipe_smem_bytes<NormUpdateSched>(), env.stream, p, env.status);
    }
    if (e != cudaSuccess) return e;
  }
  const dim3 fin(unsigned(a.d), unsigned(a.n_udocs));
  return launch_pdl(norm_finalize_kernel, fin, dim3(256), 0, env.stream,
                    static_cast<const float*>(a.state), static_cast<const float*>(a.partial),
                    a.snap, a.state_out, a.docs, a.upd_docs, a.state_out ? 1 : 0, a.d, a.f,
                    p.nparts);
}

}  // namespace ittt
