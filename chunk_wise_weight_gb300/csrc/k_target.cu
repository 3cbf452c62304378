// k_target.cu -- the next-token-aligned value target
//   eta * Vhat = eta * Conv1D(X0) W_target^T
// ("[논문리뷰] In-Place Test-Time Training", Method §2 eq. (5); causal
// padding from Method §3), in two variants with identical results:
//
// Split (default): conv3_kernel streams X0 once into Xc (TMA boxes of 66
// rows x 256 channels through a shared-memory ring; a thread owns 8 channels
// of 8 consecutive token rows: fp32 taps, one bf16 rounding), and the target
// GEMM then TMA-loads Xc as its A operand.
//
// Fused: the GEMM builds each A tile itself.  Per 64-channel K block the
// producer loads, besides the W_target tile, a TMA box of the 130 X0 rows
// [m0 - 1, m0 + 128] (the tile's rows plus one halo row on each side; rows
// outside the tensor read zero) and, with a bulk copy, the block's 64 x 3
// fp32 conv weights.  Eight builder warps turn them into the bf16 A tile in
// shared memory: each thread owns 8 channels of 4 consecutive rows, reads the
// 6 X0 rows it needs, applies the taps in fp32, rounds once to bf16 and
// writes the 128-byte-swizzled K-major layout the tensor core reads.  The
// convolution never touches HBM, but it is repeated for every 256-column
// output tile on CUDA cores and the larger stage leaves room for 3 stages
// instead of 4, which makes this variant slower on GB300.
//
// In both, a tap that reaches outside the current chunk (or, in sequence
// mode, outside the sequence) reads zero, and the epilogue scales by the
// fast-weight learning rate before the bf16 rounding, so the output is
// eta * Vhat: the update's left operand with eta folded in (the identity
// eta K^T(KW - V) = K~^T(K~W - V~) of the "ViT^3" review's design insights,
// here with the whole eta on the value side).
#include "kernels.h"
#include "pipeline.cuh"
#include "pipeline_pair.cuh"

namespace ittt {
namespace {

constexpr int kHaloRows = kBM + 2;                     // 130 X0 rows per stage
constexpr uint32_t kX0BoxBytes = kHaloRows * 128;      // 16640
constexpr uint32_t kConvWBytes = kBK * 3 * 4;          // 64 channels x 3 fp32 taps
constexpr uint32_t kX0StageBytes = kX0BoxBytes + kConvWBytes;  // 17408 = 17 KiB

__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
  return uint64_t(__float_as_uint(lo)) | (uint64_t(__float_as_uint(hi)) << 32);
}

// bf16x2 word -> two fp32 lanes (exact).
__device__ __forceinline__ uint64_t bf16x2_widen(uint32_t w) {
  return uint64_t(w << 16) | (uint64_t(w & 0xffff0000u) << 32);
}

__device__ __forceinline__ uint32_t f32x2_to_bf16x2(uint64_t v) {
  return pack_bf16x2(__uint_as_float(uint32_t(v)), __uint_as_float(uint32_t(v >> 32)));
}

// conv3_kernel: persistent, two CTAs per SM.  A unit is a tile of 64 token
// rows x 256 channels.  One producer lane TMA-loads the tile's X0 box with
// one halo row on each side (66 x 256; rows outside [0, rows) and channels
// past d read zero) into a ring of three 33 KB shared-memory stages, so about
// 200 KB per SM are in flight however many registers the compute threads
// use.  Eight compute warps take eight rows each; lane g owns channels
// 8g..8g+7 (16 bytes): a warp reads one 512-byte box row without bank
// conflicts and writes 512 contiguous bytes of Xc per row.  (Measured at
// 2 x 32k tokens, d 2560: 0.110 ms against 0.115 ms with 32-row tiles and six
// stages and 0.178 ms for a thread-per-window kernel without the ring; a
// plain device copy of the same bytes takes 0.105 ms.)
constexpr int kConvCols = int(kConvMapBoxCols);         // 256
constexpr int kConvBoxRows = int(kConvMapBoxRows);      // 66
constexpr int kConvTileRows = kConvBoxRows - 2;         // 64
constexpr uint32_t kConvRowBytes = kConvCols * 2;                    // 512
constexpr uint32_t kConvBoxBytes = kConvBoxRows * kConvRowBytes;     // 33792
constexpr int kConvStages = 3;
constexpr int kConvComputeWarps = 8;
constexpr int kConvRowsPerWarp = kConvTileRows / kConvComputeWarps;  // 8
constexpr int kConvThreads = 32 * (kConvComputeWarps + 1);
constexpr int kConvCtasPerSm = 2;
static_assert(kConvBoxBytes % 128 == 0, "stages stay 128-byte aligned for TMA");

struct __align__(8) ConvSync {
  uint64_t full[kConvStages];
  uint64_t empty[kConvStages];
  int abort_flag;
};

constexpr size_t kConvSmemBytes = 128 + size_t(kConvStages) * kConvBoxBytes + sizeof(ConvSync);

// Tokens [lo, hi) a tap of token t may read: its document and, with chunk
// padding, its chunk (chunks start at the document's first token; the last
// one ends with the document).
struct TapSpan {
  int lo, hi;
};

__device__ __forceinline__ TapSpan tap_span(const DocMap& docs, int t, int pad_mode) {
  const int k = docs.doc_of_token(t);
  int lo = docs.start(k);
  int hi = lo + docs.len(k);
  if (pad_mode == 0) {
    lo += ((t - lo) / docs.C) * docs.C;
    hi = min(lo + docs.C, hi);
  }
  return {lo, hi};
}

__global__ void __launch_bounds__(kConvThreads, kConvCtasPerSm)
    conv3_kernel(const __grid_constant__ CUtensorMap tm_x0, const float* __restrict__ conv_w,
                 __nv_bfloat16* __restrict__ xc, int rows, DocMap docs, int d, int pad_mode,
                 unsigned int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  ConvSync* sync = reinterpret_cast<ConvSync*>(smem + size_t(kConvStages) * kConvBoxBytes);
  volatile int* abort_flag = &sync->abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kConvStages; ++s) {
      mbar_init(&sync->full[s], 1);
      mbar_init(&sync->empty[s], 32 * kConvComputeWarps);
    }
    sync->abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  griddep_wait();  // programmatic launch: the previous grid is done
  griddep_launch_dependents();
  const int ctiles = (d + kConvCols - 1) / kConvCols;
  const int64_t nunits = int64_t((rows + kConvTileRows - 1) / kConvTileRows) * ctiles;

  if (warp == kConvComputeWarps) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      tma_prefetch_desc(&tm_x0);
      int stage = 0;
      uint32_t phase = 0, issued = 0;
      for (int64_t u = blockIdx.x; u < nunits && !*abort_flag; u += gridDim.x) {
        if (!mbar_wait(&sync->empty[stage], phase ^ 1u, abort_flag)) {
          raise_abort(abort_flag, status, kStatusTimeout);
          break;
        }
        const int mt = int(u / ctiles);
        const int ct = int(u - int64_t(mt) * ctiles);
        mbar_arrive_expect_tx(&sync->full[stage], kConvBoxBytes);
        tma_load_2d(smem + size_t(stage) * kConvBoxBytes, &tm_x0, &sync->full[stage],
                    ct * kConvCols, mt * kConvTileRows - 1);
        ++issued;
        if (++stage == kConvStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // Let every load still in flight land before the CTA can exit.
      const int zero = 0;
      const uint32_t tail = issued < uint32_t(kConvStages) ? issued : uint32_t(kConvStages);
      for (uint32_t q = issued - tail; q < issued; ++q) {
        if (!mbar_wait(&sync->full[q % kConvStages], (q / kConvStages) & 1u, &zero))
          atomicOr(status, kStatusTimeout);
      }
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
  int stage = 0;
  uint32_t phase = 0;
  for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
    if (!mbar_wait(&sync->full[stage], phase, abort_flag)) {
      if (lane == 0) raise_abort(abort_flag, status, kStatusTimeout);
      break;
    }
    const int mt = int(u / ctiles);
    const int ct = int(u - int64_t(mt) * ctiles);
    const int t0 = mt * kConvTileRows + warp * kConvRowsPerWarp;
    const int c = ct * kConvCols + lane * 8;
    const bool active = c < d && t0 < rows;
    // Box rows warp*8 .. warp*8+9 hold tokens t0-1 .. t0+8.
    const uint8_t* box = smem + size_t(stage) * kConvBoxBytes +
                         size_t(warp * kConvRowsPerWarp) * kConvRowBytes + lane * 16;
    uint4 o[kConvRowsPerWarp];
    if (active) {
      uint4 x[kConvRowsPerWarp + 2];
#pragma unroll
      for (int j = 0; j < kConvRowsPerWarp + 2; ++j)
        x[j] = *reinterpret_cast<const uint4*>(box + j * kConvRowBytes);
      float w[24];
      const float4* w4 = reinterpret_cast<const float4*>(conv_w + size_t(c) * 3);
#pragma unroll
      for (int q = 0; q < 6; ++q) {
        const float4 v = __ldg(w4 + q);
        w[4 * q] = v.x;
        w[4 * q + 1] = v.y;
        w[4 * q + 2] = v.z;
        w[4 * q + 3] = v.w;
      }
      TapSpan sp = tap_span(docs, t0, pad_mode);
#pragma unroll
      for (int j = 0; j < kConvRowsPerWarp; ++j) {
        const int t = t0 + j;
        if (t < rows && t >= sp.hi) sp = tap_span(docs, t, pad_mode);  // next chunk or document
        const uint4 xm = t - 1 >= sp.lo ? x[j] : zero4;
        const uint4 xp = t + 1 < sp.hi ? x[j + 2] : zero4;
        const uint4 xx = x[j + 1];
        const uint32_t am[4] = {xm.x, xm.y, xm.z, xm.w};
        const uint32_t a0[4] = {xx.x, xx.y, xx.z, xx.w};
        const uint32_t ap[4] = {xp.x, xp.y, xp.z, xp.w};
        uint32_t r[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 fm = unpack_bf16x2(am[q]);
          const float2 f0 = unpack_bf16x2(a0[q]);
          const float2 fp = unpack_bf16x2(ap[q]);
          const int c0 = 2 * q, c1 = 2 * q + 1;  // channel within the group of 8
          float y0 = w[3 * c0] * fm.x;
          y0 = fmaf(w[3 * c0 + 1], f0.x, y0);
          y0 = fmaf(w[3 * c0 + 2], fp.x, y0);
          float y1 = w[3 * c1] * fm.y;
          y1 = fmaf(w[3 * c1 + 1], f0.y, y1);
          y1 = fmaf(w[3 * c1 + 2], fp.y, y1);
          r[q] = pack_bf16x2(y0, y1);
        }
        o[j] = make_uint4(r[0], r[1], r[2], r[3]);
      }
    }
    // Every value this lane read from the stage is consumed above.  Order
    // those reads before the next TMA write into the stage (a different
    // proxy), then release the stage: each lane arrives for itself.
    fence_proxy_async_smem();
    mbar_arrive(&sync->empty[stage]);
    if (++stage == kConvStages) {
      stage = 0;
      phase ^= 1u;
    }
    if (active) {
#pragma unroll
      for (int j = 0; j < kConvRowsPerWarp; ++j)
        if (t0 + j < rows)
          *reinterpret_cast<uint4*>(xc + size_t(t0 + j) * size_t(d) + size_t(c)) = o[j];
    }
  }
  fence_proxy_async_global();  // the target GEMM reads Xc through TMA
}

struct TargetParams {
  CUtensorMap tm_a;      // split: Xc [M, d] box {64, 128}; fused: X0 [M, d] box {64, 130}
  CUtensorMap tm_wt;     // W_target [d, d]  box {64, 256}
  CUtensorMap tm_vs;     // eta*Vhat [M, d]  box {64, 128}  (TMA store, split variant)
  const float* conv_w;   // [d, 3]
  const float* eta_tok;  // [M] per-token rate weights or nullptr
  __nv_bfloat16* vhat;   // eta * Vhat [M, d]
  float eta;
  int M, T, d, C, pad_mode;
  int m_tiles, n_tiles, kblocks, raster;
};

// The update's rate for token row gm: eta, times its per-token weight.
__device__ __forceinline__ float target_row_rate(const TargetParams& p, int gm) {
  return p.eta_tok == nullptr ? p.eta : (gm < p.M ? p.eta * __ldg(p.eta_tok + gm) : 0.0f);
}

// Split variant's epilogue: 256 columns of rows m0.. as four 64-column TMA
// stores (rows >= M and columns >= d are not written).
__device__ __forceinline__ void target_epilogue(const TargetParams& p, int m0, int n0, int row,
                                                uint32_t trow, EpiStager& st) {
  const float scale = target_row_rate(p, m0 + row);
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
               make_uint4(pack_bf16x2(scale * __uint_as_float(v[8 * q]),
                                      scale * __uint_as_float(v[8 * q + 1])),
                          pack_bf16x2(scale * __uint_as_float(v[8 * q + 2]),
                                      scale * __uint_as_float(v[8 * q + 3])),
                          pack_bf16x2(scale * __uint_as_float(v[8 * q + 4]),
                                      scale * __uint_as_float(v[8 * q + 5])),
                          pack_bf16x2(scale * __uint_as_float(v[8 * q + 6]),
                                      scale * __uint_as_float(v[8 * q + 7]))));
    }
    st.commit(buf, [&](uint8_t* src) { tma_store_2d(&p.tm_vs, src, n0 + g * 64, m0); });
  }
}

template <bool kFused>
struct TargetSched : SchedDefaults {
  using Params = TargetParams;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN, false, false);
  static constexpr int kNumStages = kFused ? 3 : 4;
  static constexpr uint32_t kExtraStageBytes = kFused ? kX0StageBytes : 0;
  static constexpr int kBuilderWarps = kFused ? 8 : 0;
  static constexpr bool kStagedStores = !kFused;  // the fused stage leaves no room
  static_assert(kX0StageBytes % 1024 == 0, "stage alignment");

  const Params& p;
  int m0 = 0, n0 = 0, acc = 0;

  __device__ explicit TargetSched(const Params& pp) : p(pp) {}
  __device__ int num_units() const { return p.m_tiles * p.n_tiles; }
  __device__ void begin_unit(int u, int local) {
    int m, n;
    raster_grouped(u, p.m_tiles, p.n_tiles, p.raster, m, n);
    m0 = m * kBM;
    n0 = n * kBN;
    acc = local & 1;
  }
  __device__ int num_segments() const { return 1; }
  __device__ int seg_acc(int) const { return acc; }
  __device__ int seg_kblocks(int) const { return p.kblocks; }
  __device__ bool seg_fresh(int) const { return true; }

  // Conv weights of the K block's channels (fewer in a ragged last block).
  __device__ uint32_t conv_w_bytes(int kb) const {
    return uint32_t(min(kBK, p.d - kb * kBK)) * 12u;
  }
  __device__ uint32_t tma_bytes(int, int kb) const {
    if constexpr (kFused) return kBTileBytes + kX0BoxBytes + conv_w_bytes(kb);
    return kStageBytes;
  }
  __device__ void load(int, int kb, uint8_t* stage, uint64_t* bar) const {
    const int k = kb * kBK;
    tma_load_2d(stage + kATileBytes, &p.tm_wt, bar, k, n0);
    if constexpr (kFused) {
      tma_load_2d(stage + kStageBytes, &p.tm_a, bar, k, m0 - 1);
      bulk_load(stage + kStageBytes + kX0BoxBytes, p.conv_w + size_t(k) * 3, conv_w_bytes(kb),
                bar);
    } else {
      tma_load_2d(stage, &p.tm_a, bar, k, m0);
    }
  }

  // Conv of 8 channels x 4 rows per thread (256 threads cover 128 x 64).
  __device__ void build_a(int, int kb, uint8_t* stage, int tid) const {
    const int c8 = tid & 7;          // 16-byte chunk = channels k0 .. k0+7
    const int r0 = (tid >> 3) * 4;   // first of this thread's 4 rows
    const int k0 = kb * kBK + c8 * 8;
    const uint8_t* xbox = stage + kStageBytes;  // box row j = token row m0 - 1 + j
    uint8_t* atile = stage;

    // Taps of channel pairs (2j, 2j+1): tap index 0 = t-1, 1 = t, 2 = t+1;
    // the stage carries this K block's weights right after the X0 box.
    uint64_t w[3][4];
    if (k0 < p.d) {
      float wf[24];
      const float4* src =
          reinterpret_cast<const float4*>(stage + kStageBytes + kX0BoxBytes + c8 * 96);
#pragma unroll
      for (int q = 0; q < 6; ++q) {
        const float4 v = src[q];
        wf[4 * q] = v.x;
        wf[4 * q + 1] = v.y;
        wf[4 * q + 2] = v.z;
        wf[4 * q + 3] = v.w;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int tap = 0; tap < 3; ++tap)
          w[tap][j] = f32x2_pack(wf[3 * (2 * j) + tap], wf[3 * (2 * j + 1) + tap]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) w[0][j] = w[1][j] = w[2][j] = 0ull;
    }

    // Six X0 rows r0-1 .. r0+4 (box rows r0 .. r0+5), widened to fp32.
    uint64_t x[6][4];
#pragma unroll
    for (int j = 0; j < 6; ++j) {
      const int br = r0 + j;
      const uint4 q = *reinterpret_cast<const uint4*>(xbox + br * 128 + ((c8 ^ (br & 7)) << 4));
      x[j][0] = bf16x2_widen(q.x);
      x[j][1] = bf16x2_widen(q.y);
      x[j][2] = bf16x2_widen(q.z);
      x[j][3] = bf16x2_widen(q.w);
    }
    // The 4 rows share one chunk (C and m0 are multiples of 64 and 128): only
    // the halo rows can fall outside it.
    const int t0 = (m0 + r0) % p.T;  // token index of row r0 in its sequence
    bool prev_ok, next_ok;
    if (p.pad_mode == 0) {
      const int pc = t0 % p.C;
      prev_ok = pc > 0;
      next_ok = pc + 4 < min(p.C, p.T - (t0 - pc));  // a partial last chunk ends at T
    } else {
      prev_ok = t0 > 0;
      next_ok = t0 + 4 < p.T;
    }
    if (!prev_ok) x[0][0] = x[0][1] = x[0][2] = x[0][3] = 0ull;
    if (!next_ok) x[5][0] = x[5][1] = x[5][2] = x[5][3] = 0ull;

#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint64_t y = f32x2_mul(w[0][j], x[i][j]);
        y = f32x2_fma(w[1][j], x[i + 1][j], y);
        y = f32x2_fma(w[2][j], x[i + 2][j], y);
        o[j] = f32x2_to_bf16x2(y);
      }
      const int r = r0 + i;
      *reinterpret_cast<uint4*>(atile + r * 128 + ((c8 ^ (r & 7)) << 4)) =
          make_uint4(o[0], o[1], o[2], o[3]);
    }
  }

  static __device__ uint64_t a_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }
  static __device__ uint64_t b_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }

  __device__ float row_rate(int gm) const { return target_row_rate(p, gm); }

  // Split variant: 256 columns as four 64-column TMA stores (rows >= M and
  // columns >= d are not written).
  __device__ void epilogue(int, int row, uint32_t trow, EpiStager& st) const {
    target_epilogue(p, m0, n0, row, trow, st);
  }

  // Fused variant: direct 16-byte stores.
  __device__ void epilogue(int, int row, uint32_t trow) const {
    const int gm = m0 + row;
    const bool row_ok = gm < p.M;
    const float scale = row_rate(gm);
    __nv_bfloat16* vrow = p.vhat + size_t(row_ok ? gm : 0) * size_t(p.d);
#pragma unroll 1
    for (int c = 0; c < kBN; c += 32) {
      uint32_t v[32];
      tmem_ld_32cols(trow + uint32_t(c), v);
      tmem_wait_ld();
      pin_regs(v);
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        pk[j] = pack_bf16x2(scale * __uint_as_float(v[2 * j]),
                            scale * __uint_as_float(v[2 * j + 1]));
      if (row_ok) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int col = n0 + c + 8 * q;
          if (col < p.d)
            *reinterpret_cast<uint4*>(vrow + col) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
    }
  }
};

template <bool kFused>
__global__ void __launch_bounds__(PipeShape<TargetSched<kFused>>::kThreads, 1)
    target_kernel(const __grid_constant__ TargetParams p, unsigned int* status) {
  run_pipeline<TargetSched<kFused>>(p, status);
}

// CTA pairs (split convolution only): a unit is a 256-row x 256-column
// tile; each CTA keeps its 128 Xc rows and 128 of the W_target rows.
struct TargetPairSched : PairDefaults {
  using Params = TargetParams;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(2 * kBM, kBN, false, false);
  static constexpr bool kStagedStores = true;

  const Params& p;
  const int rank;
  int m0 = 0, n0 = 0, acc = 0;

  __device__ TargetPairSched(const Params& pp, uint32_t r) : p(pp), rank(int(r)) {}
  __device__ int num_units() const { return p.m_tiles * p.n_tiles; }
  __device__ void begin_unit(int u, int local) {
    int m, n;
    raster_grouped(u, p.m_tiles, p.n_tiles, p.raster, m, n);
    m0 = m * (2 * kBM) + rank * kBM;
    n0 = n * kBN;
    acc = local & 1;
  }
  __device__ int num_segments() const { return 1; }
  __device__ int seg_acc(int) const { return acc; }
  __device__ int seg_kblocks(int) const { return p.kblocks; }
  __device__ bool seg_fresh(int) const { return true; }
  __device__ void load(int, int kb, uint8_t* stage, uint32_t bar) const {
    const int k = kb * kBK;
    tma_load_2d_pair(stage, &p.tm_a, bar, k, m0);
    tma_load_2d_pair(stage + kPairATileBytes, &p.tm_wt, bar, k, n0 + rank * kBM);
  }
  static __device__ uint64_t a_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }
  static __device__ uint64_t b_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }
  __device__ void epilogue(int, int row, uint32_t trow, EpiStager& st) const {
    target_epilogue(p, m0, n0, row, trow, st);
  }
};

__global__ void __launch_bounds__(kBaseThreads, 1)
    target_pair_kernel(const __grid_constant__ TargetParams p, unsigned int* status) {
  run_pipeline_pair<TargetPairSched>(p, status);
}

template <bool kFused>
cudaError_t launch_target_variant(const LaunchEnv& env, const TargetParams& p, int units) {
  using S = TargetSched<kFused>;
  cudaError_t e = cudaFuncSetAttribute(target_kernel<kFused>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(pipe_smem_bytes<S>()));
  if (e != cudaSuccess) return e;
  const int grid = units < env.num_sms ? units : env.num_sms;
  return launch_pdl(target_kernel<kFused>, dim3(grid), dim3(PipeShape<S>::kThreads),
                    pipe_smem_bytes<S>(), env.stream, p, env.status);
}

}  // namespace

cudaError_t launch_conv(const LaunchEnv& env, const CUtensorMap& tm_x0, const float* conv_w,
                        __nv_bfloat16* xc, int64_t rows, const DocMap& docs, int d,
                        int pad_mode) {
  const int64_t units = (rows + kConvTileRows - 1) / kConvTileRows * ((d + kConvCols - 1) / kConvCols);
  if (units == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(conv3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(kConvSmemBytes));
  if (e != cudaSuccess) return e;
  int64_t grid = int64_t(env.num_sms) * kConvCtasPerSm;
  if (grid > units) grid = units;
  return launch_pdl(conv3_kernel, dim3(unsigned(grid)), dim3(kConvThreads), kConvSmemBytes,
                    env.stream, tm_x0, conv_w, xc, int(rows), docs, d, pad_mode, env.status);
}

cudaError_t launch_target_pair(const LaunchEnv& env, const CUtensorMap& tm_xc,
                               const CUtensorMap& tm_wt, const CUtensorMap& tm_vs,
                               const float* eta_tok, __nv_bfloat16* vhat, float eta, int M,
                               int d, int K) {
  if (K <= 0) K = d;
  TargetParams p;
  memset(&p, 0, sizeof(p));
  p.eta_tok = eta_tok;
  p.tm_a = tm_xc;
  p.tm_wt = tm_wt;
  p.tm_vs = tm_vs;
  p.vhat = vhat;
  p.eta = eta;
  p.M = M;
  p.d = d;
  p.m_tiles = (M + 2 * kBM - 1) / (2 * kBM);
  p.n_tiles = (d + kBN - 1) / kBN;
  p.kblocks = (K + kBK - 1) / kBK;
  p.raster = p.n_tiles < 16 ? p.n_tiles : 16;
  const int units = p.m_tiles * p.n_tiles;
  if (units == 0) return cudaSuccess;
  const size_t smem = pair_smem_bytes<TargetPairSched>();
  cudaError_t e = cudaFuncSetAttribute(target_pair_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  static std::atomic<int> resident{-1};
  int pairs = 0;
  if ((e = max_pairs(reinterpret_cast<const void*>(target_pair_kernel), smem, env, &pairs,
                     &resident)) != cudaSuccess)
    return e;
  if (pairs < 1) return cudaErrorNotSupported;
  if (units < pairs) pairs = units;
  return launch_on_pairs(reinterpret_cast<const void*>(target_pair_kernel), pairs, smem, env, &p);
}

cudaError_t launch_target(const LaunchEnv& env, const CUtensorMap& tm_a, const CUtensorMap& tm_wt,
                          const CUtensorMap& tm_vs, const float* conv_w, const float* eta_tok,
                          __nv_bfloat16* vhat, float eta, int M, int T, int d, int C, int pad_mode,
                          bool fused, int K) {
  if (K <= 0 || fused) K = d;
  TargetParams p;
  p.eta_tok = eta_tok;
  p.tm_a = tm_a;
  p.tm_wt = tm_wt;
  p.tm_vs = tm_vs;
  p.conv_w = conv_w;
  p.vhat = vhat;
  p.eta = eta;
  p.M = M;
  p.T = T;
  p.d = d;
  p.C = C;
  p.pad_mode = pad_mode;
  p.m_tiles = (M + kBM - 1) / kBM;
  p.n_tiles = (d + kBN - 1) / kBN;
  p.kblocks = (K + kBK - 1) / kBK;
  p.raster = p.n_tiles < 16 ? p.n_tiles : 16;
  const int units = p.m_tiles * p.n_tiles;
  if (units == 0) return cudaSuccess;
  return fused ? launch_target_variant<true>(env, p, units)
               : launch_target_variant<false>(env, p, units);
}

}  // namespace ittt
