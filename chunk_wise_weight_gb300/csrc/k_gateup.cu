// k_gateup.cu -- gate/up GEMM with the SiLU (.) mul epilogue:
//   Z = SiLU(H W_gate^T) (.) (H W_up^T)
// ("[논문리뷰] In-Place Test-Time Training", Method §1 eq. (2), phi = SiLU).
//
// Each MMA tile computes 128 gate columns and the matching 128 up columns
// for the same f-range, so the accumulator holds gate pre-activations in
// TMEM columns 0..127 and up pre-activations in 128..255; the epilogue pairs
// column j with column j + 128 and writes 128 bf16 Z columns.
//
// On CTA pairs (the default) a unit is 256 rows: each CTA keeps its 128 H
// rows, the leader loads the 128 W_gate rows of the f-range and its peer the
// 128 W_up rows (the pair MMA's two B halves).  On a single CTA (fallback)
// the producer stacks both into one 256-row B tile of a 128-row unit.
#include "kernels.h"
#include "pipeline.cuh"
#include "pipeline_pair.cuh"

namespace ittt {
namespace {

constexpr int kGateUpTileN = 128;

struct GateUpParams {
  CUtensorMap tm_h;   // H      [M, K]  box {64, 128}
  CUtensorMap tm_wg;  // W_gate [f, K]  box {64, 128}
  CUtensorMap tm_wu;  // W_up   [f, K]  box {64, 128}
  CUtensorMap tm_zs;  // Z      [M, f]  box {64, 128}  (TMA store)
  int M, f;
  int m_tiles, n_tiles, kblocks, raster;
};

// 128 Z columns as two 64-column TMA stores; rows >= M and columns >= f
// fall outside the tensor map and are not written.
__device__ __forceinline__ void gateup_epilogue(const GateUpParams& p, int m0, int n0,
                                                uint32_t trow, EpiStager& st) {
#pragma unroll 1
  for (int g = 0; g < kGateUpTileN / 64; ++g) {
    uint8_t* buf = st.acquire();
#pragma unroll 1
    for (int hc = 0; hc < 2; ++hc) {
      const int c = g * 64 + hc * 32;
      uint32_t gv[32], uv[32];
      tmem_ld_32cols(trow + uint32_t(c), gv);
      tmem_ld_32cols(trow + uint32_t(kGateUpTileN + c), uv);
      tmem_wait_ld();
      pin_regs(gv);
      pin_regs(uv);
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float g0 = __uint_as_float(gv[2 * j]), g1 = __uint_as_float(gv[2 * j + 1]);
        const float u0 = __uint_as_float(uv[2 * j]), u1 = __uint_as_float(uv[2 * j + 1]);
        // CUDA's full-precision expf: against the fast __expf intrinsic it
        // measured no slower and the same Z and O error (both dominated by
        // the bf16 rounding of Z).
        const float z0 = g0 / (1.0f + expf(-g0)) * u0;
        const float z1 = g1 / (1.0f + expf(-g1)) * u1;
        pk[j] = pack_bf16x2(z0, z1);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st.put(buf, hc * 4 + q, make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]));
    }
    st.commit(buf, [&](uint8_t* src) { tma_store_2d(&p.tm_zs, src, n0 + g * 64, m0); });
  }
}

struct GateUpSched : SchedDefaults {
  using Params = GateUpParams;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN, false, false);
  static constexpr bool kStagedStores = true;

  const Params& p;
  int m0 = 0, n0 = 0, acc = 0;

  __device__ explicit GateUpSched(const Params& pp) : p(pp) {}
  __device__ int num_units() const { return p.m_tiles * p.n_tiles; }
  __device__ void begin_unit(int u, int local) {
    int m, n;
    raster_grouped(u, p.m_tiles, p.n_tiles, p.raster, m, n);
    m0 = m * kBM;
    n0 = n * kGateUpTileN;
    acc = local & 1;
  }
  __device__ int num_segments() const { return 1; }
  __device__ int seg_acc(int) const { return acc; }
  __device__ int seg_kblocks(int) const { return p.kblocks; }
  __device__ bool seg_fresh(int) const { return true; }

  __device__ void load(int, int kb, uint8_t* stage, uint64_t* bar) const {
    const int k = kb * kBK;
    tma_load_2d(stage, &p.tm_h, bar, k, m0);
    tma_load_2d(stage + kATileBytes, &p.tm_wg, bar, k, n0);
    tma_load_2d(stage + kATileBytes + kBTileBytes / 2, &p.tm_wu, bar, k, n0);
  }

  // K-major, 128-byte swizzle: the k-th 16-wide slice starts 32 bytes in.
  static __device__ uint64_t a_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }
  static __device__ uint64_t b_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }

  __device__ void epilogue(int, int, uint32_t trow, EpiStager& st) const {
    gateup_epilogue(p, m0, n0, trow, st);
  }
};

__global__ void __launch_bounds__(PipeShape<GateUpSched>::kThreads, 1)
    gateup_kernel(const __grid_constant__ GateUpParams p, unsigned int* status) {
  run_pipeline<GateUpSched>(p, status);
}

struct GateUpPairSched : PairDefaults {
  using Params = GateUpParams;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(2 * kBM, kBN, false, false);
  static constexpr bool kStagedStores = true;

  const Params& p;
  const int rank;
  int m0 = 0, n0 = 0, acc = 0;

  __device__ GateUpPairSched(const Params& pp, uint32_t r) : p(pp), rank(int(r)) {}
  __device__ int num_units() const { return p.m_tiles * p.n_tiles; }
  __device__ void begin_unit(int u, int local) {
    int m, n;
    raster_grouped(u, p.m_tiles, p.n_tiles, p.raster, m, n);
    m0 = m * (2 * kBM) + rank * kBM;
    n0 = n * kGateUpTileN;
    acc = local & 1;
  }
  __device__ int num_segments() const { return 1; }
  __device__ int seg_acc(int) const { return acc; }
  __device__ int seg_kblocks(int) const { return p.kblocks; }
  __device__ bool seg_fresh(int) const { return true; }
  __device__ void load(int, int kb, uint8_t* stage, uint32_t bar) const {
    const int k = kb * kBK;
    tma_load_2d_pair(stage, &p.tm_h, bar, k, m0);
    tma_load_2d_pair(stage + kPairATileBytes, rank == 0 ? &p.tm_wg : &p.tm_wu, bar, k, n0);
  }
  static __device__ uint64_t a_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }
  static __device__ uint64_t b_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }
  __device__ void epilogue(int, int, uint32_t trow, EpiStager& st) const {
    gateup_epilogue(p, m0, n0, trow, st);
  }
};

__global__ void __launch_bounds__(kBaseThreads, 1)
    gateup_pair_kernel(const __grid_constant__ GateUpParams p, unsigned int* status) {
  run_pipeline_pair<GateUpPairSched>(p, status);
}

}  // namespace

cudaError_t launch_gateup_pair(const LaunchEnv& env, const CUtensorMap& tm_h,
                               const CUtensorMap& tm_wg, const CUtensorMap& tm_wu,
                               const CUtensorMap& tm_zs, int M, int f, int K) {
  GateUpParams p;
  p.tm_h = tm_h;
  p.tm_wg = tm_wg;
  p.tm_wu = tm_wu;
  p.tm_zs = tm_zs;
  p.M = M;
  p.f = f;
  p.m_tiles = (M + 2 * kBM - 1) / (2 * kBM);
  p.n_tiles = (f + kGateUpTileN - 1) / kGateUpTileN;
  p.kblocks = (K + kBK - 1) / kBK;
  // Column tiles in the fewest even bands of at most 40 (each band re-reads
  // H once; 76 tiles -> 2 x 38: a same-box sweep gave 3.67 ms at 38, 3.70 at
  // 16 and 4.16 at 76, where the band's weights no longer stay in L2).
  {
    const int bands = (p.n_tiles + 39) / 40;
    p.raster = (p.n_tiles + bands - 1) / bands;
  }
  const int units = p.m_tiles * p.n_tiles;
  if (units == 0) return cudaSuccess;
  const size_t smem = pair_smem_bytes<GateUpPairSched>();
  cudaError_t e = cudaFuncSetAttribute(gateup_pair_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  static std::atomic<int> resident{-1};
  int pairs = 0;
  if ((e = max_pairs(reinterpret_cast<const void*>(gateup_pair_kernel), smem, env, &pairs,
                     &resident)) != cudaSuccess)
    return e;
  if (pairs < 1) return cudaErrorNotSupported;
  if (units < pairs) pairs = units;
  return launch_on_pairs(reinterpret_cast<const void*>(gateup_pair_kernel), pairs, smem, env, &p);
}

cudaError_t launch_gateup(const LaunchEnv& env, const CUtensorMap& tm_h, const CUtensorMap& tm_wg,
                          const CUtensorMap& tm_wu, const CUtensorMap& tm_zs, int M, int f, int K) {
  GateUpParams p;
  p.tm_h = tm_h;
  p.tm_wg = tm_wg;
  p.tm_wu = tm_wu;
  p.tm_zs = tm_zs;
  p.M = M;
  p.f = f;
  p.m_tiles = (M + kBM - 1) / kBM;
  p.n_tiles = (f + kGateUpTileN - 1) / kGateUpTileN;
  p.kblocks = (K + kBK - 1) / kBK;
  p.raster = p.n_tiles < 16 ? p.n_tiles : 16;
  const int units = p.m_tiles * p.n_tiles;
  if (units == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(pipe_smem_bytes<GateUpSched>()));
  if (e != cudaSuccess) return e;
  const int grid = units < env.num_sms ? units : env.num_sms;
  return launch_pdl(gateup_kernel, dim3(grid), dim3(PipeShape<GateUpSched>::kThreads),
                    pipe_smem_bytes<GateUpSched>(), env.stream, p, env.status);
}

}  // namespace ittt
