// k_target.cu -- the next-token-aligned value target
//   Vhat = Conv1D(X0) W_target^T
// ("[논문리뷰] In-Place Test-Time Training", Method §2 eq. (5); causal
// padding from Method §3).
//
// The depthwise three-tap convolution runs on CUDA cores: one thread per
// 8 channels of a token row, 128-bit loads of the rows t-1, t, t+1, fp32
// arithmetic, one rounding to bf16 (the tensor-core operand).  Taps outside
// the current chunk (or, in sequence mode, outside the sequence) read zero.
// The projection is a tcgen05 GEMM over the result.  Its epilogue scales by
// the fast-weight learning rate before the bf16 rounding, so the tensor
// stores eta * Vhat: the update's left operand with eta folded in (the
// identity eta K^T(KW - V) = K~^T(K~W - V~), K~ = sqrt(eta) K, of the "ViT^3"
// review's design insights, here with the whole eta on the value side).
#include "kernels.h"
#include "pipeline.cuh"

namespace ittt {
namespace {

__global__ void __launch_bounds__(256)
    conv3_kernel(const __nv_bfloat16* __restrict__ x0, const float* __restrict__ conv_w,
                 __nv_bfloat16* __restrict__ xc, int64_t rows, int T, int d, int C,
                 int pad_mode) {
  const int groups = d >> 3;
  const int64_t total = rows * groups;
  for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = idx / groups;
    const int g = int(idx - r * groups);
    const int t = int(r % T);
    int lo = 0, hi = T;
    if (pad_mode == 0) {
      lo = (t / C) * C;
      hi = lo + C;
    }
    const size_t base = size_t(r) * size_t(d) + size_t(g) * 8;
    const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
    const uint4 xm = (t - 1 >= lo) ? __ldg(reinterpret_cast<const uint4*>(x0 + base - d)) : zero4;
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(x0 + base));
    const uint4 xp = (t + 1 < hi) ? __ldg(reinterpret_cast<const uint4*>(x0 + base + d)) : zero4;
    float w[24];
    const float4* w4 = reinterpret_cast<const float4*>(conv_w + size_t(g) * 24);
#pragma unroll
    for (int q = 0; q < 6; ++q) {
      const float4 v = __ldg(w4 + q);
      w[4 * q] = v.x;
      w[4 * q + 1] = v.y;
      w[4 * q + 2] = v.z;
      w[4 * q + 3] = v.w;
    }
    const uint32_t am[4] = {xm.x, xm.y, xm.z, xm.w};
    const uint32_t a0[4] = {x.x, x.y, x.z, x.w};
    const uint32_t ap[4] = {xp.x, xp.y, xp.z, xp.w};
    uint32_t o[4];
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
      o[q] = pack_bf16x2(y0, y1);
    }
    *reinterpret_cast<uint4*>(xc + base) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

struct TargetParams {
  CUtensorMap tm_xc;  // Xc       [M, d]  box {64, 128}
  CUtensorMap tm_wt;  // W_target [d, d]  box {64, 256}
  __nv_bfloat16* vhat;  // eta * Vhat [M, d]
  float eta;
  int M, d;
  int m_tiles, n_tiles, kblocks, raster;
};

struct TargetSched {
  using Params = TargetParams;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN, false, false);
  static constexpr bool kPreload = false;

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

  __device__ void load(int, int kb, void* a, void* b, uint64_t* bar) const {
    const int k = kb * kBK;
    tma_load_2d(a, &p.tm_xc, bar, k, m0);
    tma_load_2d(b, &p.tm_wt, bar, k, n0);
  }
  static __device__ uint64_t a_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }
  static __device__ uint64_t b_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }

  __device__ void epilogue(int, int row, uint32_t trow) const {
    const int gm = m0 + row;
    const bool row_ok = gm < p.M;
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
        pk[j] = pack_bf16x2(p.eta * __uint_as_float(v[2 * j]),
                            p.eta * __uint_as_float(v[2 * j + 1]));
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

__global__ void __launch_bounds__(kNumThreads, 1)
    target_kernel(const __grid_constant__ TargetParams p, unsigned int* status) {
  run_pipeline<TargetSched>(p, status);
}

}  // namespace

cudaError_t launch_conv(const LaunchEnv& env, const __nv_bfloat16* x0, const float* conv_w,
                        __nv_bfloat16* xc, int64_t rows, int T, int d, int C, int pad_mode) {
  const int64_t total = rows * (d / 8);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = int64_t(env.num_sms) * 8;
  if (blocks > cap) blocks = cap;
  conv3_kernel<<<int(blocks), 256, 0, env.stream>>>(x0, conv_w, xc, rows, T, d, C, pad_mode);
  return cudaGetLastError();
}

cudaError_t launch_target(const LaunchEnv& env, const CUtensorMap& tm_xc, const CUtensorMap& tm_wt,
                          __nv_bfloat16* vhat, float eta, int M, int d) {
  TargetParams p;
  p.tm_xc = tm_xc;
  p.tm_wt = tm_wt;
  p.vhat = vhat;
  p.eta = eta;
  p.M = M;
  p.d = d;
  p.m_tiles = (M + kBM - 1) / kBM;
  p.n_tiles = (d + kBN - 1) / kBN;
  p.kblocks = (d + kBK - 1) / kBK;
  p.raster = p.n_tiles < 16 ? p.n_tiles : 16;
  const int units = p.m_tiles * p.n_tiles;
  if (units == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(target_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(kPipeSmemBytes));
  if (e != cudaSuccess) return e;
  const int grid = units < env.num_sms ? units : env.num_sms;
  target_kernel<<<grid, kNumThreads, kPipeSmemBytes, env.stream>>>(p, env.status);
  return cudaGetLastError();
}

}  // namespace ittt
