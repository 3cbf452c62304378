// k_fp32_inputs.cu -- fp32 activations and weights on the bf16 tensor cores.
//
// When H, X0, W_gate, W_up and W_target arrive as fp32, rounding them to
// bf16 once would add an input error of about 2^-9 relative to every
// product.  Instead each fp32 value x is split into two bf16 parts,
//   hi = bf16(x),  lo = bf16(x - hi),
// so hi + lo carries 16 of x's 24 significand bits, and a product becomes
//   x y ~= hi_x hi_y + hi_x lo_y + lo_x hi_y
// (the dropped lo_x lo_y term is below 2^-16 relative).  The three terms are
// one contraction over a concatenated K = 3 d: the A operand is stored as
// [A_hi | A_hi | A_lo] and the B operand as [B_hi | B_lo | B_hi], on the
// same kernels and tile schedules as bf16 inputs; only K changes.  Both
// GEMMs take this form: gate/up with A = H and B = W_gate, W_up; the target
// with A = Xc (the depthwise convolution of the fp32 X0, computed in fp32
// and split like an input) and B = W_target.
#include "kernels.h"
#include "sm103.cuh"

namespace ittt {
namespace {

__device__ __forceinline__ void split_hi_lo(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

// dst[r, k*cols + c] = part k of src[r, c] for k < nseg: the lo part when
// bit k of lo_mask is set, else the hi part.  Four columns per thread step
// (cols is a multiple of 8).
__global__ void __launch_bounds__(256)
    split_bf16_kernel(const float* __restrict__ src, int64_t rows, int cols,
                      __nv_bfloat16* __restrict__ dst, int nseg, unsigned lo_mask) {
  griddep_wait();  // programmatic launch: the previous grid is done
  griddep_launch_dependents();
  const int q4 = cols >> 2;
  const int64_t total = rows * q4;
  for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = idx / q4;
    const int c = int(idx - r * q4) * 4;
    const float4 v = __ldg(reinterpret_cast<const float4*>(src + r * cols + c));
    const float x[4] = {v.x, v.y, v.z, v.w};
    __nv_bfloat16 h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) split_hi_lo(x[j], h[j], l[j]);
    uint2 hi, lo;
    hi.x = uint32_t(__bfloat16_as_ushort(h[0])) | (uint32_t(__bfloat16_as_ushort(h[1])) << 16);
    hi.y = uint32_t(__bfloat16_as_ushort(h[2])) | (uint32_t(__bfloat16_as_ushort(h[3])) << 16);
    lo.x = uint32_t(__bfloat16_as_ushort(l[0])) | (uint32_t(__bfloat16_as_ushort(l[1])) << 16);
    lo.y = uint32_t(__bfloat16_as_ushort(l[2])) | (uint32_t(__bfloat16_as_ushort(l[3])) << 16);
    for (int k = 0; k < nseg; ++k)
      *reinterpret_cast<uint2*>(dst + r * int64_t(nseg) * cols + int64_t(k) * cols + c) =
          (lo_mask >> k) & 1u ? lo : hi;
  }
  fence_proxy_async_global();  // the GEMMs read dst through TMA
}

// Xc = three-tap depthwise conv of an fp32 X0 (as conv3_kernel: taps at
// t-1, t, t+1 inside the token's document and, with chunk padding, its
// chunk; fp32 taps in the same order), written as the split A operand of
// the target GEMM: row t of xc3 (3 d wide) is [Xc_hi | Xc_hi | Xc_lo].  A
// thread owns four channels of one row.
__global__ void __launch_bounds__(256)
    conv3_fp32_kernel(const float* __restrict__ x0, const float* __restrict__ conv_w,
                      __nv_bfloat16* __restrict__ xc3, int rows, DocMap docs, int d,
                      int pad_mode) {
  griddep_wait();
  griddep_launch_dependents();
  const int q4 = d >> 2;
  const int64_t total = int64_t(rows) * q4;
  for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int t = int(idx / q4);
    const int c = int(idx - int64_t(t) * q4) * 4;
    const int k = docs.doc_of_token(t);
    int t_lo = docs.start(k);
    int t_hi = t_lo + docs.len(k);
    if (pad_mode == 0) {
      t_lo += ((t - t_lo) / docs.C) * docs.C;
      t_hi = min(t_lo + docs.C, t_hi);
    }
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 xm = t - 1 >= t_lo ? __ldg(reinterpret_cast<const float4*>(x0 + size_t(t - 1) * d + c)) : zero;
    const float4 x = __ldg(reinterpret_cast<const float4*>(x0 + size_t(t) * d + c));
    const float4 xp = t + 1 < t_hi ? __ldg(reinterpret_cast<const float4*>(x0 + size_t(t + 1) * d + c)) : zero;
    const float am[4] = {xm.x, xm.y, xm.z, xm.w};
    const float a0[4] = {x.x, x.y, x.z, x.w};
    const float ap[4] = {xp.x, xp.y, xp.z, xp.w};
    float y[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float* w = conv_w + size_t(c + j) * 3;
      float v = __ldg(w) * am[j];
      v = fmaf(__ldg(w + 1), a0[j], v);
      y[j] = fmaf(__ldg(w + 2), ap[j], v);
    }
    __nv_bfloat16 h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) split_hi_lo(y[j], h[j], l[j]);
    uint2 hi, lo;
    hi.x = uint32_t(__bfloat16_as_ushort(h[0])) | (uint32_t(__bfloat16_as_ushort(h[1])) << 16);
    hi.y = uint32_t(__bfloat16_as_ushort(h[2])) | (uint32_t(__bfloat16_as_ushort(h[3])) << 16);
    lo.x = uint32_t(__bfloat16_as_ushort(l[0])) | (uint32_t(__bfloat16_as_ushort(l[1])) << 16);
    lo.y = uint32_t(__bfloat16_as_ushort(l[2])) | (uint32_t(__bfloat16_as_ushort(l[3])) << 16);
    __nv_bfloat16* row = xc3 + size_t(t) * (3 * size_t(d));
    *reinterpret_cast<uint2*>(row + c) = hi;
    *reinterpret_cast<uint2*>(row + d + c) = hi;
    *reinterpret_cast<uint2*>(row + 2 * d + c) = lo;
  }
  fence_proxy_async_global();  // the target GEMM reads xc3 through TMA
}

int64_t grid_for(int64_t items, int num_sms) {
  int64_t blocks = (items + 255) / 256;
  const int64_t cap = int64_t(num_sms) * 8;
  return blocks > cap ? cap : (blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_split_bf16(const LaunchEnv& env, const float* src, int64_t rows, int cols,
                              __nv_bfloat16* dst, int nseg, unsigned lo_mask) {
  const int64_t items = rows * (cols / 4);
  if (items == 0) return cudaSuccess;
  return launch_pdl(split_bf16_kernel, dim3(unsigned(grid_for(items, env.num_sms))), dim3(256),
                    0, env.stream, src, rows, cols, dst, nseg, lo_mask);
}

cudaError_t launch_conv_fp32(const LaunchEnv& env, const float* x0, const float* conv_w,
                             __nv_bfloat16* xc3, int64_t rows, const DocMap& docs, int d,
                             int pad_mode) {
  const int64_t items = rows * (d / 4);
  if (items == 0) return cudaSuccess;
  return launch_pdl(conv3_fp32_kernel, dim3(unsigned(grid_for(items, env.num_sms))), dim3(256),
                    0, env.stream, x0, conv_w, xc3, int(rows), docs, d, pad_mode);
}

}  // namespace ittt
