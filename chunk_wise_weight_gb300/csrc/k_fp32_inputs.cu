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

__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 a, __nv_bfloat16 b) {
  return uint32_t(__bfloat16_as_ushort(a)) | (uint32_t(__bfloat16_as_ushort(b)) << 16);
}

// Eight fp32 values -> their bf16 hi and lo parts, 16 bytes each.
__device__ __forceinline__ void split8(const float (&x)[8], uint4& hi, uint4& lo) {
  __nv_bfloat16 h[8], l[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) split_hi_lo(x[j], h[j], l[j]);
  hi = make_uint4(pack2(h[0], h[1]), pack2(h[2], h[3]), pack2(h[4], h[5]), pack2(h[6], h[7]));
  lo = make_uint4(pack2(l[0], l[1]), pack2(l[2], l[3]), pack2(l[4], l[5]), pack2(l[6], l[7]));
}

__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
  const float4 a = __ldcs(reinterpret_cast<const float4*>(p));  // read once: streaming
  const float4 b = __ldcs(reinterpret_cast<const float4*>(p + 4));
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// dst[r, k*cols + c] = part k of src[r, c] for k < nseg: the lo part when
// bit k of lo_mask is set, else the hi part.  One thread per eight columns
// of a row (cols is a multiple of 8): 16-byte loads and stores, one item per
// thread on a grid as large as the work (the block scheduler then balances
// the SMs; a single wave of grid-stride blocks measured 10-15% slower).  The
// loop only strides past a grid capped at kMaxGridBlocks.
__global__ void __launch_bounds__(256)
    split_bf16_kernel(const float* __restrict__ src, int64_t rows, int cols,
                      __nv_bfloat16* __restrict__ dst, int nseg, unsigned lo_mask) {
  griddep_wait();  // programmatic launch: the previous grid is done
  griddep_launch_dependents();
  const int q8 = cols >> 3;
  const int64_t total = rows * q8;
  for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = idx / q8;
    const int c = int(idx - r * q8) * 8;
    float x[8];
    load8(src + r * cols + c, x);
    uint4 hi, lo;
    split8(x, hi, lo);
    __nv_bfloat16* row = dst + r * int64_t(nseg) * cols + c;
    for (int k = 0; k < nseg; ++k)
      *reinterpret_cast<uint4*>(row + int64_t(k) * cols) = (lo_mask >> k) & 1u ? lo : hi;
  }
  fence_proxy_async_global();  // the GEMMs read dst through TMA
}

constexpr int kConvFp32Rows = 4;  // rows per thread: a 6-row window of loads
constexpr int64_t kMaxGridBlocks = int64_t(1) << 30;

struct TapRange {
  int lo, hi;  // taps read rows in [lo, hi)
};

// The rows a token's taps may read: its document and, with chunk padding,
// its chunk (as conv3_kernel).
__device__ __forceinline__ TapRange tap_range(const DocMap& docs, int t, int pad_mode) {
  const int k = docs.doc_of_token(t);
  int lo = docs.start(k);
  int hi = lo + docs.len(k);
  if (pad_mode == 0) {
    lo += ((t - lo) / docs.C) * docs.C;
    hi = min(lo + docs.C, hi);
  }
  return {lo, hi};
}

// Xc = three-tap depthwise conv of an fp32 X0 (as conv3_kernel: taps at
// t-1, t, t+1 inside the token's document and, with chunk padding, its
// chunk; fp32 taps in the same order), written as the split A operand of
// the target GEMM: row t of xc3 (3 d wide) is [Xc_hi | Xc_hi | Xc_lo].  A
// thread owns eight channels of kConvFp32Rows consecutive rows and loads
// their window of kConvFp32Rows + 2 rows once (one row per thread, each row
// read three times, measured 2.3x slower).
__global__ void __launch_bounds__(256)
    conv3_fp32_kernel(const float* __restrict__ x0, const float* __restrict__ conv_w,
                      __nv_bfloat16* __restrict__ xc3, int rows, DocMap docs, int d,
                      int pad_mode) {
  griddep_wait();
  griddep_launch_dependents();
  const int q8 = d >> 3;
  const int64_t total = int64_t((rows + kConvFp32Rows - 1) / kConvFp32Rows) * q8;
  for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int rb = int(idx / q8);
    const int c = int(idx - int64_t(rb) * q8) * 8;
    const int t0 = rb * kConvFp32Rows;
    float w0[8], w1[8], w2[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      w0[j] = __ldg(conv_w + size_t(c + j) * 3);
      w1[j] = __ldg(conv_w + size_t(c + j) * 3 + 1);
      w2[j] = __ldg(conv_w + size_t(c + j) * 3 + 2);
    }
    float x[kConvFp32Rows + 2][8];  // rows t0-1 .. t0+kConvFp32Rows
#pragma unroll
    for (int i = 0; i < kConvFp32Rows + 2; ++i) {
      const int t = t0 - 1 + i;
      if (t >= 0 && t < rows) {
        load8(x0 + size_t(t) * d + c, x[i]);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[i][j] = 0.f;
      }
    }
    TapRange tr = tap_range(docs, t0, pad_mode);
#pragma unroll
    for (int i = 0; i < kConvFp32Rows; ++i) {
      const int t = t0 + i;
      if (t < rows) {
        if (t >= tr.hi) tr = tap_range(docs, t, pad_mode);  // next chunk or document
        const bool has_m = t - 1 >= tr.lo, has_p = t + 1 < tr.hi;
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float v = w0[j] * (has_m ? x[i][j] : 0.f);
          v = fmaf(w1[j], x[i + 1][j], v);
          y[j] = fmaf(w2[j], has_p ? x[i + 2][j] : 0.f, v);
        }
        uint4 hi, lo;
        split8(y, hi, lo);
        __nv_bfloat16* row = xc3 + size_t(t) * (3 * size_t(d)) + c;
        *reinterpret_cast<uint4*>(row) = hi;
        *reinterpret_cast<uint4*>(row + d) = hi;
        *reinterpret_cast<uint4*>(row + 2 * d) = lo;
      }
    }
  }
  fence_proxy_async_global();  // the target GEMM reads xc3 through TMA
}

}  // namespace

cudaError_t launch_split_bf16(const LaunchEnv& env, const float* src, int64_t rows, int cols,
                              __nv_bfloat16* dst, int nseg, unsigned lo_mask) {
  const int64_t items = rows * (cols / 8);
  if (items == 0) return cudaSuccess;
  const int64_t blocks = (items + 255) / 256;
  return launch_pdl(split_bf16_kernel, dim3(unsigned(blocks < kMaxGridBlocks ? blocks : kMaxGridBlocks)), dim3(256), 0,
                    env.stream, src, rows, cols, dst, nseg, lo_mask);
}

cudaError_t launch_conv_fp32(const LaunchEnv& env, const float* x0, const float* conv_w,
                             __nv_bfloat16* xc3, int64_t rows, const DocMap& docs, int d,
                             int pad_mode) {
  const int64_t items = (rows + kConvFp32Rows - 1) / kConvFp32Rows * (d / 8);
  if (items == 0) return cudaSuccess;
  const int64_t blocks = (items + 255) / 256;
  return launch_pdl(conv3_fp32_kernel, dim3(unsigned(blocks < kMaxGridBlocks ? blocks : kMaxGridBlocks)), dim3(256), 0,
                    env.stream, x0, conv_w, xc3, int(rows), docs, d, pad_mode);
}

}  // namespace ittt
