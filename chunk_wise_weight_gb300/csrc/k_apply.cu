// k_apply.cu -- apply step for every chunk of every sequence in one launch:
//   O_[i] = Z_[i] W_i^T
// ("[논문리뷰] In-Place Test-Time Training", Method §1 eq. (3); all chunks in
// parallel as in Method §3 stage 3).
//
// W_i is the bf16 snapshot the update kernel wrote (slot 0 holds W_0).  A
// work unit is (sequence b, chunk i, 128-row tile of the chunk, 256-column
// tile of d_model); rows past the chunk's end belong to another chunk and are
// computed but not stored, so any chunk size that is a multiple of 64 works,
// and the last chunk may be the shorter remainder of the sequence.
#include "kernels.h"
#include "pipeline.cuh"

namespace ittt {
namespace {

struct ApplyParams {
  CUtensorMap tm_z;     // Z          [B*T, f]    box {64, 128}
  CUtensorMap tm_snap;  // snapshots  [B*n*d, f]  box {64, 256}
  CUtensorMap tm_os;    // bf16 O as [B][T rows][d cols], box {64, 64, 1} (store)
  void* out;            // O [B*T, d], bf16 or fp32
  int out_fp32;
  int B, T, d, f, C, n;
  int mt_per_chunk, nt, kblocks;
};

struct ApplySched : SchedDefaults {
  using Params = ApplyParams;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN, false, false);
  static constexpr bool kStagedStores = true;

  const Params& p;
  int arow0 = 0, brow0 = 0, rows_valid = 0, n0 = 0, acc = 0, seq = 0, srow0 = 0;

  __device__ explicit ApplySched(const Params& pp) : p(pp) {}
  __device__ int num_units() const { return p.B * p.n * p.mt_per_chunk * p.nt; }
  __device__ void begin_unit(int u, int local) {
    const int nt = u % p.nt;
    int r = u / p.nt;
    const int mt = r % p.mt_per_chunk;
    r /= p.mt_per_chunk;
    const int i = r % p.n;
    const int b = r / p.n;
    arow0 = b * p.T + i * p.C + mt * kBM;
    brow0 = (b * p.n + i) * p.d + nt * kBN;
    rows_valid = min(kBM, min(p.C, p.T - i * p.C) - mt * kBM);
    n0 = nt * kBN;
    seq = b;
    srow0 = i * p.C + mt * kBM;
    acc = local & 1;
  }
  // Row tiles past the end of a partial last chunk have nothing to do.
  __device__ int num_segments() const { return rows_valid > 0 ? 1 : 0; }
  __device__ int seg_acc(int) const { return acc; }
  __device__ int seg_kblocks(int) const { return p.kblocks; }
  __device__ bool seg_fresh(int) const { return true; }

  __device__ void load(int, int kb, uint8_t* stage, uint64_t* bar) const {
    const int k = kb * kBK;
    tma_load_2d(stage, &p.tm_z, bar, k, arow0);
    tma_load_2d(stage + kATileBytes, &p.tm_snap, bar, k, brow0);
  }
  static __device__ uint64_t a_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }
  static __device__ uint64_t b_desc(uint32_t base, int k) {
    return sdesc_sw128(base + uint32_t(k) * 32u, 16u, 1024u);
  }

  // bf16 O: 64-column TMA stores of 64-row halves through a [B][T][d] map:
  // the second half is stored only when the chunk reaches it (chunk lengths
  // are multiples of 64), rows >= T and columns >= d are clipped.  fp32 O:
  // direct 16-byte stores.
  __device__ void epilogue(int, int row, uint32_t trow, EpiStager& st) const {
    if (!p.out_fp32) {
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
          tma_store_3d(&p.tm_os, src, n0 + g * 64, srow0, seq);
          if (rows_valid > 64) tma_store_3d(&p.tm_os, src + 64 * 128, n0 + g * 64, srow0 + 64, seq);
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
};

__global__ void __launch_bounds__(PipeShape<ApplySched>::kThreads, 1)
    apply_kernel(const __grid_constant__ ApplyParams p, unsigned int* status) {
  run_pipeline<ApplySched>(p, status);
}

}  // namespace

cudaError_t launch_apply(const LaunchEnv& env, const CUtensorMap& tm_z, const CUtensorMap& tm_snap,
                         const CUtensorMap& tm_os, void* out, bool out_fp32, int B, int T, int d,
                         int f, int C) {
  ApplyParams p;
  p.tm_z = tm_z;
  p.tm_snap = tm_snap;
  p.tm_os = tm_os;
  p.out = out;
  p.out_fp32 = out_fp32 ? 1 : 0;
  p.B = B;
  p.T = T;
  p.d = d;
  p.f = f;
  p.C = C;
  p.n = (T + C - 1) / C;
  p.mt_per_chunk = (C + kBM - 1) / kBM;
  p.nt = (d + kBN - 1) / kBN;
  p.kblocks = (f + kBK - 1) / kBK;
  const int64_t units = int64_t(B) * p.n * p.mt_per_chunk * p.nt;
  if (units == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(pipe_smem_bytes<ApplySched>()));
  if (e != cudaSuccess) return e;
  const int grid = units < env.num_sms ? int(units) : env.num_sms;
  apply_kernel<<<grid, PipeShape<ApplySched>::kThreads, pipe_smem_bytes<ApplySched>(), env.stream>>>(p, env.status);
  return cudaGetLastError();
}

}  // namespace ittt
