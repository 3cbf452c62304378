// ittt_noalloc.cu -- ittt_forward_noalloc: the layer forward for callers
// that must not allocate device memory.
//
// Some callers cannot call cudaMalloc, cudaMallocAsync or any other
// allocating routine once they are running: a serving loop whose device
// memory budget is fixed and fully partitioned at start-up, a process whose
// device memory belongs to another framework's caching allocator (a raw
// allocation would fail or fragment it), or a real-time path that forbids
// allocation after initialisation.  ittt_forward takes its scratch from a
// stream-ordered pool, which these callers cannot use.
//
// This entry point runs the same kernels as ittt_forward on the same
// arguments, but all of its scratch (Z, the convolved X0, eta*Vhat and the
// bf16 weight snapshots) lives in one file-scope device array of
// kNoAllocScratchBytes.  Consequences for the caller:
//   - every GPU that loads this library holds that array until the process
//     exits;
//   - a call whose scratch would not fit is rejected (ITTT_ERR_UNSUPPORTED)
//     before anything is enqueued;
//   - every call shares the one array, so calls that overlap on the GPU
//     (different streams, or different host threads) race on it: serialise
//     them on one stream;
//   - the first call on a device does a one-time set-up (it looks up the
//     array's device address with cudaGetSymbolAddress); make that first call
//     before any stream capture.
// Nothing in the scratch has to start at zero: every region is written in
// full before it is read.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "ittt.h"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
// The pair GEMMs' unit counters, zeroed at the start of every call (shared
// like the scratch: calls are serialised on one stream).
static __device__ __align__(16) unsigned int g_noalloc_tickets[ittt::kNumTickets];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct NoAllocDevice {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
  unsigned int* tickets = nullptr;   // device address of g_noalloc_tickets
  unsigned int* status = nullptr;
  int num_sms = 0;
};

std::mutex g_na_mutex;
EncodeTiledFn g_na_encode = nullptr;
NoAllocDevice g_na_dev[kMaxDevices];

ittt_status na_fail(ittt_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  ittt::set_last_error(buf);
  return s;
}

// One-time per-device set-up, with that device current.
ittt_status na_setup(NoAllocDevice** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return na_fail(ITTT_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return na_fail(ITTT_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lock(g_na_mutex);
  NoAllocDevice& nd = g_na_dev[dev];
  if (!nd.ready) {
    if (g_na_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
        return na_fail(ITTT_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
      g_na_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return na_fail(ITTT_ERR_UNSUPPORTED, "built for sm_103a (GB300); device %d is sm_%d%d", dev,
                     major, minor);
    e = cudaDeviceGetAttribute(&nd.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
      return na_fail(ITTT_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    // In host code g_noalloc_scratch names a host-side stand-in; the kernels
    // need the array's device address.
    void* scratch = nullptr;
    e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
    if (e != cudaSuccess)
      return na_fail(ITTT_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    nd.scratch = static_cast<unsigned char*>(scratch);
    void* tickets = nullptr;
    e = cudaGetSymbolAddress(&tickets, g_noalloc_tickets);
    if (e != cudaSuccess)
      return na_fail(ITTT_ERR_CUDA, "cudaGetSymbolAddress(tickets): %s", cudaGetErrorString(e));
    nd.tickets = static_cast<unsigned int*>(tickets);
    e = ittt::status_word_address(&nd.status);
    if (e != cudaSuccess)
      return na_fail(ITTT_ERR_CUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
    nd.ready = true;
  }
  *out = &nd;
  return ITTT_OK;
}

ittt_status na_check(const ittt_tensor* t, const char* name, int ndim, const int64_t* shape,
                     bool allow_bf16, bool allow_fp32) {
  if (t == nullptr || t->data == nullptr)
    return na_fail(ITTT_ERR_INVALID_ARG, "%s: null descriptor or data pointer", name);
  if (!((t->dtype == ITTT_BF16 && allow_bf16) || (t->dtype == ITTT_FP32 && allow_fp32)))
    return na_fail(ITTT_ERR_INVALID_ARG, "%s: unsupported dtype %d", name, int(t->dtype));
  if (t->ndim != ndim)
    return na_fail(ITTT_ERR_INVALID_ARG, "%s: expected %d dims, got %d", name, ndim,
                   int(t->ndim));
  int64_t expect = 1;
  for (int k = ndim - 1; k >= 0; --k) {
    if (t->shape[k] != shape[k])
      return na_fail(ITTT_ERR_INVALID_ARG, "%s: dim %d is %lld, expected %lld", name, k,
                     (long long)t->shape[k], (long long)shape[k]);
    if (t->stride[k] != expect && t->shape[k] != 1)
      return na_fail(ITTT_ERR_INVALID_ARG, "%s: not dense row-major", name);
    expect *= shape[k];
  }
  if (reinterpret_cast<uintptr_t>(t->data) % 16 != 0)
    return na_fail(ITTT_ERR_INVALID_ARG, "%s: data pointer not 16-byte aligned", name);
  return ITTT_OK;
}

size_t na_bytes(const ittt_tensor* t) {
  size_t n = t->dtype == ITTT_FP32 ? 4 : 2;
  for (int k = 0; k < t->ndim; ++k) n *= size_t(t->shape[k]);
  return n;
}

size_t na_round(size_t x) { return (x + 255) & ~size_t(255); }

// 3-D bf16 map {inner, mid, outer} of a dense tensor, 128-byte swizzle.
ittt_status na_map_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t mid,
                   uint64_t outer, uint32_t box_inner, uint32_t box_mid, const char* what) {
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {inner * 2, inner * mid * 2};
  cuuint32_t box[3] = {box_inner, box_mid, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_na_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return na_fail(ITTT_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, int(r));
  return ITTT_OK;
}

ittt_status na_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                   uint32_t box_inner, uint32_t box_outer, const char* what,
                   CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_na_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return na_fail(ITTT_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, int(r));
  return ITTT_OK;
}

// The target and gate/up GEMMs on CTA pairs where two can be resident.
cudaError_t target_pair_or_single(const ittt::LaunchEnv& env, const CUtensorMap& tm_xc,
                                  const CUtensorMap& tm_wt, const CUtensorMap& tm_wt128,
                                  const CUtensorMap& tm_vs, const float* conv_w,
                                  __nv_bfloat16* vhat, float eta, int M, int T, int d, int C) {
  cudaError_t e = ittt::launch_target_pair(env, tm_xc, tm_wt128, tm_vs, nullptr, vhat, eta, M, d);
  if (e != cudaErrorNotSupported) return e;
  cudaGetLastError();
  return ittt::launch_target(env, tm_xc, tm_wt, tm_vs, conv_w, nullptr, vhat, eta, M, T, d, C,
                             ITTT_PAD_CHUNK, false);
}

cudaError_t gateup_pair_or_single(const ittt::LaunchEnv& env, const CUtensorMap& tm_h,
                                  const CUtensorMap& tm_wg, const CUtensorMap& tm_wu,
                                  const CUtensorMap& tm_zk, int M, int f, int d) {
  cudaError_t e = ittt::launch_gateup_pair(env, tm_h, tm_wg, tm_wu, tm_zk, M, f, d);
  if (e != cudaErrorNotSupported) return e;
  cudaGetLastError();
  return ittt::launch_gateup(env, tm_h, tm_wg, tm_wu, tm_zk, M, f, d);
}

}  // namespace

extern "C" ittt_status ittt_forward_noalloc(const ittt_tensor* H, const ittt_tensor* X0,
                                            const ittt_tensor* W_gate, const ittt_tensor* W_up,
                                            const ittt_tensor* W_down0,
                                            const ittt_tensor* W_target,
                                            const ittt_tensor* conv_w, float eta, int64_t chunk,
                                            ittt_tensor* out, ittt_stream_t stream_) {
  ittt::set_last_error("");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (H == nullptr || H->ndim != 3 || W_gate == nullptr || W_gate->ndim != 2)
    return na_fail(ITTT_ERR_INVALID_ARG, "H must be [B,T,d] and W_gate [f,d]");
  const int64_t B = H->shape[0], T = H->shape[1], d = H->shape[2], f = W_gate->shape[0];
  if (B <= 0 || T <= 0 || d <= 0 || f <= 0)
    return na_fail(ITTT_ERR_INVALID_ARG, "sizes must be positive");
  if (chunk <= 0) return na_fail(ITTT_ERR_INVALID_ARG, "chunk must be positive");
  if (d % 8 != 0 || f % 8 != 0)
    return na_fail(ITTT_ERR_UNSUPPORTED, "d_model and d_ff must be multiples of 8");
  if (B * T >= (int64_t(1) << 31))
    return na_fail(ITTT_ERR_UNSUPPORTED, "B*T exceeds 32-bit token coordinates");
  if (!std::isfinite(eta)) return na_fail(ITTT_ERR_INVALID_ARG, "eta is not finite");
  const int64_t n = (T + chunk - 1) / chunk;  // the last chunk may be partial
  const int64_t sh_btd[3] = {B, T, d}, sh_fd[2] = {f, d}, sh_df[2] = {d, f}, sh_dd[2] = {d, d},
                sh_d3[2] = {d, 3};
  ittt_status s;
  if ((s = na_check(H, "H", 3, sh_btd, true, false))) return s;
  if ((s = na_check(X0, "X0", 3, sh_btd, true, false))) return s;
  if ((s = na_check(W_gate, "W_gate", 2, sh_fd, true, false))) return s;
  if ((s = na_check(W_up, "W_up", 2, sh_fd, true, false))) return s;
  if ((s = na_check(W_down0, "W_down0", 2, sh_df, true, true))) return s;
  if ((s = na_check(W_target, "W_target", 2, sh_dd, true, false))) return s;
  if ((s = na_check(conv_w, "conv_w", 2, sh_d3, false, true))) return s;
  if ((s = na_check(out, "out", 3, sh_btd, true, true))) return s;
  const ittt_tensor* ins[] = {H, X0, W_gate, W_up, W_down0, W_target, conv_w};
  const uintptr_t o0 = reinterpret_cast<uintptr_t>(out->data), o1 = o0 + na_bytes(out);
  for (const ittt_tensor* t : ins) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(t->data), a1 = a0 + na_bytes(t);
    if (a0 < o1 && o0 < a1) return na_fail(ITTT_ERR_INVALID_ARG, "out overlaps an input");
  }
  // Scratch plan inside the static array: Z, Xc, eta*Vhat, snapshots.
  const size_t z_bytes = na_round(size_t(B) * T * f * 2);
  const size_t act_bytes = na_round(size_t(B) * T * d * 2);
  const size_t snap_bytes = na_round(size_t(B) * n * d * f * 2);
  const size_t need = z_bytes + 2 * act_bytes + snap_bytes;
  if (need > kNoAllocScratchBytes)
    return na_fail(ITTT_ERR_UNSUPPORTED,
                   "this call needs %zu bytes of scratch; ittt_forward_noalloc holds at most %zu "
                   "(64 MiB) -- use ittt_forward or ittt_forward_ex with a workspace",
                   need, kNoAllocScratchBytes);

  NoAllocDevice* nd = nullptr;
  if ((s = na_setup(&nd))) return s;
  auto* z = reinterpret_cast<__nv_bfloat16*>(nd->scratch);
  auto* xc = reinterpret_cast<__nv_bfloat16*>(nd->scratch + z_bytes);
  auto* vhat = reinterpret_cast<__nv_bfloat16*>(nd->scratch + z_bytes + act_bytes);
  auto* snap = reinterpret_cast<__nv_bfloat16*>(nd->scratch + z_bytes + 2 * act_bytes);

  const uint64_t M = uint64_t(B * T);
  CUtensorMap tm_h, tm_wg, tm_wu, tm_x0, tm_xc, tm_wt, tm_wt128, tm_vmn, tm_zmn, tm_zk, tm_snap,
      tm_snap_pair, tm_w0d, tm_w0d_pair;
  // As in ittt_forward: a bf16 W_0 is read by the apply itself (no slot-0
  // copy), the GEMMs run on CTA pairs where two can be resident.
  const bool w0_direct = W_down0->dtype == ITTT_BF16;
  if ((s = na_map(&tm_h, H->data, d, M, 64, 128, "H"))) return s;
  if ((s = na_map(&tm_wg, W_gate->data, d, f, 64, 128, "W_gate"))) return s;
  if ((s = na_map(&tm_wu, W_up->data, d, f, 64, 128, "W_up"))) return s;
  if ((s = na_map(&tm_x0, X0->data, d, M, ittt::kConvMapBoxCols, ittt::kConvMapBoxRows,
                  "X0 (conv)", CU_TENSOR_MAP_SWIZZLE_NONE)))
    return s;
  if ((s = na_map(&tm_xc, xc, d, M, 64, 128, "Xc"))) return s;
  if ((s = na_map(&tm_wt, W_target->data, d, d, 64, 256, "W_target"))) return s;
  if ((s = na_map(&tm_wt128, W_target->data, d, d, 64, 128, "W_target (pair)"))) return s;
  if ((s = na_map(&tm_vmn, vhat, d, M, 64, 64, "Vhat"))) return s;
  if ((s = na_map(&tm_zmn, z, f, M, 64, 64, "Z (update)"))) return s;
  if ((s = na_map(&tm_zk, z, f, M, 64, 128, "Z (apply)"))) return s;
  if ((s = na_map(&tm_snap, snap, f, uint64_t(B * n * d), 64, 256, "snapshots"))) return s;
  if ((s = na_map(&tm_snap_pair, snap, f, uint64_t(B * n * d), 64, 128, "snapshots (pair)")))
    return s;
  if (w0_direct) {
    if ((s = na_map(&tm_w0d, W_down0->data, f, uint64_t(d), 64, 256, "W_0"))) return s;
    if ((s = na_map(&tm_w0d_pair, W_down0->data, f, uint64_t(d), 64, 128, "W_0 (pair)")))
      return s;
  }
  CUtensorMap tm_vs, tm_ss, tm_os;
  memset(&tm_os, 0, sizeof(tm_os));
  if ((s = na_map(&tm_vs, vhat, d, M, 64, 128, "Vhat (store)"))) return s;
  if ((s = na_map_3d(&tm_ss, snap, f, d, uint64_t(B * n), 64, 128, "snapshots (store)")))
    return s;
  if (out->dtype == ITTT_BF16 && (s = na_map(&tm_os, out->data, d, M, 64, 64, "O (store)")))
    return s;

  const ittt::LaunchEnv env{stream, nd->num_sms, nd->status, nd->tickets};
  ittt::DocMap docs;
  memset(&docs, 0, sizeof(docs));
  docs.ndocs = int(B);
  docs.nchunks = int(B * n);
  docs.T = int(T);
  docs.n = int(n);
  docs.C = int(chunk);
  docs.mtc = int((chunk + 127) / 128);
  docs.tiles_per_seq = int((n - 1) * docs.mtc + (T - (n - 1) * chunk + 127) / 128);
  docs.ntiles = int(B) * docs.tiles_per_seq;
  docs.mtc2 = int((chunk + 255) / 256);
  docs.tiles_per_seq2 = int((n - 1) * docs.mtc2 + (T - (n - 1) * chunk + 255) / 256);
  docs.ntiles2 = int(B) * docs.tiles_per_seq2;
  const bool w0_fp32 = W_down0->dtype == ITTT_FP32;
  cudaError_t e;
  const char* what = nullptr;
  if ((e = cudaMemsetAsync(nd->tickets, 0, ittt::kNumTickets * sizeof(unsigned int), stream)) !=
      cudaSuccess) {
    what = "unit counters";
  } else if ((e = ittt::launch_conv(env, tm_x0, static_cast<const float*>(conv_w->data), xc,
                             int64_t(M), docs, int(d), ITTT_PAD_CHUNK)) != cudaSuccess) {
    what = "conv";
  } else if ((e = target_pair_or_single(env, tm_xc, tm_wt, tm_wt128, tm_vs,
                                         static_cast<const float*>(conv_w->data), vhat, eta,
                                         int(M), int(T), int(d), int(chunk))) != cudaSuccess) {
    what = "target";
  } else if ((e = gateup_pair_or_single(env, tm_h, tm_wg, tm_wu, tm_zk, int(M), int(f),
                                        int(d))) != cudaSuccess) {
    what = "gate/up";
  } else if (!w0_direct && (e = ittt::launch_snapshot0(env, W_down0->data, w0_fp32, 0, snap, docs,
                                                       int(d), int(f))) != cudaSuccess) {
    what = "snapshot";
  } else {
    ittt::UpdateArgs ua;
    ua.docs = docs;
    ua.upd_docs = nullptr;
    ua.n_udocs = n > 1 ? int(B) : 0;
    ua.final_update = false;
    ua.d = int(d);
    ua.f = int(f);
    ua.w0 = W_down0->data;
    ua.w0_fp32 = w0_fp32;
    ua.w0_bstride = 0;
    ua.state_out = nullptr;
    ua.allow_pairs = chunk % 64 == 0;  // every updated chunk is a whole chunk
    if ((e = ittt::launch_update(env, tm_vmn, tm_zmn, tm_ss, ua)) != cudaSuccess) {
      what = "update";
    } else {
      e = ittt::launch_apply_pair(env, tm_zk, tm_snap_pair, w0_direct ? &tm_w0d_pair : nullptr,
                                  tm_os, out->data, out->dtype == ITTT_FP32, docs, int(d), int(f));
      if (e == cudaErrorNotSupported) {
        cudaGetLastError();
        e = ittt::launch_apply(env, tm_zk, tm_snap, w0_direct ? &tm_w0d : nullptr, tm_os,
                               out->data, out->dtype == ITTT_FP32, docs, int(d), int(f));
      }
      if (e != cudaSuccess) what = "apply";
    }
  }
  if (what != nullptr)
    return na_fail(ITTT_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
  return ITTT_OK;
}
