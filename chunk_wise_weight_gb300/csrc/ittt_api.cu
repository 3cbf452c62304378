// ittt_api.cu -- the C-ABI of libittt.so (declared in include/ittt.h).
//
// Validates every descriptor before anything is enqueued, takes the scratch
// it needs (stream-ordered, from a library-private memory pool, or from a
// caller workspace), encodes the TMA tensor maps and launches the kernels in
// data-flow order on the caller's stream:
//   conv3 (Xc) ; target GEMM (eta*Vhat) ; gate/up GEMM (Z) ; snapshot 0 ;
//   update walk (snapshots W_1..W_{n-1}) ; apply GEMM (O).
// With ITTT_FLAG_FUSED_CONV the target GEMM computes the conv itself.  (Run
// beside the gate/up GEMM on a second stream, the conv slowed that GEMM by
// more than its own 0.2 ms at the 32k-token workload, so it runs in line.)
// No host synchronisation happens inside a forward call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "ittt.h"
#include "kernels.h"
#include "sm103.cuh"

namespace {

constexpr int kMaxDevices = 64;

thread_local std::string g_last_error;

ittt_status fail(ittt_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

ittt_status cuda_fail(cudaError_t e, const char* what) {
  return fail(e == cudaErrorMemoryAllocation ? ITTT_ERR_OOM : ITTT_ERR_CUDA, "%s: %s (%s)", what,
              cudaGetErrorName(e), cudaGetErrorString(e));
}

// Device status word the kernels record failures in (kStatusTimeout).
__device__ unsigned int g_device_status;

// cuTensorMapEncodeTiled, fetched from the driver once.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  unsigned int* status = nullptr;
  cudaMemPool_t pool = nullptr;
};

std::mutex g_mutex;
EncodeTiledFn g_encode = nullptr;
DeviceState g_dev[kMaxDevices];

ittt_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ITTT_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& ds = g_dev[dev];
  if (!ds.ready) {
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
        return fail(ITTT_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return fail(ITTT_ERR_UNSUPPORTED,
                  "libittt.so is built for sm_103a (GB300); device %d is sm_%d%d", dev, major,
                  minor);
    e = cudaDeviceGetAttribute(&ds.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    void* sym = nullptr;
    e = cudaGetSymbolAddress(&sym, g_device_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    ds.status = static_cast<unsigned int*>(sym);
    cudaMemPoolProps props;
    memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    e = cudaMemPoolCreate(&ds.pool, &props);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
    uint64_t keep = ~0ull;  // keep freed scratch mapped for the next call
    cudaMemPoolSetAttribute(ds.pool, cudaMemPoolAttrReleaseThreshold, &keep);
    ds.ready = true;
  }
  *out = &ds;
  return ITTT_OK;
}

// ---------------------------------------------------------------- validation
size_t dtype_size(int32_t dt) { return dt == ITTT_FP32 ? 4 : 2; }

ittt_status check_tensor(const ittt_tensor* t, const char* name, int ndim, const int64_t* shape,
                         bool allow_bf16, bool allow_fp32) {
  if (t == nullptr) return fail(ITTT_ERR_INVALID_ARG, "%s: null descriptor", name);
  if (t->data == nullptr) return fail(ITTT_ERR_INVALID_ARG, "%s: null data pointer", name);
  if (!((t->dtype == ITTT_BF16 && allow_bf16) || (t->dtype == ITTT_FP32 && allow_fp32)))
    return fail(ITTT_ERR_INVALID_ARG, "%s: unsupported dtype %d", name, int(t->dtype));
  if (t->ndim != ndim)
    return fail(ITTT_ERR_INVALID_ARG, "%s: expected %d dims, got %d", name, ndim, int(t->ndim));
  int64_t expect_stride = 1;
  for (int k = ndim - 1; k >= 0; --k) {
    if (t->shape[k] != shape[k])
      return fail(ITTT_ERR_INVALID_ARG, "%s: dim %d is %lld, expected %lld", name, k,
                  (long long)t->shape[k], (long long)shape[k]);
    if (t->stride[k] != expect_stride && t->shape[k] != 1)
      return fail(ITTT_ERR_INVALID_ARG, "%s: not dense row-major (dim %d stride %lld)", name, k,
                  (long long)t->stride[k]);
    expect_stride *= shape[k];
  }
  if (reinterpret_cast<uintptr_t>(t->data) % 16 != 0)
    return fail(ITTT_ERR_INVALID_ARG, "%s: data pointer not 16-byte aligned", name);
  return ITTT_OK;
}

size_t tensor_bytes(const ittt_tensor* t) {
  size_t n = dtype_size(t->dtype);
  for (int k = 0; k < t->ndim; ++k) n *= size_t(t->shape[k]);
  return n;
}

bool overlaps(const ittt_tensor* a, const ittt_tensor* b) {
  if (a == nullptr || b == nullptr) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a->data), a1 = a0 + tensor_bytes(a);
  const uintptr_t b0 = reinterpret_cast<uintptr_t>(b->data), b1 = b0 + tensor_bytes(b);
  return a0 < b1 && b0 < a1;
}

ittt_status check_sizes(int64_t B, int64_t T, int64_t d, int64_t f, int64_t chunk) {
  if (B <= 0 || T <= 0 || d <= 0 || f <= 0)
    return fail(ITTT_ERR_INVALID_ARG, "sizes must be positive (B=%lld T=%lld d=%lld f=%lld)",
                (long long)B, (long long)T, (long long)d, (long long)f);
  if (chunk <= 0) return fail(ITTT_ERR_INVALID_ARG, "chunk %lld must be positive", (long long)chunk);
  if (chunk % 64 != 0 || T % 64 != 0)
    return fail(ITTT_ERR_UNSUPPORTED, "chunk %lld and T %lld must be multiples of 64",
                (long long)chunk, (long long)T);
  if (d % 8 != 0 || f % 8 != 0)
    return fail(ITTT_ERR_UNSUPPORTED, "d_model=%lld and d_ff=%lld must be multiples of 8",
                (long long)d, (long long)f);
  const int64_t n = (T + chunk - 1) / chunk;
  if (B * T >= (int64_t(1) << 31) || B * n * d >= (int64_t(1) << 31) || d * f >= (int64_t(1) << 40))
    return fail(ITTT_ERR_UNSUPPORTED, "sizes exceed 32-bit tile coordinates");
  return ITTT_OK;
}

// --------------------------------------------------------------- workspace
struct Layout {
  size_t z = 0, vhat = 0, xc = 0, snap = 0, scores = 0, w0b = 0, total = 0;
};

size_t round_up(size_t x) { return (x + 255) & ~size_t(255); }

Layout plan_workspace(int64_t B, int64_t T, int64_t d, int64_t f, int64_t chunk, bool need_z,
                      bool need_vhat, bool need_xc, bool need_snap) {
  Layout L;
  const int64_t n = (T + chunk - 1) / chunk;
  size_t off = 0;
  if (need_z) {
    L.z = off;
    off += round_up(size_t(B) * T * f * 2);
  }
  if (need_vhat) {
    L.vhat = off;
    off += round_up(size_t(B) * T * d * 2);
  }
  if (need_xc) {
    L.xc = off;
    off += round_up(size_t(B) * T * d * 2);
  }
  if (need_snap) {
    L.snap = off;
    off += round_up(size_t(B) * n * d * f * 2);
  }
  L.total = off;
  return L;
}

// ------------------------------------------------------------- tensor maps
// 3-D bf16 map {inner, mid, outer} of a dense tensor, 128-byte swizzle.
ittt_status make_map_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t mid,
                   uint64_t outer, uint32_t box_inner, uint32_t box_mid, const char* what) {
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {inner * 2, inner * mid * 2};
  cuuint32_t box[3] = {box_inner, box_mid, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(ITTT_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, int(r));
  return ITTT_OK;
}

ittt_status make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                     uint32_t box_inner, uint32_t box_outer, const char* what) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(ITTT_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, int(r));
  return ITTT_OK;
}

struct ScratchGuard {
  void* ptr = nullptr;
  cudaStream_t stream = nullptr;
  ~ScratchGuard() {
    if (ptr) cudaFreeAsync(ptr, stream);
  }
};

ittt_status forward_impl(const ittt_tensor* H, const ittt_tensor* X0, const ittt_tensor* W_gate,
                         const ittt_tensor* W_up, const ittt_tensor* W_down0,
                         const ittt_tensor* W_target, const ittt_tensor* conv_w, float eta,
                         int64_t chunk, ittt_tensor* out, cudaStream_t stream,
                         const ittt_opts* opts) {
  g_last_error.clear();
  ittt_opts o;
  memset(&o, 0, sizeof(o));
  if (opts) o = *opts;
  if (o.pad_mode != ITTT_PAD_CHUNK && o.pad_mode != ITTT_PAD_SEQUENCE)
    return fail(ITTT_ERR_INVALID_ARG, "pad_mode %d", int(o.pad_mode));
  if (o.flags & ~int32_t(ITTT_FLAG_FUSED_CONV | ITTT_FLAG_DUAL))
    return fail(ITTT_ERR_INVALID_ARG, "unknown flags 0x%x", unsigned(o.flags));
  const bool fused = (o.flags & ITTT_FLAG_FUSED_CONV) != 0;
  const bool dual = (o.flags & ITTT_FLAG_DUAL) != 0;
  if (dual && (o.state_out || o.snap_buf))
    return fail(ITTT_ERR_UNSUPPORTED,
                "the dual form forms no fast-weight state: no state_out or snap_buf");
  if (H == nullptr || H->ndim != 3)
    return fail(ITTT_ERR_INVALID_ARG, "H: expected a [B,T,d] descriptor");
  const int64_t B = H->shape[0], T = H->shape[1], d = H->shape[2];
  if (W_gate == nullptr || W_gate->ndim != 2)
    return fail(ITTT_ERR_INVALID_ARG, "W_gate: expected a [f,d] descriptor");
  const int64_t f = W_gate->shape[0];
  ittt_status s = check_sizes(B, T, d, f, chunk);
  if (s != ITTT_OK) return s;
  if (!std::isfinite(eta)) return fail(ITTT_ERR_INVALID_ARG, "eta is not finite");
  const int64_t n = (T + chunk - 1) / chunk;  // the last chunk may be partial
  if (dual && T % chunk != 0)
    return fail(ITTT_ERR_UNSUPPORTED, "the dual form needs chunk to divide T");

  const int64_t sh_btd[3] = {B, T, d}, sh_fd[2] = {f, d}, sh_df[2] = {d, f}, sh_dd[2] = {d, d},
                sh_d3[2] = {d, 3}, sh_bdf[3] = {B, d, f}, sh_btf[3] = {B, T, f},
                sh_bndf[4] = {B, n, d, f};
  if ((s = check_tensor(H, "H", 3, sh_btd, true, false))) return s;
  if ((s = check_tensor(X0, "X0", 3, sh_btd, true, false))) return s;
  if ((s = check_tensor(W_gate, "W_gate", 2, sh_fd, true, false))) return s;
  if ((s = check_tensor(W_up, "W_up", 2, sh_fd, true, false))) return s;
  if (o.state_in) {
    if ((s = check_tensor(o.state_in, "state_in", 3, sh_bdf, false, true))) return s;
  } else if ((s = check_tensor(W_down0, "W_down0", 2, sh_df, true, true))) {
    return s;
  }
  if ((s = check_tensor(W_target, "W_target", 2, sh_dd, true, false))) return s;
  if ((s = check_tensor(conv_w, "conv_w", 2, sh_d3, false, true))) return s;
  if ((s = check_tensor(out, "out", 3, sh_btd, true, true))) return s;
  if (o.state_out && (s = check_tensor(o.state_out, "state_out", 3, sh_bdf, false, true))) return s;
  if (o.z_buf && (s = check_tensor(o.z_buf, "z_buf", 3, sh_btf, true, false))) return s;
  if (o.vhat_buf && (s = check_tensor(o.vhat_buf, "vhat_buf", 3, sh_btd, true, false))) return s;
  if (o.snap_buf && (s = check_tensor(o.snap_buf, "snap_buf", 4, sh_bndf, true, false))) return s;
  const int64_t sh_bt[2] = {B, T};
  if (o.eta_tok && (s = check_tensor(o.eta_tok, "eta_tok", 2, sh_bt, false, true))) return s;

  const ittt_tensor* inputs[] = {H,        X0,     W_gate,   W_up, o.state_in ? o.state_in : W_down0,
                                 W_target, conv_w, o.eta_tok};
  const ittt_tensor* writes[] = {out, o.state_out, o.z_buf, o.vhat_buf, o.snap_buf};
  for (const ittt_tensor* w : writes) {
    for (const ittt_tensor* in : inputs)
      if (overlaps(w, in)) return fail(ITTT_ERR_INVALID_ARG, "an output overlaps an input");
  }
  for (int a = 0; a < 5; ++a)
    for (int b = a + 1; b < 5; ++b)
      if (overlaps(writes[a], writes[b]))
        return fail(ITTT_ERR_INVALID_ARG, "two output buffers overlap");

  DeviceState* ds = nullptr;
  if ((s = device_state(&ds))) return s;

  // Scratch.
  // The dual form needs the scores and, unless W_0 is one bf16 matrix
  // already, a bf16 copy of each sequence's W_0 instead of the snapshots.
  const bool w0_is_bf16 = !o.state_in && W_down0->dtype == ITTT_BF16;
  Layout L = plan_workspace(B, T, d, f, chunk, o.z_buf == nullptr, o.vhat_buf == nullptr, !fused,
                            !dual && o.snap_buf == nullptr);
  if (dual) {
    L.scores = L.total;
    L.total += round_up(size_t(B) * T * T * 2);
    if (!w0_is_bf16) {
      L.w0b = L.total;
      L.total += round_up(size_t(o.state_in ? B : 1) * d * f * 2);
    }
  }
  ScratchGuard guard;
  uint8_t* ws = nullptr;
  if (o.workspace) {
    if (o.workspace_bytes < L.total)
      return fail(ITTT_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu needed",
                  o.workspace_bytes, L.total);
    if (reinterpret_cast<uintptr_t>(o.workspace) % 256 != 0)
      return fail(ITTT_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    ws = static_cast<uint8_t*>(o.workspace);
  } else {
    void* p = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&p, L.total, ds->pool, stream);
    if (e != cudaSuccess) return cuda_fail(e, "scratch allocation");
    guard.ptr = p;
    guard.stream = stream;
    ws = static_cast<uint8_t*>(p);
  }
  auto* z = o.z_buf ? static_cast<__nv_bfloat16*>(o.z_buf->data)
                    : reinterpret_cast<__nv_bfloat16*>(ws + L.z);
  auto* vhat = o.vhat_buf ? static_cast<__nv_bfloat16*>(o.vhat_buf->data)
                          : reinterpret_cast<__nv_bfloat16*>(ws + L.vhat);
  auto* xc = reinterpret_cast<__nv_bfloat16*>(ws + L.xc);
  auto* snap = o.snap_buf ? static_cast<__nv_bfloat16*>(o.snap_buf->data)
                          : reinterpret_cast<__nv_bfloat16*>(ws + L.snap);

  // Tensor maps.
  const uint64_t M = uint64_t(B * T);
  CUtensorMap tm_h, tm_wg, tm_wu, tm_a, tm_wt, tm_vmn, tm_zmn, tm_zk, tm_snap;
  if ((s = make_map(&tm_h, H->data, d, M, 64, 128, "H"))) return s;
  if ((s = make_map(&tm_wg, W_gate->data, d, f, 64, 128, "W_gate"))) return s;
  if ((s = make_map(&tm_wu, W_up->data, d, f, 64, 128, "W_up"))) return s;
  if (fused) {
    if ((s = make_map(&tm_a, X0->data, d, M, 64, 130, "X0"))) return s;
  } else if ((s = make_map(&tm_a, xc, d, M, 64, 128, "Xc"))) {
    return s;
  }
  if ((s = make_map(&tm_wt, W_target->data, d, d, 64, 256, "W_target"))) return s;
  // Output maps for the epilogues' TMA stores (Z's is tm_zk).
  CUtensorMap tm_vs, tm_ss, tm_os;
  memset(&tm_ss, 0, sizeof(tm_ss));
  memset(&tm_os, 0, sizeof(tm_os));
  if ((s = make_map(&tm_vs, vhat, d, M, 64, 128, "Vhat (store)"))) return s;
  if (out->dtype == ITTT_BF16 &&
      (s = make_map_3d(&tm_os, out->data, d, T, uint64_t(B), 64, 64, "O (store)")))
    return s;
  if ((s = make_map(&tm_vmn, vhat, d, M, 64, 64, "Vhat"))) return s;
  if ((s = make_map(&tm_zmn, z, f, M, 64, 64, "Z (update)"))) return s;
  if ((s = make_map(&tm_zk, z, f, M, 64, 128, "Z (apply)"))) return s;
  CUtensorMap tm_zs, tm_w0b, tm_sc;
  auto* scores = reinterpret_cast<__nv_bfloat16*>(ws + L.scores);
  const void* w0b = w0_is_bf16 ? W_down0->data : static_cast<const void*>(ws + L.w0b);
  if (dual) {
    if ((s = make_map(&tm_zs, z, f, M, 64, 256, "Z (scores)"))) return s;
    if ((s = make_map(&tm_w0b, w0b, f, uint64_t((o.state_in ? B : 1) * d), 64, 256, "bf16 W_0")))
      return s;
    if ((s = make_map(&tm_sc, scores, uint64_t(T), M, 64, 128, "scores"))) return s;
  } else {
    if ((s = make_map(&tm_snap, snap, f, uint64_t(B * n * d), 64, 256, "snapshots"))) return s;
    if ((s = make_map_3d(&tm_ss, snap, f, d, uint64_t(B * n), 64, 128, "snapshots (store)")))
      return s;
  }

  const ittt::LaunchEnv env{stream, ds->num_sms, ds->status};
  const void* w0 = o.state_in ? o.state_in->data : W_down0->data;
  const bool w0_fp32 = o.state_in ? true : (W_down0->dtype == ITTT_FP32);
  const int64_t w0_bstride = o.state_in ? d * f : 0;

  cudaEvent_t const* ev = reinterpret_cast<cudaEvent_t const*>(o.events);
  auto rec = [&](int slot, cudaStream_t st) -> cudaError_t {
    return ev ? cudaEventRecord(ev[slot], st) : cudaSuccess;
  };
  const float* cw = static_cast<const float*>(conv_w->data);

  cudaError_t e = cudaSuccess;
  const char* what = nullptr;
#define ITTT_STEP(call, name) \
  if (what == nullptr && (e = (call)) != cudaSuccess) what = name
  ITTT_STEP(rec(2 * ITTT_PHASE_CONV, stream), "event record");
  if (!fused) {
    ITTT_STEP(ittt::launch_conv(env, static_cast<const __nv_bfloat16*>(X0->data), cw, xc,
                                int64_t(M), int(T), int(d), int(chunk), int(o.pad_mode)),
              "conv launch");
  }
  ITTT_STEP(rec(2 * ITTT_PHASE_CONV + 1, stream), "event record");
  ITTT_STEP(rec(2 * ITTT_PHASE_TARGET, stream), "event record");
  ITTT_STEP(ittt::launch_target(env, tm_a, tm_wt, tm_vs, cw,
                                o.eta_tok ? static_cast<const float*>(o.eta_tok->data) : nullptr,
                                vhat, eta, int(M), int(T), int(d), int(chunk), int(o.pad_mode),
                                fused),
            "target launch");
  ITTT_STEP(rec(2 * ITTT_PHASE_TARGET + 1, stream), "event record");
  ITTT_STEP(rec(2 * ITTT_PHASE_GATEUP, stream), "event record");
  ITTT_STEP(ittt::launch_gateup(env, tm_h, tm_wg, tm_wu, tm_zk, int(M), int(f), int(d)),
            "gate/up launch");
  ITTT_STEP(rec(2 * ITTT_PHASE_GATEUP + 1, stream), "event record");
  ITTT_STEP(rec(2 * ITTT_PHASE_SNAPSHOT0, stream), "event record");
  if (!dual) {
    ITTT_STEP(ittt::launch_snapshot0(env, w0, w0_fp32, w0_bstride, snap, int(B), int(n), int(d),
                                     int(f)),
              "snapshot launch");
  } else if (!w0_is_bf16) {
    ITTT_STEP(ittt::launch_snapshot0(env, w0, w0_fp32, w0_bstride,
                                     static_cast<__nv_bfloat16*>(const_cast<void*>(w0b)),
                                     int(o.state_in ? B : 1), 1, int(d), int(f)),
              "W_0 copy launch");
  }
  ITTT_STEP(rec(2 * ITTT_PHASE_SNAPSHOT0 + 1, stream), "event record");
  if (!dual) {
    ittt::UpdateArgs ua;
    ua.B = int(B);
    ua.T = int(T);
    ua.d = int(d);
    ua.f = int(f);
    ua.C = int(chunk);
    ua.n = int(n);
    ua.n_upd = o.state_out ? int(n) : int(n - 1);
    ua.w0 = w0;
    ua.w0_fp32 = w0_fp32;
    ua.w0_bstride = w0_bstride;
    ua.snap = snap;
    ua.state_out = o.state_out ? static_cast<float*>(o.state_out->data) : nullptr;
    ITTT_STEP(rec(2 * ITTT_PHASE_UPDATE, stream), "event record");
    ITTT_STEP(ittt::launch_update(env, tm_vmn, tm_zmn, tm_ss, ua), "update launch");
    ITTT_STEP(rec(2 * ITTT_PHASE_UPDATE + 1, stream), "event record");
    ITTT_STEP(rec(2 * ITTT_PHASE_APPLY, stream), "event record");
    ITTT_STEP(ittt::launch_apply(env, tm_zk, tm_snap, tm_os, out->data,
                                 out->dtype == ITTT_FP32, int(B), int(T), int(d), int(f),
                                 int(chunk)),
              "apply launch");
    ITTT_STEP(rec(2 * ITTT_PHASE_APPLY + 1, stream), "event record");
  } else {
    ITTT_STEP(rec(2 * ITTT_PHASE_UPDATE, stream), "event record");
    ITTT_STEP(ittt::launch_scores(env, tm_zk, tm_zs, scores, int(B), int(T), int(f), int(chunk)),
              "scores launch");
    ITTT_STEP(rec(2 * ITTT_PHASE_UPDATE + 1, stream), "event record");
    ITTT_STEP(rec(2 * ITTT_PHASE_APPLY, stream), "event record");
    ITTT_STEP(ittt::launch_dual_apply(env, tm_zk, tm_w0b, tm_sc, tm_vmn, o.state_in != nullptr,
                                      out->data, out->dtype == ITTT_FP32, int(B), int(T), int(d),
                                      int(f), int(chunk)),
              "dual apply launch");
    ITTT_STEP(rec(2 * ITTT_PHASE_APPLY + 1, stream), "event record");
  }
#undef ITTT_STEP
  if (what != nullptr) return cuda_fail(e, what);
  return ITTT_OK;
}

}  // namespace

namespace ittt {

// Address of this library's device status word on the current device, for
// entry points defined in other translation units (no other set-up).
cudaError_t status_word_address(unsigned int** out) {
  void* sym = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&sym, g_device_status);
  if (e == cudaSuccess) *out = static_cast<unsigned int*>(sym);
  return e;
}

// Records `msg` as the calling thread's ittt_last_error() text.
void set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }

}  // namespace ittt

extern "C" {

ittt_status ittt_forward(const ittt_tensor* H, const ittt_tensor* X0, const ittt_tensor* W_gate,
                         const ittt_tensor* W_up, const ittt_tensor* W_down0,
                         const ittt_tensor* W_target, const ittt_tensor* conv_w, float eta,
                         int64_t chunk, ittt_tensor* out, ittt_stream_t stream) {
  return forward_impl(H, X0, W_gate, W_up, W_down0, W_target, conv_w, eta, chunk, out,
                      reinterpret_cast<cudaStream_t>(stream), nullptr);
}

ittt_status ittt_forward_ex(const ittt_tensor* H, const ittt_tensor* X0,
                            const ittt_tensor* W_gate, const ittt_tensor* W_up,
                            const ittt_tensor* W_down0, const ittt_tensor* W_target,
                            const ittt_tensor* conv_w, float eta, int64_t chunk,
                            ittt_tensor* out, ittt_stream_t stream, const ittt_opts* opts) {
  return forward_impl(H, X0, W_gate, W_up, W_down0, W_target, conv_w, eta, chunk, out,
                      reinterpret_cast<cudaStream_t>(stream), opts);
}

size_t ittt_workspace_bytes(int64_t B, int64_t T, int64_t d, int64_t f, int64_t chunk) {
  const std::string saved = g_last_error;
  if (check_sizes(B, T, d, f, chunk) != ITTT_OK) {
    g_last_error = saved;
    return 0;
  }
  return plan_workspace(B, T, d, f, chunk, true, true, true, true).total;
}

ittt_status ittt_stream_status(ittt_stream_t stream) {
  g_last_error.clear();
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "pending CUDA error");
  DeviceState* ds = nullptr;
  ittt_status s = device_state(&ds);
  if (s != ITTT_OK) return s;
  unsigned int word = 0;
  e = cudaMemcpy(&word, ds->status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  if (word != 0) {
    const unsigned int zero = 0;
    cudaMemcpy(ds->status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (word & ittt::kStatusTimeout)
      return fail(ITTT_ERR_TIMEOUT, "a kernel's bounded wait ran out (status 0x%x)", word);
    return fail(ITTT_ERR_CUDA, "device status 0x%x", word);
  }
  return ITTT_OK;
}

const char* ittt_last_error(void) { return g_last_error.c_str(); }

int32_t ittt_version(void) { return 100; }

int32_t ittt_launch_count(int64_t B, int64_t T, int64_t d, int64_t f, int64_t chunk) {
  const std::string saved = g_last_error;
  if (check_sizes(B, T, d, f, chunk) != ITTT_OK) {
    g_last_error = saved;
    return 0;
  }
  // conv, target, gate/up, snapshot 0, update (when a chunk updates), apply
  return (T / chunk > 1) ? 6 : 5;
}

}  // extern "C"
