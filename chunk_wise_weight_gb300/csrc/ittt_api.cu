// ittt_api.cu -- the C-ABI of libittt.so (declared in include/ittt.h).
//
// Validates every descriptor before anything is enqueued, plans the call
// (documents, snapshot slots, scratch), takes the scratch it needs
// (stream-ordered, from a library-private memory pool, or from a caller
// workspace), encodes the TMA tensor maps and launches the kernels in
// data-flow order on the caller's stream:
//   [packed documents: table staging] ; conv3 (Xc) ; target GEMM (eta*Vhat) ;
//   gate/up GEMM (Z) ; [snapshot 0, when W_0 is not one shared bf16 matrix or
//   the caller wants the snapshots] ; update walk (snapshots W_1..W_{n-1}) ;
//   apply GEMM (O).
// The GEMMs run on CTA pairs where two can be resident (and the update walk
// when every updated chunk is a multiple of 64 tokens), else on single CTAs.
// With ITTT_FLAG_FUSED_CONV the target GEMM computes the conv itself; in the
// dual form (forced by ITTT_FLAG_DUAL, or chosen by the planner for short
// sequences, T < 2.5 d f / (d + f), where it measured faster) scores Z Z^T and
// the dual apply replace walk and apply; with ITTT_FLAG_L2_NORM the walk runs
// one launch per chunk.  (Run beside the
// gate/up GEMM on a second stream, the conv slowed that GEMM by more than its
// own 0.2 ms at the 32k-token workload, so it runs in line.)  No host
// synchronisation happens inside a forward call; the packed-document staging
// waits only for a staging buffer's previous copy.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "ittt.h"
#include "kernels.h"
#include "sm103.cuh"

namespace {

constexpr int kMaxDevices = 64;

thread_local std::string g_last_error;

// Scratch bytes one call may allocate (0: no cap); ittt_set_scratch_limit.
std::atomic<size_t> g_scratch_limit{0};

// An NVTX range for the lifetime of the object: the host side of each phase
// shows up by name on a profiler's timeline (no cost without a tool).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// One NVTX range per phase of a forward call (opened at the phase's start
// event, closed at its end); ranges still open when the call returns early
// are closed then.
struct PhaseRanges {
  int open = 0;
  void mark(int slot) {
    static const char* const kNames[ITTT_NUM_PHASES] = {
        "ittt conv", "ittt target", "ittt gate/up", "ittt snapshot 0", "ittt update",
        "ittt apply"};
    if (slot % 2 == 0) {
      nvtxRangePushA(kNames[slot / 2]);
      ++open;
    } else if (open > 0) {
      nvtxRangePop();
      --open;
    }
  }
  ~PhaseRanges() {
    for (; open > 0; --open) nvtxRangePop();
  }
};

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

// Pinned, device-mapped host buffers that packed-document tables are staged
// from.  A small kernel on the caller's stream copies a table into device
// scratch: unlike a host-to-device memcpy it never queues behind the
// caller's bulk uploads on the copy engines.  A buffer is rewritten only
// after the kernel that last read it has finished, so several calls can be
// in flight on the device.
constexpr int kStagingSlots = 4;
struct StagingSlot {
  void* host = nullptr;
  int* dev = nullptr;  // device address of `host`
  size_t bytes = 0;
  cudaEvent_t done = nullptr;
  bool pending = false;
};

__global__ void __launch_bounds__(256)
    stage_table_kernel(const int* __restrict__ src, int* __restrict__ dst, int count) {
  ittt::griddep_wait();  // programmatic launch: the previous grid is done
  ittt::griddep_launch_dependents();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < count; i += gridDim.x * blockDim.x)
    dst[i] = src[i];
}

// The bounded waits' failure path, on purpose: one CTA of two warps waits
// on an mbarrier that nothing arrives on.  Warp 0 gives up after limit_ns,
// records kStatusTimeout and raises the CTA's abort flag; warp 1, allowed
// four times as long, unwinds as soon as it sees the flag (as the roles of
// a pipeline do), so the kernel ends after about limit_ns.
__global__ void __launch_bounds__(64, 1) wait_check_kernel(uint64_t limit_ns,
                                                           unsigned int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ittt::mbar_init(&bar, 1);
    abort_flag = 0;
    ittt::fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  const bool got = ittt::mbar_wait(&bar, 0u, &abort_flag, warp == 0 ? limit_ns : 4 * limit_ns);
  if (!got && warp == 0 && (threadIdx.x & 31) == 0)
    ittt::raise_abort(&abort_flag, status, ittt::kStatusTimeout);
}

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  unsigned int* status = nullptr;
  cudaMemPool_t pool = nullptr;
  StagingSlot staging[kStagingSlots];
  int next_slot = 0;
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

// Copies `count` ints of host data to device `dst` in stream order: into a
// pinned staging buffer on the host, then by stage_table_kernel.
ittt_status stage_table(DeviceState* ds, int* dst, const int* src, size_t count,
                        cudaStream_t stream) {
  const size_t bytes = count * sizeof(int);
  std::lock_guard<std::mutex> lock(g_mutex);
  StagingSlot& sl = ds->staging[ds->next_slot];
  ds->next_slot = (ds->next_slot + 1) % kStagingSlots;
  cudaError_t e = cudaSuccess;
  if (sl.pending) {
    e = cudaEventSynchronize(sl.done);
    if (e != cudaSuccess) return cuda_fail(e, "waiting for a staging buffer");
    sl.pending = false;
  }
  if (sl.done == nullptr) {
    e = cudaEventCreateWithFlags(&sl.done, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
  }
  if (sl.bytes < bytes) {
    if (sl.host) cudaFreeHost(sl.host);
    sl.host = nullptr;
    sl.dev = nullptr;
    sl.bytes = 0;
    const size_t want = std::max(bytes, size_t(64) << 10);
    e = cudaHostAlloc(&sl.host, want, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) return cuda_fail(e, "cudaHostAlloc (staging)");
    void* dp = nullptr;
    e = cudaHostGetDevicePointer(&dp, sl.host, 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaHostGetDevicePointer (staging)");
    sl.dev = static_cast<int*>(dp);
    sl.bytes = want;
  }
  memcpy(sl.host, src, bytes);
  const int blocks = int(std::min<size_t>((count + 255) / 256, 64));
  e = ittt::launch_pdl(stage_table_kernel, dim3(blocks), dim3(256), 0, stream,
                       static_cast<const int*>(sl.dev), dst, int(count));
  if (e != cudaSuccess) return cuda_fail(e, "document table staging");
  e = cudaEventRecord(sl.done, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord (staging)");
  sl.pending = true;
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
  if (d % 8 != 0 || f % 8 != 0)
    return fail(ITTT_ERR_UNSUPPORTED, "d_model=%lld and d_ff=%lld must be multiples of 8",
                (long long)d, (long long)f);
  if (B * T >= (int64_t(1) << 31) || d * f >= (int64_t(1) << 40))
    return fail(ITTT_ERR_UNSUPPORTED, "sizes exceed 32-bit tile coordinates");
  return ITTT_OK;
}

// --------------------------------------------------------------- planning
struct Layout {
  size_t z = 0, vhat = 0, xc = 0, snap = 0, scores = 0, w0b = 0, table = 0, state = 0,
         partial = 0, walk_part = 0, walk_arrive = 0, total = 0;
  // fp32 inputs: the bf16 split operands of the gate/up and target GEMMs
  size_t h3 = 0, wg3 = 0, wu3 = 0, wt3 = 0;
  size_t tickets = 0;  // the pair GEMMs' unit counters (zeroed by the call)
  bool has_tickets = false;
  size_t apply_part = 0;  // fp32 partials of the apply's split last round
  bool has_apply_part = false;
};

size_t round_up(size_t x) { return (x + 255) & ~size_t(255); }

// Everything a call needs to know before it touches the device: documents,
// snapshot slots, the packed-document table and the scratch layout.
struct Plan {
  int64_t B = 0, T = 0, d = 0, f = 0, C = 0, M = 0;
  bool fused = false, dual = false, packed = false, l2norm = false;
  bool update_only = false;  // fold every chunk into state_out, no apply
  bool reuse = false;        // Z and eta*Vhat come in through z_buf / vhat_buf
  bool fp32_in = false;      // H, X0, W_gate, W_up, W_target are fp32 (hi/lo split)
  int64_t ndocs = 0;   // documents: B, or the packed count
  int64_t nslots = 0;  // snapshot slots = chunks over all documents
  int64_t n = 0;       // chunks per sequence (regular)
  bool final_update = false;
  bool ragged_walk = false;  // an updated chunk is not a multiple of 64 tokens
  int n_udocs = 0;     // documents that run at least one update
  int64_t ntiles = 0;   // 128-row tiles over all chunks (the apply's row units)
  int64_t ntiles2 = 0;  // 256-row tiles over all chunks (row units on CTA pairs)
  // L2 normalisation: launches of the walk, and how many documents are
  // still updating at each (documents sorted by update count).
  std::vector<int> active;
  // Packed: starts[ndocs+1] | chunk_base[ndocs+1] | chunk_doc[nslots] |
  // tile_base[nslots+1] | tile_base2[nslots+1] | upd_docs[n_udocs], staged
  // into the scratch at L.table.
  std::vector<int> table;
  Layout L;
};

// w0_bf16: W_down0 is one bf16 matrix (the dual form then needs no bf16
// copy of it; pass false when unknown, which plans the larger scratch).
ittt_status make_plan(int64_t B, int64_t T, int64_t d, int64_t f, int64_t chunk,
                      const ittt_opts& o, bool w0_bf16, Plan* P) {
  ittt_status s = check_sizes(B, T, d, f, chunk);
  if (s != ITTT_OK) return s;
  if (o.pad_mode != ITTT_PAD_CHUNK && o.pad_mode != ITTT_PAD_SEQUENCE)
    return fail(ITTT_ERR_INVALID_ARG, "pad_mode %d", int(o.pad_mode));
  if (o.flags & ~int32_t(ITTT_FLAG_FUSED_CONV | ITTT_FLAG_DUAL | ITTT_FLAG_L2_NORM |
                          ITTT_FLAG_SINGLE_CTA | ITTT_FLAG_UPDATE_ONLY | ITTT_FLAG_REUSE_ZV |
                          ITTT_FLAG_PRIMAL | ITTT_FLAG_FP32_INPUTS))
    return fail(ITTT_ERR_INVALID_ARG, "unknown flags 0x%x", unsigned(o.flags));
  if ((o.flags & ITTT_FLAG_DUAL) && (o.flags & ITTT_FLAG_PRIMAL))
    return fail(ITTT_ERR_INVALID_ARG, "ITTT_FLAG_DUAL and ITTT_FLAG_PRIMAL exclude each other");
  P->B = B;
  P->T = T;
  P->d = d;
  P->f = f;
  P->C = chunk;
  P->M = B * T;
  P->fused = (o.flags & ITTT_FLAG_FUSED_CONV) != 0;
  P->dual = (o.flags & ITTT_FLAG_DUAL) != 0;
  P->packed = o.cu_seqlens != nullptr;
  P->l2norm = (o.flags & ITTT_FLAG_L2_NORM) != 0;
  P->fp32_in = (o.flags & ITTT_FLAG_FP32_INPUTS) != 0;
  if (P->fp32_in && P->fused)
    return fail(ITTT_ERR_UNSUPPORTED,
                "fp32 inputs run with the split convolution (no ITTT_FLAG_FUSED_CONV)");
  // Form choice by measured cost: the dual form for short sequences, where
  // the walk's per-chunk d x f snapshots cost more than the dual form's
  // T^2 terms.  The two forms' FLOPs are equal at T = 2 d f / (d + f); the
  // walk's snapshot traffic moves the measured crossover on GB300 to
  // 1.25-1.3 times that length.
  if (!P->dual && !(o.flags & ITTT_FLAG_PRIMAL) && !P->fused && !P->packed && !P->l2norm &&
      o.state_out == nullptr && o.snap_buf == nullptr && !(o.flags & ITTT_FLAG_UPDATE_ONLY) &&
      chunk % 64 == 0 && T % chunk == 0 && T / chunk >= 2 &&
      double(T) * double(d + f) < 2.5 * double(d) * double(f))
    P->dual = true;
  if (P->l2norm && P->dual)
    return fail(ITTT_ERR_UNSUPPORTED,
                "the normalised update has no dual form (the update is not additive)");
  P->update_only = (o.flags & ITTT_FLAG_UPDATE_ONLY) != 0;
  P->reuse = (o.flags & ITTT_FLAG_REUSE_ZV) != 0;
  if (P->update_only) {
    if (o.state_out == nullptr)
      return fail(ITTT_ERR_INVALID_ARG, "ITTT_FLAG_UPDATE_ONLY needs state_out");
    if (o.snap_buf != nullptr)
      return fail(ITTT_ERR_INVALID_ARG, "ITTT_FLAG_UPDATE_ONLY forms no snapshots: no snap_buf");
    if (P->dual || P->l2norm)
      return fail(ITTT_ERR_UNSUPPORTED,
                  "ITTT_FLAG_UPDATE_ONLY needs the additive primal update (no dual, no L2 norm)");
  }
  if (P->reuse && (o.z_buf == nullptr || o.vhat_buf == nullptr))
    return fail(ITTT_ERR_INVALID_ARG, "ITTT_FLAG_REUSE_ZV needs z_buf and vhat_buf");
  P->final_update = o.state_out != nullptr;
  if (P->dual && (o.state_out || o.snap_buf))
    return fail(ITTT_ERR_UNSUPPORTED,
                "the dual form forms no fast-weight state: no state_out or snap_buf");
  if (!P->packed && o.num_docs != 0)
    return fail(ITTT_ERR_INVALID_ARG, "num_docs is set but cu_seqlens is NULL");
  if (P->packed) {
    if (P->fused || P->dual)
      return fail(ITTT_ERR_UNSUPPORTED,
                  "packed documents run with the split convolution and the primal form only");
    if (B != 1)
      return fail(ITTT_ERR_INVALID_ARG, "packed documents need B = 1 (got %lld)", (long long)B);
    const int64_t nd = o.num_docs;
    const int64_t* cu = o.cu_seqlens;
    if (nd < 1) return fail(ITTT_ERR_INVALID_ARG, "num_docs %lld must be >= 1", (long long)nd);
    if (nd >= (int64_t(1) << 30))
      return fail(ITTT_ERR_UNSUPPORTED, "num_docs %lld is too large", (long long)nd);
    if (cu[0] != 0) return fail(ITTT_ERR_INVALID_ARG, "cu_seqlens[0] must be 0");
    if (cu[nd] != T)
      return fail(ITTT_ERR_INVALID_ARG, "cu_seqlens[num_docs] = %lld, expected T = %lld",
                  (long long)cu[nd], (long long)T);
    int64_t slots = 0;
    for (int64_t k = 0; k < nd; ++k) {
      if (cu[k + 1] <= cu[k])
        return fail(ITTT_ERR_INVALID_ARG,
                    "cu_seqlens must increase strictly (document %lld is empty or negative)",
                    (long long)k);
      slots += (cu[k + 1] - cu[k] + chunk - 1) / chunk;
    }
    P->ndocs = nd;
    P->nslots = slots;
    // Documents that update, most updates first (the update kernel walks
    // them in this order, so the longest walks start first).
    std::vector<std::pair<int64_t, int>> upd;
    for (int64_t k = 0; k < nd; ++k) {
      const int64_t nk = (cu[k + 1] - cu[k] + chunk - 1) / chunk;
      const int64_t nu = P->final_update ? nk : nk - 1;
      if (nu > 0) upd.push_back({-nu, int(k)});
    }
    std::stable_sort(upd.begin(), upd.end(),
                     [](const std::pair<int64_t, int>& a, const std::pair<int64_t, int>& b) {
                       return a.first < b.first;
                     });
    P->n_udocs = int(upd.size());
    if (P->l2norm && !upd.empty()) {
      P->active.assign(size_t(-upd[0].first), 0);
      for (const auto& u : upd)
        for (int64_t i = 0; i < -u.first; ++i) ++P->active[size_t(i)];
    }
    std::vector<int>& t = P->table;
    t.resize(size_t(2 * (nd + 1) + 3 * slots + 2 + P->n_udocs));
    int* starts = t.data();
    int* base = starts + (nd + 1);
    int* cdoc = base + (nd + 1);
    int* tbase = cdoc + slots;
    int* tbase2 = tbase + slots + 1;
    int* ud = tbase2 + slots + 1;
    int64_t g = 0, tiles = 0, tiles2 = 0;
    for (int64_t k = 0; k <= nd; ++k) {
      starts[k] = int(cu[k]);
      base[k] = int(g);
      if (k < nd) {
        const int64_t L = cu[k + 1] - cu[k];
        const int64_t nk = (L + chunk - 1) / chunk;
        for (int64_t j = 0; j < nk; ++j) {
          const int64_t len = std::min<int64_t>(chunk, L - j * chunk);
          tbase[g] = int(tiles);
          tbase2[g] = int(tiles2);
          tiles += (len + 127) / 128;
          tiles2 += (len + 255) / 256;
          cdoc[g++] = int(k);
        }
      }
    }
    tbase[slots] = int(tiles);
    tbase2[slots] = int(tiles2);
    P->ntiles = tiles;
    P->ntiles2 = tiles2;
    for (int q = 0; q < P->n_udocs; ++q) ud[q] = upd[size_t(q)].second;
    P->ragged_walk = chunk % 64 != 0;
    if (P->update_only) {
      // One contraction over each document's tokens.
      P->n_udocs = int(nd);
      P->ragged_walk = false;
      for (int64_t k = 0; k < nd; ++k)
        if ((cu[k + 1] - cu[k]) % 64 != 0) P->ragged_walk = true;
    } else if (P->final_update)
      for (int64_t k = 0; k < nd; ++k) {
        const int64_t L = cu[k + 1] - cu[k];
        if ((L - ((L + chunk - 1) / chunk - 1) * chunk) % 64 != 0) P->ragged_walk = true;
      }
  } else {
    P->ndocs = B;
    P->n = (T + chunk - 1) / chunk;  // the last chunk may be partial
    P->nslots = B * P->n;
    P->n_udocs = (P->final_update || P->n > 1) ? int(B) : 0;
    if (P->l2norm && P->n_udocs > 0)
      P->active.assign(size_t(P->final_update ? P->n : P->n - 1), int(B));
    const int64_t last = T - (P->n - 1) * chunk;
    P->ragged_walk = chunk % 64 != 0 || (P->final_update && last % 64 != 0);
    if (P->update_only) P->ragged_walk = T % 64 != 0;  // one contraction over T tokens
    P->ntiles = B * ((P->n - 1) * ((chunk + 127) / 128) + (last + 127) / 128);
    P->ntiles2 = B * ((P->n - 1) * ((chunk + 255) / 256) + (last + 255) / 256);
  }
  // The fused convolution forms its A tile from 4-row groups inside one
  // chunk; the dual form's scores are blocked by 64-token chunks.
  if (P->fused && (chunk % 64 != 0 || T % 64 != 0))
    return fail(ITTT_ERR_UNSUPPORTED, "the fused convolution needs chunk and T multiples of 64");
  if (P->dual && (chunk % 64 != 0 || T % chunk != 0))
    return fail(ITTT_ERR_UNSUPPORTED,
                "the dual form needs chunk a multiple of 64 that divides T");
  const int64_t apply_units = P->ntiles * ((d + 255) / 256);
  if (P->nslots * d >= (int64_t(1) << 31) || apply_units >= (int64_t(1) << 31))
    return fail(ITTT_ERR_UNSUPPORTED, "too many chunks for 32-bit tile coordinates");

  // Scratch.  The dual form needs the scores and, unless W_0 is one bf16
  // matrix already, a bf16 copy of each sequence's W_0 instead of the
  // snapshots.
  Layout& L = P->L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += round_up(bytes);
    return at;
  };
  // The unit counter of the apply on CTA pairs (it takes its units
  // dynamically): every call that runs the primal apply.
  L.has_tickets = !P->update_only && !P->dual;
  if (L.has_tickets) L.tickets = take(ittt::kNumTickets * sizeof(unsigned int));
  // Partials for splitting the apply's partial last round, where it can have
  // one: at least two full rounds of its 256 x 256 units on the GPU's pairs.
  const int64_t apply_pair_units = P->ntiles2 * ((d + 255) / 256);
  L.has_apply_part = L.has_tickets && apply_pair_units >= 2 * ittt::kMaxApplyTailPieces;
  if (L.has_apply_part) L.apply_part = take(ittt::kApplyPartBytes);
  if (o.z_buf == nullptr) L.z = take(size_t(P->M) * f * 2);
  if (o.vhat_buf == nullptr) L.vhat = take(size_t(P->M) * d * 2);
  if (!P->fused && !P->reuse) L.xc = take(size_t(P->M) * d * 2 * (P->fp32_in ? 3 : 1));
  if (P->fp32_in && !P->reuse) {
    L.h3 = take(size_t(P->M) * 3 * d * 2);
    L.wg3 = take(size_t(f) * 3 * d * 2);
    L.wu3 = take(size_t(f) * 3 * d * 2);
    L.wt3 = take(size_t(d) * 3 * d * 2);
  }
  if (!P->dual && !P->update_only && o.snap_buf == nullptr)
    L.snap = take(size_t(P->nslots) * d * f * 2);
  if (P->dual) {
    L.scores = take(size_t(B) * T * T * 2);
    if (o.state_in || !w0_bf16) L.w0b = take(size_t(o.state_in ? B : 1) * d * f * 2);
  }
  if (P->packed) L.table = take(P->table.size() * sizeof(int));
  if (P->l2norm && P->n_udocs > 0) {
    L.state = take(size_t(P->ndocs) * ((d + 127) / 128) * ((f + 31) / 32) * 128 * 32 * 4);
    // row partial sums per 256-column block of the state, in two 128-column parts
    L.partial = take(size_t(2) * P->ndocs * 2 * ((f + 255) / 256) * d * 4);
    if (!P->packed) {  // the walk with the state in TMEM (used when the pairs fit)
      L.walk_part = take(ittt::norm_walk_part_bytes(int(f), ittt::kNormWalkMaxPairs));
      L.walk_arrive = take(ittt::norm_walk_arrive_bytes(ittt::kNormWalkMaxPairs));
    }
  }
  L.total = off;
  return ITTT_OK;
}

// ------------------------------------------------------------- tensor maps
// 3-D map {inner, mid, outer} of a dense bf16 (or fp32) tensor, 128-byte
// swizzle.
ittt_status make_map_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t mid,
                        uint64_t outer, uint32_t box_inner, uint32_t box_mid, const char* what,
                        bool fp32 = false) {
  const uint64_t es = fp32 ? 4 : 2;
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {inner * es, inner * mid * es};
  cuuint32_t box[3] = {box_inner, box_mid, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(ITTT_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, int(r));
  return ITTT_OK;
}

ittt_status make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                     uint32_t box_inner, uint32_t box_outer, const char* what,
                     CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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
  if (H == nullptr || H->ndim != 3)
    return fail(ITTT_ERR_INVALID_ARG, "H: expected a [B,T,d] descriptor");
  const int64_t B = H->shape[0], T = H->shape[1], d = H->shape[2];
  if (W_gate == nullptr || W_gate->ndim != 2)
    return fail(ITTT_ERR_INVALID_ARG, "W_gate: expected a [f,d] descriptor");
  const int64_t f = W_gate->shape[0];
  if (!std::isfinite(eta)) return fail(ITTT_ERR_INVALID_ARG, "eta is not finite");
  // fp32 inputs follow from H's dtype; the flag alone (bf16 H) is an error.
  const bool fp32_in = H->dtype == ITTT_FP32;
  if ((o.flags & ITTT_FLAG_FP32_INPUTS) && !fp32_in)
    return fail(ITTT_ERR_INVALID_ARG, "ITTT_FLAG_FP32_INPUTS is set but H is not fp32");
  if (fp32_in) o.flags |= ITTT_FLAG_FP32_INPUTS;
  const bool w0_bf16 = W_down0 != nullptr && W_down0->dtype == ITTT_BF16;
  Plan P;
  ittt_status s = make_plan(B, T, d, f, chunk, o, w0_bf16, &P);
  if (s != ITTT_OK) return s;
  const bool fused = P.fused, dual = P.dual;
  const bool single = (o.flags & ITTT_FLAG_SINGLE_CTA) != 0;
  const bool update_only = P.update_only, reuse = P.reuse;
  const int64_t S = P.ndocs;  // per-document state count

  const int64_t sh_btd[3] = {B, T, d}, sh_fd[2] = {f, d}, sh_df[2] = {d, f}, sh_dd[2] = {d, d},
                sh_d3[2] = {d, 3}, sh_sdf[3] = {S, d, f}, sh_btf[3] = {B, T, f},
                sh_snap[4] = {B, P.nslots / B, d, f};
  if ((s = check_tensor(H, "H", 3, sh_btd, !fp32_in, fp32_in))) return s;
  if ((s = check_tensor(X0, "X0", 3, sh_btd, !fp32_in, fp32_in))) return s;
  if ((s = check_tensor(W_gate, "W_gate", 2, sh_fd, !fp32_in, fp32_in))) return s;
  if ((s = check_tensor(W_up, "W_up", 2, sh_fd, !fp32_in, fp32_in))) return s;
  // Folding chunks only, with neither state_in nor W_down0, starts from zero.
  const bool zero_start = update_only && o.state_in == nullptr && W_down0 == nullptr;
  if (o.state_in) {
    if ((s = check_tensor(o.state_in, "state_in", 3, sh_sdf, false, true))) return s;
  } else if (!zero_start && (s = check_tensor(W_down0, "W_down0", 2, sh_df, true, true))) {
    return s;
  }
  if ((s = check_tensor(W_target, "W_target", 2, sh_dd, !fp32_in, fp32_in))) return s;
  if ((s = check_tensor(conv_w, "conv_w", 2, sh_d3, false, true))) return s;
  // Nothing is applied when folding chunks only: out is ignored.
  if (update_only) out = nullptr;
  if (!update_only && (s = check_tensor(out, "out", 3, sh_btd, true, true))) return s;
  if (o.state_out && (s = check_tensor(o.state_out, "state_out", 3, sh_sdf, false, true))) return s;
  if (o.z_buf && (s = check_tensor(o.z_buf, "z_buf", 3, sh_btf, true, false))) return s;
  if (o.vhat_buf && (s = check_tensor(o.vhat_buf, "vhat_buf", 3, sh_btd, true, false))) return s;
  if (o.snap_buf && (s = check_tensor(o.snap_buf, "snap_buf", 4, sh_snap, true, false))) return s;
  const int64_t sh_bt[2] = {B, T};
  if (o.eta_tok && (s = check_tensor(o.eta_tok, "eta_tok", 2, sh_bt, false, true))) return s;

  const ittt_tensor* inputs[] = {H,        X0,     W_gate,   W_up, o.state_in ? o.state_in : W_down0,
                                 W_target, conv_w, o.eta_tok};
  const ittt_tensor* writes[] = {out, o.state_out, o.z_buf, o.vhat_buf, o.snap_buf};
  // state_out may be state_in itself: every kernel reads a block of the
  // initial state before that block's final state is written (the walk's
  // unit preloads the block it later stores; the snapshot-0 copy runs first;
  // the normalised walk writes state_out after its last launch).
  const bool in_place = o.state_in && o.state_out && o.state_in->data == o.state_out->data &&
                        tensor_bytes(o.state_in) == tensor_bytes(o.state_out);
  for (const ittt_tensor* w : writes) {
    for (const ittt_tensor* in : inputs) {
      if (in_place && w == o.state_out && in == o.state_in) continue;
      if (overlaps(w, in)) return fail(ITTT_ERR_INVALID_ARG, "an output overlaps an input");
    }
  }
  // Reused Z and eta*Vhat are read by the walk and the apply: no written
  // buffer may overlap them (the check above covers out, state_out and
  // snap_buf against each other and against z_buf / vhat_buf).
  for (int a = 0; a < 5; ++a)
    for (int b = a + 1; b < 5; ++b)
      if (overlaps(writes[a], writes[b]))
        return fail(ITTT_ERR_INVALID_ARG, "two output buffers overlap");

  const Layout& L = P.L;
  const size_t cap = g_scratch_limit.load();
  if (o.workspace == nullptr && cap != 0 && L.total > cap)
    return fail(ITTT_ERR_OOM, "the call needs %zu bytes of scratch, over the limit of %zu",
                L.total, cap);

  DeviceState* ds = nullptr;
  if ((s = device_state(&ds))) return s;

  const bool w0_is_bf16 = !o.state_in && w0_bf16;
  ScratchGuard guard;
  uint8_t* ws = nullptr;
  if (o.workspace) {
    if (o.workspace_bytes < L.total)
      return fail(ITTT_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu needed",
                  o.workspace_bytes, L.total);
    if (reinterpret_cast<uintptr_t>(o.workspace) % 256 != 0)
      return fail(ITTT_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    ws = static_cast<uint8_t*>(o.workspace);
  } else if (L.total > 0) {
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

  // Documents (the packed tables are staged at the start of the conv phase).
  ittt::DocMap docs;
  memset(&docs, 0, sizeof(docs));
  docs.ndocs = int(P.ndocs);
  docs.nchunks = int(P.nslots);
  docs.ntiles = int(P.ntiles);
  docs.T = int(T);
  docs.n = int(P.n);
  docs.C = int(chunk);
  docs.ntiles2 = int(P.ntiles2);
  docs.mtc = int((chunk + 127) / 128);
  docs.mtc2 = int((chunk + 255) / 256);
  if (!P.packed) {
    docs.tiles_per_seq = int(P.ntiles / B);
    docs.tiles_per_seq2 = int(P.ntiles2 / B);
  }
  const int* upd_docs = nullptr;
  int* tab = reinterpret_cast<int*>(ws + L.table);
  if (P.packed) {
    docs.starts = tab;
    docs.chunk_base = tab + (P.ndocs + 1);
    docs.chunk_doc = tab + 2 * (P.ndocs + 1);
    docs.tile_base = docs.chunk_doc + P.nslots;
    docs.tile_base2 = docs.tile_base + P.nslots + 1;
    upd_docs = docs.tile_base2 + P.nslots + 1;
  }

  // Tensor maps.
  const uint64_t M = uint64_t(P.M);
  CUtensorMap tm_h, tm_wg, tm_wu, tm_a, tm_wt, tm_wt128, tm_vmn, tm_zmn, tm_zk, tm_snap;
  // Output maps for the epilogues' TMA stores (Z's is tm_zk).
  CUtensorMap tm_vs, tm_ss, tm_os;
  memset(&tm_ss, 0, sizeof(tm_ss));
  memset(&tm_os, 0, sizeof(tm_os));
  // fp32 inputs: the GEMMs read bf16 hi/lo split copies over K = 3d,
  // A as [A_hi|A_hi|A_lo] (H; Xc) and B as [B_hi|B_lo|B_hi] (W_gate, W_up;
  // W_target), so each product is hi*hi + hi*lo + lo*hi.
  const int64_t k_gu = fp32_in ? 3 * d : d, k_t = fp32_in ? 3 * d : d;
  auto* h3 = reinterpret_cast<__nv_bfloat16*>(ws + L.h3);
  auto* wg3 = reinterpret_cast<__nv_bfloat16*>(ws + L.wg3);
  auto* wu3 = reinterpret_cast<__nv_bfloat16*>(ws + L.wu3);
  auto* wt3 = reinterpret_cast<__nv_bfloat16*>(ws + L.wt3);
  if (!reuse) {  // the producers of Z and eta*Vhat
    const void* a_h = fp32_in ? static_cast<const void*>(h3) : H->data;
    const void* a_wg = fp32_in ? static_cast<const void*>(wg3) : W_gate->data;
    const void* a_wu = fp32_in ? static_cast<const void*>(wu3) : W_up->data;
    const void* a_wt = fp32_in ? static_cast<const void*>(wt3) : W_target->data;
    if ((s = make_map(&tm_h, a_h, k_gu, M, 64, 128, "H"))) return s;
    if ((s = make_map(&tm_wg, a_wg, k_gu, f, 64, 128, "W_gate"))) return s;
    if ((s = make_map(&tm_wu, a_wu, k_gu, f, 64, 128, "W_up"))) return s;
    if (fused) {
      if ((s = make_map(&tm_a, X0->data, d, M, 64, 130, "X0"))) return s;
    } else if ((s = make_map(&tm_a, xc, k_t, M, 64, 128, "Xc"))) {
      return s;
    }
    if ((s = make_map(&tm_wt, a_wt, k_t, d, 64, 256, "W_target"))) return s;
    if ((s = make_map(&tm_wt128, a_wt, k_t, d, 64, 128, "W_target (pair)"))) return s;
    if ((s = make_map(&tm_vs, vhat, d, M, 64, 128, "Vhat (store)"))) return s;
  }
  if (out && out->dtype == ITTT_BF16 &&
      (s = make_map(&tm_os, out->data, d, M, 64, 64, "O (store)")))
    return s;
  if ((s = make_map(&tm_vmn, vhat, d, M, 64, 64, "Vhat"))) return s;
  if ((s = make_map(&tm_zmn, z, f, M, 64, 64, "Z (update)"))) return s;
  if ((s = make_map(&tm_zk, z, f, M, 64, 128, "Z (apply)"))) return s;
  CUtensorMap tm_zs, tm_w0b, tm_w0b_pair, tm_sc, tm_snap_pair, tm_w0d, tm_w0d_pair;
  // The apply reads a shared bf16 W_0 itself for first chunks, so slot 0 of
  // each document need not be copied (unless the caller asked for the
  // snapshots).
  const bool w0_direct = !dual && w0_is_bf16 && o.snap_buf == nullptr;
  auto* scores = reinterpret_cast<__nv_bfloat16*>(ws + L.scores);
  const void* w0b = w0_is_bf16 ? W_down0->data : static_cast<const void*>(ws + L.w0b);
  if (dual) {
    if ((s = make_map(&tm_zs, z, f, M, 64, 256, "Z (scores)"))) return s;
    if ((s = make_map(&tm_w0b, w0b, f, uint64_t((o.state_in ? B : 1) * d), 64, 256, "bf16 W_0")))
      return s;
    if ((s = make_map(&tm_w0b_pair, w0b, f, uint64_t((o.state_in ? B : 1) * d), 64, 128,
                      "bf16 W_0 (pair)")))
      return s;
    if ((s = make_map(&tm_sc, scores, uint64_t(T), M, 64, 128, "scores"))) return s;
  } else if (update_only) {
    // No snapshot is formed; the walk's store map only needs valid memory.
    if ((s = make_map_3d(&tm_ss, o.state_out->data, f, d, 1, 64, 128, "snapshots (unused)")))
      return s;
  } else {
    if ((s = make_map(&tm_snap, snap, f, uint64_t(P.nslots * d), 64, 256, "snapshots"))) return s;
    if ((s = make_map(&tm_snap_pair, snap, f, uint64_t(P.nslots * d), 64, 128,
                      "snapshots (pair)")))
      return s;
    if (w0_direct) {
      if ((s = make_map(&tm_w0d, W_down0->data, f, uint64_t(d), 64, 256, "W_0 (apply)"))) return s;
      if ((s = make_map(&tm_w0d_pair, W_down0->data, f, uint64_t(d), 64, 128, "W_0 (apply, pair)")))
        return s;
    }
    if ((s = make_map_3d(&tm_ss, snap, f, d, uint64_t(P.nslots), 64, 128, "snapshots (store)")))
      return s;
  }

  auto* tickets = L.has_tickets ? reinterpret_cast<unsigned int*>(ws + L.tickets) : nullptr;
  ittt::LaunchEnv env{stream, ds->num_sms, ds->status, tickets};
  if (L.has_apply_part) env.apply_part = reinterpret_cast<float*>(ws + L.apply_part);
  // w0 == nullptr: the walk starts from zero (folding chunks only).
  const void* w0 = o.state_in ? o.state_in->data : (zero_start ? nullptr : W_down0->data);
  const bool w0_fp32 = o.state_in ? true : (!zero_start && W_down0->dtype == ITTT_FP32);
  const int64_t w0_bstride = o.state_in ? d * f : 0;

  cudaEvent_t const* ev = reinterpret_cast<cudaEvent_t const*>(o.events);
  NvtxRange call_range("ittt_forward");
  PhaseRanges ranges;
  auto rec = [&](int slot, cudaStream_t st) -> cudaError_t {
    ranges.mark(slot);
    return (ev && ev[slot]) ? cudaEventRecord(ev[slot], st) : cudaSuccess;
  };
  const float* cw = static_cast<const float*>(conv_w->data);

  cudaError_t e = cudaSuccess;
  const char* what = nullptr;
#define ITTT_STEP(call, name) \
  if (what == nullptr && (e = (call)) != cudaSuccess) what = name
  if (tickets != nullptr)
    ITTT_STEP(cudaMemsetAsync(tickets, 0, ittt::kNumTickets * sizeof(unsigned int), stream),
              "unit counter reset");
  ITTT_STEP(rec(2 * ITTT_PHASE_CONV, stream), "event record");
  if (what == nullptr && P.packed &&
      (s = stage_table(ds, tab, P.table.data(), P.table.size(), stream)) != ITTT_OK)
    return s;
  if (!fused && !reuse && fp32_in) {
    // hi/lo split copies of the fp32 operands, then the fp32 convolution,
    // split the same way into [Xc_hi | Xc_hi | Xc_lo].
    ITTT_STEP(ittt::launch_split_bf16(env, static_cast<const float*>(H->data), int64_t(M), int(d),
                                      h3, 3, 4u),
              "split launch (H)");
    ITTT_STEP(ittt::launch_split_bf16(env, static_cast<const float*>(W_gate->data), f, int(d),
                                      wg3, 3, 2u),
              "split launch (W_gate)");
    ITTT_STEP(ittt::launch_split_bf16(env, static_cast<const float*>(W_up->data), f, int(d), wu3,
                                      3, 2u),
              "split launch (W_up)");
    ITTT_STEP(ittt::launch_split_bf16(env, static_cast<const float*>(W_target->data), d, int(d),
                                      wt3, 3, 2u),
              "split launch (W_target)");
    ITTT_STEP(ittt::launch_conv_fp32(env, static_cast<const float*>(X0->data), cw, xc, int64_t(M),
                                     docs, int(d), int(o.pad_mode)),
              "conv launch (fp32)");
  } else if (!fused && !reuse) {
    CUtensorMap tm_x0;
    if (what == nullptr &&
        (s = make_map(&tm_x0, X0->data, d, M, ittt::kConvMapBoxCols, ittt::kConvMapBoxRows,
                      "X0 (conv)", CU_TENSOR_MAP_SWIZZLE_NONE)))
      return s;
    ITTT_STEP(ittt::launch_conv(env, tm_x0, cw, xc, int64_t(M), docs, int(d), int(o.pad_mode)),
              "conv launch");
  }
  ITTT_STEP(rec(2 * ITTT_PHASE_CONV + 1, stream), "event record");
  ITTT_STEP(rec(2 * ITTT_PHASE_TARGET, stream), "event record");
  if (what == nullptr && !reuse) {
    const float* et = o.eta_tok ? static_cast<const float*>(o.eta_tok->data) : nullptr;
    // CTA pairs where two can be resident (split convolution), else one CTA.
    e = fused || single ? cudaErrorNotSupported
                        : ittt::launch_target_pair(env, tm_a, tm_wt128, tm_vs, et, vhat, eta,
                                                   int(M), int(d), int(k_t));
    if (e == cudaErrorNotSupported) {
      cudaGetLastError();
      e = ittt::launch_target(env, tm_a, tm_wt, tm_vs, cw, et, vhat, eta, int(M), int(T), int(d),
                              int(chunk), int(o.pad_mode), fused, int(k_t));
    }
    if (e != cudaSuccess) what = "target launch";
  }
  ITTT_STEP(rec(2 * ITTT_PHASE_TARGET + 1, stream), "event record");
  ITTT_STEP(rec(2 * ITTT_PHASE_GATEUP, stream), "event record");
  if (what == nullptr && !reuse) {
    e = single ? cudaErrorNotSupported
               : ittt::launch_gateup_pair(env, tm_h, tm_wg, tm_wu, tm_zk, int(M), int(f),
                                          int(k_gu));
    if (e == cudaErrorNotSupported) {
      cudaGetLastError();
      e = ittt::launch_gateup(env, tm_h, tm_wg, tm_wu, tm_zk, int(M), int(f), int(k_gu));
    }
    if (e != cudaSuccess) what = "gate/up launch";
  }
  ITTT_STEP(rec(2 * ITTT_PHASE_GATEUP + 1, stream), "event record");
  ITTT_STEP(rec(2 * ITTT_PHASE_SNAPSHOT0, stream), "event record");
  if (!dual) {
    // Slot 0 of each document, unless the apply reads a shared bf16 W_0
    // itself or nothing is applied.
    if (!w0_direct && !update_only)
      ITTT_STEP(ittt::launch_snapshot0(env, w0, w0_fp32, w0_bstride, snap, docs, int(d), int(f)),
                "snapshot launch");
  } else if (!w0_is_bf16) {
    // The dual form's bf16 copy of each W_0.
    ittt::DocMap w0docs;
    memset(&w0docs, 0, sizeof(w0docs));
    w0docs.ndocs = int(o.state_in ? B : 1);
    w0docs.nchunks = w0docs.ndocs;
    w0docs.T = 1;
    w0docs.n = 1;
    w0docs.C = 1;
    ITTT_STEP(ittt::launch_snapshot0(env, w0, w0_fp32, w0_bstride,
                                     static_cast<__nv_bfloat16*>(const_cast<void*>(w0b)), w0docs,
                                     int(d), int(f)),
              "W_0 copy launch");
  }
  ITTT_STEP(rec(2 * ITTT_PHASE_SNAPSHOT0 + 1, stream), "event record");
  if (!dual) {
    ittt::UpdateArgs ua;
    ua.docs = docs;
    if (update_only) {
      // The update is additive, so folding every chunk is one contraction
      // over each document's tokens: walk with a single chunk of T tokens
      // (no boundary, so no snapshot) and keep the final state.
      ua.docs.C = int(T);
      ua.docs.n = 1;
      ua.docs.nchunks = int(P.ndocs);
      ua.docs.chunk_base = nullptr;
      ua.docs.chunk_doc = nullptr;
    }
    ua.upd_docs = upd_docs;
    ua.n_udocs = P.n_udocs;
    ua.final_update = P.final_update;
    ua.d = int(d);
    ua.f = int(f);
    ua.w0 = w0;
    ua.w0_fp32 = w0_fp32;
    ua.w0_bstride = w0_bstride;
    ua.state_out = o.state_out ? static_cast<float*>(o.state_out->data) : nullptr;
    ua.allow_pairs = !P.ragged_walk && !single;
    ITTT_STEP(rec(2 * ITTT_PHASE_UPDATE, stream), "event record");
    if (P.l2norm) {
      ittt::NormUpdateArgs na;
      na.docs = docs;
      na.upd_docs = upd_docs;
      na.n_udocs = P.n_udocs;
      na.n_steps = int(P.active.size());
      na.active = P.active.data();
      na.d = int(d);
      na.f = int(f);
      na.w0 = w0;
      na.w0_fp32 = w0_fp32;
      na.w0_bstride = w0_bstride;
      na.state = reinterpret_cast<float*>(ws + L.state);
      na.partial = reinterpret_cast<float*>(ws + L.partial);
      na.walk_part = P.packed ? nullptr : reinterpret_cast<float*>(ws + L.walk_part);
      na.walk_arrive = P.packed ? nullptr : reinterpret_cast<unsigned int*>(ws + L.walk_arrive);
      na.walk_pairs = ittt::kNormWalkMaxPairs;
      na.snap = snap;
      na.state_out = ua.state_out;
      na.allow_pairs = !P.ragged_walk && !single && d % 256 == 0;
      ITTT_STEP(ittt::launch_norm_update(env, tm_vmn, tm_zmn, tm_ss, na),
                "normalised update launch");
    } else {
      ITTT_STEP(ittt::launch_update(env, tm_vmn, tm_zmn, tm_ss, ua), "update launch");
    }
    ITTT_STEP(rec(2 * ITTT_PHASE_UPDATE + 1, stream), "event record");
    ITTT_STEP(rec(2 * ITTT_PHASE_APPLY, stream), "event record");
    if (what == nullptr && !update_only) {
      // CTA pairs where two can be resident, else one CTA per tile.
      e = single ? cudaErrorNotSupported
                 : ittt::launch_apply_pair(env, tm_zk, tm_snap_pair,
                                           w0_direct ? &tm_w0d_pair : nullptr, tm_os, out->data,
                                           out->dtype == ITTT_FP32, docs, int(d), int(f));
      if (e == cudaErrorNotSupported) {
        cudaGetLastError();
        e = ittt::launch_apply(env, tm_zk, tm_snap, w0_direct ? &tm_w0d : nullptr, tm_os,
                               out->data, out->dtype == ITTT_FP32, docs, int(d), int(f));
      }
      if (e != cudaSuccess) what = "apply launch";
    }
    ITTT_STEP(rec(2 * ITTT_PHASE_APPLY + 1, stream), "event record");
  } else {
    ITTT_STEP(rec(2 * ITTT_PHASE_UPDATE, stream), "event record");
    ITTT_STEP(ittt::launch_scores(env, tm_zk, tm_zs, scores, int(B), int(T), int(f), int(chunk),
                                  !single),
              "scores launch");
    ITTT_STEP(rec(2 * ITTT_PHASE_UPDATE + 1, stream), "event record");
    ITTT_STEP(rec(2 * ITTT_PHASE_APPLY, stream), "event record");
    ITTT_STEP(ittt::launch_dual_apply(env, tm_zk, tm_w0b, tm_w0b_pair, tm_sc, tm_vmn,
                                      o.state_in != nullptr, out->data, out->dtype == ITTT_FP32,
                                      int(B), int(T), int(d), int(f), int(chunk), !single),
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

ittt_status ittt_state_prefix(const ittt_tensor* W_start, const ittt_tensor* deltas,
                              int32_t count, ittt_tensor* state, ittt_stream_t stream) {
  g_last_error.clear();
  if (deltas == nullptr || deltas->ndim != 4)
    return fail(ITTT_ERR_INVALID_ARG, "deltas: expected an [R,S,d,f] descriptor");
  const int64_t R = deltas->shape[0], S = deltas->shape[1], d = deltas->shape[2],
                f = deltas->shape[3];
  if (R <= 0 || S <= 0 || d <= 0 || f <= 0)
    return fail(ITTT_ERR_INVALID_ARG, "deltas: sizes must be positive");
  if (d % 8 != 0 || f % 8 != 0)
    return fail(ITTT_ERR_UNSUPPORTED, "d_model=%lld and d_ff=%lld must be multiples of 8",
                (long long)d, (long long)f);
  if (count < 0 || count > R)
    return fail(ITTT_ERR_INVALID_ARG, "count %d outside 0..%lld", int(count), (long long)R);
  const int64_t sh_r[4] = {R, S, d, f}, sh_s[3] = {S, d, f}, sh_df[2] = {d, f};
  ittt_status s;
  if ((s = check_tensor(deltas, "deltas", 4, sh_r, false, true))) return s;
  if ((s = check_tensor(state, "state", 3, sh_s, false, true))) return s;
  int kind = 0;
  if (W_start != nullptr) {
    if (W_start->ndim == 2) {
      if ((s = check_tensor(W_start, "W_start", 2, sh_df, true, true))) return s;
      kind = W_start->dtype == ITTT_BF16 ? 1 : 2;
    } else {
      if ((s = check_tensor(W_start, "W_start", 3, sh_s, false, true))) return s;
      kind = 3;
    }
  }
  if (overlaps(state, deltas) || overlaps(state, W_start))
    return fail(ITTT_ERR_INVALID_ARG, "state overlaps an input");
  DeviceState* ds = nullptr;
  if ((s = device_state(&ds))) return s;
  const ittt::LaunchEnv env{reinterpret_cast<cudaStream_t>(stream), ds->num_sms, ds->status};
  const cudaError_t e = ittt::launch_state_prefix(
      env, W_start ? W_start->data : nullptr, kind, static_cast<const float*>(deltas->data),
      int(count), static_cast<float*>(state->data), S, d * f);
  if (e != cudaSuccess) return cuda_fail(e, "state prefix launch");
  return ITTT_OK;
}

void ittt_set_scratch_limit(size_t bytes) { g_scratch_limit.store(bytes); }

ittt_status ittt_check_wait_timeout(uint64_t limit_ns, ittt_stream_t stream) {
  g_last_error.clear();
  if (limit_ns < 1000 || limit_ns > 1000000000ull)
    return fail(ITTT_ERR_INVALID_ARG, "limit_ns %llu outside [1e3, 1e9]",
                static_cast<unsigned long long>(limit_ns));
  DeviceState* ds = nullptr;
  ittt_status s = device_state(&ds);
  if (s != ITTT_OK) return s;
  wait_check_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, ds->status);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "wait check launch");
  return ITTT_OK;
}

int32_t ittt_plan_form(int64_t B, int64_t T, int64_t d, int64_t f, int64_t chunk,
                       const ittt_opts* opts) {
  const std::string saved = g_last_error;
  ittt_opts o;
  memset(&o, 0, sizeof(o));
  if (opts) o = *opts;
  Plan P;
  if (make_plan(B, T, d, f, chunk, o, false, &P) != ITTT_OK) {
    g_last_error = saved;
    return -1;
  }
  return P.dual ? ITTT_FORM_DUAL : ITTT_FORM_PRIMAL;
}

size_t ittt_workspace_bytes(int64_t B, int64_t T, int64_t d, int64_t f, int64_t chunk) {
  return ittt_workspace_bytes_ex(B, T, d, f, chunk, nullptr);
}

size_t ittt_workspace_bytes_ex(int64_t B, int64_t T, int64_t d, int64_t f, int64_t chunk,
                               const ittt_opts* opts) {
  const std::string saved = g_last_error;
  ittt_opts o;
  memset(&o, 0, sizeof(o));
  if (opts) o = *opts;
  Plan P;
  if (make_plan(B, T, d, f, chunk, o, false, &P) != ITTT_OK) {
    g_last_error = saved;
    return 0;
  }
  return P.L.total;
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
  // conv, target, gate/up, update (when a chunk updates), apply -- or, in
  // the dual form (which needs two chunks or more), conv, target, gate/up,
  // scores, dual apply; with a shared bf16 W_down0 and no snapshot buffer
  // neither form copies W_0
  return ((T + chunk - 1) / chunk > 1) ? 5 : 4;
}

}  // extern "C"
