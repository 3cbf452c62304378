// pipeline.cuh -- persistent, warp-specialised tcgen05 GEMM pipeline shared by
// the layer's tensor-core kernels.
//
// One CTA per SM (the shared-memory footprint forces it).  Roles:
//   warp 0, lane 0 : TMA producer -- fills a ring of operand stages
//   warp 1         : allocates 512 TMEM columns; lane 0 issues tcgen05.mma
//   warps 2..5     : epilogue -- drains the fp32 accumulator from TMEM
//   warps 6..      : optional A-tile builders (S::kBuilderWarps > 0): they
//                    compute the A tile in shared memory from raw data the
//                    producer loaded into the stage, instead of TMA loading it
//
// Tiles are 128 (M) x 256 (N), K staged 64 at a time with the 128-byte
// swizzle.  TMEM holds two 128 x 256 fp32 accumulators, so the epilogue of
// one accumulation overlaps the MMAs of the next.
//
// A kernel plugs in a schedule class `S` (deriving from SchedDefaults) that
// describes its work:
//   S(const Params&)                     construct from the kernel parameters
//   int  num_units()                     persistent work units
//   void begin_unit(int unit, int local) local = how many units this CTA did
//   int  num_segments()                  accumulations in the current unit
//   int  seg_acc(int s)                  accumulator (0/1) segment s uses
//   int  seg_kblocks(int s)              64-wide K blocks of segment s
//   bool seg_fresh(int s)                segment starts from a zero accumulator
//   void load(int s, int kb, uint8_t* stage, uint64_t* bar)     (TMA issue)
//   void epilogue(int s, int row, uint32_t tmem_row_base)       (per thread)
//   static uint64_t a_desc(uint32_t a_smem, int k16)
//   static uint64_t b_desc(uint32_t b_smem, int k16)
//   static constexpr uint32_t kIdesc
// A stage holds the A tile at offset 0, the B tile at kATileBytes and
// S::kExtraStageBytes of kernel-specific data at kStageBytes.
// Segments let one accumulator keep accumulating across several epilogue
// reads (the fast-weight state walks the chunks of a sequence).
//
// With kPreload the epilogue also writes each unit's starting accumulator
// values into TMEM before the unit's first MMA:
//   int  unit_accs()                               accumulators the unit uses
//   void preload(int acc, int row, uint32_t tmem_row_base)   (per thread)
// Each MMA use of an accumulator then waits for exactly one epilogue arrival:
// the release after the previous segment's read inside a unit, or the
// preload for a unit's first use (the last read of a unit is not released;
// the next unit's preload stands for it).  The epilogue preloads accumulator
// h for the CTA's next unit as soon as it has read h's last value in the
// current one, so the MMA rolls from one unit into the next without waiting.
//
// With kBuilderWarps > 0 the producer's copies complete on a `loaded`
// barrier (tma_bytes(s, kb) per stage); the builder warps wait for it, call
//   void build_a(int s, int kb, uint8_t* stage, int tid)  (tid < 32*warps)
// then each makes its writes visible to the tensor core and arrives on
// `full` (32 * kBuilderWarps arrivals per stage).
#pragma once

#include "sm103.cuh"

namespace ittt {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kUmmaK = 16;
constexpr int kMaxStages = 4;
constexpr uint32_t kATileBytes = kBM * kBK * 2;  // 16 KiB
constexpr uint32_t kBTileBytes = kBN * kBK * 2;  // 32 KiB
constexpr uint32_t kStageBytes = kATileBytes + kBTileBytes;
constexpr uint32_t kTmemCols = 512;
constexpr int kBaseThreads = 192;
constexpr int kEpilogueThreads = 128;

// Epilogue output staging for TMA stores: two 128-row x 128-byte tiles.
constexpr uint32_t kStagingTileBytes = kBM * 128;
constexpr uint32_t kStagingBytes = 2 * kStagingTileBytes;

// Helper the epilogue threads use to write a 128 x 64 bf16 output tile
// through shared memory: every thread fills its row (8 x 16 bytes, 128-byte
// swizzle), then one thread issues the TMA store.  Two staging buffers
// alternate; a buffer is refilled only after the store that read it two
// tiles ago has finished reading shared memory.  With two epilogue groups
// (kEpilogueGroups) each group has its own pair of buffers and its own
// named barrier.
struct EpiStager {
  uint8_t* buf;
  int tid;  // 0..127 = tile row
  uint32_t issued;
  int group = 0;  // epilogue group (named barrier 1 + group)

  // Next buffer to fill (every thread of the group must call this).
  __device__ __forceinline__ uint8_t* acquire() {
    if (tid == 0 && issued >= 2) bulk_wait_group_read<1>();
    epilogue_group_bar(group);
    return buf + (issued & 1u) * kStagingTileBytes;
  }
  // Writes 16-byte chunk c (0..7) of this thread's row.
  __device__ __forceinline__ void put(uint8_t* b, int c, uint4 v) const {
    *reinterpret_cast<uint4*>(b + tid * 128 + ((c ^ (tid & 7)) << 4)) = v;
  }
  // Publishes the buffer; `store(buf)` runs on one thread and issues the TMA.
  template <class F>
  __device__ __forceinline__ void commit(uint8_t* b, F&& store) {
    fence_proxy_async_smem();
    epilogue_group_bar(group);
    if (tid == 0) {
      store(b);
      bulk_commit_group();
    }
    ++issued;
  }
  __device__ __forceinline__ void finish() const {
    if (tid == 0) bulk_wait_group_all();
  }
};

struct SchedDefaults {
  static constexpr int kNumStages = 4;
  static constexpr uint32_t kExtraStageBytes = 0;
  static constexpr int kBuilderWarps = 0;
  static constexpr bool kPreload = false;
  // Epilogue writes bf16 tiles through EpiStager (TMA stores); then
  //   void epilogue(int s, int row, uint32_t tmem_row_base, EpiStager& st)
  static constexpr bool kStagedStores = false;
  // With kStagedPreload (needs kStagedStores) the preload may store through
  // the staging tiles too:
  //   void preload(int acc, int row, uint32_t tmem_row_base, EpiStager& st)
  static constexpr bool kStagedPreload = false;
  // With kMixedOperands the MMA asks the schedule for each K block's
  // instruction and shared-memory descriptors (operand major-ness may change
  // inside one accumulation):
  //   uint32_t idesc(int s, int kb); uint64_t a_desc(int s, int kb, uint32_t
  //   base, int k16); uint64_t b_desc(int s, int kb, uint32_t base, int k16)
  static constexpr bool kMixedOperands = false;
  // With kRaggedK a K block may hold fewer than 64 valid K indices (the end
  // of a chunk that is not a multiple of 64 tokens long).  The MMA thread
  // then zeroes the operand lines of the invalid K indices inside the last
  // 16-wide slice it issues and skips the slices after it:
  //   int  k_valid(int s, int kb)                       1..64
  //   void clear_k(uint8_t* stage, int from, int to)    (generic stores)
  static constexpr bool kRaggedK = false;
  // Groups of four epilogue warps (CTA-pair pipeline only): each group runs
  // the epilogue and preload on the same accumulator lanes, on its share of
  // the columns (EpiStager::group tells the schedule which).
  static constexpr int kEpilogueGroups = 1;
  // Transaction bytes the producer's copies deliver into a stage.
  __device__ uint32_t tma_bytes(int, int) const { return kStageBytes; }
  // With kBindsSync (CTA-pair pipeline only) the epilogue's schedule gets
  // the CTA's abort flag and the device status word before its first unit:
  //   void bind_sync(volatile int* abort_flag, unsigned int* status)
  // for epilogues that wait on other CTAs.
  static constexpr bool kBindsSync = false;
  // With kAccTeams (CTA-pair pipeline, two epilogue groups) epilogue group g
  // alone drains, preloads and releases accumulator g, all of its columns:
  // the two accumulators' epilogues then run side by side instead of in
  // turn on the same warps.
  static constexpr bool kAccTeams = false;
  // With kDynamicUnits (CTA-pair pipeline only; not with kPreload or
  // kAccTeams) the pairs take units in increasing order from a counter in
  // global memory, zero at launch, instead of each walking a fixed stride:
  //   unsigned int* unit_ticket()
  // Units then start in index order whatever the pairs' speeds, so the
  // units in flight stay within about one round of each other.
  static constexpr bool kDynamicUnits = false;
  // With kEarlyRelease (CTA-pair pipeline, kStagedStores) the epilogue gets
  // a callable to invoke once its last TMEM read has completed; it hands the
  // accumulator on (releases it, or preloads the next unit's initial state
  // into it and releases it), so the next MMAs can start while the epilogue
  // still converts and stores:
  //   template <class F> void epilogue(int s, int row, uint32_t tmem_row_base,
  //                                    EpiStager& st, F&& handoff)
  static constexpr bool kEarlyRelease = false;
  // With kPrefetchPreload (CTA-pair pipeline, kPreload, fixed stride) the
  // epilogue asks the next unit's schedule, as each unit starts, to pull
  // what its preload will read into L2:   void prefetch_preload(int row)
  static constexpr bool kPrefetchPreload = false;
};

template <class S>
struct PipeShape {
  static_assert(S::kNumStages >= 2 && S::kNumStages <= kMaxStages, "stage count");
  static_assert((kStageBytes + S::kExtraStageBytes) % 1024 == 0, "stages stay 1 KiB aligned");
  static_assert(S::kEpilogueGroups == 1, "one epilogue group on single CTAs");
  static constexpr uint32_t kStageStride = kStageBytes + S::kExtraStageBytes;
  static constexpr int kThreads = kBaseThreads + 32 * S::kBuilderWarps;
};

struct __align__(8) PipeSync {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t loaded[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int vote[4];  // epilogue warps' go/unwind votes (staged-store kernels)
};

template <class S>
__host__ __device__ constexpr size_t pipe_staging_bytes() {
  return S::kStagedStores ? kStagingBytes * S::kEpilogueGroups : 0;
}

template <class S>
__host__ __device__ constexpr size_t pipe_smem_bytes() {
  return 1024 + size_t(S::kNumStages) * PipeShape<S>::kStageStride + pipe_staging_bytes<S>() +
         sizeof(PipeSync);
}

template <class S>
__device__ __forceinline__ void run_pipeline(const typename S::Params& p, unsigned int* status) {
  constexpr int NS = S::kNumStages;
  constexpr uint32_t kStride = PipeShape<S>::kStageStride;
  constexpr bool kBuild = S::kBuilderWarps > 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + size_t(NS) * kStride;  // 1 KiB aligned
  PipeSync* sync = reinterpret_cast<PipeSync*>(staging + pipe_staging_bytes<S>());
  volatile int* abort_flag = &sync->abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sync->full[s], kBuild ? 32 * S::kBuilderWarps : 1);
      mbar_init(&sync->empty[s], 1);
      mbar_init(&sync->loaded[s], 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&sync->acc_full[h], 1);
      mbar_init(&sync->acc_empty[h], kEpilogueThreads);
    }
    mbar_init(&sync->drain, 1);
    sync->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sync->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sync->tmem_base;
  // Set-up done: only now touch memory the previous grid may still write or
  // read (launched with programmatic serialization, this grid's set-up
  // overlapped that grid's last CTAs).
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      S sched(p);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      const int nunits = sched.num_units();
      int local = 0;
      for (int u = blockIdx.x; u < nunits && !*abort_flag; u += gridDim.x, ++local) {
        sched.begin_unit(u, local);
        const int nseg = sched.num_segments();
        for (int s = 0; s < nseg && !*abort_flag; ++s) {
          const int nkb = sched.seg_kblocks(s);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&sync->empty[stage], phase ^ 1u, abort_flag)) {
              raise_abort(abort_flag, status, kStatusTimeout);
              break;
            }
            uint64_t* bar = kBuild ? &sync->loaded[stage] : &sync->full[stage];
            mbar_arrive_expect_tx(bar, sched.tma_bytes(s, kb));
            sched.load(s, kb, smem + size_t(stage) * kStride, bar);
            ++issued;
            if (++stage == NS) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // Let every load still in flight land before the CTA can exit.
      const int zero = 0;
      const uint32_t tail = issued < uint32_t(NS) ? issued : uint32_t(NS);
      for (uint32_t q = issued - tail; q < issued; ++q) {
        const int st = int(q % NS);
        const uint32_t par = (q / NS) & 1u;
        uint64_t* bar = kBuild ? &sync->loaded[st] : &sync->full[st];
        if (!mbar_wait(bar, par, &zero)) atomicOr(status, kStatusTimeout);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------------- MMA
      S sched(p);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_use[2] = {0u, 0u};
      const int nunits = sched.num_units();
      int local = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++local) {
        sched.begin_unit(u, local);
        const int nseg = sched.num_segments();
        for (int s = 0; s < nseg && ok; ++s) {
          const int h = sched.seg_acc(s);
          const uint32_t empty_parity = S::kPreload ? (acc_use[h] & 1u) : ((acc_use[h] & 1u) ^ 1u);
          if (!mbar_wait(&sync->acc_empty[h], empty_parity, abort_flag)) {
            raise_abort(abort_flag, status, kStatusTimeout);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem + uint32_t(h * kBN);
          const int nkb = sched.seg_kblocks(s);
          const bool fresh = sched.seg_fresh(s);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&sync->full[stage], phase, abort_flag)) {
              raise_abort(abort_flag, status, kStatusTimeout);
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t a_base = smem_u32(smem + size_t(stage) * kStride);
            const uint32_t b_base = a_base + kATileBytes;
            if constexpr (S::kRaggedK) {
              const int kv = sched.k_valid(s, kb);
              if (kv < kBK) {
                const int kv16 = (kv + kUmmaK - 1) / kUmmaK * kUmmaK;
                if (kv < kv16) {
                  sched.clear_k(smem + size_t(stage) * kStride, kv, kv16);
                  fence_proxy_async_smem();  // generic stores -> tensor core
                }
#pragma unroll
                for (int k = 0; k < kBK / kUmmaK; ++k) {
                  if (k * kUmmaK < kv)
                    mma_bf16(d_tmem, S::a_desc(a_base, k), S::b_desc(b_base, k), S::kIdesc,
                             (fresh && kb == 0 && k == 0) ? 0u : 1u);
                }
                mma_commit(&sync->empty[stage]);
                if (++stage == NS) {
                  stage = 0;
                  phase ^= 1u;
                }
                continue;
              }
            }
            if constexpr (S::kMixedOperands) {
              const uint32_t id = sched.idesc(s, kb);
#pragma unroll
              for (int k = 0; k < kBK / kUmmaK; ++k) {
                mma_bf16(d_tmem, sched.a_desc(s, kb, a_base, k), sched.b_desc(s, kb, b_base, k),
                         id, (fresh && kb == 0 && k == 0) ? 0u : 1u);
              }
            } else {
#pragma unroll
              for (int k = 0; k < kBK / kUmmaK; ++k) {
                mma_bf16(d_tmem, S::a_desc(a_base, k), S::b_desc(b_base, k), S::kIdesc,
                         (fresh && kb == 0 && k == 0) ? 0u : 1u);
              }
            }
            mma_commit(&sync->empty[stage]);
            if (++stage == NS) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(&sync->acc_full[h]);
          ++acc_use[h];
        }
      }
      // Every MMA issued so far completes before TMEM is released.
      mma_commit(&sync->drain);
      const int zero = 0;
      if (!mbar_wait(&sync->drain, 0u, &zero)) atomicOr(status, kStatusTimeout);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------- epilogue
    S sched(p);
    S next(p);  // lookahead for the preload of the CTA's next unit
    const int quad = warp & 3;  // TMEM lanes this warp may touch: 32*quad..+31
    const int row = quad * 32 + lane;
    EpiStager stager{staging, row, 0u};
    const uint32_t tlane = tmem + (uint32_t(quad * 32) << 16);
    uint32_t acc_use[2] = {0u, 0u};
    bool preloaded[2] = {false, false};
    const int nunits = sched.num_units();
    int local = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++local) {
      sched.begin_unit(u, local);
      const int nseg = sched.num_segments();
      if constexpr (S::kPreload) {
        for (int h = 0; h < sched.unit_accs(); ++h) {
          if (!preloaded[h]) {
            if constexpr (S::kStagedPreload) {
              sched.preload(h, row, tlane + uint32_t(h * kBN), stager);
            } else {
              sched.preload(h, row, tlane + uint32_t(h * kBN));
            }
            tmem_wait_st();
            tc_fence_before_sync();
            mbar_arrive(&sync->acc_empty[h]);
          }
        }
        preloaded[0] = preloaded[1] = false;
      }
      for (int s = 0; s < nseg; ++s) {
        const int h = sched.seg_acc(s);
        // The TMEM loads below are warp-collective: the whole warp proceeds
        // or the whole warp unwinds.  Staged stores also synchronise the four
        // epilogue warps with a named barrier, so there the four warps vote
        // and proceed or unwind together.
        bool got = __all_sync(0xffffffffu, mbar_wait(&sync->acc_full[h], acc_use[h] & 1u,
                                                     abort_flag));
        if constexpr (S::kStagedStores) {
          if (lane == 0) sync->vote[quad] = got ? 1 : 0;
          epilogue_bar();
          got = (sync->vote[0] & sync->vote[1] & sync->vote[2] & sync->vote[3]) != 0;
          epilogue_bar();
        }
        if (!got) {
          raise_abort(abort_flag, status, kStatusTimeout);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t trow = tlane + uint32_t(h * kBN);
        if constexpr (S::kStagedStores) {
          sched.epilogue(s, row, trow, stager);
        } else {
          sched.epilogue(s, row, trow);
        }
        bool release = true;
        if constexpr (S::kPreload) {
          release = s < nseg - sched.unit_accs();
          const int un = u + int(gridDim.x);
          if (!release && un < nunits) {
            next.begin_unit(un, local + 1);
            if (h < next.unit_accs()) {
              if constexpr (S::kStagedPreload) {
                next.preload(h, row, trow, stager);
              } else {
                next.preload(h, row, trow);
              }
              tmem_wait_st();
              tc_fence_before_sync();
              mbar_arrive(&sync->acc_empty[h]);
              preloaded[h] = true;
            }
          }
        }
        if (release) {
          tc_fence_before_sync();
          mbar_arrive(&sync->acc_empty[h]);
        }
        ++acc_use[h];
      }
    }
    // Shared memory must outlive the TMA stores that read it.
    if constexpr (S::kStagedStores) stager.finish();
  } else if constexpr (kBuild) {
    // ------------------------------------------------------- A-tile builders
    S sched(p);
    const int tid = int(threadIdx.x) - kBaseThreads;
    int stage = 0;
    uint32_t phase = 0;
    const int nunits = sched.num_units();
    int local = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++local) {
      sched.begin_unit(u, local);
      const int nseg = sched.num_segments();
      for (int s = 0; s < nseg && ok; ++s) {
        const int nkb = sched.seg_kblocks(s);
        for (int kb = 0; kb < nkb; ++kb) {
          const bool got =
              __all_sync(0xffffffffu, mbar_wait(&sync->loaded[stage], phase, abort_flag));
          if (!got) {
            raise_abort(abort_flag, status, kStatusTimeout);
            ok = false;
            break;
          }
          sched.build_a(s, kb, smem + size_t(stage) * kStride, tid);
          fence_proxy_async_smem();  // generic-proxy writes -> tensor core
          mbar_arrive(&sync->full[stage]);
          if (++stage == NS) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace ittt
