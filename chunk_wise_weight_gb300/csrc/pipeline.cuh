// pipeline.cuh -- persistent, warp-specialised tcgen05 GEMM pipeline shared by
// the layer's four tensor-core kernels.
//
// One CTA per SM (the shared-memory footprint forces it).  Roles:
//   warp 0, lane 0 : TMA producer -- fills a ring of kStages operand stages
//   warp 1         : allocates 512 TMEM columns; lane 0 issues tcgen05.mma
//   warps 2..5     : epilogue -- drains the fp32 accumulator from TMEM
//
// Tiles are 128 (M) x 256 (N), K staged 64 at a time with the 128-byte
// swizzle.  TMEM holds two 128 x 256 fp32 accumulators, so the epilogue of
// one accumulation overlaps the MMAs of the next.
//
// A kernel plugs in a schedule class `S` that describes its work:
//   S(const Params&)                     construct from the kernel parameters
//   int  num_units()                     persistent work units
//   void begin_unit(int unit, int local) local = how many units this CTA did
//   int  num_segments()                  accumulations in the current unit
//   int  seg_acc(int s)                  accumulator (0/1) segment s uses
//   int  seg_kblocks(int s)              64-wide K blocks of segment s
//   bool seg_fresh(int s)                segment starts from a zero accumulator
//   void load(int s, int kb, void* a, void* b, uint64_t* bar)   (TMA issue)
//   void epilogue(int s, int row, uint32_t tmem_row_base)       (per thread)
//   static uint64_t a_desc(uint32_t a_smem, int k16)
//   static uint64_t b_desc(uint32_t b_smem, int k16)
//   static constexpr uint32_t kIdesc
//   static constexpr bool kPreload
// Segments let one accumulator keep accumulating across several epilogue
// reads (the fast-weight state walks the chunks of a sequence).
//
// With kPreload the epilogue also writes each unit's starting accumulator
// values into TMEM before the unit's first MMA:
//   int  unit_accs()                               accumulators the unit uses
//   void preload(int acc, int row, uint32_t tmem_row_base)   (per thread)
// Each MMA use of an accumulator then waits for exactly one epilogue arrival:
// the release after the previous segment's read inside a unit, or the
// preload at a unit's start (the last read of a unit is not released; the
// next unit's preload stands for it).
#pragma once

#include "sm103.cuh"

namespace ittt {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kUmmaK = 16;
constexpr int kStages = 4;
constexpr uint32_t kATileBytes = kBM * kBK * 2;  // 16 KiB
constexpr uint32_t kBTileBytes = kBN * kBK * 2;  // 32 KiB
constexpr uint32_t kStageBytes = kATileBytes + kBTileBytes;
constexpr uint32_t kTmemCols = 512;
constexpr int kNumThreads = 192;
constexpr int kEpilogueThreads = 128;

struct __align__(8) PipeSync {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t kPipeSmemBytes = 1024 + size_t(kStages) * kStageBytes + sizeof(PipeSync);

template <class S>
__device__ __forceinline__ void run_pipeline(const typename S::Params& p, unsigned int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PipeSync* sync = reinterpret_cast<PipeSync*>(smem + size_t(kStages) * kStageBytes);
  volatile int* abort_flag = &sync->abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sync->full[s], 1);
      mbar_init(&sync->empty[s], 1);
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
            uint8_t* sa = smem + size_t(stage) * kStageBytes;
            mbar_arrive_expect_tx(&sync->full[stage], kStageBytes);
            sched.load(s, kb, sa, sa + kATileBytes, &sync->full[stage]);
            ++issued;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // Let every load still in flight land before the CTA can exit.
      const int zero = 0;
      const uint32_t tail = issued < uint32_t(kStages) ? issued : uint32_t(kStages);
      for (uint32_t q = issued - tail; q < issued; ++q) {
        const int st = int(q % kStages);
        const uint32_t par = (q / kStages) & 1u;
        if (!mbar_wait(&sync->full[st], par, &zero)) atomicOr(status, kStatusTimeout);
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
            const uint32_t a_base = smem_u32(smem + size_t(stage) * kStageBytes);
            const uint32_t b_base = a_base + kATileBytes;
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k) {
              mma_bf16(d_tmem, S::a_desc(a_base, k), S::b_desc(b_base, k), S::kIdesc,
                       (fresh && kb == 0 && k == 0) ? 0u : 1u);
            }
            mma_commit(&sync->empty[stage]);
            if (++stage == kStages) {
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
  } else {
    // ------------------------------------------------------------- epilogue
    S sched(p);
    const int quad = warp & 3;  // TMEM lanes this warp may touch: 32*quad..+31
    const int row = quad * 32 + lane;
    uint32_t acc_use[2] = {0u, 0u};
    const int nunits = sched.num_units();
    int local = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++local) {
      sched.begin_unit(u, local);
      const int nseg = sched.num_segments();
      if constexpr (S::kPreload) {
        for (int h = 0; h < sched.unit_accs(); ++h) {
          sched.preload(h, row, tmem + (uint32_t(quad * 32) << 16) + uint32_t(h * kBN));
          tmem_wait_st();
          tc_fence_before_sync();
          mbar_arrive(&sync->acc_empty[h]);
        }
      }
      for (int s = 0; s < nseg; ++s) {
        const int h = sched.seg_acc(s);
        // The TMEM loads below are warp-collective: the whole warp proceeds
        // or the whole warp unwinds.
        const bool got = __all_sync(0xffffffffu, mbar_wait(&sync->acc_full[h], acc_use[h] & 1u,
                                                           abort_flag));
        if (!got) {
          raise_abort(abort_flag, status, kStatusTimeout);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t trow = tmem + (uint32_t(quad * 32) << 16) + uint32_t(h * kBN);
        sched.epilogue(s, row, trow);
        bool release = true;
        if constexpr (S::kPreload) release = s < nseg - sched.unit_accs();
        if (release) {
          tc_fence_before_sync();
          mbar_arrive(&sync->acc_empty[h]);
        }
        ++acc_use[h];
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
