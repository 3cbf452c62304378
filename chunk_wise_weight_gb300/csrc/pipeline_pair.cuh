// pipeline_pair.cuh -- the persistent warp-specialised tcgen05 pipeline on
// CTA pairs (clusters of two CTAs on two SMs).
//
// A pair computes 256 x 256 output tiles with tcgen05.mma.cta_group::2:
// each CTA keeps half of the A tile (its 128 rows) and half of the B tile
// (128 of the 256 columns) in its own shared memory, and the accumulator
// rows of its half in its own TMEM.  A stage is 32 KB per CTA instead of
// the 48 KB a single CTA needs for a 128 x 256 tile, so six stages fit
// where four did: the operand ring covers half again as much TMA latency,
// and each SM reads a third less operand data per FLOP.
//
// Roles per CTA (as in pipeline.cuh):
//   warp 0, lane 0 : TMA producer for this CTA's halves.  Its copies count
//                    their bytes on the LEADER's (even CTA's) full barrier;
//                    the leader's producer posts the pair's expected bytes.
//   warp 1         : TMEM allocation for the pair; in the leader, lane 0
//                    issues the pair MMAs and commits them to the barriers
//                    of both CTAs (multicast).
//   warps 2..5     : epilogue on this CTA's accumulator rows (with two epilogue
//   (and 6..9)       groups, each group on its share of the columns); a release
//                    arrives on the leader's acc_empty barrier.
// Both CTAs walk the same units in the same order: a fixed stride of the
// unit index, or (kDynamicUnits) the units the leader's producer draws from
// a global counter and hands to every role of both CTAs through a small ring
// in shared memory (unit_full: the slot holds the next unit; unit_empty:
// every reader took it).  Every wait is bounded
// (kWaitLimitNs); a CTA that gives up records kStatusTimeout and unwinds,
// and its peer's waits then run out too.  Cluster barriers after set-up and
// before TMEM release keep each CTA's barriers and shared memory alive while
// the other can still reach them.
//
// A schedule S for this pipeline provides, beside SchedDefaults' members:
//   S(const Params&, uint32_t rank)       rank = this CTA's place in the pair
//   int  num_units(); void begin_unit(int u, int local)
//   int  num_segments(); int seg_acc(int s); int seg_kblocks(int s);
//   bool seg_fresh(int s)
//   void load(int s, int kb, uint8_t* stage, uint32_t full_bar)
//        (this CTA's two 16 KB halves: A at 0, B at kPairATileBytes)
//   static uint64_t a_desc(uint32_t a_smem, int k16), b_desc(...)
//   static constexpr uint32_t kIdesc        (M = 256)
//   epilogue / preload / unit_accs as in pipeline.cuh, on this CTA's rows.
#pragma once

#include <atomic>
#include <cstring>

#include "kernels.h"
#include "pipeline.cuh"

namespace ittt {

constexpr int kMaxPairStages = 8;
constexpr int kUnitRing = 8;  // units handed out ahead of the slowest reader
constexpr uint32_t kPairATileBytes = 128 * kBK * 2;  // 16 KiB: 128 rows of A
constexpr uint32_t kPairBTileBytes = 128 * kBK * 2;  // 16 KiB: 128 rows of B
constexpr uint32_t kPairStageBytes = kPairATileBytes + kPairBTileBytes;

struct PairDefaults : SchedDefaults {
  static constexpr int kNumStages = 6;
};

// Threads of a CTA: producer, MMA and one or two groups of epilogue warps.
template <class S>
__host__ __device__ constexpr int pair_threads() {
  static_assert(S::kEpilogueGroups == 1 || S::kEpilogueGroups == 2, "epilogue groups");
  return kBaseThreads + kEpilogueThreads * (S::kEpilogueGroups - 1);
}

struct __align__(8) PairSync {
  uint64_t full[kMaxPairStages];   // leader: both CTAs' operand bytes landed
  uint64_t empty[kMaxPairStages];  // both: the pair MMAs reading the stage are done
  uint64_t acc_full[2];            // both: the pair accumulation is complete
  uint64_t acc_empty[2];           // leader: both CTAs' epilogues released it
  uint64_t drain;                  // leader: every pair MMA is done
  uint32_t tmem_base;
  int abort_flag;
  int vote[8];                     // epilogue warps' go/unwind votes, four per group
  uint64_t unit_full[kUnitRing];   // both: the slot holds the next unit (kDynamicUnits)
  uint64_t unit_empty[kUnitRing];  // leader: every reader of both CTAs took the slot
  int unit_ring[kUnitRing];        // the unit, or -1 once the counter passed the last
};

// Readers of a unit slot: the leader's MMA thread, the peer's producer and
// every epilogue warp of both CTAs (the leader's producer writes it).
template <class S>
__host__ __device__ constexpr uint32_t unit_readers() {
  return 2u + 2u * 4u * uint32_t(S::kEpilogueGroups);
}

template <class S>
__host__ __device__ constexpr size_t pair_smem_bytes() {
  static_assert(S::kNumStages >= 2 && S::kNumStages <= kMaxPairStages, "stage count");
  return 1024 + size_t(S::kNumStages) * kPairStageBytes + pipe_staging_bytes<S>() +
         sizeof(PairSync);
}

template <class S>
__device__ __forceinline__ void run_pipeline_pair(const typename S::Params& p,
                                                  unsigned int* status) {
  constexpr int NS = S::kNumStages;
  constexpr uint16_t kBoth = 0x3;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + size_t(NS) * kPairStageBytes;  // 1 KiB aligned
  PairSync* sync = reinterpret_cast<PairSync*>(staging + pipe_staging_bytes<S>());
  volatile int* abort_flag = &sync->abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = int(blockIdx.x >> 1);
  const int npairs = int(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sync->full[s], 1);
      mbar_init(&sync->empty[s], 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&sync->acc_full[h], 1);
      mbar_init(&sync->acc_empty[h],
                2 * kEpilogueThreads * (S::kAccTeams ? 1 : S::kEpilogueGroups));
    }
    mbar_init(&sync->drain, 1);
    if constexpr (S::kDynamicUnits) {
      static_assert(!S::kPreload && !S::kAccTeams, "dynamic units need neither");
      for (int r = 0; r < kUnitRing; ++r) {
        mbar_init(&sync->unit_full[r], 1);
        mbar_init(&sync->unit_empty[r], unit_readers<S>());
      }
    }
    sync->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&sync->tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync();  // both CTAs' barriers exist before either reaches across
  tc_fence_after_sync();
  const uint32_t tmem = sync->tmem_base;
  // Set-up done: only now touch memory the previous grid may still write or
  // read (see pipeline.cuh).
  griddep_wait();
  griddep_launch_dependents();

  // The unit of this CTA's `local`-th step: a fixed stride, or
  // (kDynamicUnits) the ring's slot.  -1: no more units; -2: a wait ran out.
  // take_unit waits and reads; give_unit (after every reader of the calling
  // warp or thread has read) frees the slot.
  auto take_unit = [&](int local, int nunits) -> int {
    if constexpr (S::kDynamicUnits) {
      const int slot = local % kUnitRing;
      if (!mbar_wait_cluster(&sync->unit_full[slot], uint32_t(local / kUnitRing) & 1u,
                             abort_flag))
        return -2;
      return *reinterpret_cast<volatile int*>(&sync->unit_ring[slot]);
    } else {
      const int u = pair + local * npairs;
      return u < nunits ? u : -1;
    }
  };
  auto give_unit = [&](int local) {
    if constexpr (S::kDynamicUnits)
      mbar_arrive_cluster(mapa_shared(smem_u32(&sync->unit_empty[local % kUnitRing]), 0));
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      S sched(p, rank);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      const int nunits = sched.num_units();
      for (int local = 0; !*abort_flag; ++local) {
        int u = -1;
        bool drawn = false;
        if constexpr (S::kDynamicUnits) {
          if (leader) {
            // Draw the next unit and hand it to both CTAs.
            const int slot = local % kUnitRing;
            if (!mbar_wait_cluster(&sync->unit_empty[slot],
                                   (uint32_t(local / kUnitRing) & 1u) ^ 1u, abort_flag)) {
              raise_abort(abort_flag, status, kStatusTimeout);
              break;
            }
            u = int(atomicAdd(sched.unit_ticket(), 1u));
            if (u >= nunits) u = -1;
            sync->unit_ring[slot] = u;
            st_shared_cluster_s32(mapa_shared(smem_u32(&sync->unit_ring[slot]), 1), u);
            mbar_arrive_cluster(mapa_shared(smem_u32(&sync->unit_full[slot]), 0));
            mbar_arrive_cluster(mapa_shared(smem_u32(&sync->unit_full[slot]), 1));
            drawn = true;
          }
        }
        if (!drawn) {
          u = take_unit(local, nunits);
          if (u == -2) {
            raise_abort(abort_flag, status, kStatusTimeout);
            break;
          }
          give_unit(local);
        }
        if (u < 0) break;
        sched.begin_unit(u, local);
        const int nseg = sched.num_segments();
        for (int s = 0; s < nseg && !*abort_flag; ++s) {
          const int nkb = sched.seg_kblocks(s);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&sync->empty[stage], phase ^ 1u, abort_flag)) {
              raise_abort(abort_flag, status, kStatusTimeout);
              break;
            }
            if (leader) mbar_arrive_expect_tx(&sync->full[stage], 2 * kPairStageBytes);
            sched.load(s, kb, smem + size_t(stage) * kPairStageBytes,
                       mapa_shared(smem_u32(&sync->full[stage]), 0));
            ++issued;
            if (++stage == NS) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // The leader's full barriers count both CTAs' copies: let every copy
      // still in flight land before the pair can exit.
      if (leader) {
        const int zero = 0;
        const uint32_t tail = issued < uint32_t(NS) ? issued : uint32_t(NS);
        for (uint32_t q = issued - tail; q < issued; ++q) {
          if (!mbar_wait(&sync->full[q % NS], (q / NS) & 1u, &zero))
            atomicOr(status, kStatusTimeout);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ----------------------------------------------------------------- MMA
      S sched(p, rank);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_use[2] = {0u, 0u};
      const int nunits = sched.num_units();
      bool ok = true;
      for (int local = 0; ok; ++local) {
        const int u = take_unit(local, nunits);
        if (u == -2) {
          raise_abort(abort_flag, status, kStatusTimeout);
          break;
        }
        give_unit(local);
        if (u < 0) break;
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
            const uint32_t a_base = smem_u32(smem + size_t(stage) * kPairStageBytes);
            const uint32_t b_base = a_base + kPairATileBytes;
            if constexpr (S::kMixedOperands) {
              const uint32_t id = sched.idesc(s, kb);
#pragma unroll
              for (int k = 0; k < kBK / kUmmaK; ++k) {
                mma_bf16_pair(d_tmem, sched.a_desc(s, kb, a_base, k),
                              sched.b_desc(s, kb, b_base, k), id,
                              (fresh && kb == 0 && k == 0) ? 0u : 1u);
              }
            } else {
#pragma unroll
              for (int k = 0; k < kBK / kUmmaK; ++k) {
                mma_bf16_pair(d_tmem, S::a_desc(a_base, k), S::b_desc(b_base, k), S::kIdesc,
                              (fresh && kb == 0 && k == 0) ? 0u : 1u);
              }
            }
            mma_commit_pair(&sync->empty[stage], kBoth);
            if (++stage == NS) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit_pair(&sync->acc_full[h], kBoth);
          ++acc_use[h];
        }
      }
      // Every pair MMA issued so far completes before TMEM is released.
      mma_commit_pair(&sync->drain, 0x1);
      const int zero = 0;
      if (!mbar_wait(&sync->drain, 0u, &zero)) atomicOr(status, kStatusTimeout);
    }
  } else if (warp < 2 + 4 * S::kEpilogueGroups) {
    // ------------------------------------------------------------- epilogue
    S sched(p, rank);
    S next(p, rank);
    if constexpr (S::kBindsSync) sched.bind_sync(abort_flag, status);
    const int group = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    EpiStager stager{staging + size_t(group) * kStagingBytes, row, 0u, group};
    const uint32_t tlane = tmem + (uint32_t(quad * 32) << 16);
    const uint32_t acc_empty_leader[2] = {mapa_shared(smem_u32(&sync->acc_empty[0]), 0),
                                          mapa_shared(smem_u32(&sync->acc_empty[1]), 0)};
    uint32_t acc_use[2] = {0u, 0u};
    bool preloaded[2] = {false, false};
    // The warps that meet at epilogue barriers agree on whether a wait
    // succeeded, so that they unwind together.
    auto agree = [&](bool got) -> bool {
      if constexpr (S::kBindsSync && !S::kAccTeams) {
        // One vote over both groups: such an epilogue meets the other
        // group at CTA-wide barriers.
        static_assert(S::kEpilogueGroups == 2, "CTA-wide vote over two groups");
        volatile int* vote = sync->vote;
        if (lane == 0) vote[warp - 2] = got ? 1 : 0;
        epilogue_all_bar();
        got = (vote[0] & vote[1] & vote[2] & vote[3] & vote[4] & vote[5] & vote[6] & vote[7]) != 0;
        epilogue_all_bar();
      } else if constexpr (S::kStagedStores) {
        volatile int* vote = sync->vote + 4 * group;
        if (lane == 0) vote[quad] = got ? 1 : 0;
        epilogue_group_bar(group);
        got = (vote[0] & vote[1] & vote[2] & vote[3]) != 0;
        epilogue_group_bar(group);
      }
      return got;
    };
    const int nunits = sched.num_units();
    bool ok = true;
    for (int local = 0; ok; ++local) {
      int u;
      if constexpr (S::kDynamicUnits) {
        const int slot = local % kUnitRing;
        const bool got = agree(__all_sync(
            0xffffffffu, mbar_wait_cluster(&sync->unit_full[slot],
                                           uint32_t(local / kUnitRing) & 1u, abort_flag)));
        if (!got) {
          raise_abort(abort_flag, status, kStatusTimeout);
          ok = false;
          break;
        }
        u = *reinterpret_cast<volatile int*>(&sync->unit_ring[slot]);
        __syncwarp();
        if (lane == 0) give_unit(local);
      } else {
        u = take_unit(local, nunits);
      }
      if (u < 0) break;
      sched.begin_unit(u, local);
      const int nseg = sched.num_segments();
      if constexpr (S::kPrefetchPreload) {
        static_assert(S::kPreload && !S::kDynamicUnits, "prefetches the next stride unit");
        if (u + npairs < nunits) {
          next.begin_unit(u + npairs, local + 1);
          next.prefetch_preload(row);
        }
      }
      if constexpr (S::kPreload) {
        for (int h = 0; h < sched.unit_accs(); ++h) {
          if (!preloaded[h] && (!S::kAccTeams || h == group)) {
            if constexpr (S::kStagedPreload) {
              sched.preload(h, row, tlane + uint32_t(h * kBN), stager);
            } else {
              sched.preload(h, row, tlane + uint32_t(h * kBN));
            }
            tmem_wait_st();
            tc_fence_before_sync();
            mbar_arrive_cluster(acc_empty_leader[h]);
          }
        }
        preloaded[0] = preloaded[1] = false;
      }
      for (int s = 0; s < nseg; ++s) {
        const int h = sched.seg_acc(s);
        if constexpr (S::kAccTeams) {
          static_assert(S::kEpilogueGroups == 2, "one epilogue group per accumulator");
          if (h != group) continue;  // the other group's accumulator
        }
        const bool got = agree(__all_sync(
            0xffffffffu, mbar_wait(&sync->acc_full[h], acc_use[h] & 1u, abort_flag)));
        if (!got) {
          raise_abort(abort_flag, status, kStatusTimeout);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t trow = tlane + uint32_t(h * kBN);
        // The unit's last segments keep their accumulators for the next
        // unit's preload (kPreload); every other segment releases its own.
        // The hand-off runs once: called by a kEarlyRelease epilogue after
        // its last TMEM read, else here after the epilogue.
        bool release = true;
        if constexpr (S::kPreload) release = s < nseg - sched.unit_accs();
        bool handed = false;
        auto handoff = [&]() {
          if (handed) return;
          handed = true;
          if (release) {
            tc_fence_before_sync();
            mbar_arrive_cluster(acc_empty_leader[h]);
            return;
          }
          if constexpr (S::kPreload) {
            const int un = u + npairs;
            if (un < nunits) {
              next.begin_unit(un, local + 1);
              if (h < next.unit_accs()) {
                if constexpr (S::kStagedPreload) {
                  next.preload(h, row, trow, stager);
                } else {
                  next.preload(h, row, trow);
                }
                tmem_wait_st();
                tc_fence_before_sync();
                mbar_arrive_cluster(acc_empty_leader[h]);
                preloaded[h] = true;
              }
            }
          }
        };
        if constexpr (S::kStagedStores && S::kEarlyRelease) {
          sched.epilogue(s, row, trow, stager, handoff);
        } else if constexpr (S::kStagedStores) {
          sched.epilogue(s, row, trow, stager);
        } else {
          sched.epilogue(s, row, trow);
        }
        handoff();
        ++acc_use[h];
      }
    }
    if constexpr (S::kStagedStores) stager.finish();
  }

  __syncwarp();
  tc_fence_before_sync();
  cluster_sync();  // the leader's MMAs (reading both CTAs) are done
  tc_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
// attr: room for two attributes (the cluster shape and, with `pdl`,
// programmatic stream serialization as in launch_pdl).
inline cudaLaunchConfig_t pair_launch_config(int pairs, size_t smem, const LaunchEnv& env,
                                             cudaLaunchAttribute* attr,
                                             int threads = kBaseThreads, bool pdl = false) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(unsigned(2 * pairs), 1, 1);
  cfg.blockDim = dim3(unsigned(threads), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = env.stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (pdl) {
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  return cfg;
}

// Number of CTA pairs of `kernel` that can be resident at once (0: none).
// Asked once per kernel and device configuration, then remembered.
inline cudaError_t max_pairs(const void* kernel, size_t smem, const LaunchEnv& env, int* out,
                             std::atomic<int>* cache, int threads = kBaseThreads) {
  int n = cache->load();
  if (n < 0) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_launch_config(env.num_sms / 2, smem, env, attr, threads);
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (e != cudaSuccess) return e;
    cache->store(n);
  }
  *out = n;
  return cudaSuccess;
}

template <class P>
inline cudaError_t launch_on_pairs(const void* kernel, int pairs, size_t smem,
                                   const LaunchEnv& env, const P* params,
                                   int threads = kBaseThreads) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_launch_config(pairs, smem, env, attr, threads, true);
  unsigned int* status = env.status;
  void* args[] = {const_cast<P*>(params), &status};
  return cudaLaunchKernelExC(&cfg, kernel, args);
}

}  // namespace ittt
