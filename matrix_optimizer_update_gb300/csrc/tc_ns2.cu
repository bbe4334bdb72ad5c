// tc_ns2.cu - the Newton-Schulz products on CTA pairs: two-SM UMMA
// (tcgen05 cta_group::2), 256 x 256 output tiles.
//
// Same phases and the same per-tile epilogue as tc_ns.cu (gram / poly /
// gemm, epi::epilogue_tile: TMA-stored output boxes, prefetched W blocks on
// the last step). A
// cluster of two CTAs on neighbouring SMs owns one tile: each CTA loads its
// 128 rows of A and one half (128 rows, or 128 columns for the MN-major X
// operand of the gemm) of B into its own shared memory, the leader CTA
// (cluster rank 0) issues tcgen05.mma.cta_group::2 with M = 256, N = 256,
// and the 256 x 256 fp32 accumulator lands half in each CTA's TMEM. Per SM
// that moves 32 KB of operands per 4.2 MFLOP instead of 48 KB with one-SM
// 128 x 256 tiles.
//
// Synchronisation across the pair:
//  - full[s] lives in the leader; both CTAs' TMA loads count their bytes on
//    it (.cta_group::2 lets a load signal the peer's barrier), the leader
//    alone sets the expected byte count;
//  - empty[s] and tfull[a] live in both CTAs; the leader's commits arrive
//    on both (multicast::cluster);
//  - tempty[a] lives in the leader and collects one arrival per epilogue
//    warp of both CTAs;
//  - cluster barriers after set-up and before TMEM is released, so that no
//    CTA signals an uninitialised barrier or leaves while the leader's MMAs
//    still read its shared memory or write its TMEM.
// Tiles: the leader's TMA thread claims them from the launch's counter (or
// deals them, pair b taking items b, b + pairs, ...) and writes each item into
// a ring in both CTAs (sched_full in each CTA, one arrival from the leader);
// the leader's MMA thread, the peer's TMA thread and the epilogue warps of
// both take it from their own ring and arrive on the leader's sched_empty.
// All mbarrier waits are bounded as in tc_ns.cu.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "tc_epilogue.cuh"

namespace dmuon {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kPairBM = 256;                   // rows of a pair tile (128 per CTA)
constexpr int kPairBN = 256;                   // columns of a pair tile
constexpr uint32_t kHalfA = 128 * kTcBK * 2;   // 16 KB: this CTA's 128 rows of A
constexpr uint32_t kHalfB = 128 * kTcBK * 2;   // 16 KB: this CTA's half of B
constexpr int kStages = 6;
constexpr uint32_t kTmemCols = 2 * kPairBN;    // two 128 x 256 fp32 accumulators per CTA
constexpr int kEpiWarps = 8;
constexpr int kEpiChunks = kPairBN / 2 / 32;

constexpr int kSchedDepth = 8;                     // items in flight between the claim and the epilogue
constexpr uint32_t kSchedConsumers = 2 + 2 * kEpiWarps;  // leader's MMA thread, peer's TMA thread, epilogue warps

struct PairShared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint64_t sched_full[kSchedDepth];   // this CTA's ring slot written (1 arrival: the leader's TMA thread)
  uint64_t sched_empty[kSchedDepth];  // used in the leader: the slot read by every consumer of both CTAs
  int ring[kSchedDepth];              // item index, -1 = no more tiles
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(PairShared) <= 1024, "barriers must fit their 1 KB");
using epi::kStageBox;

// Consumer side of the item ring: the j-th item of this pair (false when the CTA gives up).
// lead_empty: cluster address of the leader's sched_empty[0].
__device__ __forceinline__ bool pair_take(PairShared* sh, uint32_t j, int& w, uint32_t lead_empty,
                                          volatile int* abortf, const TcParams& p) {
  const uint32_t slot = j % kSchedDepth;
  if (!ptx::mbar_wait_cluster(&sh->sched_full[slot], (j / kSchedDepth) & 1u, abortf, p.status, p.timeout_ns))
    return false;
  w = *reinterpret_cast<volatile int*>(&sh->ring[slot]);
  ptx::mbar_arrive_cluster(lead_empty + slot * static_cast<uint32_t>(sizeof(uint64_t)));
  return true;
}

template <int PHASE>
__global__ void __launch_bounds__(kTcThreads, 1) tc_ns_pair_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + kStages * kHalfA;
  PairShared* sh = reinterpret_cast<PairShared*>(sB + kStages * kHalfB);
  // epilogue staging: two 2 KB boxes per epilogue warp, after the barriers' 1 KB
  uint8_t* stg_all = sB + kStages * kHalfB + 1024;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abortf = &sh->abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&sh->full[s], 1);
      ptx::mbar_init(&sh->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&sh->tfull[a], 1);
      ptx::mbar_init(&sh->tempty[a], 2 * kEpiWarps);
    }
    ptx::mbar_init(&sh->mma_done, 1);
    for (int k = 0; k < kSchedDepth; ++k) {
      ptx::mbar_init(&sh->sched_full[k], 1);
      ptx::mbar_init(&sh->sched_empty[k], kSchedConsumers);
    }
    sh->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(&sh->tmem_base, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int npairs = static_cast<int>(gridDim.x >> 1);
  const uint32_t lead_empty = ptx::mapa_shared(ptx::smem_u32(&sh->sched_empty[0]), 0);
  const uint64_t t_start = ptx::globaltimer();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer (both CTAs)
      const uint32_t lead_full = ptx::mapa_shared(ptx::smem_u32(&sh->full[0]), 0);
      uint32_t stage = 0, phase = 0;
      uint32_t fills = 0;  // stages filled so far: fill f went to stage f % stages
      auto load_tile = [&](int w) -> bool {
        const int4 it = p.items[w];
        const TcBucket& B = p.bk[it.x];
        const int nk = (B.kdim + kTcBK - 1) / kTcBK;
        // a diagonal pair tile of a matrix with itself: each CTA's A rows are its B rows
        const bool a_in_b = PHASE != kPhaseGemm && B.same_ab && it.w == 0;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait_cluster(&sh->empty[stage], phase ^ 1u, abortf, p.status, p.timeout_ns)) return false;
          if (leader) ptx::mbar_arrive_expect_tx(&sh->full[stage], 2 * ((a_in_b ? 0u : kHalfA) + kHalfB));
          const uint32_t fb = lead_full + stage * static_cast<uint32_t>(sizeof(uint64_t));
          const int k0 = kb * kTcBK;
          if (!a_in_b)
            ptx::tma_load_3d_pair(sA + stage * kHalfA, &B.tmA, fb, k0, it.z * kPairBM + rank * 128, it.y);
          if (PHASE == kPhaseGemm) {  // one copy: this CTA's two 64-column chunks of 64 k-rows
            ptx::tma_load_4d_pair(sB + stage * kHalfB, &B.tmB, fb, 0, k0, (it.w * kPairBN + rank * 128) / 64, it.y);
          } else {  // symmetric products list a row pair's tiles from its diagonal block on
            ptx::tma_load_3d_pair(sB + stage * kHalfB, &B.tmB, fb, k0, (it.z + it.w) * kPairBN + rank * 128, it.y);
          }
          ++fills;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        return true;
      };
      if (leader) {
        // Also the pair's tile scheduler: with p.sched, tiles are claimed from the launch's counter in
        // list order as the pair gets to them, one claim ahead of the loads; without it, pair b takes
        // items b, b + pairs, ... Each item goes into both CTAs' rings; -1 ends the list.
        const uint32_t peer_ring = ptx::mapa_shared(ptx::smem_u32(&sh->ring[0]), 1);
        const uint32_t peer_full = ptx::mapa_shared(ptx::smem_u32(&sh->sched_full[0]), 1);
        auto claim = [&](uint32_t j) -> int {
          if (p.sched == nullptr) {
            const int64_t w = pair + static_cast<int64_t>(j) * npairs;
            return w < p.n_items ? static_cast<int>(w) : -1;
          }
          const unsigned w = atomicAdd(p.sched, 1u);
          return w < static_cast<unsigned>(p.n_items) ? static_cast<int>(w) : -1;
        };
        int w = claim(0);
        for (uint32_t j = 0;; ++j) {
          const uint32_t slot = j % kSchedDepth;
          if (!ptx::mbar_wait_cluster(&sh->sched_empty[slot], ((j / kSchedDepth) & 1u) ^ 1u, abortf, p.status,
                                      p.timeout_ns))
            break;
          sh->ring[slot] = w;
          ptx::st_shared_cluster_s32(peer_ring + slot * 4u, w);
          ptx::mbar_arrive(&sh->sched_full[slot]);
          ptx::mbar_arrive_cluster(peer_full + slot * static_cast<uint32_t>(sizeof(uint64_t)));  // orders the store
          if (w < 0) break;
          const int next = claim(j + 1);  // its latency hides under this tile's loads
          if (!load_tile(w)) break;
          w = next;
        }
      } else {
        for (uint32_t j = 0;; ++j) {
          int w;
          if (!pair_take(sh, j, w, lead_empty, abortf, p) || w < 0) break;
          if (!load_tile(w)) break;
        }
      }
      // The leader's full barriers count both CTAs' bytes: once their last
      // phases complete, no load of either CTA is still in flight.
      if (leader) {
        for (uint32_t s = 0; s < kStages; ++s) {
          if (fills > s) {
            const uint32_t n = (fills - 1u - s) / kStages + 1u;  // fills of stage s
            int zero = 0;
            ptx::mbar_wait_cluster(&sh->full[s], (n - 1u) & 1u, &zero, p.status, p.timeout_ns);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ MMA issuer (leader only)
      constexpr uint32_t idesc = ptx::idesc_bf16(kPairBM, kPairBN, PHASE == kPhaseGemm);
      uint32_t stage = 0, phase = 0, local = 0;
      bool ok = true;
      for (int w; ok && pair_take(sh, local, w, lead_empty, abortf, p) && w >= 0; ++local) {
        const int4 it = p.items[w];
        const TcBucket& B = p.bk[it.x];
        const int nk = (B.kdim + kTcBK - 1) / kTcBK;
        const uint32_t acc = local & 1u;
        const bool a_in_b = PHASE != kPhaseGemm && B.same_ab && it.w == 0;
        if (!ptx::mbar_wait_cluster(&sh->tempty[acc], ((local >> 1) & 1u) ^ 1u, abortf, p.status, p.timeout_ns))
          break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + acc * kPairBN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait_cluster(&sh->full[stage], phase, abortf, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t b0 = ptx::smem_u32(sB + stage * kHalfB);
          const uint32_t a0 = a_in_b ? b0 : ptx::smem_u32(sA + stage * kHalfA);
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk) {
            const uint64_t adesc = ptx::sw128_desc(a0 + kk * 32, 16, 1024);
            const uint64_t bdesc = (PHASE == kPhaseGemm) ? ptx::sw128_desc(b0 + kk * 2048, 64 * kTcBK * 2, 1024)
                                                         : ptx::sw128_desc(b0 + kk * 32, 16, 1024);
            ptx::umma_f16_pair(d, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::umma_commit_pair(&sh->empty[stage], 0x3);  // frees the stage in both CTAs
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::umma_commit_pair(&sh->tfull[acc], 0x3);  // accumulator halves ready in both CTAs
      }
      ptx::umma_commit_pair(&sh->mma_done, 0x1);
      int zero = 0;
      ptx::mbar_wait(&sh->mma_done, 0, &zero, p.status, p.timeout_ns);
    }
  } else {
    // -------------------------------------------------------------- epilogue (both CTAs)
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t lead_tempty = ptx::mapa_shared(ptx::smem_u32(&sh->tempty[0]), 0);
    uint8_t* stg = stg_all + (warp - 2) * (2 * kStageBox);
    uint32_t local = 0, nbox = 0;
    for (;; ++local) {
      int w = -2;  // -2: the CTA gave up
      if (lane == 0 && !pair_take(sh, local, w, lead_empty, abortf, p)) w = -2;
      w = __shfl_sync(0xffffffffu, w, 0);
      if (w < 0) break;
      const uint32_t acc = local & 1u;
      const int4 it = p.items[w];
      const TcBucket& B = p.bk[it.x];
      const int i0 = it.z * kPairBM + static_cast<int>(rank) * 128 + q * 32;
      const int jbase = (PHASE == kPhaseGemm ? it.w : it.z + it.w) * kPairBN + half * (kPairBN / 2);
      const uint32_t tbase = tmem + acc * kPairBN + half * (kPairBN / 2) + ((uint32_t)(q * 32) << 16);
      const bool ok = epi::epilogue_tile<PHASE, kEpiChunks>(p, B, it, i0, jbase, tbase, lane, stg, nbox, [&]() {
        return ptx::mbar_wait_cluster(&sh->tfull[acc], (local >> 1) & 1u, abortf, p.status, p.timeout_ns);
      });
      if (!ok) break;
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(lead_tempty + acc * static_cast<uint32_t>(sizeof(uint64_t)));
    }
    ptx::bulk_wait_all();      // every bulk store of this warp (TMA boxes, W rows) has landed
    ptx::cp_async_wait<0>();   // and every W copy (matters only after an abort)
  }

  __syncthreads();
  if (threadIdx.x == 0) {
    if (p.cta_times != nullptr && blockIdx.x < kMaxCtaRecords) {  // profiling: this CTA's start and end
      p.cta_times[2 * blockIdx.x] = t_start;
      p.cta_times[2 * blockIdx.x + 1] = ptx::globaltimer();
    }
    if (p.sched != nullptr) {
      // Every claim of a leader precedes its arrival here; the last CTA to arrive leaves both words
      // at zero for the next launch that uses them.
      __threadfence();
      if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
        p.sched[0] = 0u;
        p.sched[1] = 0u;
      }
    }
  }
  ptx::cluster_sync();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, kTmemCols);
  }
}

template <int PHASE>
cudaError_t launch_pair_phase(const TcParams& p, int pairs, cudaStream_t s) {
  const size_t smem = 1024 + kStages * (kHalfA + kHalfB) + 1024 + kEpiWarps * kStageBox * 2;
  cudaError_t e = cudaFuncSetAttribute(tc_ns_pair_kernel<PHASE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_ns_pair_kernel<PHASE>, p);
}

}  // namespace

cudaError_t launch_tc_pair(int phase, const TcParams& p, int pairs, cudaStream_t s) {
  switch (phase) {
    case kPhaseGram:
      return launch_pair_phase<kPhaseGram>(p, pairs, s);
    case kPhasePoly:
      return launch_pair_phase<kPhasePoly>(p, pairs, s);
    case kPhaseGemm:
      return launch_pair_phase<kPhaseGemm>(p, pairs, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace dmuon
