// tc_ns.cu - the three Newton-Schulz products on the 5th-generation tensor
// cores (tcgen05), one persistent launch per phase over every bucket.
//
// Per step k of the quintic iteration (X is m x n, m <= n, bf16 in HBM):
//   gram:  A = X X^T            (only tiles touching the upper triangle are
//                                computed; each value is written to (i,j)
//                                and mirrored to (j,i): the symmetric-Gram /
//                                SYRK execution path of "DMuon: Efficient
//                                Distributed Muon Training with Near-Adam
//                                Overhead", gist.science summary section 2,
//                                "Benutting van Symmetrie")
//   poly:  P = a*I + b*A + c*(A A^T)
//                               (A is symmetric, so A A = A A^T: the same
//                                symmetric product on A; b*A from the same
//                                bf16 A tile and a on the diagonal are added
//                                in the epilogue)
//   gemm:  X' = P X = a*X + (b*A + c*A^2) X
//                               (on the last step the epilogue applies
//                                W -= lr*scale*X' instead of storing X'.
//                                With DMUON_FLAG_EPILOGUE_AX the poly leaves
//                                out a*I and the gemm epilogue adds a*X.)
// At step 0 the Frobenius normalisation is folded in: the workspace holds the
// unnormalised U and X0 = s*U with s = 1/(||U||_F + eps), so the gram epilogue
// multiplies by s^2 and the gemm epilogue by s.
//
// The same three kernels also run the Gram-space form of the iteration
// (gist.science summary section 2, "Gram Space Recurrence"): G = X0 X0^T once,
// then per step P = a I + b G + c G^2 (poly with a diagonal term),
// Q <- P Q and G <- (P G) P (symmetric products of commuting symmetric
// matrices: the gram kernel with two different operands), and finally
// X = Q X0 (gemm with a = 0) with the W update fused.
//
// CTA layout (320 threads, one CTA per SM, persistent over a cost-ordered
// tile list): warp 0 issues TMA loads of 64-wide K slices into a 4-stage ring
// of shared-memory buffers (128B swizzle); warp 1 allocates 512 TMEM columns
// (two 128 x 256 fp32 accumulators) and one thread issues tcgen05.mma
// (M=128, N=256, K=16); warps 2..9 drain an accumulator with tcgen05.ld
// (two warps per TMEM lane quarter, one per column half) while the MMA warp
// fills the other one. The epilogue warps stage their 32 x 32 output chunks
// in shared memory and write them with TMA stores (a symmetric chunk also as
// its mirror image); on the last step they prefetch the weights' blocks with
// cp.async and update them in shared memory. Every wait is bounded (see
// ptx.cuh).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "tc_epilogue.cuh"

namespace dmuon {
namespace {

using bf16 = __nv_bfloat16;

constexpr uint32_t kStageA = kTcBM * kTcBK * 2;  // 16 KB: 128 rows x 128 B
constexpr int kEpiWarps = 8;                      // two per TMEM lane quarter
using epi::kStageBox;

// Tile width N of one CTA (the UMMA N): 256, or 128 where the planner's
// tile-count cost favours it. Shared-memory stages fill the same 192 KB
// either way; 32 KB of epilogue staging and 1 KB of barriers follow them.
template <int BN>
struct TcCfg {
  static constexpr uint32_t kStageB = BN * kTcBK * 2;  // BN rows x 128 B (or BN/64 x [64 k-rows x 128 B])
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr uint32_t kTmemCols = 2 * BN;        // two fp32 accumulators of BN columns
  static constexpr int kEpiChunks = BN / 2 / 32;       // 32-column chunks per epilogue warp
};

// Tiles claimed by the TMA thread reach the MMA thread and the epilogue warps
// through a ring of this many item indices.
constexpr int kSchedDepth = 8;

template <int STAGES>
struct TcShared {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint64_t sched_full[kSchedDepth];   // item published (1 arrival: the TMA thread)
  uint64_t sched_empty[kSchedDepth];  // item read by the MMA thread and every epilogue warp
  int ring[kSchedDepth];              // item index, -1 = no more tiles
  uint32_t tmem_base;
  int abort_flag;
};

static_assert(sizeof(TcShared<6>) <= 1024, "barriers must fit their 1 KB");

// Consumer side of the item ring: the j-th item of this CTA (false when the CTA gives up).
template <int STAGES>
__device__ __forceinline__ bool ring_take(TcShared<STAGES>* sh, uint32_t j, int& w, volatile int* abortf,
                                          const TcParams& p) {
  const uint32_t slot = j % kSchedDepth;
  if (!ptx::mbar_wait(&sh->sched_full[slot], (j / kSchedDepth) & 1u, abortf, p.status, p.timeout_ns)) return false;
  w = *reinterpret_cast<volatile int*>(&sh->ring[slot]);
  ptx::mbar_arrive(&sh->sched_empty[slot]);
  return true;
}

// A symmetric product of one matrix with itself (X X^T, A A^T): a tile that starts at its diagonal
// block (tj = 0) has A rows 128 ti.. equal to the first 128 of its B rows, so the A operand is read
// from the B stage and not loaded. (The same holds per CTA of a two-SM tile.)
__device__ __forceinline__ bool a_rows_in_b(const TcBucket& B, const int4& it) { return B.same_ab && it.w == 0; }

// First output column of a symmetric-product tile (bucket, slot, ti, tj):
// the planner lists each row block's tiles from its diagonal block on.
template <int BN>
__device__ __forceinline__ int sym_col0(const int4& it) {
  return it.z * kTcBM + it.w * BN;
}

template <int PHASE, int BN>
__global__ void __launch_bounds__(kTcThreads, 1) tc_ns_kernel(const __grid_constant__ TcParams p) {
  using C = TcCfg<BN>;
  constexpr int kTcStages = C::kStages;
  constexpr uint32_t kStageB = C::kStageB;
  constexpr uint32_t kTmemCols = C::kTmemCols;
  constexpr int kEpiChunks = C::kEpiChunks;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + kTcStages * kStageA;
  TcShared<kTcStages>* sh = reinterpret_cast<TcShared<kTcStages>*>(sB + kTcStages * kStageB);
  // Epilogue staging for TMA stores: two 2 KB boxes (32 x 32 bf16) per epilogue warp, after the
  // barriers' 1 KB.
  uint8_t* stg_all = sB + kTcStages * kStageB + 1024;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abortf = &sh->abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      ptx::mbar_init(&sh->full[s], 1);
      ptx::mbar_init(&sh->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&sh->tfull[a], 1);
      ptx::mbar_init(&sh->tempty[a], kEpiWarps);
    }
    ptx::mbar_init(&sh->mma_done, 1);
    for (int k = 0; k < kSchedDepth; ++k) {
      ptx::mbar_init(&sh->sched_full[k], 1);
      ptx::mbar_init(&sh->sched_empty[k], 1 + kEpiWarps);
    }
    sh->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&sh->tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sh->tmem_base;

  const uint64_t t_start = ptx::globaltimer();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      // Also the tile scheduler: with p.sched, tiles are claimed from the launch's counter in
      // list order (largest cost first) as this CTA gets to them, one claim ahead of the loads;
      // without it, CTA b takes items b, b + grid, b + 2*grid, ... Either way each claimed item
      // goes into the ring for the MMA thread and the epilogue warps; -1 ends the list.
      auto claim = [&](uint32_t j) -> int {
        if (p.sched == nullptr) {
          const int64_t w = blockIdx.x + static_cast<int64_t>(j) * gridDim.x;
          return w < p.n_items ? static_cast<int>(w) : -1;
        }
        const unsigned w = atomicAdd(p.sched, 1u);
        return w < static_cast<unsigned>(p.n_items) ? static_cast<int>(w) : -1;
      };
      uint32_t stage = 0, phase = 0, j = 0;
      uint32_t fills = 0;  // stages filled so far: fill f went to stage f % stages
      int w = claim(0);
      for (;;) {
        const uint32_t slot = j % kSchedDepth;
        if (!ptx::mbar_wait(&sh->sched_empty[slot], ((j / kSchedDepth) & 1u) ^ 1u, abortf, p.status, p.timeout_ns))
          break;
        sh->ring[slot] = w;
        ptx::mbar_arrive(&sh->sched_full[slot]);
        ++j;
        if (w < 0) break;
        const int next = claim(j);  // its latency hides under this tile's loads
        const int4 it = p.items[w];
        const TcBucket& B = p.bk[it.x];
        const int nk = (B.kdim + kTcBK - 1) / kTcBK;
        const bool a_in_b = a_rows_in_b(B, it);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait(&sh->empty[stage], phase ^ 1u, abortf, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&sh->full[stage], (a_in_b ? 0u : kStageA) + kStageB);
          const int k0 = kb * kTcBK;
          if (!a_in_b) ptx::tma_load_3d(sA + stage * kStageA, &B.tmA, &sh->full[stage], k0, it.z * kTcBM, it.y);
          if (PHASE == kPhaseGemm) {  // one copy: BN/64 chunks of 64 columns x 64 k-rows, 8 KB apart
            ptx::tma_load_4d(sB + stage * kStageB, &B.tmB, &sh->full[stage], 0, k0, it.w * (BN / 64), it.y);
          } else {  // rows of the tile's columns; rows past the matrix's edge are zero-filled
            ptx::tma_load_3d(sB + stage * kStageB, &B.tmB, &sh->full[stage], k0, sym_col0<BN>(it), it.y);
          }
          ++fills;
          if (++stage == kTcStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        w = next;
      }
      // Every issued copy must land before the CTA may exit (matters only after an abort).
      for (uint32_t s = 0; s < kTcStages; ++s) {
        if (fills > s) {
          const uint32_t n = (fills - 1u - s) / kTcStages + 1u;  // fills of stage s
          int zero = 0;
          ptx::mbar_wait(&sh->full[s], (n - 1u) & 1u, &zero, p.status, p.timeout_ns);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc_full = ptx::idesc_bf16(kTcBM, BN, PHASE == kPhaseGemm);
      constexpr uint32_t idesc_half = ptx::idesc_bf16(kTcBM, BN / 2, PHASE == kPhaseGemm);
      uint32_t stage = 0, phase = 0, local = 0;
      bool ok = true;
      for (int w; ok && ring_take(sh, local, w, abortf, p) && w >= 0; ++local) {
        const int4 it = p.items[w];
        const TcBucket& B = p.bk[it.x];
        const int nk = (B.kdim + kTcBK - 1) / kTcBK;
        const uint32_t acc = local & 1u;
        // A symmetric tile whose right half lies wholly past the matrix's edge multiplies only its
        // left half (the first BN/2 rows of the B stage); the epilogue stores nothing of the rest.
        const uint32_t idesc =
            (PHASE != kPhaseGemm && BN == 256 && sym_col0<BN>(it) + BN / 2 >= B.m) ? idesc_half : idesc_full;
        const bool a_in_b = a_rows_in_b(B, it);
        if (!ptx::mbar_wait(&sh->tempty[acc], ((local >> 1) & 1u) ^ 1u, abortf, p.status, p.timeout_ns)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait(&sh->full[stage], phase, abortf, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t b0 = ptx::smem_u32(sB + stage * kStageB);
          const uint32_t a0 = a_in_b ? b0 : ptx::smem_u32(sA + stage * kStageA);
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk) {
            // K-major 128B-swizzled rows: a K step of 16 bf16 is 32 bytes inside the swizzle atom;
            // 8-row groups are 1024 bytes apart.
            const uint64_t adesc = ptx::sw128_desc(a0 + kk * 32, 16, 1024);
            uint64_t bdesc;
            if (PHASE == kPhaseGemm) {
              // MN-major: 64-column chunks 8 KB apart (leading), 8 k-rows 1024 B apart (stride);
              // a K step of 16 rows is 2048 bytes.
              bdesc = ptx::sw128_desc(b0 + kk * 2048, 64 * kTcBK * 2, 1024);
            } else {
              bdesc = ptx::sw128_desc(b0 + kk * 32, 16, 1024);
            }
            ptx::umma_f16(d, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::umma_commit(&sh->empty[stage]);  // frees the smem stage once these MMAs have read it
          if (++stage == kTcStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::umma_commit(&sh->tfull[acc]);  // accumulator ready for the epilogue
      }
      // All MMAs must be complete before TMEM is released.
      ptx::umma_commit(&sh->mma_done);
      int zero = 0;
      ptx::mbar_wait(&sh->mma_done, 0, &zero, p.status, p.timeout_ns);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    // Two warps per TMEM lane quarter (warp % 4), each on one half of the 256 columns.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* stg = stg_all + (warp - 2) * (2 * kStageBox);
    uint32_t local = 0, nbox = 0;
    for (;; ++local) {
      int w = -2;  // -2: the CTA gave up
      if (lane == 0 && !ring_take(sh, local, w, abortf, p)) w = -2;
      w = __shfl_sync(0xffffffffu, w, 0);
      if (w < 0) break;
      const uint32_t acc = local & 1u;
      const int4 it = p.items[w];
      const TcBucket& B = p.bk[it.x];
      const int i0 = it.z * kTcBM + q * 32;
      const int jbase = (PHASE == kPhaseGemm ? it.w * BN : sym_col0<BN>(it)) + half * (BN / 2);
      const uint32_t tbase = tmem + acc * BN + half * (BN / 2) + ((uint32_t)(q * 32) << 16);
      const bool ok = epi::epilogue_tile<PHASE, kEpiChunks>(p, B, it, i0, jbase, tbase, lane, stg, nbox, [&]() {
        return ptx::mbar_wait(&sh->tfull[acc], (local >> 1) & 1u, abortf, p.status, p.timeout_ns);
      });
      if (!ok) break;
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sh->tempty[acc]);
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
      // Every claim of this CTA precedes its arrival here; the last CTA to arrive leaves both
      // words at zero for the next launch that uses them.
      __threadfence();
      if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
        p.sched[0] = 0u;
        p.sched[1] = 0u;
      }
    }
  }
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int PHASE, int BN>
size_t smem_bytes() {
  using C = TcCfg<BN>;
  return 1024 + C::kStages * (kStageA + C::kStageB) + 1024 + kEpiWarps * kStageBox * 2;
}

template <int PHASE, int BN>
cudaError_t launch_phase(const TcParams& p, int grid, cudaStream_t s) {
  const size_t smem = smem_bytes<PHASE, BN>();
  cudaError_t e = cudaFuncSetAttribute(tc_ns_kernel<PHASE, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  tc_ns_kernel<PHASE, BN><<<grid, kTcThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <int BN>
cudaError_t launch_bn(int phase, const TcParams& p, int grid, cudaStream_t s) {
  switch (phase) {
    case kPhaseGram:
      return launch_phase<kPhaseGram, BN>(p, grid, s);
    case kPhasePoly:
      return launch_phase<kPhasePoly, BN>(p, grid, s);
    case kPhaseGemm:
      return launch_phase<kPhaseGemm, BN>(p, grid, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_tc(int phase, int bn, const TcParams& p, int grid, cudaStream_t s) {
  if (bn == 256) return launch_bn<256>(phase, p, grid, s);
  if (bn == 128) return launch_bn<128>(phase, p, grid, s);
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ self-test
// A barrier that nothing ever arrives on: the bounded wait must give up,
// record DMUON_DEV_WAIT_TIMEOUT and let the kernel return.
__global__ void wait_timeout_selftest_kernel(unsigned* status, int64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile int* af = &abort_flag;
    ptx::mbar_wait(&bar, 0, af, status, limit_ns);
  }
}

cudaError_t launch_wait_timeout_selftest(unsigned* status, int64_t limit_ns, cudaStream_t s) {
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace dmuon

static_assert(sizeof(dmuon::TcParams) <= 4000, "tensor-core launch parameters must fit the 4 KB kernel-parameter space");
