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
//   poly:  B = b*A + c*(A A^T)  (A is symmetric, so A A = A A^T: the same
//                                symmetric product on A, b*A added in the
//                                epilogue from the same bf16 A tile)
//   gemm:  X' = a*X + B X       (a*X added in the epilogue; on the last step
//                                the epilogue applies W -= lr*scale*X' instead
//                                of storing X')
// At step 0 the Frobenius normalisation is folded in: the workspace holds the
// unnormalised U and X0 = s*U with s = 1/(||U||_F + eps), so the gram epilogue
// multiplies by s^2 and the gemm epilogue by s.
//
// CTA layout (192 threads, one CTA per SM, persistent over a cost-ordered
// tile list): warp 0 issues TMA loads of 64-wide K slices into a 4-stage ring
// of shared-memory buffers (128B swizzle); warp 1 allocates 512 TMEM columns
// (two 128 x 256 fp32 accumulators) and one thread issues tcgen05.mma
// (M=128, N=256, K=16); warps 2..5 drain an accumulator with tcgen05.ld while
// the MMA warp fills the other one. Every wait is bounded (see ptx.cuh).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace dmuon {
namespace {

using bf16 = __nv_bfloat16;

constexpr uint32_t kStageA = kTcBM * kTcBK * 2;  // 16 KB: 128 rows x 128 B
constexpr uint32_t kStageB = kTcBN * kTcBK * 2;  // 32 KB: 256 rows x 128 B (or 4 x [64 k-rows x 128 B])
constexpr uint32_t kTmemCols = 2 * kTcBN;        // two fp32 accumulators of 256 columns
constexpr int kEpiWarps = 4;

struct TcShared {
  uint64_t full[kTcStages];
  uint64_t empty[kTcStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void load_row_bf16(const bf16* src, int j0, int lim, float (&x)[32]) {
  if (j0 + 32 <= lim) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src + j0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 u = s4[q];
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float2 f = __bfloat1622float2(h[e]);
        x[q * 8 + 2 * e] = f.x;
        x[q * 8 + 2 * e + 1] = f.y;
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < 32; ++k) x[k] = (j0 + k < lim) ? __bfloat162float(src[j0 + k]) : 0.f;
  }
}

__device__ __forceinline__ void store_row_bf16(bf16* dst, int j0, int jmin, int lim, const float (&v)[32]) {
  if (j0 >= jmin && j0 + 32 <= lim) {
    uint4* d4 = reinterpret_cast<uint4*>(dst + j0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 u;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
      for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(v[q * 8 + 2 * e], v[q * 8 + 2 * e + 1]);
      d4[q] = u;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const int j = j0 + k;
      if (j >= jmin && j < lim) dst[j] = __float2bfloat16_rn(v[k]);
    }
  }
}

// Epilogue of one 32-column chunk of one accumulator row.
template <int PHASE>
__device__ __forceinline__ void epilogue_chunk(const TcParams& p, const TcBucket& B, const MatDev& md, int gm,
                                               int slot, int i, int j0, float sc, float (&v)[32]) {
  if (PHASE == kPhaseGram || PHASE == kPhasePoly) {
    const int m = B.m;
    if (i >= m || j0 >= m || j0 + 31 < i) return;  // nothing of the upper triangle here
    bf16* out = reinterpret_cast<bf16*>(B.out + slot * B.out_mat_stride);
    if (PHASE == kPhasePoly) {
      const bf16* A = reinterpret_cast<const bf16*>(B.aux + slot * B.aux_mat_stride) + (int64_t)i * B.aux_ld;
      float a[32];
      load_row_bf16(A, j0, m, a);
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = p.b * a[k] + p.c * v[k];
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] *= sc;
    }
    // own row: columns j >= i; mirror: (j, i) for j > i (coalesced across the warp's 32 rows)
    store_row_bf16(out + (int64_t)i * B.out_ld, j0, i, m, v);
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const int j = j0 + k;
      if (j > i && j < m) out[(int64_t)j * B.out_ld + i] = __float2bfloat16_rn(v[k]);
    }
  } else {  // gemm
    const int m = B.m, n = B.n;
    if (i >= m || j0 >= n) return;
    const bf16* X = reinterpret_cast<const bf16*>(B.aux + slot * B.aux_mat_stride) + (int64_t)i * B.aux_ld;
    float x[32];
    load_row_bf16(X, j0, n, x);
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = (p.a * x[k] + v[k]) * sc;
    if (!p.last) {
      bf16* out = reinterpret_cast<bf16*>(B.out + slot * B.out_mat_stride) + (int64_t)i * B.out_ld;
      store_row_bf16(out, j0, 0, n, v);
      return;
    }
    const float step = p.lr * md.scale;
    void* W = reinterpret_cast<void*>(p.ptrs[gm]);
    if (!md.transposed) {  // W is m x n, row i
      if (p.param_bf16) {
        bf16* w = reinterpret_cast<bf16*>(W) + (int64_t)i * n;
        if (j0 + 32 <= n && (n & 7) == 0) {
          uint4* w4 = reinterpret_cast<uint4*>(w + j0);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 u = w4[q];
            __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float2 f = __bfloat1622float2(h[e]);
              f.x -= step * v[q * 8 + 2 * e];
              f.y -= step * v[q * 8 + 2 * e + 1];
              h[e] = __floats2bfloat162_rn(f.x, f.y);
            }
            w4[q] = u;
          }
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (j0 + k < n) w[j0 + k] = __float2bfloat16_rn(__bfloat162float(w[j0 + k]) - step * v[k]);
        }
      } else {
        float* w = reinterpret_cast<float*>(W) + (int64_t)i * n;
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (j0 + k < n) w[j0 + k] -= step * v[k];
      }
    } else {  // W is n x m: element (j, i); consecutive lanes write consecutive i
      if (p.param_bf16) {
        bf16* w = reinterpret_cast<bf16*>(W);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int j = j0 + k;
          if (j < n) {
            bf16* e = w + (int64_t)j * m + i;
            *e = __float2bfloat16_rn(__bfloat162float(*e) - step * v[k]);
          }
        }
      } else {
        float* w = reinterpret_cast<float*>(W);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int j = j0 + k;
          if (j < n) w[(int64_t)j * m + i] -= step * v[k];
        }
      }
    }
    if (p.capture != nullptr && md.cap_off >= 0) {
      float* cap = p.capture + md.cap_off;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int j = j0 + k;
        if (j < n) cap[md.transposed ? (int64_t)j * m + i : (int64_t)i * n + j] = v[k];
      }
    }
  }
}

template <int PHASE>
__global__ void __launch_bounds__(kTcThreads, 1) tc_ns_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + kTcStages * kStageA;
  TcShared* sh = reinterpret_cast<TcShared*>(sB + kTcStages * kStageB);
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

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      uint32_t stage = 0, phase = 0;
      uint32_t issued[kTcStages];
      for (int s = 0; s < kTcStages; ++s) issued[s] = 0;
      for (int w = blockIdx.x; w < p.n_items; w += gridDim.x) {
        const int4 it = p.items[w];
        const TcBucket& B = p.bk[it.x];
        const int nk = (B.kdim + kTcBK - 1) / kTcBK;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait(&sh->empty[stage], phase ^ 1u, abortf, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&sh->full[stage], kStageA + kStageB);
          const int k0 = kb * kTcBK;
          ptx::tma_load_3d(sA + stage * kStageA, &B.tmA, &sh->full[stage], k0, it.z * kTcBM, it.y);
          if (PHASE == kPhaseGemm) {
#pragma unroll
            for (int q = 0; q < kTcBN / 64; ++q)
              ptx::tma_load_3d(sB + stage * kStageB + q * (64 * kTcBK * 2), &B.tmB, &sh->full[stage],
                               it.w * kTcBN + q * 64, k0, it.y);
          } else {
            ptx::tma_load_3d(sB + stage * kStageB, &B.tmB, &sh->full[stage], k0, it.w * kTcBN, it.y);
          }
          ++issued[stage];
          if (++stage == kTcStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      // Every issued copy must land before the CTA may exit (matters only after an abort).
      for (int s = 0; s < kTcStages; ++s) {
        if (issued[s]) {
          int zero = 0;
          ptx::mbar_wait(&sh->full[s], (issued[s] - 1u) & 1u, &zero, p.status, p.timeout_ns);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = ptx::idesc_bf16(kTcBM, kTcBN, PHASE == kPhaseGemm);
      uint32_t stage = 0, phase = 0, local = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < p.n_items && ok; w += gridDim.x, ++local) {
        const int4 it = p.items[w];
        const TcBucket& B = p.bk[it.x];
        const int nk = (B.kdim + kTcBK - 1) / kTcBK;
        const uint32_t acc = local & 1u;
        if (!ptx::mbar_wait(&sh->tempty[acc], ((local >> 1) & 1u) ^ 1u, abortf, p.status, p.timeout_ns)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + acc * kTcBN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait(&sh->full[stage], phase, abortf, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(sA + stage * kStageA);
          const uint32_t b0 = ptx::smem_u32(sB + stage * kStageB);
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
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint32_t local = 0;
    for (int w = blockIdx.x; w < p.n_items; w += gridDim.x, ++local) {
      const uint32_t acc = local & 1u;
      if (!ptx::mbar_wait(&sh->tfull[acc], (local >> 1) & 1u, abortf, p.status, p.timeout_ns)) break;
      ptx::tc_fence_after();
      const int4 it = p.items[w];
      const TcBucket& B = p.bk[it.x];
      const int gm = B.slot_mat[it.y];
      const MatDev md = p.mats[gm];
      float sc = 1.f;
      if (p.first) {
        const float s = p.s_norm[gm];
        sc = (PHASE == kPhaseGram) ? s * s : s;
      }
      const int i = it.z * kTcBM + q * 32 + lane;
      const uint32_t tbase = tmem + acc * kTcBN + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int ch = 0; ch < kTcBN / 32; ++ch) {
        float v[32];
        ptx::tmem_ld_32x32b_x32(tbase + ch * 32, v);
        epilogue_chunk<PHASE>(p, B, md, gm, it.y, i, it.w * kTcBN + ch * 32, sc, v);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sh->tempty[acc]);
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int PHASE>
cudaError_t launch_phase(const TcParams& p, int grid, cudaStream_t s) {
  static bool configured = false;
  const size_t smem = tc_smem_bytes();
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(tc_ns_kernel<PHASE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  tc_ns_kernel<PHASE><<<grid, kTcThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t tc_smem_bytes() { return 1024 + kTcStages * (kStageA + kStageB) + sizeof(TcShared); }

cudaError_t launch_tc(int phase, const TcParams& p, int grid, cudaStream_t s) {
  switch (phase) {
    case kPhaseGram:
      return launch_phase<kPhaseGram>(p, grid, s);
    case kPhasePoly:
      return launch_phase<kPhasePoly>(p, grid, s);
    case kPhaseGemm:
      return launch_phase<kPhaseGemm>(p, grid, s);
    default:
      return cudaErrorInvalidValue;
  }
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
