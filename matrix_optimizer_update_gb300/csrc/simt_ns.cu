// simt_ns.cu - fp32 arithmetic mode of the Newton-Schulz products.
//
// Same three phases as the tensor-core path (gram A = X X^T on upper tiles
// with mirrored stores; poly B = b*A + c*A A^T; gemm X' = a*X + B X with the
// W update fused into the last step), computed with fp32 FFMA on CUDA cores:
// TF32 tensor math keeps only 10 mantissa bits and cannot reach fp32-level
// agreement. One kSimtBM x kSimtBN output tile per CTA, 256 threads in a 16 x 16
// grid, each with (kSimtBM / 16) x (kSimtBN / 16) outputs, K staged kSimtBK at a
// time through shared memory. Each output is summed over K in increasing order
// by one thread, so neither the tile shape nor the stage depth changes the result.
#include <cuda_bf16.h>

#include "simt.h"

namespace dmuon {
namespace {

template <int PHASE>
__global__ void __launch_bounds__(kSimtThreads) simt_ns_kernel(const __grid_constant__ SimtParams p) {
  __shared__ float As[kSimtBK][kSimtBM + 4];  // As[k][row]
  __shared__ float Bs[kSimtBK][kSimtBN + 4];  // Bs[k][col]
  const int4 it = p.items[blockIdx.x];
  const SimtBucket& B = p.bk[it.x];
  const int slot = it.y;
  // symmetric products list their tiles from the diagonal block on: column tile it.w counts from it.z
  const int row0 = it.z * kSimtBM, col0 = (PHASE == kPhaseGemm) ? it.w * kSimtBN : row0 + it.w * kSimtBN;
  const float* opA = B.opA + slot * B.a_mat_stride;
  const float* opB = B.opB + slot * B.b_mat_stride;
  constexpr int TM = kSimtBM / 16, TN = kSimtBN / 16;  // outputs per thread along rows / columns
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m = B.m, kdim = B.kdim;
  // output columns are bounded by m (gram/poly) or n (gemm)
  const int ncols = (PHASE == kPhaseGemm) ? B.n : B.m;

  float acc[TM][TN];
#pragma unroll
  for (int r = 0; r < TM; ++r)
#pragma unroll
    for (int c = 0; c < TN; ++c) acc[r][c] = 0.f;

  // Operand elements this thread moves per K stage, and the stages whose loads are issued together:
  // the loads of up to kSimtGroup stages go out at once into registers, so a short K waits on memory
  // about once; each stage then passes through shared memory in turn.
  constexpr int kPerA = kSimtBM * kSimtBK / kSimtThreads, kPerB = kSimtBN * kSimtBK / kSimtThreads;
  static_assert(kPerA * kSimtThreads == kSimtBM * kSimtBK && kPerB * kSimtThreads == kSimtBN * kSimtBK,
                "tiles must split evenly over the threads");
  // A operand element e of a stage: row e / BK, k e % BK (rows of opA, K contiguous in memory).
  auto load_a = [&](int k0, int q) -> float {
    const int e = tid + q * kSimtThreads;
    const int gr = row0 + e / kSimtBK, gk = k0 + e % kSimtBK;
    return (gr < m && gk < kdim) ? opA[(int64_t)gr * B.a_ld + gk] : 0.f;
  };
  // B operand element e: gemm, X_k row k (K) e / BN, column e % BN (columns contiguous in memory);
  // symmetric products, row col0 + e / BK of the same matrix, k e % BK.
  auto load_b = [&](int k0, int q) -> float {
    const int e = tid + q * kSimtThreads;
    if (PHASE == kPhaseGemm) {
      const int gk = k0 + e / kSimtBN, gc = col0 + e % kSimtBN;
      return (gk < kdim && gc < ncols) ? opB[(int64_t)gk * B.b_ld + gc] : 0.f;
    }
    const int gc = col0 + e / kSimtBK, gk = k0 + e % kSimtBK;
    return (gc < ncols && gk < kdim) ? opB[(int64_t)gc * B.b_ld + gk] : 0.f;
  };
  for (int g0 = 0; g0 < kdim; g0 += kSimtGroup * kSimtBK) {
    float ra[kSimtGroup][kPerA], rb[kSimtGroup][kPerB];
#pragma unroll
    for (int st = 0; st < kSimtGroup; ++st) {
      const int k0 = g0 + st * kSimtBK;
#pragma unroll
      for (int q = 0; q < kPerA; ++q) ra[st][q] = (k0 < kdim) ? load_a(k0, q) : 0.f;
#pragma unroll
      for (int q = 0; q < kPerB; ++q) rb[st][q] = (k0 < kdim) ? load_b(k0, q) : 0.f;
    }
#pragma unroll
    for (int st = 0; st < kSimtGroup; ++st) {
      if (g0 + st * kSimtBK >= kdim) break;
#pragma unroll
      for (int q = 0; q < kPerA; ++q) {
        const int e = tid + q * kSimtThreads;
        As[e % kSimtBK][e / kSimtBK] = ra[st][q];
      }
#pragma unroll
      for (int q = 0; q < kPerB; ++q) {
        const int e = tid + q * kSimtThreads;
        if (PHASE == kPhaseGemm)
          Bs[e / kSimtBN][e % kSimtBN] = rb[st][q];
        else
          Bs[e % kSimtBK][e / kSimtBK] = rb[st][q];
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kSimtBK; ++k) {
        float a[TM], b[TN];
#pragma unroll
        for (int r = 0; r < TM; ++r) a[r] = As[k][ty * TM + r];
#pragma unroll
        for (int c = 0; c < TN; ++c) b[c] = Bs[k][tx * TN + c];
#pragma unroll
        for (int r = 0; r < TM; ++r)
#pragma unroll
          for (int c = 0; c < TN; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
      }
      __syncthreads();
    }
  }

  const int gm = B.slot_mat[slot];
  const MatDev md = p.mats[gm];
  float sc = 1.f;
  if (p.first) {
    const float s = p.s_norm[gm];
    sc = (PHASE == kPhaseGram) ? s * s : (PHASE == kPhaseGemm ? s : 1.f);
  }
  float* out = B.out ? B.out + slot * B.out_mat_stride : nullptr;
  const float* aux = B.aux ? B.aux + slot * B.aux_mat_stride : nullptr;
#pragma unroll
  for (int r = 0; r < TM; ++r) {
    const int i = row0 + ty * TM + r;
    if (i >= m) continue;
#pragma unroll
    for (int c = 0; c < TN; ++c) {
      const int j = col0 + tx * TN + c;
      if (j >= ncols) continue;
      float v = acc[r][c];
      if (PHASE == kPhaseGram || PHASE == kPhasePoly) {
        if (j < i) continue;
        v = (PHASE == kPhaseGram) ? v * sc
                                  : p.b * aux[(int64_t)i * B.aux_ld + j] + p.c * v + (i == j ? p.diag : 0.f);
        out[(int64_t)i * B.out_ld + j] = v;
        out[(int64_t)j * B.out_ld + i] = v;
      } else {
        v = ((p.a != 0.f ? p.a * aux[(int64_t)i * B.aux_ld + j] : 0.f) + v) * sc;
        if (!p.last) {
          out[(int64_t)i * B.out_ld + j] = v;
          continue;
        }
        const float step = p.lr * md.scale;
        const int64_t widx = md.transposed ? (int64_t)j * m + i : (int64_t)i * B.n + j;
        if (p.param_bf16) {
          __nv_bfloat16* w = reinterpret_cast<__nv_bfloat16*>(p.ptrs[gm]);
          w[widx] = __float2bfloat16_rn(__bfloat162float(w[widx]) - step * v);
        } else {
          float* w = reinterpret_cast<float*>(p.ptrs[gm]);
          w[widx] -= step * v;
        }
        if (p.capture != nullptr && md.cap_off >= 0) p.capture[md.cap_off + widx] = v;
      }
    }
  }
}

}  // namespace

cudaError_t launch_simt(int phase, const SimtParams& p, int grid, cudaStream_t s) {
  switch (phase) {
    case kPhaseGram:
      simt_ns_kernel<kPhaseGram><<<grid, kSimtThreads, 0, s>>>(p);
      break;
    case kPhasePoly:
      simt_ns_kernel<kPhasePoly><<<grid, kSimtThreads, 0, s>>>(p);
      break;
    case kPhaseGemm:
      simt_ns_kernel<kPhaseGemm><<<grid, kSimtThreads, 0, s>>>(p);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace dmuon
