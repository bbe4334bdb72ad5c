// momentum.cu - the streaming pass in front of Newton-Schulz.
//
// One launch over every matrix of the batch:
//   M <- mu*M + G;  U = G + mu*M (Nesterov) or U = M      (fp32 math, M in place)
//   U is written to the matrix's workspace slot in the compute dtype, already
//   in the short-side orientation (transposed through shared memory when
//   rows > cols), and each work unit writes its fp32 partial of sum(U^2).
// A second, small launch (norm_finalize_kernel) adds each matrix's partials
// in a fixed order in fp64 and stores s = 1 / (sqrt(sum) + eps): the sum is
// deterministic, and the streaming pass carries no fence or atomic per unit
// (a ticket per unit, with the fence it needs, cost about a third of the
// pass's bandwidth).
// The Newton-Schulz kernels fold s into their first-step epilogues, so U is
// never rescaled in HBM. ("momentum-aggregated gradients", "DMuon: Efficient
// Distributed Muon Training with Near-Adam Overhead", gist.science summary
// section 1.)
//
// HBM-bound: per element it reads G (2 or 4 B) and M (4 B) and writes M (4 B)
// and U (2 or 4 B). Work units: 8192 contiguous elements when the stored
// matrix and its slot share a layout (rows <= cols, cols % 8 == 0), else
// 64 x 128 tiles of the stored matrix.
#include <cuda_bf16.h>

#include "internal.h"
#include "stream_tile.cuh"

namespace dmuon {
namespace {

using bf16 = __nv_bfloat16;
using stile::load1_grad;
using stile::store1_x;
using stile::store8_x;

__device__ __forceinline__ int find_matrix(const int64_t* unit_begin, int n_mats, int64_t u) {
  int lo = 0, hi = n_mats;  // unit_begin[lo] <= u < unit_begin[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (unit_begin[mid] <= u)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

template <bool GB>
__device__ __forceinline__ void load8_grad(const void* g, int64_t e, float (&x)[8]) {
  if (GB) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(reinterpret_cast<const bf16*>(g) + e));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      x[2 * k] = f.x;
      x[2 * k + 1] = f.y;
    }
  } else {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(g) + e));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(g) + e + 4));
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
  }
}


// 8 consecutive U values from the slot (bf16 or fp32), as fp32.
__device__ __forceinline__ void load8_x(const char* X, int64_t e, float (&x)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const bf16*>(X) + e);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __bfloat1622float2(h[k]);
    x[2 * k] = f.x;
    x[2 * k + 1] = f.y;
  }
}




__device__ __forceinline__ double block_sum_d(double v, double* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0)
    for (int k = 0; k < kStreamThreads / 32; ++k) t += red[k];
  return t;
}

// Resident CTAs per SM the momentum kernel is compiled for: more warps keep its loads in flight when
// the SM clock drops (as it does under the power limit right after the tensor-core phases).
constexpr int kMomentumCtasPerSm = 4;

template <bool GB, bool XB>
__global__ void __launch_bounds__(kStreamThreads, kMomentumCtasPerSm) momentum_kernel(const __grid_constant__ StreamParams p) {
  __shared__ float tileU[kTileR][kTileC + 1];
  const float mu = p.mu;
  const bool nest = p.nesterov != 0;

  for (int64_t u = blockIdx.x; u < p.n_units; u += gridDim.x) {
    const int mat = find_matrix(p.unit_begin, p.n_mats, u);
    const MatDev md = p.mats[mat];
    const int64_t local = u - md.unit_begin;
    const void* G = reinterpret_cast<const void*>(p.ptrs[p.n_mats + mat]);
    float* M = reinterpret_cast<float*>(p.ptrs[2 * p.n_mats + mat]);
    void* X = p.ws + md.x0_off;
    float ss = 0.f;

    if (md.flat) {
      const int64_t total = (int64_t)md.rows * md.cols;
      const int64_t e0 = local * kFlatUnit;
      const int64_t e1 = min(e0 + kFlatUnit, total);
      constexpr int kV = kFlatUnit / (8 * kStreamThreads);  // 8-element vectors per thread
      constexpr int kH = 2;                                   // of which in flight together
      if (e0 + kFlatUnit <= total) {
        // full unit, kH vectors at a time: every load of a group is issued before its stores, and
        // the registers this takes leave room for 4 CTAs per SM
#pragma unroll
        for (int h = 0; h < kV; h += kH) {
          float g[kH][8];
          float4 m0[kH], m1[kH];
#pragma unroll
          for (int k = 0; k < kH; ++k) {
            const int64_t e = e0 + (int64_t)(threadIdx.x + (h + k) * kStreamThreads) * 8;
            load8_grad<GB>(G, e, g[k]);
            m0[k] = __ldcs(reinterpret_cast<const float4*>(M + e));
            m1[k] = __ldcs(reinterpret_cast<const float4*>(M + e + 4));
          }
#pragma unroll
          for (int k = 0; k < kH; ++k) {
            const int64_t e = e0 + (int64_t)(threadIdx.x + (h + k) * kStreamThreads) * 8;
            float mv[8] = {m0[k].x, m0[k].y, m0[k].z, m0[k].w, m1[k].x, m1[k].y, m1[k].z, m1[k].w};
            float uu[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              mv[q] = fmaf(mu, mv[q], g[k][q]);
              uu[q] = nest ? fmaf(mu, mv[q], g[k][q]) : mv[q];
              ss = fmaf(uu[q], uu[q], ss);
            }
            __stcs(reinterpret_cast<float4*>(M + e), make_float4(mv[0], mv[1], mv[2], mv[3]));
            __stcs(reinterpret_cast<float4*>(M + e + 4), make_float4(mv[4], mv[5], mv[6], mv[7]));
            store8_x<XB>(X, e, uu);
          }
        }
      } else {
        for (int64_t q = e0 + threadIdx.x; q < e1; q += kStreamThreads) {
          const float g = load1_grad<GB>(G, q);
          const float mv = fmaf(mu, M[q], g);
          const float uu = nest ? fmaf(mu, mv, g) : mv;
          M[q] = mv;
          store1_x<XB>(X, q, uu);
          ss = fmaf(uu, uu, ss);
        }
      }
    } else {
      const int r0 = static_cast<int>(local / md.tiles_c) * kTileR, c0 = static_cast<int>(local % md.tiles_c) * kTileC;
      ss = stile::tile_update<GB>(G, M, md.rows, md.cols, md.vec_ok != 0, r0, c0, mu, nest, tileU);
      __syncthreads();
      stile::tile_store<XB>(X, md.x_ld, md.rows, md.cols, md.transposed != 0, true, r0, c0, tileU);
    }

    // the unit's partial sums of squares, one per warp (the sum over the matrix is the finalize
    // launch's): no barrier between units
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) p.partial[u * kPartialsPerUnit + (threadIdx.x >> 5)] = ss;
    if (!md.flat) __syncthreads();  // tileU is refilled by the next unit
  }
}

// s = 1 / (||U||_F + eps) per matrix from its units' partials, added in fp64
// in a fixed order (thread t takes partials t, t + 256, ...; then a fixed
// tree), so the result does not depend on the launch configuration.
__global__ void __launch_bounds__(kStreamThreads) norm_finalize_kernel(const __grid_constant__ StreamParams p) {
  __shared__ double redd[kStreamThreads / 32];
  for (int mat = blockIdx.x; mat < p.n_mats; mat += gridDim.x) {
    const MatDev md = p.mats[mat];
    double acc = 0.0;
    for (int64_t k = threadIdx.x; k < md.unit_count * kPartialsPerUnit; k += kStreamThreads)
      acc += static_cast<double>(p.partial[md.unit_begin * kPartialsPerUnit + k]);
    const double tot = block_sum_d(acc, redd);
    if (threadIdx.x == 0) {
      const float nrm = static_cast<float>(sqrt(tot));
      if (!isfinite(nrm)) atomicOr(p.status, DMUON_DEV_NONFINITE_NORM);
      p.s_norm[mat] = 1.0f / (nrm + p.eps);
    }
    __syncthreads();  // redd is reused by the next matrix
  }
}

// ns_steps == 0: W -= lr * scale * s * U (U read back from the slot), one
// rounding into W, the same arithmetic per element on every path. Flat units
// with bf16 weights and U move 8 elements per 16-byte access; tiles of
// transposed matrices read U^T along its rows, turn it through shared memory
// and update W rows 8 elements at a time; everything else goes element by
// element.
__device__ __forceinline__ float w_load(const void* W, bool wb, int64_t e) {
  return wb ? __bfloat162float(reinterpret_cast<const bf16*>(W)[e]) : reinterpret_cast<const float*>(W)[e];
}
__device__ __forceinline__ void w_store(void* W, bool wb, int64_t e, float v) {
  if (wb)
    reinterpret_cast<bf16*>(W)[e] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float*>(W)[e] = v;
}

// 8 consecutive bf16 weights w[e..e+7] -= f * x[0..7].
__device__ __forceinline__ void w_update8_bf16(bf16* w, int64_t e, float f, const float (&x)[8]) {
  uint4 u = *reinterpret_cast<const uint4*>(w + e);
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float2 v = __bfloat1622float2(h[k]);
    v.x -= f * x[2 * k];
    v.y -= f * x[2 * k + 1];
    h[k] = __floats2bfloat162_rn(v.x, v.y);
  }
  *reinterpret_cast<uint4*>(w + e) = u;
}

template <bool XB>
__global__ void __launch_bounds__(kStreamThreads) update0_kernel(const __grid_constant__ StreamParams p) {
  __shared__ float tileT[kTileC][kTileR + 1];  // U^T tile of a transposed matrix: [column][row]
  for (int64_t u = blockIdx.x; u < p.n_units; u += gridDim.x) {
    const int mat = find_matrix(p.unit_begin, p.n_mats, u);
    const MatDev md = p.mats[mat];
    const int64_t local = u - md.unit_begin;
    const float sn = p.s_norm[mat];
    const float f = p.lr * md.scale * sn;
    const char* X = p.ws + md.x0_off;
    void* W = reinterpret_cast<void*>(p.ptrs[mat]);
    const bool wb = p.param_bf16 != 0;
    float* cap = (p.capture != nullptr && md.cap_off >= 0) ? p.capture + md.cap_off : nullptr;
    if (md.flat) {
      const int64_t total = (int64_t)md.rows * md.cols;
      const int64_t e0 = local * kFlatUnit, e1 = min(e0 + kFlatUnit, total);
      if (XB && wb && e1 - e0 == kFlatUnit) {
        constexpr int kV = kFlatUnit / (8 * kStreamThreads);
#pragma unroll
        for (int k = 0; k < kV; ++k) {
          const int64_t e = e0 + (int64_t)(threadIdx.x + k * kStreamThreads) * 8;
          float x[8];
          load8_x(X, e, x);
          w_update8_bf16(reinterpret_cast<bf16*>(W), e, f, x);
          if (cap != nullptr)
#pragma unroll
            for (int q = 0; q < 8; ++q) cap[e + q] = sn * x[q];
        }
      } else {
        for (int64_t q = e0 + threadIdx.x; q < e1; q += kStreamThreads) {
          const float x = XB ? __bfloat162float(reinterpret_cast<const bf16*>(X)[q]) : reinterpret_cast<const float*>(X)[q];
          w_store(W, wb, q, w_load(W, wb, q) - f * x);
          if (cap != nullptr) cap[q] = sn * x;
        }
      }
      continue;
    }
    const int r0 = static_cast<int>(local / md.tiles_c) * kTileR;
    const int c0 = static_cast<int>(local % md.tiles_c) * kTileC;
    const bool full = r0 + kTileR <= md.rows && c0 + kTileC <= md.cols;
    if (XB && wb && md.transposed && full && (md.cols & 7) == 0 && (md.x_ld & 7) == 0) {
      // U^T rows c0..c0+127 (slot row pitch x_ld), 64 consecutive r each: 8 r per thread and vector
#pragma unroll
      for (int k = 0; k < (kTileC * kTileR / 8) / kStreamThreads; ++k) {
        const int v = threadIdx.x + k * kStreamThreads;
        const int cc = v / (kTileR / 8), rr = (v % (kTileR / 8)) * 8;
        float x[8];
        load8_x(X, (int64_t)(c0 + cc) * md.x_ld + r0 + rr, x);
#pragma unroll
        for (int q = 0; q < 8; ++q) tileT[cc][rr + q] = x[q];
      }
      __syncthreads();
      // W rows r0..r0+63, 8 consecutive columns per thread and vector
#pragma unroll
      for (int k = 0; k < (kTileR * kTileC / 8) / kStreamThreads; ++k) {
        const int v = threadIdx.x + k * kStreamThreads;
        const int rr = v / (kTileC / 8), cc = (v % (kTileC / 8)) * 8;
        float x[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = tileT[cc + q][rr];
        const int64_t e = (int64_t)(r0 + rr) * md.cols + c0 + cc;
        w_update8_bf16(reinterpret_cast<bf16*>(W), e, f, x);
        if (cap != nullptr)
#pragma unroll
          for (int q = 0; q < 8; ++q) cap[e + q] = sn * x[q];
      }
      __syncthreads();  // tileT is refilled by the next unit
      continue;
    }
    for (int q = threadIdx.x; q < kTileR * kTileC; q += kStreamThreads) {
      const int r = r0 + q / kTileC, c = c0 + q % kTileC;
      if (r >= md.rows || c >= md.cols) continue;
      const int64_t widx = (int64_t)r * md.cols + c;
      const int64_t xidx = md.transposed ? (int64_t)c * md.x_ld + r : (int64_t)r * md.x_ld + c;
      const float x = XB ? __bfloat162float(reinterpret_cast<const bf16*>(X)[xidx])
                         : reinterpret_cast<const float*>(X)[xidx];
      w_store(W, wb, widx, w_load(W, wb, widx) - f * x);
      if (cap != nullptr) cap[widx] = sn * x;
    }
  }
}

}  // namespace

int momentum_blocks_per_sm(int grad_bf16, int x_bf16) {
  int n = 0;
  cudaError_t e;
  if (grad_bf16 && x_bf16)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, momentum_kernel<true, true>, kStreamThreads, 0);
  else if (grad_bf16)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, momentum_kernel<true, false>, kStreamThreads, 0);
  else if (x_bf16)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, momentum_kernel<false, true>, kStreamThreads, 0);
  else
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, momentum_kernel<false, false>, kStreamThreads, 0);
  return (e == cudaSuccess && n > 0) ? n : 1;
}

cudaError_t launch_momentum(const StreamParams& p, int grid, cudaStream_t s) {
  if (p.grad_bf16 && p.x_bf16)
    momentum_kernel<true, true><<<grid, kStreamThreads, 0, s>>>(p);
  else if (p.grad_bf16)
    momentum_kernel<true, false><<<grid, kStreamThreads, 0, s>>>(p);
  else if (p.x_bf16)
    momentum_kernel<false, true><<<grid, kStreamThreads, 0, s>>>(p);
  else
    momentum_kernel<false, false><<<grid, kStreamThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_norm_finalize(const StreamParams& p, int grid, cudaStream_t s) {
  norm_finalize_kernel<<<grid, kStreamThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_update0(const StreamParams& p, int grid, cudaStream_t s) {
  if (p.x_bf16)
    update0_kernel<true><<<grid, kStreamThreads, 0, s>>>(p);
  else
    update0_kernel<false><<<grid, kStreamThreads, 0, s>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ status readout
// Copies the device status word to mapped, page-locked host memory and clears it. A kernel rather
// than a copy: a copy of the word would queue on the copy engines behind whatever large transfers
// other streams have in flight (a step's weights going back to the host, say).
__global__ void status_readout_kernel(unsigned* status, volatile unsigned* host_out) {
  const unsigned v = *status;
  *status = 0u;
  *host_out = v;
  __threadfence_system();
}

cudaError_t launch_status_readout(unsigned* status, unsigned* host_out_dev, cudaStream_t s) {
  status_readout_kernel<<<1, 1, 0, s>>>(status, host_out_dev);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ tuning data
// Fills n bf16 elements (n a multiple of 8, dst 16-byte aligned) with values in [-1/64, 1/64) from a
// counter-based hash of the element index: operands for bind-time tuning probes, so that the tensor
// cores are timed on data whose bits toggle like real operands (on zeros they draw less power and
// run at a clock the real step does not get). Not part of the update's arithmetic.
__global__ void __launch_bounds__(kStreamThreads) tuning_fill_kernel(uint4* dst, int64_t n8, uint32_t seed) {
  for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < n8; v += (int64_t)gridDim.x * blockDim.x) {
    uint32_t h[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t x = static_cast<uint32_t>(v) * 4u + q + seed * 0x9E3779B9u;
      x ^= x >> 16;
      x *= 0x7FEB352Du;
      x ^= x >> 15;
      x *= 0x846CA68Bu;
      x ^= x >> 16;
      // two bf16 values from the hash's halves: sign, exponent 2^-7..2^-14, 7 mantissa bits
      const uint32_t lo = (x & 0x807Fu) | ((0x78u - ((x >> 8) & 7u)) << 7);
      const uint32_t hi = ((x >> 16) & 0x807Fu) | ((0x78u - ((x >> 24) & 7u)) << 7);
      h[q] = lo | (hi << 16);
    }
    dst[v] = make_uint4(h[0], h[1], h[2], h[3]);
  }
}

cudaError_t launch_tuning_fill(void* dst, int64_t bytes, uint32_t seed, int grid, cudaStream_t s) {
  const int64_t n8 = bytes / 16;
  if (n8 <= 0) return cudaSuccess;
  tuning_fill_kernel<<<grid, kStreamThreads, 0, s>>>(reinterpret_cast<uint4*>(dst), n8, seed);
  return cudaGetLastError();
}

}  // namespace dmuon
