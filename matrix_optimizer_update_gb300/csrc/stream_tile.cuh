// stream_tile.cuh - one 64 x 128 tile of the momentum pass, shared by the
// workspace pass (momentum.cu) and the pass without a workspace (noalloc.cu):
//   M <- mu*M + G;  U = G + mu*M (Nesterov) or U = M   (fp32, M in place)
// U goes through shared memory so that it can be written in the short-side
// orientation (transposed when rows > cols) with 16-byte stores.
#pragma once

#include <cuda_bf16.h>

#include "internal.h"

namespace dmuon {
namespace stile {

using bf16 = __nv_bfloat16;
using Tile = float[kTileR][kTileC + 1];

template <bool GB>
__device__ __forceinline__ float load1_grad(const void* g, int64_t e) {
  return GB ? __bfloat162float(reinterpret_cast<const bf16*>(g)[e]) : reinterpret_cast<const float*>(g)[e];
}

template <bool XB>
__device__ __forceinline__ void store8_x(void* dst, int64_t e, const float (&u)[8]) {
  if (XB) {
    uint4 o;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(u[2 * k], u[2 * k + 1]);
    *reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(dst) + e) = o;
  } else {
    float* d = reinterpret_cast<float*>(dst) + e;
    *reinterpret_cast<float4*>(d) = make_float4(u[0], u[1], u[2], u[3]);
    *reinterpret_cast<float4*>(d + 4) = make_float4(u[4], u[5], u[6], u[7]);
  }
}

template <bool XB>
__device__ __forceinline__ void store1_x(void* dst, int64_t e, float v) {
  if (XB)
    reinterpret_cast<bf16*>(dst)[e] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float*>(dst)[e] = v;
}

// Rows r0.. (64) and columns c0.. (128) of the stored rows x cols matrix:
// update M, leave U in `tile` (zero outside the matrix) and return this
// thread's sum of U^2. Each thread takes 4 consecutive columns of 8 rows;
// with vec (cols % 4 == 0 and aligned G, M) a full tile issues the loads of
// half its rows before their stores, then the other half's. Ends before the
// __syncthreads that publishes `tile`.
template <bool GB>
__device__ __forceinline__ float tile_update(const void* G, float* M, int rows, int cols, bool vec, int r0, int c0,
                                             float mu, bool nest, Tile& tile) {
  float ss = 0.f;
  const int cc = (threadIdx.x & 31) * 4;
  if (vec && r0 + kTileR <= rows && c0 + kTileC <= cols) {
    constexpr int kP = kTileR / 8;  // passes of 8 rows
    constexpr int kH = kP / 2;      // passes whose loads are in flight together
#pragma unroll
    for (int h = 0; h < kP; h += kH) {
      float g[kH][4];
      float4 m4[kH];
#pragma unroll
      for (int k = 0; k < kH; ++k) {
        const int rr = (h + k) * 8 + (threadIdx.x >> 5);
        const int64_t e = (int64_t)(r0 + rr) * cols + c0 + cc;
        if (GB) {
          const uint2 raw = __ldcs(reinterpret_cast<const uint2*>(reinterpret_cast<const bf16*>(G) + e));
          const __nv_bfloat162* hh = reinterpret_cast<const __nv_bfloat162*>(&raw);
          const float2 f0 = __bfloat1622float2(hh[0]), f1 = __bfloat1622float2(hh[1]);
          g[k][0] = f0.x, g[k][1] = f0.y, g[k][2] = f1.x, g[k][3] = f1.y;
        } else {
          const float4 f = __ldcs(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(G) + e));
          g[k][0] = f.x, g[k][1] = f.y, g[k][2] = f.z, g[k][3] = f.w;
        }
        m4[k] = __ldcs(reinterpret_cast<const float4*>(M + e));
      }
#pragma unroll
      for (int k = 0; k < kH; ++k) {
        const int rr = (h + k) * 8 + (threadIdx.x >> 5);
        const int64_t e = (int64_t)(r0 + rr) * cols + c0 + cc;
        float mv[4] = {m4[k].x, m4[k].y, m4[k].z, m4[k].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          mv[q] = fmaf(mu, mv[q], g[k][q]);
          const float uu = nest ? fmaf(mu, mv[q], g[k][q]) : mv[q];
          ss = fmaf(uu, uu, ss);
          tile[rr][cc + q] = uu;
        }
        __stcs(reinterpret_cast<float4*>(M + e), make_float4(mv[0], mv[1], mv[2], mv[3]));
      }
    }
  } else {
    for (int pass = 0; pass < kTileR / 8; ++pass) {
      const int rr = pass * 8 + (threadIdx.x >> 5);
      const int r = r0 + rr, c = c0 + cc;
      float uu[4] = {0.f, 0.f, 0.f, 0.f};
      if (r < rows) {
        const int64_t e = (int64_t)r * cols + c;
        for (int q = 0; q < 4 && c + q < cols; ++q) {
          const float g = load1_grad<GB>(G, e + q);
          const float mv = fmaf(mu, M[e + q], g);
          M[e + q] = mv;
          uu[q] = nest ? fmaf(mu, mv, g) : mv;
          ss = fmaf(uu[q], uu[q], ss);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) tile[rr][cc + q] = uu[q];
    }
  }
  return ss;
}

// Write the tile's U (after a __syncthreads) to X with row pitch x_ld:
// transposed, X(c, r) at c*x_ld + r with 8 consecutive r per thread (16-byte
// stores when vec); else X(r, c) at r*x_ld + c with 4 consecutive c per
// thread (one 8- or 16-byte store when vec and x_ld % 4 == 0). vec requires X
// 16-byte aligned.
template <bool XB>
__device__ __forceinline__ void tile_store(void* X, int64_t x_ld, int rows, int cols, bool transposed, bool vec,
                                           int r0, int c0, const Tile& tile) {
  if (transposed) {
#pragma unroll
    for (int pass = 0; pass < kTileC / 32; ++pass) {
      const int jj = pass * 32 + (threadIdx.x >> 3);
      const int ii = (threadIdx.x & 7) * 8;
      const int c = c0 + jj, r = r0 + ii;
      if (c >= cols) continue;
      const int64_t e = (int64_t)c * x_ld + r;
      float v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = tile[ii + q][jj];
      if (vec && r + 8 <= rows) {
        store8_x<XB>(X, e, v);
      } else {
        for (int q = 0; q < 8 && r + q < rows; ++q) store1_x<XB>(X, e + q, v[q]);
      }
    }
  } else {
#pragma unroll 2
    for (int pass = 0; pass < kTileR / 8; ++pass) {
      const int rr = pass * 8 + (threadIdx.x >> 5);
      const int cc = (threadIdx.x & 31) * 4;
      const int r = r0 + rr, c = c0 + cc;
      if (r >= rows) continue;
      const int64_t e = (int64_t)r * x_ld + c;
      if (vec && c + 4 <= cols && (x_ld & 3) == 0) {  // 4 consecutive elements in one store
        const float4 f = make_float4(tile[rr][cc], tile[rr][cc + 1], tile[rr][cc + 2], tile[rr][cc + 3]);
        if (XB) {
          uint2 o;
          __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
          h[0] = __floats2bfloat162_rn(f.x, f.y);
          h[1] = __floats2bfloat162_rn(f.z, f.w);
          *reinterpret_cast<uint2*>(reinterpret_cast<bf16*>(X) + e) = o;
        } else {
          *reinterpret_cast<float4*>(reinterpret_cast<float*>(X) + e) = f;
        }
      } else {
        for (int q = 0; q < 4 && c + q < cols; ++q) store1_x<XB>(X, e + q, tile[rr][cc + q]);
      }
    }
  }
}

}  // namespace stile
}  // namespace dmuon
