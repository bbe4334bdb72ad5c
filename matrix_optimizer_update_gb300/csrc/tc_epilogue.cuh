// tc_epilogue.cuh - epilogue of the Newton-Schulz tensor-core kernels: one
// 32-column chunk of one accumulator row (fp32, read from TMEM) turned into
// the phase's output (symmetric store with mirror, polynomial term, a*X term,
// or the fused weight update).
#pragma once

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace dmuon {
namespace epi {

using bf16 = __nv_bfloat16;

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

// STREAM: mark the stores evict-first (st.global.cs). The symmetric products'
// outputs (A, B) are read again only by the next launch, after far more than
// the L2 holds has streamed through it; marking them keeps the operand rows
// that other CTAs are still reading in L2.
template <bool STREAM>
__device__ __forceinline__ void store_row_bf16(bf16* dst, int j0, int jmin, int lim, const float (&v)[32]) {
  if (j0 >= jmin && j0 + 32 <= lim) {
    uint4* d4 = reinterpret_cast<uint4*>(dst + j0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 u;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
      for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(v[q * 8 + 2 * e], v[q * 8 + 2 * e + 1]);
      if (STREAM)
        __stcs(d4 + q, u);
      else
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

__device__ __forceinline__ void unpack_bf16x32(const uint4 (&u)[4], float (&x)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u[q]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      x[q * 8 + 2 * e] = f.x;
      x[q * 8 + 2 * e + 1] = f.y;
    }
  }
}

// ---- staging of a 32 x 32 bf16 box for a TMA store (64-byte rows, 64-byte
// swizzle: the 16-byte piece c of row r sits at piece c ^ ((r >> 1) & 3)).
// Lane r holds row r's 32 values (columns 0..31 of the box).
__device__ __forceinline__ void stage_row_sw64(uint8_t* box, int r, const float (&v)[32]) {
  uint8_t* row = box + r * 64;
  const int x = (r >> 1) & 3;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(v[c * 8 + 2 * e], v[c * 8 + 2 * e + 1]);
    *reinterpret_cast<uint4*>(row + ((c ^ x) << 4)) = u;
  }
}

// The transpose: lane r's value k goes to row k, column r, so that the box
// stored at (x = row origin, y = column origin) is the mirror image.
__device__ __forceinline__ void stage_col_sw64(uint8_t* box, int r, const float (&v)[32]) {
  const int c = r >> 3, off = (r & 7) * 2;
#pragma unroll
  for (int k = 0; k < 32; ++k)
    *reinterpret_cast<bf16*>(box + k * 64 + ((c ^ ((k >> 1) & 3)) << 4) + off) = __float2bfloat16_rn(v[k]);
}

// Poly's b*A operand of one chunk as this lane's row (a[k] = A[i][j0 + k]).
// `blk` holds the chunk's 32 x 32 block of A as fetched (lane: row
// (lane >> 2) + 8u, piece lane & 3); it is turned into rows through `box`
// (64-byte swizzled rows), which must be free. Chunks past the matrix's
// right edge read their row directly.
__device__ __forceinline__ void poly_aux_rows(const TcBucket& B, const bf16* abase, int i, int j0, int lane,
                                              const uint4 (&blk)[4], uint8_t* box, float (&a)[32]) {
  if (j0 + 32 <= B.m) {
    const int i0 = i - lane;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int rr = (lane >> 2) + 8 * u;
      if (i0 + rr < B.m) *reinterpret_cast<uint4*>(box + rr * 64 + (((lane & 3) ^ ((rr >> 1) & 3)) << 4)) = blk[u];
    }
    __syncwarp();
    uint4 r[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) r[c] = *reinterpret_cast<const uint4*>(box + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4));
    unpack_bf16x32(r, a);
    __syncwarp();  // every lane has its row before the box is reused
  } else if (i < B.m) {
    load_row_bf16(abase + (int64_t)i * B.aux_ld, j0, B.m, a);
  } else {
#pragma unroll
    for (int k = 0; k < 32; ++k) a[k] = 0.f;
  }
}

// Values of a chunk strictly above the diagonal (no diagonal term): gram
// s^2-scaled (sc), poly b*A + c*(A A^T).
template <int PHASE>
__device__ __forceinline__ void sym_values(const TcParams& p, float sc, const float (&a)[32], float (&v)[32]) {
#pragma unroll
  for (int k = 0; k < 32; ++k) v[k] = (PHASE == kPhasePoly) ? p.b * a[k] + p.c * v[k] : v[k] * sc;
}

// A chunk on the diagonal: values with the diagonal term, then the own row
// for columns j >= i and the mirror (j, i) for j > i, per element.
template <int PHASE>
__device__ __forceinline__ void sym_diag_chunk(const TcParams& p, const TcBucket& B, int slot, int i, int j0,
                                               float sc, const float (&a)[32], float (&v)[32]) {
  const int m = B.m;
  if (i >= m) return;
#pragma unroll
  for (int k = 0; k < 32; ++k)
    v[k] = (PHASE == kPhasePoly) ? p.b * a[k] + p.c * v[k] + (j0 + k == i ? p.diag : 0.f) : v[k] * sc;
  bf16* out = reinterpret_cast<bf16*>(B.out + slot * B.out_mat_stride);
  store_row_bf16<true>(out + (int64_t)i * B.out_ld, j0, i, m, v);
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    const int j = j0 + k;
    if (j > i && j < m)
      __stcs(reinterpret_cast<unsigned short*>(out + (int64_t)j * B.out_ld + i),
             __bfloat16_as_ushort(__float2bfloat16_rn(v[k])));
  }
}

// ---- last step on bf16 weights: W -= lr * scale * X, one 32 x 32 chunk of X
// (rows i0.., columns j0.. in the iteration's orientation) at a time. The
// chunk's W block is copied into shared memory ahead of time (cp.async, 16
// bytes per lane and row segment), updated there from the fp32 X each lane
// holds (one rounding per element), and written back by one TMA store of the
// box through the matrix's own tensor map (p.wmaps), so the warp does not wait
// on the stores and the TMA unit sees one operation per chunk. Box layout: 32
// rows of 64 bytes, piece c of row r at piece c ^ ((r >> 1) & 3) (the 64-byte
// swizzle of the map). Box rows are W rows: i0 + r for W = m x n, j0 + r for
// W = n x m (stored transposed).

// Whole chunk inside W with 16-byte aligned row segments (else the per-row path).
__device__ __forceinline__ bool w_chunk_vec(const MatDev& md, int m, int n, int i0, int j0) {
  return md.transposed ? ((m & 7) == 0 && i0 + 32 <= m && j0 < n) : ((n & 7) == 0 && j0 + 32 <= n && i0 < m);
}

// Offset of the 16-byte W segment that lane copies for box row rr, or -1 past W's edge.
__device__ __forceinline__ int64_t w_seg(const MatDev& md, int m, int n, int i0, int j0, int rr, int pc) {
  if (md.transposed) return (j0 + rr < n) ? (int64_t)(j0 + rr) * m + i0 + 8 * pc : -1;
  return (i0 + rr < m) ? (int64_t)(i0 + rr) * n + j0 + 8 * pc : -1;
}

__device__ __forceinline__ uint8_t* box_piece(uint8_t* box, int r, int c) {
  return box + r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
}

__device__ __forceinline__ void w_chunk_fetch(const TcParams& p, const MatDev& md, int gm, int m, int n, int i0,
                                              int j0, int lane, uint8_t* box) {
  if (!w_chunk_vec(md, m, n, i0, j0)) return;
  const bf16* W = reinterpret_cast<const bf16*>(p.ptrs[gm]);
  const int pc = lane & 3;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int rr = (lane >> 2) + 8 * u;
    const int64_t off = w_seg(md, m, n, i0, j0, rr, pc);
    if (off >= 0) ptx::cp_async16(box_piece(box, rr, pc), W + off);
  }
}

// The copies of this chunk must have landed (cp_async_wait + __syncwarp) before
// the call. Lane 0 commits one bulk group (the box's store to W); the box is
// free again once that group has read it (lane 0 bulk_wait_read + __syncwarp).
__device__ __forceinline__ void w_chunk_apply(const TcParams& p, const MatDev& md, int gm, int m, int n, int i0,
                                              int j0, int lane, const float (&v)[32], uint8_t* box) {
  const float step = p.lr * md.scale;
  if (!md.transposed) {  // box row = this lane's row
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4* pp = reinterpret_cast<uint4*>(box_piece(box, lane, c));
      uint4 u = *pp;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float2 f = __bfloat1622float2(h[e]);
        f.x -= step * v[8 * c + 2 * e];
        f.y -= step * v[8 * c + 2 * e + 1];
        h[e] = __floats2bfloat162_rn(f.x, f.y);
      }
      *pp = u;
    }
  } else {  // box column = this lane's row: element (k, lane)
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      bf16* e = reinterpret_cast<bf16*>(box_piece(box, k, lane >> 3)) + (lane & 7);
      *e = __float2bfloat16_rn(__bfloat162float(*e) - step * v[k]);
    }
  }
  ptx::fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {  // W rows past the matrix's edge are clipped by the map
    if (md.transposed) ptx::tma_store_2d(&p.wmaps[gm], box, i0, j0);
    else ptx::tma_store_2d(&p.wmaps[gm], box, j0, i0);
    ptx::bulk_commit();
  }
}

// The linear term and the normalisation of the last product's chunk: v = (a x + v) s.
__device__ __forceinline__ void gemm_values(const TcParams& p, const TcBucket& B, int slot, int i, int j0, float sc,
                                            float (&v)[32], const uint4 (&pre)[4]) {
  if (p.a != 0.f && i < B.m) {
    float x[32];
    if (j0 + 32 <= B.n) {
      unpack_bf16x32(pre, x);
    } else {
      const bf16* X = reinterpret_cast<const bf16*>(B.aux + slot * B.aux_mat_stride) + (int64_t)i * B.aux_ld;
      load_row_bf16(X, j0, B.n, x);
    }
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = (p.a * x[k] + v[k]) * sc;
  } else {
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] *= sc;
  }
}

__device__ __forceinline__ void capture_row(const TcParams& p, const MatDev& md, int i, int j0, int m, int n,
                                            const float (&v)[32]) {
  if (p.capture == nullptr || md.cap_off < 0 || i >= m) return;
  float* cap = p.capture + md.cap_off;
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    const int j = j0 + k;
    if (j < n) cap[md.transposed ? (int64_t)j * m + i : (int64_t)i * n + j] = v[k];
  }
}

// Epilogue of one 32-column chunk of one accumulator row. `pre` holds the
// chunk's bf16 operand of the linear term (A for poly, X_k for gemm) when the
// whole chunk lies inside the matrix (fetched before the accumulator was
// ready); otherwise the operand is read here element by element.
template <int PHASE>
__device__ __forceinline__ void epilogue_chunk(const TcParams& p, const TcBucket& B, const MatDev& md, int gm,
                                               int slot, int i, int j0, float sc, float (&v)[32],
                                               const uint4 (&pre)[4]) {
  if (PHASE == kPhaseGram || PHASE == kPhasePoly) {
    const int m = B.m;
    if (i >= m || j0 >= m || j0 + 31 < i) return;  // nothing of the upper triangle here
    bf16* out = reinterpret_cast<bf16*>(B.out + slot * B.out_mat_stride);
    if (PHASE == kPhasePoly) {
      float a[32];
      if (j0 + 32 <= m) {
        unpack_bf16x32(pre, a);
      } else {
        const bf16* A = reinterpret_cast<const bf16*>(B.aux + slot * B.aux_mat_stride) + (int64_t)i * B.aux_ld;
        load_row_bf16(A, j0, m, a);
      }
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = p.b * a[k] + p.c * v[k] + (j0 + k == i ? p.diag : 0.f);
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] *= sc;
    }
    // own row: columns j >= i; mirror: (j, i) for j > i (coalesced across the warp's 32 rows)
    store_row_bf16<true>(out + (int64_t)i * B.out_ld, j0, i, m, v);
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const int j = j0 + k;
      if (j > i && j < m)
        __stcs(reinterpret_cast<unsigned short*>(out + (int64_t)j * B.out_ld + i),
               __bfloat16_as_ushort(__float2bfloat16_rn(v[k])));
    }
  } else {  // gemm
    const int m = B.m, n = B.n;
    if (i >= m || j0 >= n) return;
    float x[32];
    if (p.a == 0.f) {
#pragma unroll
      for (int k = 0; k < 32; ++k) x[k] = 0.f;
    } else if (j0 + 32 <= n) {
      unpack_bf16x32(pre, x);
    } else {
      const bf16* X = reinterpret_cast<const bf16*>(B.aux + slot * B.aux_mat_stride) + (int64_t)i * B.aux_ld;
      load_row_bf16(X, j0, n, x);
    }
    #pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = (p.a * x[k] + v[k]) * sc;
    if (!p.last) {
      bf16* out = reinterpret_cast<bf16*>(B.out + slot * B.out_mat_stride) + (int64_t)i * B.out_ld;
      store_row_bf16<false>(out, j0, 0, n, v);
      return;
    }
    // W update: every load of the chunk is issued before any store, so the
    // read-modify-write costs one memory round trip, not 32 dependent ones.
    const float step = p.lr * md.scale;
    void* W = reinterpret_cast<void*>(p.ptrs[gm]);
    if (!md.transposed) {  // W is m x n, row i
      if (p.param_bf16) {
        bf16* w = reinterpret_cast<bf16*>(W) + (int64_t)i * n;
        if (j0 + 32 <= n && (n & 7) == 0) {
          uint4* w4 = reinterpret_cast<uint4*>(w + j0);
          uint4 u[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) u[q] = w4[q];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u[q]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float2 f = __bfloat1622float2(h[e]);
              f.x -= step * v[q * 8 + 2 * e];
              f.y -= step * v[q * 8 + 2 * e + 1];
              h[e] = __floats2bfloat162_rn(f.x, f.y);
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) w4[q] = u[q];
        } else {
          float old[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) old[k] = (j0 + k < n) ? __bfloat162float(w[j0 + k]) : 0.f;
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (j0 + k < n) w[j0 + k] = __float2bfloat16_rn(old[k] - step * v[k]);
        }
      } else {
        float* w = reinterpret_cast<float*>(W) + (int64_t)i * n;
        float old[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) old[k] = (j0 + k < n) ? w[j0 + k] : 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (j0 + k < n) w[j0 + k] = old[k] - step * v[k];
      }
    } else {  // W is n x m: element (j, i); consecutive lanes touch consecutive i
      // two halves of 16 columns keep the live addresses and values in registers
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int jh = j0 + hh * 16;
        if (p.param_bf16) {
          bf16* w = reinterpret_cast<bf16*>(W) + (int64_t)jh * m + i;
          float old[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) old[k] = (jh + k < n) ? __bfloat162float(w[k * m]) : 0.f;
#pragma unroll
          for (int k = 0; k < 16; ++k)
            if (jh + k < n) w[k * m] = __float2bfloat16_rn(old[k] - step * v[hh * 16 + k]);
        } else {
          float* w = reinterpret_cast<float*>(W) + (int64_t)jh * m + i;
          float old[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) old[k] = (jh + k < n) ? w[k * m] : 0.f;
#pragma unroll
          for (int k = 0; k < 16; ++k)
            if (jh + k < n) w[k * m] = old[k] - step * v[hh * 16 + k];
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

// ---- the per-tile epilogue of one epilogue warp, shared by the one-SM and
// the two-SM kernels. The warp owns 32 accumulator rows (its TMEM lane
// quarter) and kChunks 32-column chunks of them: output rows i0 + lane,
// columns jbase + 32 ch (tbase: the chunks' TMEM address). wait_acc() waits
// for the accumulator (false when the CTA gave up). Before that wait the
// operands that do not depend on the accumulator are fetched: the linear
// term's first two chunks, and on the last step the first two W blocks. Then
// each chunk is drained and written: through a staged TMA box (X', symmetric
// chunks above the diagonal, with the mirror image), through the staged W
// update, or per row (diagonal chunks, matrix edges, fp32 weights, a*X in
// the epilogue). stg: this warp's two staging boxes; nbox counts the X' boxes
// (their double buffering spans tiles).
constexpr int kStageBox = 32 * 32 * 2;  // one 32 x 32 bf16 box staged for a TMA store

template <int PHASE, int kChunks, class WaitAcc>
__device__ __forceinline__ bool epilogue_tile(const TcParams& p, const TcBucket& B, const int4& it, int i0, int jbase,
                                              uint32_t tbase, int lane, uint8_t* stg, uint32_t& nbox,
                                              WaitAcc&& wait_acc) {
  const int i = i0 + lane;
  // The linear term's operand does not depend on the accumulator: the first
  // two chunks are fetched while the MMAs of this tile are still running,
  // each later chunk while the chunk two places before it is processed.
  // Poly (b*A): the chunk's 32 x 32 block of A, coalesced (lane: row
  // (lane >> 2) + 8u, 16-byte piece lane & 3), only where the chunk touches
  // the upper triangle. Gemm with a*X in the epilogue: this lane's row.
  const int lim = (PHASE == kPhasePoly) ? B.m : B.n;
  const bf16* abase = reinterpret_cast<const bf16*>(B.aux + it.y * B.aux_mat_stride);
  const bf16* row = abase + (int64_t)i * B.aux_ld;
  // gemm with a == 0 (the last product of the Gram-space recurrence) has no linear term
  const bool need_aux = PHASE == kPhasePoly || (PHASE == kPhaseGemm && p.a != 0.f);
  uint4 cur[4], nxt[4];
  auto fetch = [&](int ch, uint4 (&dst)[4]) {
    const int j0 = jbase + ch * 32;
    if (PHASE == kPhasePoly) {
      if (j0 + 32 <= B.m && j0 + 31 >= i0) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ii = i0 + (lane >> 2) + 8 * u;
          if (ii < B.m)
            dst[u] = __ldg(reinterpret_cast<const uint4*>(abase + (int64_t)ii * B.aux_ld + j0 + 8 * (lane & 3)));
        }
      }
    } else if (need_aux && i < B.m && j0 + 32 <= lim) {
      const uint4* s4 = reinterpret_cast<const uint4*>(row + j0);
#pragma unroll
      for (int u = 0; u < 4; ++u) dst[u] = __ldg(s4 + u);
    }
  };
  fetch(0, cur);
  fetch(1, nxt);
  const int gm = B.slot_mat[it.y];
  const MatDev md = p.mats[gm];
  // last step on bf16 weights: the W blocks of the first two chunks are copied in while the
  // MMAs still run; chunk ch + 2's while chunk ch is processed (one copy group per chunk)
  const bool w_last = PHASE == kPhaseGemm && p.last && p.param_bf16 && p.wmaps != nullptr;
  if (w_last) {
    if (lane == 0) {
      ptx::bulk_wait_read<0>();  // the previous tile's stores to W are done with both boxes
      ptx::fence_tensormap_acquire(&p.wmaps[gm]);
    }
    __syncwarp();
    w_chunk_fetch(p, md, gm, B.m, B.n, i0, jbase, lane, stg);
    ptx::cp_async_commit();
    w_chunk_fetch(p, md, gm, B.m, B.n, i0, jbase + 32, lane, stg + kStageBox);
    ptx::cp_async_commit();
  }
  if (!wait_acc()) return false;
  ptx::tc_fence_after();
  float sc = 1.f;
  if (p.first) {
    const float s = p.s_norm[gm];
    sc = (PHASE == kPhaseGram) ? s * s : s;
  }
  // Output chunks leave through shared memory and TMA stores (one 32 x 32 box per chunk, and
  // its mirror image for the symmetric products): X' of the gemm (not on the last step, which
  // updates W, nor when a*X is added here), and every chunk of a symmetric product strictly
  // above the diagonal. On the last step bf16 weights are updated in shared memory from
  // prefetched blocks. Diagonal chunks, matrix edges and fp32 weights take the per-row path.
  const bool gemm_tma = PHASE == kPhaseGemm && !p.last && !need_aux;
#pragma unroll 1
  for (int ch = 0; ch < kChunks; ++ch) {
    float v[32];
    ptx::tmem_ld_32x32b_x32(tbase + ch * 32, v);
    const int j0 = jbase + ch * 32;
    if (PHASE == kPhaseGemm && gemm_tma) {
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] *= sc;
      uint8_t* box = stg + (nbox & 1u) * kStageBox;
      if (lane == 0) ptx::bulk_wait_read<1>();  // the store that last read this box is done with it
      __syncwarp();
      stage_row_sw64(box, lane, v);
      ptx::fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
        if (i0 < B.m && j0 < B.n) ptx::tma_store_3d(&B.tmOut, box, j0, i0, it.y);
        ptx::bulk_commit();  // one group per box, stored or not, so the count above holds
      }
      ++nbox;
    } else if (PHASE == kPhaseGemm && w_last) {
      uint8_t* box = stg + (ch & 1) * kStageBox;
      ptx::cp_async_wait<1>();  // this chunk's copies (all but the newest group) have landed
      __syncwarp();
      if (w_chunk_vec(md, B.m, B.n, i0, j0)) {
        gemm_values(p, B, it.y, i, j0, sc, v, cur);
        capture_row(p, md, i, j0, B.m, B.n, v);
        w_chunk_apply(p, md, gm, B.m, B.n, i0, j0, lane, v, box);
      } else {
        epilogue_chunk<PHASE>(p, B, md, gm, it.y, i, j0, sc, v, cur);  // matrix edges
      }
      if (ch + 2 < kChunks) {
        if (lane == 0) ptx::bulk_wait_read<0>();  // this chunk's store has read the box
        __syncwarp();
        w_chunk_fetch(p, md, gm, B.m, B.n, i0, j0 + 64, lane, box);
      }
      ptx::cp_async_commit();
    } else if (PHASE != kPhaseGemm && i0 < B.m && j0 < B.m && j0 + 31 >= i0) {
      // a chunk of a symmetric product touching the upper triangle
      if (lane == 0) ptx::bulk_wait_read<0>();  // both boxes free again
      __syncwarp();
      float a[32];
      if (PHASE == kPhasePoly) poly_aux_rows(B, abase, i, j0, lane, cur, stg, a);
      if (j0 >= i0 + 32) {  // strictly above the diagonal: the chunk and its mirror as TMA boxes
        sym_values<PHASE>(p, sc, a, v);
        stage_row_sw64(stg, lane, v);
        stage_col_sw64(stg + kStageBox, lane, v);
        ptx::fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_3d(&B.tmOut, stg, j0, i0, it.y);
          ptx::tma_store_3d(&B.tmOut, stg + kStageBox, i0, j0, it.y);
          ptx::bulk_commit();
        }
      } else {  // on the diagonal: per-row stores keep the result exactly symmetric
        sym_diag_chunk<PHASE>(p, B, it.y, i, j0, sc, a, v);
      }
    } else if (PHASE == kPhaseGemm) {
      epilogue_chunk<PHASE>(p, B, md, gm, it.y, i, j0, sc, v, cur);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) cur[u] = nxt[u];
    if (ch + 2 < kChunks) fetch(ch + 2, nxt);
  }
  return true;
}

}  // namespace epi
}  // namespace dmuon
