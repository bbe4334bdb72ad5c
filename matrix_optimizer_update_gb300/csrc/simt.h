// simt.h - the fp32 arithmetic mode of the Newton-Schulz products (CUDA-core FFMA): tile shape,
// launch parameters and launcher, shared by the host planner and the SIMT kernel.
#pragma once

#include "internal.h"

namespace dmuon {

// fp32 SIMT tile: 32 x 32 outputs per CTA of 256 threads (2 x 2 per thread), K staged 64 at a time.
// Small tiles and a deep K stage suit the short, latency-bound products this mode runs on.
constexpr int kSimtBM = 32;
constexpr int kSimtBN = 32;
constexpr int kSimtBK = 64;
constexpr int kSimtThreads = 256;
constexpr int kSimtGroup = 4;  // K stages whose loads a thread issues together (K up to 256 at once)

// One bucket as seen by a fp32 SIMT launch.
struct SimtBucket {
  const int32_t* slot_mat;
  const float* opA;   // gram: X (m x n); poly: A (m x m); gemm: B (m x m)
  const float* opB;   // gram: X; poly: A; gemm: X_k
  float* out;
  const float* aux;
  int64_t a_mat_stride, b_mat_stride, out_mat_stride, aux_mat_stride;  // elements
  int32_t a_ld, b_ld, out_ld, aux_ld;
  int32_t m, n, kdim, pad;
};

struct SimtParams {
  SimtBucket bk[kMaxBucketsPerLaunch];
  const int4* items;
  int32_t n_items;
  int32_t first, last;
  float a, b, c, lr;
  float diag;  // poly phase: added on the diagonal
  const MatDev* mats;
  const uint64_t* ptrs;
  const float* s_norm;
  float* capture;
  int32_t param_bf16;
};

cudaError_t launch_simt(int phase, const SimtParams& p, int grid, cudaStream_t s);

}  // namespace dmuon
