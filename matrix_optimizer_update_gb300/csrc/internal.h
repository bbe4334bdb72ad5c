// internal.h - structures shared by the host planner and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dmuon.h"

namespace dmuon {

constexpr int kMaxBucketsPerLaunch = 7;  // 7 x 512 B of bucket descriptors fit the 4 KB of launch parameters

// Tensor-core tile: 128 rows (UMMA M) x 256 or 128 columns (UMMA N, chosen per
// bucket), K staged 64 at a time.
constexpr int kTcBM = 128;
constexpr int kTcBN = 256;  // default tile width
constexpr int kTcBK = 64;
constexpr int kTcThreads = 320;  // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2..9 epilogue

// Streaming unit of the momentum pass: 8192 contiguous elements (flat mode)
// or a 64 x 128 tile of the stored matrix (tiled mode).
constexpr int kFlatUnit = 8192;
constexpr int kTileR = 64;
constexpr int kTileC = 128;
constexpr int kStreamThreads = 256;
constexpr int kPartialsPerUnit = kStreamThreads / 32;  // one sum of squares per warp and unit

enum Phase : int { kPhaseGram = 1, kPhasePoly = 2, kPhaseGemm = 3 };

// Per-matrix description (device table, uploaded once at bind).
struct MatDev {
  int32_t rows, cols;   // stored shape (rows = dim 0)
  int32_t m, n;         // short and long side
  int32_t transposed;   // rows > cols: the iteration runs on the transpose
  int32_t bucket, slot; // bucket index and position inside it
  int32_t x_ld;         // row pitch (elements) of the U/X copies in the workspace
  float scale;          // sqrt(max(1, rows/cols))
  int32_t flat;         // momentum pass mode: 1 = flat contiguous, 0 = 64x128 tiles
  int32_t tiles_c;      // tiled mode: tiles along cols
  int32_t vec_ok;       // tiled mode: cols % 4 == 0 (vector loads allowed)
  int64_t x0_off;       // byte offset from the workspace base of this matrix's X0 (= U)
  int64_t unit_begin;   // first momentum-pass unit of this matrix
  int64_t unit_count;
  int64_t cap_off;      // element offset in the capture buffer, -1 when not captured
};

// Momentum / normalisation pass.
struct StreamParams {
  const MatDev* mats;
  const int64_t* unit_begin;  // [n_mats + 1]
  const uint64_t* ptrs;       // [3 * n_mats]: W, G, M device pointers
  char* ws;
  float* partial;             // [n_units * kPartialsPerUnit]: per warp and unit, sums of squares of U
  float* s_norm;              // [n_mats]: 1 / (||U||_F + eps)
  unsigned* status;
  float* capture;
  int64_t n_units;
  int32_t n_mats;
  float mu, eps, lr;
  int32_t nesterov;
  int32_t grad_bf16, x_bf16, param_bf16;
};

// One bucket as seen by a tensor-core launch.
struct TcBucket {
  CUtensorMap tmA;  // A operand: 128 x 64 boxes, K-major
  CUtensorMap tmB;  // B operand: 256 x 64 boxes K-major (gram/poly), or for the gemm a 4-D map that brings
                    // BN/64 chunks of 64 columns x 64 k-rows in one copy (MN-major)
  CUtensorMap tmOut;  // output: 32 x 32 boxes, 64-byte swizzle (epilogue TMA stores)
  const int32_t* slot_mat;  // slot -> global matrix index
  char* out;                // A (gram), B (poly), X_{k+1} (gemm, not last)
  const char* aux;          // A (poly: b*A term), X_k (gemm: a*X term)
  int64_t out_mat_stride;   // bytes between consecutive matrices of out
  int64_t aux_mat_stride;
  int32_t out_ld, aux_ld;   // row pitch in elements
  int32_t m, n, kdim;
  int32_t same_ab;  // both operands are the same matrix (X X^T, A A^T): a diagonal-start tile's A rows
                    // are the first rows of its B rows
};

struct TcParams {
  TcBucket bk[kMaxBucketsPerLaunch];
  const int4* items;  // (bucket, slot, ti, tj), cost-ordered
  int32_t n_items;
  int32_t first, last;
  float a, b, c, lr;
  float diag;  // poly phase: added on the diagonal (a*I of the Gram-space polynomial)
  const MatDev* mats;
  const uint64_t* ptrs;
  const CUtensorMap* wmaps;  // last step on bf16 weights: per matrix, W as 32 x 32 boxes (64-byte swizzle)
  const float* s_norm;
  float* capture;
  unsigned* status;
  int32_t param_bf16;
  int64_t timeout_ns;
  // Dynamic tile claiming: [0] counts claimed items, [1] CTAs that finished; both zero before
  // the launch, and the last CTA leaves them zero. nullptr = CTA b (CTA pair b of the two-SM
  // kernel) takes items b, b + grid, ...
  unsigned* sched;
  unsigned long long* cta_times;  // profiling: start and end (global timer, ns) per CTA, or nullptr
};

constexpr int kMaxCtaRecords = 1024;  // CTAs per launch the per-CTA profiling records

// Kernel launchers (each returns the launch's cudaError_t).
cudaError_t launch_momentum(const StreamParams& p, int grid, cudaStream_t s);
cudaError_t launch_norm_finalize(const StreamParams& p, int grid, cudaStream_t s);
cudaError_t launch_update0(const StreamParams& p, int grid, cudaStream_t s);
int momentum_blocks_per_sm(int grad_bf16, int x_bf16);  // resident CTAs per SM of the momentum kernel
cudaError_t launch_tc(int phase, int bn, const TcParams& p, int grid, cudaStream_t s);
// Two-SM form: 256 x 256 tiles on clusters of two CTAs; `pairs` clusters.
cudaError_t launch_tc_pair(int phase, const TcParams& p, int pairs, cudaStream_t s);
cudaError_t launch_wait_timeout_selftest(unsigned* status, int64_t limit_ns, cudaStream_t s);
// status word -> mapped host word (device address of it), then cleared
cudaError_t launch_status_readout(unsigned* status, unsigned* host_out_dev, cudaStream_t s);
// bind-time tuning only: bytes (a multiple of 16) of pseudo-random bf16 operands at dst
cudaError_t launch_tuning_fill(void* dst, int64_t bytes, uint32_t seed, int grid, cudaStream_t s);

// Record the message dmuon_last_error() returns on this thread; returns st.
dmuon_status set_last_error(dmuon_status st, const char* msg);

}  // namespace dmuon
