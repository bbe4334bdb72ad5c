// noalloc.cu - the momentum / normalisation pass for ONE matrix without any
// caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// optimizer: a framework whose caching allocator has already reserved the
// whole GPU, a plugin that is handed only the tensors it must update, or a
// runtime that forbids allocation once its steady state has begun. The
// regular pass (momentum.cu) keeps its per-unit partial sums and per-matrix
// tickets in the caller's workspace; this variant keeps them in a file-scope
// static device array instead, so the caller passes only inputs and outputs.
//
// The array lives in every GPU that loads the library until the process
// exits; it holds kNoallocMaxUnits fp32 partial sums (256 KiB, plus 256 B
// kept free). All calls share it: calls that overlap on the GPU (two
// streams, or two host threads) race on it and give wrong results.
//
// One call is two launches on the caller's stream: the tile pass (the same
// 64 x 128 tile code as the workspace pass, stream_tile.cuh), where every
// tile writes its partial sum of squares, then one CTA that adds the
// partials in a fixed order in fp64 and writes s.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdio>
#include <cmath>
#include <mutex>

#include "dmuon.h"
#include "internal.h"
#include "stream_tile.cuh"

namespace dmuon {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kNoallocMaxUnits = 65536;  // 64 x 128 tiles per matrix
constexpr int kNoallocWords = kNoallocMaxUnits + 64;

// Static scratch: [0, kNoallocMaxUnits) fp32 partial sums, stored as raw words.
static __device__ __align__(256) unsigned g_noalloc_scratch[kNoallocWords];

struct NoallocParams {
  const void* grad;
  float* momentum;
  void* u;
  float* s_out;
  unsigned* scratch;  // device address of g_noalloc_scratch
  int32_t rows, cols, u_ld, tiles_c;
  int32_t n_tiles;
  int32_t transposed;
  int32_t vec_load, vec_store;  // 16-byte access allowed (alignment of the pointers, cols % 4)
  float mu, eps;
  int32_t nesterov;
};

template <bool GB, bool XB>
__global__ void __launch_bounds__(kStreamThreads) momentum_noalloc_kernel(const __grid_constant__ NoallocParams p) {
  __shared__ float tileU[kTileR][kTileC + 1];
  __shared__ float red[kStreamThreads / 32];
  float* partial = reinterpret_cast<float*>(p.scratch);
  const bool nest = p.nesterov != 0;
  for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x) {
    const int r0 = (t / p.tiles_c) * kTileR, c0 = (t % p.tiles_c) * kTileC;
    float ss = stile::tile_update<GB>(p.grad, p.momentum, p.rows, p.cols, p.vec_load != 0, r0, c0, p.mu, nest,
                                      tileU);
    __syncthreads();
    stile::tile_store<XB>(p.u, p.u_ld, p.rows, p.cols, p.transposed != 0, p.vec_store != 0, r0, c0, tileU);
    // the tile's partial, fixed-order block sum
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
      float b = 0.f;
      for (int k = 0; k < kStreamThreads / 32; ++k) b += red[k];
      partial[t] = b;
    }
    __syncthreads();  // tileU and red are reused by the next tile
  }
}

// s = 1 / (||U||_F + eps) from the tiles' partials, in fp64 and a fixed order.
__global__ void __launch_bounds__(kStreamThreads) noalloc_finalize_kernel(const __grid_constant__ NoallocParams p) {
  __shared__ double redd[kStreamThreads / 32];
  const float* partial = reinterpret_cast<const float*>(p.scratch);
  double acc = 0.0;
  for (int k = threadIdx.x; k < p.n_tiles; k += kStreamThreads) acc += static_cast<double>(partial[k]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) redd[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int k = 0; k < kStreamThreads / 32; ++k) tot += redd[k];
    *p.s_out = 1.0f / (static_cast<float>(sqrt(tot)) + p.eps);
  }
}

// Device address of the static scratch, looked up once per device and
// context. The address belongs to the context that was current when it was
// looked up: after cudaDeviceReset the device gets a new primary context,
// whose ID differs, and the address is looked up again.
constexpr int kMaxDevices = 64;
struct ScratchAddr {
  unsigned long long ctx_id = 0;  // unique over the process's lifetime; 0 = not looked up
  unsigned* addr = nullptr;
};
std::mutex g_setup_mu;
ScratchAddr g_scratch_addr[kMaxDevices];

// ID of the calling thread's current context, or 0 when none is current yet.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    looked_up = true;
  }
  if (get_cur == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

}  // namespace
}  // namespace dmuon

using namespace dmuon;

extern "C" dmuon_status dmuon_momentum_norm_noalloc(const void* grad, float* momentum, void* u_out, float* s_out,
                                                    int64_t rows, int64_t cols, int32_t grad_dtype,
                                                    int32_t u_dtype, float mu, int32_t nesterov, float eps,
                                                    void* stream) {
  if (grad == nullptr || momentum == nullptr || u_out == nullptr || s_out == nullptr)
    return set_last_error(DMUON_ERR_INVALID_ARG, "NULL pointer argument");
  if (rows < 1 || cols < 1 || rows > (1 << 20) || cols > (1 << 20) || rows * cols >= (1LL << 31))
    return set_last_error(DMUON_ERR_INVALID_ARG, "unsupported matrix shape");
  if ((grad_dtype != DMUON_F32 && grad_dtype != DMUON_BF16) || (u_dtype != DMUON_F32 && u_dtype != DMUON_BF16))
    return set_last_error(DMUON_ERR_UNSUPPORTED, "grad and u dtypes must be DMUON_F32 or DMUON_BF16");
  if (!std::isfinite(mu) || !(eps >= 0.f) || (nesterov != 0 && nesterov != 1))
    return set_last_error(DMUON_ERR_INVALID_ARG, "bad mu, eps or nesterov");
  const int64_t tiles_c = (cols + kTileC - 1) / kTileC;
  const int64_t n_tiles = ((rows + kTileR - 1) / kTileR) * tiles_c;
  if (n_tiles > kNoallocMaxUnits)
    return set_last_error(DMUON_ERR_UNSUPPORTED,
                          "matrix too large for the static scratch: ceil(rows/64)*ceil(cols/128) must be <= 65536");

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return set_last_error(DMUON_ERR_CUDA, "no usable current CUDA device");
  // An error left pending by the caller's earlier work is reported as such (and left pending),
  // not mistaken for a failure of this call's launches.
  const cudaError_t pending = cudaPeekAtLastError();
  if (pending != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof msg, "a CUDA error from earlier work is pending: %s (%s)", cudaGetErrorName(pending),
             cudaGetErrorString(pending));
    return set_last_error(DMUON_ERR_CUDA, msg);
  }
  unsigned* scratch;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    ScratchAddr& sa = g_scratch_addr[dev];
    unsigned long long ctx = current_context_id();
    if (sa.addr == nullptr || ctx == 0 || ctx != sa.ctx_id) {
      // The array's name in host code is only a host-side handle; the kernel
      // needs its device address, fetched here with this device current (this
      // also creates the device's primary context when none exists yet).
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
        return set_last_error(DMUON_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
      sa.addr = static_cast<unsigned*>(ptr);
      sa.ctx_id = current_context_id();
    }
    scratch = sa.addr;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  NoallocParams p;
  p.grad = grad;
  p.momentum = momentum;
  p.u = u_out;
  p.s_out = s_out;
  p.scratch = scratch;
  p.rows = static_cast<int32_t>(rows);
  p.cols = static_cast<int32_t>(cols);
  p.transposed = rows > cols;
  const int64_t n_long = rows > cols ? rows : cols;
  p.u_ld = static_cast<int32_t>((n_long + 7) / 8 * 8);
  p.tiles_c = static_cast<int32_t>(tiles_c);
  p.n_tiles = static_cast<int32_t>(n_tiles);
  p.mu = mu;
  p.eps = eps;
  p.nesterov = nesterov;
  const auto aligned = [](const void* q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) & (a - 1)) == 0; };
  p.vec_load = (cols % 4 == 0) && aligned(momentum, 16) && aligned(grad, grad_dtype == DMUON_BF16 ? 8 : 16);
  p.vec_store = aligned(u_out, 16);
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = static_cast<int>(std::min<int64_t>(n_tiles, 4LL * (sms > 0 ? sms : 1)));
  const bool gb = grad_dtype == DMUON_BF16, xb = u_dtype == DMUON_BF16;
  if (gb && xb)
    momentum_noalloc_kernel<true, true><<<grid, kStreamThreads, 0, s>>>(p);
  else if (gb)
    momentum_noalloc_kernel<true, false><<<grid, kStreamThreads, 0, s>>>(p);
  else if (xb)
    momentum_noalloc_kernel<false, true><<<grid, kStreamThreads, 0, s>>>(p);
  else
    momentum_noalloc_kernel<false, false><<<grid, kStreamThreads, 0, s>>>(p);
  // no error was pending before the launches, so one seen now is theirs
  if (cudaGetLastError() != cudaSuccess) return set_last_error(DMUON_ERR_CUDA, "tile-pass kernel launch failed");
  noalloc_finalize_kernel<<<1, kStreamThreads, 0, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return set_last_error(DMUON_ERR_CUDA, "norm kernel launch failed");
  return set_last_error(DMUON_OK, "");
}
