// adamw.cu - AdamW step over one flat buffer, for the parameters the Muon
// predicate does not select ("DMuon" project docs, section "DMuon 能做什么":
// the optimizer takes a separate ``adamw_lr`` for everything else, e.g.
// embeddings, norms and task heads). Decoupled weight decay, bias-corrected
// moments:
//   p <- p*(1 - lr*wd);  m <- b1*m + (1-b1)*g;  v <- b2*v + (1-b2)*g^2
//   p <- p - (lr/(1-b1^t)) * m / (sqrt(v)/sqrt(1-b2^t) + eps)
// fp32 arithmetic, fp32 moments, params and grads bf16 or fp32. HBM-bound:
// 2*|p| + |g| + 16 bytes per element; 8 elements per thread per iteration
// with 16-byte vector accesses, grid-stride over the buffer.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "dmuon.h"
#include "internal.h"

namespace dmuon {
namespace {

using bf16 = __nv_bfloat16;

struct AdamwParams {
  void* param;
  const void* grad;
  float* m;
  float* v;
  int64_t n;
  float decay;         // 1 - lr*wd
  float beta1, one_minus_beta1, beta2, one_minus_beta2;
  float step_size;     // lr / (1 - b1^t)
  float inv_sqrt_bc2;  // 1 / sqrt(1 - b2^t)
  float eps;
};

__device__ __forceinline__ float adamw_elem(const AdamwParams& a, float p, float g, float& m, float& v) {
  m = fmaf(a.beta1, m, a.one_minus_beta1 * g);
  v = fmaf(a.beta2, v, a.one_minus_beta2 * g * g);
  const float denom = sqrtf(v) * a.inv_sqrt_bc2 + a.eps;
  return p * a.decay - a.step_size * (m / denom);
}

template <bool PB, bool GB>
__global__ void __launch_bounds__(256) adamw_kernel(const __grid_constant__ AdamwParams a) {
  const int64_t nvec = a.n / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < nvec; t += stride) {
    const int64_t e = t * 8;
    float p[8], g[8], m[8], v[8];
    if (PB) {
      const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const bf16*>(a.param) + e);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(h[k]);
        p[2 * k] = f.x;
        p[2 * k + 1] = f.y;
      }
    } else {
      const float4 x = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.param) + e);
      const float4 y = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.param) + e + 4);
      p[0] = x.x, p[1] = x.y, p[2] = x.z, p[3] = x.w, p[4] = y.x, p[5] = y.y, p[6] = y.z, p[7] = y.w;
    }
    if (GB) {
      const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const bf16*>(a.grad) + e);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(h[k]);
        g[2 * k] = f.x;
        g[2 * k + 1] = f.y;
      }
    } else {
      const float4 x = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.grad) + e);
      const float4 y = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.grad) + e + 4);
      g[0] = x.x, g[1] = x.y, g[2] = x.z, g[3] = x.w, g[4] = y.x, g[5] = y.y, g[6] = y.z, g[7] = y.w;
    }
    {
      const float4 x = *reinterpret_cast<const float4*>(a.m + e), y = *reinterpret_cast<const float4*>(a.m + e + 4);
      m[0] = x.x, m[1] = x.y, m[2] = x.z, m[3] = x.w, m[4] = y.x, m[5] = y.y, m[6] = y.z, m[7] = y.w;
      const float4 z = *reinterpret_cast<const float4*>(a.v + e), w = *reinterpret_cast<const float4*>(a.v + e + 4);
      v[0] = z.x, v[1] = z.y, v[2] = z.z, v[3] = z.w, v[4] = w.x, v[5] = w.y, v[6] = w.z, v[7] = w.w;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) p[k] = adamw_elem(a, p[k], g[k], m[k], v[k]);
    *reinterpret_cast<float4*>(a.m + e) = make_float4(m[0], m[1], m[2], m[3]);
    *reinterpret_cast<float4*>(a.m + e + 4) = make_float4(m[4], m[5], m[6], m[7]);
    *reinterpret_cast<float4*>(a.v + e) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(a.v + e + 4) = make_float4(v[4], v[5], v[6], v[7]);
    if (PB) {
      uint4 u;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(p[2 * k], p[2 * k + 1]);
      *reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(a.param) + e) = u;
    } else {
      float* d = reinterpret_cast<float*>(a.param) + e;
      *reinterpret_cast<float4*>(d) = make_float4(p[0], p[1], p[2], p[3]);
      *reinterpret_cast<float4*>(d + 4) = make_float4(p[4], p[5], p[6], p[7]);
    }
  }
  // ragged tail (< 8 elements), one thread each
  const int64_t tail0 = nvec * 8;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t < a.n - tail0) {
    const int64_t e = tail0 + t;
    const float p = PB ? __bfloat162float(reinterpret_cast<const bf16*>(a.param)[e])
                       : reinterpret_cast<const float*>(a.param)[e];
    const float g = GB ? __bfloat162float(reinterpret_cast<const bf16*>(a.grad)[e])
                       : reinterpret_cast<const float*>(a.grad)[e];
    float m = a.m[e], v = a.v[e];
    const float np = adamw_elem(a, p, g, m, v);
    a.m[e] = m;
    a.v[e] = v;
    if (PB)
      reinterpret_cast<bf16*>(a.param)[e] = __float2bfloat16_rn(np);
    else
      reinterpret_cast<float*>(a.param)[e] = np;
  }
}

}  // namespace
}  // namespace dmuon

using namespace dmuon;

extern "C" dmuon_status dmuon_adamw_flat(void* param, const void* grad, float* exp_avg, float* exp_avg_sq,
                                         int64_t n, int32_t param_dtype, int32_t grad_dtype, float lr,
                                         float beta1, float beta2, float eps, float weight_decay, int32_t step,
                                         void* stream) {
  if (param == nullptr || grad == nullptr || exp_avg == nullptr || exp_avg_sq == nullptr)
    return set_last_error(DMUON_ERR_INVALID_ARG, "NULL pointer argument");
  if (n < 1) return set_last_error(DMUON_ERR_INVALID_ARG, "n must be >= 1");
  if (((reinterpret_cast<uintptr_t>(param) | reinterpret_cast<uintptr_t>(grad) |
        reinterpret_cast<uintptr_t>(exp_avg) | reinterpret_cast<uintptr_t>(exp_avg_sq)) & 15) != 0)
    return set_last_error(DMUON_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  if ((param_dtype != DMUON_F32 && param_dtype != DMUON_BF16) || (grad_dtype != DMUON_F32 && grad_dtype != DMUON_BF16))
    return set_last_error(DMUON_ERR_UNSUPPORTED, "param and grad dtypes must be DMUON_F32 or DMUON_BF16");
  if (!std::isfinite(lr) || !std::isfinite(weight_decay) || !(beta1 >= 0.f && beta1 < 1.f) ||
      !(beta2 >= 0.f && beta2 < 1.f) || !(eps >= 0.f) || step < 1)
    return set_last_error(DMUON_ERR_INVALID_ARG, "bad lr, betas, eps, weight_decay or step");
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return set_last_error(DMUON_ERR_CUDA, "no usable CUDA device");
  AdamwParams a;
  a.param = param;
  a.grad = grad;
  a.m = exp_avg;
  a.v = exp_avg_sq;
  a.n = n;
  a.decay = 1.0f - lr * weight_decay;
  a.beta1 = beta1;
  a.one_minus_beta1 = 1.0f - beta1;
  a.beta2 = beta2;
  a.one_minus_beta2 = 1.0f - beta2;
  const double bc1 = 1.0 - std::pow(static_cast<double>(beta1), step);
  const double bc2 = 1.0 - std::pow(static_cast<double>(beta2), step);
  a.step_size = static_cast<float>(lr / bc1);
  a.inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
  a.eps = eps;
  const int64_t nvec = n / 8;
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((nvec + 255) / 256, 8LL * sms));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool pb = param_dtype == DMUON_BF16, gb = grad_dtype == DMUON_BF16;
  if (pb && gb)
    adamw_kernel<true, true><<<(int)blocks, 256, 0, s>>>(a);
  else if (pb)
    adamw_kernel<true, false><<<(int)blocks, 256, 0, s>>>(a);
  else if (gb)
    adamw_kernel<false, true><<<(int)blocks, 256, 0, s>>>(a);
  else
    adamw_kernel<false, false><<<(int)blocks, 256, 0, s>>>(a);
  if (cudaGetLastError() != cudaSuccess) return set_last_error(DMUON_ERR_CUDA, "kernel launch failed");
  return set_last_error(DMUON_OK, "");
}
