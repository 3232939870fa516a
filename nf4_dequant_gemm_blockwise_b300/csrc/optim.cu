// AdamW over the LoRA adapters' float32 master weights, in place.
//
// "Layer streaming: fine-tune a model that does not fit in your card", "Measured numbers":
// the pages' runs train the adapters with an AdamW (8-bit paged state there; float32 state
// here).  The update is Adam's bias-corrected moments (Kingma & Ba, "Adam: A Method for
// Stochastic Optimization") with the weight decay decoupled from the gradient and scaled by
// the learning rate (Loshchilov & Hutter, "Decoupled Weight Decay Regularization").
//
// Purely elementwise and HBM-bound: 16 bytes read (p, g, m, v) and 12 written (p, m, v) per
// parameter.  One grid-stride launch over the whole flat buffer, four parameters per thread
// per iteration (16-byte accesses) when every pointer is 16-byte aligned.
#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "util.h"

namespace soup {
namespace {

struct AdamwConst {
  float lr, b1, b2, eps, wd, gs;
  float lr_bc1;        // lr / (1 - beta1^t)
  float inv_sqrt_bc2;  // 1 / sqrt(1 - beta2^t)
};

__device__ __forceinline__ void adamw_one(float &p, float g, float &m, float &v,
                                          const AdamwConst &a) {
  g *= a.gs;
  m = a.b1 * m + (1.f - a.b1) * g;
  v = a.b2 * v + (1.f - a.b2) * (g * g);
  const float denom = sqrtf(v) * a.inv_sqrt_bc2 + a.eps;
  p = p - a.lr * a.wd * p - a.lr_bc1 * (m / denom);
}

template <bool VEC>
__global__ void __launch_bounds__(256, 6) adamw_kernel(float *__restrict__ p,
                                                    const float *__restrict__ g,
                                                    float *__restrict__ m, float *__restrict__ v,
                                                    int64_t n, const AdamwConst a) {
  const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t head = 0;
  if constexpr (VEC) {
    const int64_t n4 = n >> 2;
    float4 *p4 = reinterpret_cast<float4 *>(p), *m4 = reinterpret_cast<float4 *>(m);
    float4 *v4 = reinterpret_cast<float4 *>(v);
    const float4 *g4 = reinterpret_cast<const float4 *>(g);
    for (int64_t i = tid; i < n4; i += stride) {
      float4 P = p4[i], M = m4[i], V = v4[i];
      const float4 G = __ldg(g4 + i);
      adamw_one(P.x, G.x, M.x, V.x, a);
      adamw_one(P.y, G.y, M.y, V.y, a);
      adamw_one(P.z, G.z, M.z, V.z, a);
      adamw_one(P.w, G.w, M.w, V.w, a);
      p4[i] = P;
      m4[i] = M;
      v4[i] = V;
    }
    head = n4 << 2;  // the last n % 4 elements go through the scalar loop
  }
  for (int64_t i = head + tid; i < n; i += stride) {
    float P = p[i], M = m[i], V = v[i];
    adamw_one(P, __ldg(g + i), M, V, a);
    p[i] = P;
    m[i] = M;
    v[i] = V;
  }
}

}  // namespace

void k_adamw(float *p, const float *g, float *m, float *v, int64_t n, float lr, float beta1,
             float beta2, float eps, float weight_decay, float grad_scale, int64_t step,
             cudaStream_t st) {
  if (n <= 0) return;
  AdamwConst a;
  a.lr = lr;
  a.b1 = beta1;
  a.b2 = beta2;
  a.eps = eps;
  a.wd = weight_decay;
  a.gs = grad_scale;
  // bias corrections in double from the float betas, rounded once
  const double bc1 = 1.0 - std::pow((double)beta1, (double)step);
  const double bc2 = 1.0 - std::pow((double)beta2, (double)step);
  a.lr_bc1 = (float)((double)lr / bc1);
  a.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
  const bool vec = ((reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(g) |
                     reinterpret_cast<uintptr_t>(m) | reinterpret_cast<uintptr_t>(v)) & 15) == 0;
  const int64_t work = vec ? (n + 3) / 4 : n;
  int64_t blocks = (work + 255) / 256;
  if (blocks > 148 * 6) blocks = 148 * 6;  // one wave: 6 resident 256-thread blocks per SM
  if (vec) adamw_kernel<true><<<(int)blocks, 256, 0, st>>>(p, g, m, v, n, a);
  else adamw_kernel<false><<<(int)blocks, 256, 0, st>>>(p, g, m, v, n, a);
  count_launches(1);
}

}  // namespace soup
