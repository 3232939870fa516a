// Memory-bound kernels of the streamed LoRA step: embedding gather, RMSNorm forward and
// backward, RoPE, SwiGLU, the rank-r LoRA projections and their gradients, the operand packs
// that fold LoRA into the base GEMM, and the vocabulary-chunked cross-entropy.
//
// Layer maths ("Layer streaming: fine-tune a model that does not fit in your card",
// "How it works": the model family's own decoder layer runs on the streamed weights;
// "Honest scope": plain LoRA on the decoder layers): pre-norm Llama block, RMSNorm
// x / sqrt(mean x^2 + eps) * w, rotate-half RoPE, SiLU-gated MLP, LoRA y += s (x A^T) B^T.
// All arithmetic is float32; every reduction has a fixed order (warp shuffles and block
// trees, never atomics), so results do not depend on scheduling.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "util.h"

namespace soup {
namespace {
using namespace soupk;

inline int cdiv(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

SOUP_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
SOUP_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ------------------------------------------------------------------ embedding
__global__ void embed_kernel(const int32_t *tok, const uint16_t *E, int V, int H, float *out) {
  const int m = blockIdx.x;
  int t = tok[m];
  t = t < 0 ? 0 : (t >= V ? V - 1 : t);
  const uint16_t *src = E + (size_t)t * H;
  float *dst = out + (size_t)m * H;
  for (int i = threadIdx.x * 8; i < H; i += blockDim.x * 8) {
    const uint4 v = *reinterpret_cast<const uint4 *>(src + i);
    *reinterpret_cast<float4 *>(dst + i) = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
    *reinterpret_cast<float4 *>(dst + i + 4) = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
  }
}

// ------------------------------------------------------------------ RMSNorm
// One row per 256-thread block: the row is read once into registers (up to RMS_V float4s per
// thread, H <= 8192) and reused after the sum of squares; the block sum adds the eight warp
// sums in warp order.
constexpr int RMS_T = 256, RMS_V = 8;

SOUP_DEV float block_sum256(float v, float *sh) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) sh[w] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < RMS_T / 32; ++i) s += sh[i];
  __syncthreads();
  return s;
}

template <bool F16>
__global__ void __launch_bounds__(RMS_T) rmsnorm_fwd_kernel(const float *h, const uint16_t *w, float eps,
                                                            int M, int H, uint16_t *out, int *err) {
  __shared__ float sh[RMS_T / 32];
  const int row = blockIdx.x;
  const float *x = h + (size_t)row * H;
  float4 v[RMS_V];
  float ss = 0.f;
#pragma unroll
  for (int it = 0; it < RMS_V; ++it) {
    const int i = (threadIdx.x + it * RMS_T) * 4;
    v[it] = i < H ? *reinterpret_cast<const float4 *>(x + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    ss += v[it].x * v[it].x + v[it].y * v[it].y + v[it].z * v[it].z + v[it].w * v[it].w;
  }
  ss = block_sum256(ss, sh);
  const float r = 1.0f / sqrtf(ss / (float)H + eps);
  uint16_t *o = out + (size_t)row * H;
  bool bad = false;
#pragma unroll
  for (int it = 0; it < RMS_V; ++it) {
    const int i = (threadIdx.x + it * RMS_T) * 4;
    if (i >= H) break;
    const uint2 wv = *reinterpret_cast<const uint2 *>(w + i);
    const float y0 = v[it].x * r * bf16_lo(wv.x), y1 = v[it].y * r * bf16_hi(wv.x);
    const float y2 = v[it].z * r * bf16_lo(wv.y), y3 = v[it].w * r * bf16_hi(wv.y);
    if (F16) bad |= half_out_of_range(y0) | half_out_of_range(y1) | half_out_of_range(y2) | half_out_of_range(y3);
    uint2 res;
    res.x = pack16x2<F16>(y0, y1);
    res.y = pack16x2<F16>(y2, y3);
    *reinterpret_cast<uint2 *>(o + i) = res;
  }
  flag_range(bad, err);
}

__global__ void __launch_bounds__(RMS_T) rmsnorm_bwd_kernel(const float *dy, const float *h, const uint16_t *w,
                                                            float eps, int M, int H, const float *dres,
                                                            float *out, uint16_t *out_bf16) {
  __shared__ float sh[RMS_T / 32];
  const int row = blockIdx.x;
  const float *x = h + (size_t)row * H;
  const float *g = dy + (size_t)row * H;
  float4 v[RMS_V], gw[RMS_V];  // x, and dy * w
  float ss = 0.f, sgh = 0.f;
#pragma unroll
  for (int it = 0; it < RMS_V; ++it) {
    const int i = (threadIdx.x + it * RMS_T) * 4;
    if (i < H) {
      v[it] = *reinterpret_cast<const float4 *>(x + i);
      const float4 d = *reinterpret_cast<const float4 *>(g + i);
      const uint2 wv = *reinterpret_cast<const uint2 *>(w + i);
      gw[it] = make_float4(d.x * bf16_lo(wv.x), d.y * bf16_hi(wv.x), d.z * bf16_lo(wv.y), d.w * bf16_hi(wv.y));
    } else {
      v[it] = gw[it] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    ss += v[it].x * v[it].x + v[it].y * v[it].y + v[it].z * v[it].z + v[it].w * v[it].w;
    sgh += gw[it].x * v[it].x + gw[it].y * v[it].y + gw[it].z * v[it].z + gw[it].w * v[it].w;
  }
  ss = block_sum256(ss, sh);
  sgh = block_sum256(sgh, sh);
  const float r = 1.0f / sqrtf(ss / (float)H + eps);
  const float c = r * r * r * sgh / (float)H;  // dx = r*g*w - x * r^3 * sum(g*w*x) / H
  float *o = out + (size_t)row * H;
  const float *dr = dres ? dres + (size_t)row * H : nullptr;
  uint16_t *ob = out_bf16 ? out_bf16 + (size_t)row * H : nullptr;
#pragma unroll
  for (int it = 0; it < RMS_V; ++it) {
    const int i = (threadIdx.x + it * RMS_T) * 4;
    if (i >= H) break;
    float4 res = make_float4(r * gw[it].x - v[it].x * c, r * gw[it].y - v[it].y * c,
                             r * gw[it].z - v[it].z * c, r * gw[it].w - v[it].w * c);
    if (dr) {
      const float4 a = *reinterpret_cast<const float4 *>(dr + i);
      res.x += a.x; res.y += a.y; res.z += a.z; res.w += a.w;
    }
    *reinterpret_cast<float4 *>(o + i) = res;
    if (ob) {
      uint2 pb;
      pb.x = pack_bf16x2(res.x, res.y);
      pb.y = pack_bf16x2(res.z, res.w);
      *reinterpret_cast<uint2 *>(ob + i) = pb;
    }
  }
}

// ------------------------------------------------------------------ RoPE (rotate-half)
// Four consecutive rotation pairs (i .. i+3, i+half .. i+half+3) per thread: 8-byte loads and
// stores of the 16-bit halves and 16-byte loads of the tables (d % 8 == 0, 16-byte aligned
// rows); 32-bit index arithmetic within a row.
template <bool F16>
__global__ void rope_fwd_kernel(uint16_t *qkv, int ld, const float *cs, const float *sn, int M,
                                int S, int nheads_rot, int d, int *err) {
  const int half = d >> 1, q4 = half >> 2, per_row = nheads_rot * q4;
  bool bad = false;
  const int64_t total = (int64_t)M * per_row;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int m = (int)(idx / per_row), r = (int)(idx - (int64_t)m * per_row);
    const int head = r / q4, i = (r - head * q4) * 4;
    const int pos = m % S;
    uint16_t *p = qkv + (size_t)m * ld + (size_t)head * d;
    const uint2 a = *reinterpret_cast<const uint2 *>(p + i);
    const uint2 b = *reinterpret_cast<const uint2 *>(p + i + half);
    const float4 c = *reinterpret_cast<const float4 *>(cs + (size_t)pos * half + i);
    const float4 sv = *reinterpret_cast<const float4 *>(sn + (size_t)pos * half + i);
    const float x1[4] = {lo16<F16>(a.x), hi16<F16>(a.x), lo16<F16>(a.y), hi16<F16>(a.y)};
    const float x2[4] = {lo16<F16>(b.x), hi16<F16>(b.x), lo16<F16>(b.y), hi16<F16>(b.y)};
    const float cc[4] = {c.x, c.y, c.z, c.w}, ss[4] = {sv.x, sv.y, sv.z, sv.w};
    float y1[4], y2[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      y1[e] = x1[e] * cc[e] - x2[e] * ss[e];
      y2[e] = x2[e] * cc[e] + x1[e] * ss[e];
      if (F16) bad |= half_out_of_range(y1[e]) | half_out_of_range(y2[e]);
    }
    *reinterpret_cast<uint2 *>(p + i) = make_uint2(pack16x2<F16>(y1[0], y1[1]), pack16x2<F16>(y1[2], y1[3]));
    *reinterpret_cast<uint2 *>(p + i + half) = make_uint2(pack16x2<F16>(y2[0], y2[1]), pack16x2<F16>(y2[2], y2[3]));
  }
  flag_range(bad, err);
}

__global__ void rope_bwd_kernel(const float *dqkv, uint16_t *out, int ld, const float *cs,
                                const float *sn, int M, int S, int nheads_rot, int nheads_all,
                                int d) {
  const int half = d >> 1, q4 = half >> 2, per_row = nheads_all * q4;
  const int64_t total = (int64_t)M * per_row;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int m = (int)(idx / per_row), r = (int)(idx - (int64_t)m * per_row);
    const int head = r / q4, i = (r - head * q4) * 4;
    const float *g = dqkv + (size_t)m * ld + (size_t)head * d;
    uint16_t *o = out + (size_t)m * ld + (size_t)head * d;
    const float4 a = *reinterpret_cast<const float4 *>(g + i);
    const float4 b = *reinterpret_cast<const float4 *>(g + i + half);
    const float d1[4] = {a.x, a.y, a.z, a.w}, d2[4] = {b.x, b.y, b.z, b.w};
    float r1[4], r2[4];
    if (head < nheads_rot) {
      const int pos = m % S;
      const float4 c = *reinterpret_cast<const float4 *>(cs + (size_t)pos * half + i);
      const float4 sv = *reinterpret_cast<const float4 *>(sn + (size_t)pos * half + i);
      const float cc[4] = {c.x, c.y, c.z, c.w}, ss[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        r1[e] = d1[e] * cc[e] + d2[e] * ss[e];
        r2[e] = d2[e] * cc[e] - d1[e] * ss[e];
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        r1[e] = d1[e];
        r2[e] = d2[e];
      }
    }
    *reinterpret_cast<uint2 *>(o + i) = make_uint2(pack_bf16x2(r1[0], r1[1]), pack_bf16x2(r1[2], r1[3]));
    *reinterpret_cast<uint2 *>(o + i + half) = make_uint2(pack_bf16x2(r2[0], r2[1]), pack_bf16x2(r2[2], r2[3]));
  }
}

// ------------------------------------------------------------------ SwiGLU
SOUP_DEV float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

template <bool F16>
__global__ void swiglu_fwd_kernel(const uint16_t *gu, int M, int I, uint16_t *act, int *err) {
  // 8 consecutive outputs per item when I % 8 == 0 (16-byte loads of gate and up)
  const int I8 = I / 8;
  bool bad = false;
  const int64_t total = (int64_t)M * I8;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = idx / I8, j = (idx % I8) * 8;
    const uint4 g = *reinterpret_cast<const uint4 *>(gu + m * 2 * I + j);
    const uint4 u = *reinterpret_cast<const uint4 *>(gu + m * 2 * I + I + j);
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float g0 = lo16<F16>(gw[e]), g1 = hi16<F16>(gw[e]);
      const float u0 = lo16<F16>(uw[e]), u1 = hi16<F16>(uw[e]);
      const float y0 = g0 * sigmoidf_(g0) * u0, y1 = g1 * sigmoidf_(g1) * u1;
      if (F16) bad |= half_out_of_range(y0) | half_out_of_range(y1);
      o[e] = pack16x2<F16>(y0, y1);
    }
    *reinterpret_cast<uint4 *>(act + m * I + j) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  flag_range(bad, err);
}

template <bool F16>
__global__ void swiglu_fwd_scalar_kernel(const uint16_t *gu, int M, int I, uint16_t *act, int *err) {
  const int64_t total = (int64_t)M * I;
  bool bad = false;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = idx / I, j = idx % I;
    const float g = ld16<F16>(gu[m * 2 * I + j]);
    const float u = ld16<F16>(gu[m * 2 * I + I + j]);
    const float y = g * sigmoidf_(g) * u;
    if (F16) bad |= half_out_of_range(y);
    act[idx] = st16<F16>(y);
  }
  flag_range(bad, err);
}

// 8 consecutive columns per item (inter % 8 == 0): 32-byte dact loads, 16-byte gate / up loads
// and dgu stores.
template <bool F16>
__global__ void swiglu_bwd_kernel(const float *dact, const uint16_t *gu, int M, int I, uint16_t *dgu) {
  const int I8 = I / 8;
  const int64_t total = (int64_t)M * I8;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = idx / I8, j = (idx % I8) * 8;
    const uint4 gv = *reinterpret_cast<const uint4 *>(gu + m * 2 * I + j);
    const uint4 uv = *reinterpret_cast<const uint4 *>(gu + m * 2 * I + I + j);
    const float4 d0 = *reinterpret_cast<const float4 *>(dact + m * I + j);
    const float4 d1 = *reinterpret_cast<const float4 *>(dact + m * I + j + 4);
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
    const float da[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
    uint32_t og[4], ou[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float dg[2], du[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float g = h ? hi16<F16>(gw[e]) : lo16<F16>(gw[e]);
        const float u = h ? hi16<F16>(uw[e]) : lo16<F16>(uw[e]);
        const float sg = sigmoidf_(g);
        dg[h] = da[2 * e + h] * u * (sg * (1.0f + g * (1.0f - sg)));
        du[h] = da[2 * e + h] * g * sg;
      }
      og[e] = pack_bf16x2(dg[0], dg[1]);
      ou[e] = pack_bf16x2(du[0], du[1]);
    }
    *reinterpret_cast<uint4 *>(dgu + m * 2 * I + j) = make_uint4(og[0], og[1], og[2], og[3]);
    *reinterpret_cast<uint4 *>(dgu + m * 2 * I + I + j) = make_uint4(ou[0], ou[1], ou[2], ou[3]);
  }
}

// ------------------------------------------------------------------ LoRA projections
// The four LoRA products are skinny GEMMs (one side is nseg * r <= 64) and run on the tensor
// cores as TF32 mma.sync (m16n8k8, float accumulation).  The 16-bit activations / gradients
// are exact in TF32; the float LoRA parameters and intermediates are rounded to TF32 (nearest,
// ties away) when they are staged.  Every reduction is split into partial tiles that a second
// kernel adds in a fixed order (no atomics).
SOUP_DEV uint32_t to_tf32(float f) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(f));
  return r;
}
SOUP_DEV void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Segment of fused output column n (the one whose range holds it; 0 if none).
SOUP_DEV int seg_of(const LoraSeg &L, int n) {
  int q = 0;
  for (int k = 1; k < L.nseg; ++k)
    if (n >= L.off[k] && n < L.off[k] + L.n[k]) q = k;
  return q;
}

// part[split][m][o] = sum over k in the split's range of X[m, k] * W_o(k), o < 64, with
//   DOWN: X = x [M, K], W_o(k) = A_seg[j, k]                       (u = x A^T)
//   DU:   X = dY [M, Ng], W_o(k) = B_seg[k - off_seg, j] inside the segment, else 0
// o = seg * r + j.  Tile: 64 rows x 64 outputs per 128-thread block (warp w: rows 16w..16w+15,
// all outputs), K in chunks of 32 staged in shared memory.  blockIdx.y picks the K range.
template <bool DU, bool XF16>
__global__ void __launch_bounds__(128) lora_part_kernel(const uint16_t *X, int ldx, int M, int K,
                                                        int KS, const LoraSeg L, float *part) {
  __shared__ uint32_t xs[64][36];  // [row][k]
  __shared__ uint32_t ws[64][36];  // [o][k]
  const int t = threadIdx.x, w = t >> 5, lane = t & 31, g = lane >> 2, q = lane & 3;
  const int m0 = blockIdx.x * 64;
  const int kb = blockIdx.y * KS, ke = min(K, kb + KS);
  const int nout = L.nseg * L.r;
  const int NT = (nout + 7) / 8;  // live 8-wide output tiles
  // the next chunk's operands are fetched into registers while the current one is computed
  uint4 xr[2];
  float wr[16];
  auto load = [&](int k0) {
#pragma unroll
    for (int it = 0; it < 2; ++it) {  // X: 64 rows x 32 k, 8 elements per item
      const int i = t + 128 * it, rr = i >> 2, c8 = (i & 3) * 8;
      const int m = m0 + rr, k = k0 + c8;
      if (m < M && k + 8 <= ke && ((ldx | k) & 7) == 0) {
        xr[it] = *reinterpret_cast<const uint4 *>(X + (size_t)m * ldx + k);
      } else {
        uint32_t h[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = (m < M && k + e < ke) ? X[(size_t)m * ldx + k + e] : 0u;
        xr[it] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
      }
    }
    if (!DU) {
#pragma unroll
      for (int it = 0; it < 4; ++it) {  // A rows: 64 o x 32 k, 4 k per item
        const int i = t + 128 * it, o = i >> 3, k4 = (i & 7) * 4;
        const int k = k0 + k4;
        float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (o < nout) {
          const float *ar = L.A[o / L.r] + (size_t)(o % L.r) * K;
          if (k + 4 <= ke && ((K | k) & 3) == 0) {
            a4 = *reinterpret_cast<const float4 *>(ar + k);
          } else {
            a4.x = k < ke ? ar[k] : 0.f;
            a4.y = k + 1 < ke ? ar[k + 1] : 0.f;
            a4.z = k + 2 < ke ? ar[k + 2] : 0.f;
            a4.w = k + 3 < ke ? ar[k + 3] : 0.f;
          }
        }
        wr[4 * it] = a4.x;
        wr[4 * it + 1] = a4.y;
        wr[4 * it + 2] = a4.z;
        wr[4 * it + 3] = a4.w;
      }
    } else {
#pragma unroll
      for (int it = 0; it < 16; ++it) {  // W[o][kk] = B_seg[k - off, j], o = seg r + j
        const int i = t + 128 * it, o = i >> 5, kk = i & 31;
        const int k = k0 + kk;
        float v = 0.f;
        if (o < nout && k < ke) {
          const int sg = o / L.r;
          if (k >= L.off[sg] && k < L.off[sg] + L.n[sg]) v = L.B[sg][(size_t)(k - L.off[sg]) * L.r + (o % L.r)];
        }
        wr[it] = v;
      }
    }
  };
  auto store = [&]() {
#pragma unroll
    for (int it = 0; it < 2; ++it) {  // 16-bit values are exact in TF32
      const int i = t + 128 * it, rr = i >> 2, c8 = (i & 3) * 8;
      const uint4 u4 = xr[it];
      const uint32_t wv[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        xs[rr][c8 + 2 * e] = __float_as_uint(lo16<XF16>(wv[e]));
        xs[rr][c8 + 2 * e + 1] = __float_as_uint(hi16<XF16>(wv[e]));
      }
    }
    if (!DU) {
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int i = t + 128 * it, o = i >> 3, k4 = (i & 7) * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) ws[o][k4 + e] = to_tf32(wr[4 * it + e]);
      }
    } else {
#pragma unroll
      for (int it = 0; it < 16; ++it) {
        const int i = t + 128 * it;
        ws[i >> 5][i & 31] = to_tf32(wr[it]);
      }
    }
  };
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  if (kb < ke) load(kb);
  for (int k0 = kb; k0 < ke; k0 += 32) {
    store();
    __syncthreads();
    if (k0 + 32 < ke) load(k0 + 32);
#pragma unroll
    for (int k8 = 0; k8 < 32; k8 += 8) {
      const uint32_t a[4] = {xs[16 * w + g][k8 + q], xs[16 * w + g + 8][k8 + q], xs[16 * w + g][k8 + q + 4],
                             xs[16 * w + g + 8][k8 + q + 4]};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
        if (nt < NT) mma_tf32(acc[nt], a, ws[8 * nt + g][k8 + q], ws[8 * nt + g][k8 + q + 4]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    if (nt >= NT) break;
    const int m = m0 + 16 * w + g, o = 8 * nt + 2 * q;
    if (m < M) {
      float *d = part + ((size_t)blockIdx.y * M + m) * 64 + o;
      d[0] = acc[nt][0];
      d[1] = acc[nt][1];
    }
    if (m + 8 < M) {
      float *d = part + ((size_t)blockIdx.y * M + m + 8) * 64 + o;
      d[0] = acc[nt][2];
      d[1] = acc[nt][3];
    }
  }
}

// out_f32[m, o] = (DU ? s : 1) * sum_split part; out16[m, o] = 16-bit(s * sum), zero padded.
// One thread per output (m, o): consecutive threads take consecutive o, so every split's loads
// are contiguous; the splits are added in split order.
template <bool DU, bool OF16>
__global__ void lora_reduce_kernel(const float *part, int nsplit, int M, const LoraSeg L,
                                   float *out_f32, uint16_t *out16, int *err) {
  pdl_trigger();
  pdl_wait();  // launched as a dependent of the partial kernel
  const int nout = L.nseg * L.r;
  const int Rp = L.Rpad();
  const int64_t total = (int64_t)M * Rp;
  const size_t plane = (size_t)M * 64;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int m = (int)(idx / Rp), o = (int)(idx % Rp);
    if (o >= nout) {
      out16[idx] = 0;
      continue;
    }
    const float *src = part + (size_t)m * 64 + o;
    float acc = src[0];
    int ks = 1;
    for (; ks + 4 <= nsplit; ks += 4) {  // four loads in flight, added in order
      const float a0 = src[(size_t)ks * plane], a1 = src[(size_t)(ks + 1) * plane];
      const float a2 = src[(size_t)(ks + 2) * plane], a3 = src[(size_t)(ks + 3) * plane];
      acc += a0;
      acc += a1;
      acc += a2;
      acc += a3;
    }
    for (; ks < nsplit; ++ks) acc += src[(size_t)ks * plane];
    out_f32[(size_t)m * nout + o] = DU ? L.s * acc : acc;
    if (OF16) flag_range(half_out_of_range(L.s * acc), err);
    out16[idx] = st16<OF16>(L.s * acc);
  }
}

template <bool F16>
__global__ void pack_fwd_kernel(const LoraSeg L, int Ng, uint16_t *vl) {
  const int Rp = L.Rpad();
  const int64_t total = (int64_t)Ng * Rp;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int n = (int)(idx / Rp), c = (int)(idx % Rp);
    float v = 0.f;
    const int seg = c / L.r;
    if (seg < L.nseg && n >= L.off[seg] && n < L.off[seg] + L.n[seg])
      v = L.B[seg][(size_t)(n - L.off[seg]) * L.r + (c % L.r)];
    vl[idx] = st16<F16>(v);
  }
}

template <bool F16>
__global__ void pack_bwd_kernel(const LoraSeg L, int K, uint16_t *acat) {
  const int Rp = L.Rpad();
  const int64_t total = (int64_t)Rp * K;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int row = (int)(idx / K), k = (int)(idx % K);
    float v = 0.f;
    if (row < L.nseg * L.r) v = L.A[row / L.r][(size_t)(row % L.r) * K + k];
    acat[idx] = st16<F16>(v);
  }
}

// All eight LoRA operand packs of one layer in one launch: blockIdx.y = 2 g + (0: the
// forward's half Vl [n_out, Rpad] of group g, 1: the dX GEMM's bf16 Acat [Rpad, n_in]); the
// same element rule as pack_fwd_kernel / pack_bwd_kernel.
struct PackJobs {
  LoraSeg L[4];
  int n_out[4], n_in[4];
  uint16_t *vl[4], *ac[4];
};
// Eight consecutive elements per thread (one 16-byte store); 32-bit index arithmetic (a pack
// holds well under 2^31 elements).  K % 8 == 0 (checked by the caller) keeps an Acat group in
// one row; a vl group never leaves its row since Rpad is a multiple of 64.
__global__ void pack_layer_kernel(const PackJobs J) {
  const int g = blockIdx.y >> 1;
  const LoraSeg &L = J.L[g];
  const int Rp = L.Rpad(), nr = L.nseg * L.r;
  const int stride = gridDim.x * blockDim.x;
  if ((blockIdx.y & 1) == 0) {
    const int per_row = Rp / 8;
    const int total = J.n_out[g] * per_row;
    uint16_t *vl = J.vl[g];
    for (int it = blockIdx.x * blockDim.x + threadIdx.x; it < total; it += stride) {
      const int n = it / per_row, c0 = (it - n * per_row) * 8;
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c = c0 + e, seg = c / L.r;
        v[e] = 0.f;
        if (c < nr && n >= L.off[seg] && n < L.off[seg] + L.n[seg])
          v[e] = L.B[seg][(size_t)(n - L.off[seg]) * L.r + (c - seg * L.r)];
      }
      *reinterpret_cast<uint4 *>(vl + (size_t)n * Rp + c0) =
          make_uint4(pack_h2(v[0], v[1]), pack_h2(v[2], v[3]), pack_h2(v[4], v[5]), pack_h2(v[6], v[7]));
    }
  } else {
    const int K = J.n_in[g], per_row = K / 8;
    const int total = Rp * per_row;
    uint16_t *acat = J.ac[g];
    for (int it = blockIdx.x * blockDim.x + threadIdx.x; it < total; it += stride) {
      const int row = it / per_row, k0 = (it - row * per_row) * 8;
      uint4 o = make_uint4(0, 0, 0, 0);
      if (row < nr) {
        const float *src = L.A[row / L.r] + (size_t)(row % L.r) * K + k0;
        const float4 x0 = *reinterpret_cast<const float4 *>(src);
        const float4 x1 = *reinterpret_cast<const float4 *>(src + 4);
        o = make_uint4(pack_bf16x2(x0.x, x0.y), pack_bf16x2(x0.z, x0.w), pack_bf16x2(x1.x, x1.y),
                       pack_bf16x2(x1.z, x1.w));
      }
      *reinterpret_cast<uint4 *>(acat + (size_t)row * K + k0) = o;
    }
  }
}

// ------------------------------------------------------------------ cross-entropy
template <int NT>
SOUP_DEV float block_reduce(float v, float *sh, bool is_max) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  v = is_max ? warp_max(v) : warp_sum(v);
  if (lane == 0) sh[w] = v;
  __syncthreads();
  if (w == 0) {
    v = lane < NT / 32 ? sh[lane] : (is_max ? -INFINITY : 0.f);
    v = is_max ? warp_max(v) : warp_sum(v);
    if (lane == 0) sh[0] = v;
  }
  __syncthreads();
  const float r = sh[0];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(256) ce_chunk_fwd_kernel(const float *z, int ldz, int v0, int vc,
                                                           const int32_t *tok, int M, int S, int first,
                                                           float *rmax, float *rsum, float *zlab) {
  __shared__ float sh[32];
  const int m = blockIdx.x;
  const float *zr = z + (size_t)m * ldz;
  float mx = -INFINITY;
  for (int i = threadIdx.x; i < vc; i += 256) mx = fmaxf(mx, zr[i]);
  mx = block_reduce<256>(mx, sh, true);
  float sm = 0.f;
  for (int i = threadIdx.x; i < vc; i += 256) sm += expf(zr[i] - mx);
  sm = block_reduce<256>(sm, sh, false);
  if (threadIdx.x == 0) {
    const int t = m % S;
    if (first) {
      rmax[m] = mx;
      rsum[m] = sm;
      zlab[m] = 0.f;
    } else {
      const float om = rmax[m], os = rsum[m];
      const float nm = fmaxf(om, mx);
      rsum[m] = os * expf(om - nm) + sm * expf(mx - nm);
      rmax[m] = nm;
    }
    if (t < S - 1) {
      const int lab = tok[m + 1];
      if (lab >= v0 && lab < v0 + vc) zlab[m] = zr[lab - v0];
    }
  }
}

__global__ void __launch_bounds__(1024) ce_finalize_kernel(const float *rmax, const float *rsum,
                                                           const float *zlab, int M, int S,
                                                           float *lse, float *loss) {
  __shared__ float sh[32];
  float acc = 0.f;
  for (int m = threadIdx.x; m < M; m += 1024) {
    const float l = rmax[m] + logf(rsum[m]);
    lse[m] = l;
    if (m % S != S - 1) acc += l - zlab[m];
  }
  acc = block_reduce<1024>(acc, sh, false);
  if (threadIdx.x == 0) {
    const int nlab = (M / S) * (S - 1);
    *loss = acc / (float)nlab;
  }
}

__global__ void ce_chunk_bwd_kernel(const float *z, int ldz, int v0, int vc, const float *lse,
                                    const int32_t *tok, int M, int S, float inv_n, uint16_t *dz) {
  const int64_t total = (int64_t)M * vc;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int m = (int)(idx / vc), c = (int)(idx % vc);
    float g = 0.f;
    if (m % S != S - 1) {
      g = expf(z[(size_t)m * ldz + c] - lse[m]);
      if (tok[m + 1] == v0 + c) g -= 1.0f;
      g *= inv_n;
    }
    dz[idx] = f_to_bf16(g);
  }
}

__global__ void cast_bf16_kernel(const float *in, uint16_t *out, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = f_to_bf16(in[i]);
}

__global__ void nf4_dequant_kernel(const uint8_t *codes, const float *absmax, int64_t n,
                                   float *out_f32, uint16_t *out_bf16, const Codebook cb) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint8_t b = codes[i >> 1];
    const int code = (i & 1) ? (b & 15) : (b >> 4);
    const float v = cb.v[code] * absmax[i >> 6];
    if (out_f32) out_f32[i] = v;
    if (out_bf16) out_bf16[i] = f_to_bf16(v);
  }
}

int grid_for(int64_t n, int threads) {
  int64_t b = (n + threads - 1) / threads;
  if (b > 148 * 32) b = 148 * 32;
  return (int)(b < 1 ? 1 : b);
}

}  // namespace

void k_embed(const int32_t *tok, const uint16_t *E, int V, int H, int M, float *out, cudaStream_t st) {
  if (M > 0) {
    embed_kernel<<<M, 128, 0, st>>>(tok, E, V, H, out);
    count_launches(1);
  }
}
void k_rmsnorm_fwd(const float *h, const uint16_t *w, float eps, int M, int H, uint16_t *out,
                   bool out_f16, int *err, cudaStream_t st) {
  if (M <= 0) return;
  if (out_f16) rmsnorm_fwd_kernel<true><<<M, RMS_T, 0, st>>>(h, w, eps, M, H, out, err);
  else rmsnorm_fwd_kernel<false><<<M, RMS_T, 0, st>>>(h, w, eps, M, H, out, err);
  count_launches(1);
}
void k_rmsnorm_bwd(const float *dy, const float *h, const uint16_t *w, float eps, int M, int H,
                   const float *dres, float *out, uint16_t *out_bf16, cudaStream_t st) {
  if (M <= 0) return;
  rmsnorm_bwd_kernel<<<M, RMS_T, 0, st>>>(dy, h, w, eps, M, H, dres, out, out_bf16);
  count_launches(1);
}
void k_rope_fwd(uint16_t *qkv, int ld, const float *cos, const float *sin, int M, int S, int nh,
                int nkv, int d, bool f16, int *err, cudaStream_t st) {
  const int64_t n = (int64_t)M * (nh + nkv) * (d / 8);  // d % 8 == 0 (checked with the configuration)
  if (n <= 0) return;
  if (f16) rope_fwd_kernel<true><<<grid_for(n, 256), 256, 0, st>>>(qkv, ld, cos, sin, M, S, nh + nkv, d, err);
  else rope_fwd_kernel<false><<<grid_for(n, 256), 256, 0, st>>>(qkv, ld, cos, sin, M, S, nh + nkv, d, err);
  count_launches(1);
}
void k_rope_bwd(const float *dqkv, uint16_t *out, int ld, const float *cos, const float *sin,
                int M, int S, int nh, int nkv, int d, cudaStream_t st) {
  const int64_t n = (int64_t)M * (nh + 2 * nkv) * (d / 8);
  if (n <= 0) return;
  rope_bwd_kernel<<<grid_for(n, 256), 256, 0, st>>>(dqkv, out, ld, cos, sin, M, S, nh + nkv,
                                                    nh + 2 * nkv, d);
  count_launches(1);
}
void k_swiglu_fwd(const uint16_t *gu, int M, int I, uint16_t *act, bool f16, int *err, cudaStream_t st) {
  const int64_t n = (int64_t)M * I;
  if (n <= 0) return;
  if (I % 8 == 0) {
    const int64_t n8 = n / 8;
    if (f16) swiglu_fwd_kernel<true><<<grid_for(n8, 256), 256, 0, st>>>(gu, M, I, act, err);
    else swiglu_fwd_kernel<false><<<grid_for(n8, 256), 256, 0, st>>>(gu, M, I, act, err);
  } else {
    if (f16) swiglu_fwd_scalar_kernel<true><<<grid_for(n, 256), 256, 0, st>>>(gu, M, I, act, err);
    else swiglu_fwd_scalar_kernel<false><<<grid_for(n, 256), 256, 0, st>>>(gu, M, I, act, err);
  }
  count_launches(1);
}
void k_swiglu_bwd(const float *dact, const uint16_t *gu, int M, int I, uint16_t *dgu, bool gu_f16,
                  cudaStream_t st) {
  const int64_t n = (int64_t)M * I;
  if (n <= 0) return;
  const int64_t n8 = n / 8;  // inter % 8 == 0 (checked with the configuration)
  if (gu_f16) swiglu_bwd_kernel<true><<<grid_for(n8, 256), 256, 0, st>>>(dact, gu, M, I, dgu);
  else swiglu_bwd_kernel<false><<<grid_for(n8, 256), 256, 0, st>>>(dact, gu, M, I, dgu);
  count_launches(1);
}

// Splits of the LoRA reductions: enough 128-thread blocks to keep several resident per SM
// (they are latency-bound), while the float partials stay well below the operand traffic.
int lora_splits(int M, int K, int *KS) {
  const int rb = cdiv(M, 64);
  int want = std::max(1, cdiv(148 * 8, rb));
  want = std::min(want, std::max(1, cdiv(K, 128)));
  int ks = cdiv(cdiv(K, want), 64) * 64;
  if (KS) *KS = ks;
  return cdiv(K, ks);
}
size_t lora_scratch_floats(int M, int dim, int nout) {
  (void)nout;
  return (size_t)lora_splits(M, dim, nullptr) * M * 64;
}

template <bool DU>
static void lora_proj(const uint16_t *X, int ldx, int M, int K, const LoraSeg &L, float *out_f32,
                      uint16_t *out16, bool x_f16, bool o_f16, float *part, int *err, cudaStream_t st) {
  if (M <= 0) return;
  // one clustered launch (lora_proj.cu) for the shapes it takes; otherwise (or if its setup
  // failed: a tensor map or attribute the driver refused) partials + an ordered reduce
  if (lora_skinny(DU, X, ldx, M, K, L, out_f32, out16, x_f16, o_f16, err, st) == 0) return;
  int KS;
  const int ns = lora_splits(M, K, &KS);
  dim3 grid(cdiv(M, 64), ns);
  if (x_f16) lora_part_kernel<DU, true><<<grid, 128, 0, st>>>(X, ldx, M, K, KS, L, part);
  else lora_part_kernel<DU, false><<<grid, 128, 0, st>>>(X, ldx, M, K, KS, L, part);
  const int64_t n = (int64_t)M * L.Rpad();  // one thread per output
  if (o_f16) launch_pdl(lora_reduce_kernel<DU, true>, dim3(grid_for(n, 256)), dim3(256), 0, st, part, ns, M, L, out_f32, out16, err);
  else launch_pdl(lora_reduce_kernel<DU, false>, dim3(grid_for(n, 256)), dim3(256), 0, st, part, ns, M, L, out_f32, out16, err);
  count_launches(2);
}
static int seg_cols(const LoraSeg &L) {
  int Ng = 0;
  for (int p = 0; p < L.nseg; ++p) Ng = L.off[p] + L.n[p] > Ng ? L.off[p] + L.n[p] : Ng;
  return Ng;
}
void k_lora_down(const uint16_t *x, int lda, int M, int K, const LoraSeg &L, float *u_f32,
                 uint16_t *ul, bool x_f16, bool ul_f16, float *part, int *err, cudaStream_t st) {
  lora_proj<false>(x, lda, M, K, L, u_f32, ul, x_f16, ul_f16, part, err, st);
}
void k_lora_du(const uint16_t *dy, int ldy, int M, const LoraSeg &L, float *du_f32, uint16_t *dul,
               bool dy_f16, bool dul_f16, float *part, cudaStream_t st) {
  lora_proj<true>(dy, ldy, M, seg_cols(L), L, du_f32, dul, dy_f16, dul_f16, part, nullptr, st);
}
void k_pack_fwd(const LoraSeg &L, int Ng, uint16_t *vl, bool f16, cudaStream_t st) {
  const int64_t n = (int64_t)Ng * L.Rpad();
  if (f16) pack_fwd_kernel<true><<<grid_for(n, 256), 256, 0, st>>>(L, Ng, vl);
  else pack_fwd_kernel<false><<<grid_for(n, 256), 256, 0, st>>>(L, Ng, vl);
  count_launches(1);
}
void k_pack_bwd(const LoraSeg &L, int K, uint16_t *acat, bool f16, cudaStream_t st) {
  const int64_t n = (int64_t)L.Rpad() * K;
  if (f16) pack_bwd_kernel<true><<<grid_for(n, 256), 256, 0, st>>>(L, K, acat);
  else pack_bwd_kernel<false><<<grid_for(n, 256), 256, 0, st>>>(L, K, acat);
  count_launches(1);
}
void k_pack_layer(const LoraSeg (&L)[4], const int n_out[4], const int n_in[4], uint16_t *const vl[4],
                  uint16_t *const ac[4], cudaStream_t st) {
  PackJobs J;
  int64_t most = 1;
  for (int g = 0; g < 4; ++g) {
    J.L[g] = L[g];
    J.n_out[g] = n_out[g];
    J.n_in[g] = n_in[g];
    J.vl[g] = vl[g];
    J.ac[g] = ac[g];
    most = std::max(most, (int64_t)L[g].Rpad() * std::max(n_out[g], n_in[g]));
  }
  bool vec = true;  // the 8-wide kernel: K % 8, 16-byte aligned A rows and packs
  for (int g = 0; g < 4; ++g) {
    vec = vec && n_in[g] % 8 == 0 && (reinterpret_cast<uintptr_t>(vl[g]) & 15) == 0 &&
          (reinterpret_cast<uintptr_t>(ac[g]) & 15) == 0;
    for (int p = 0; p < L[g].nseg; ++p) vec = vec && (reinterpret_cast<uintptr_t>(L[g].A[p]) & 15) == 0;
  }
  if (!vec) {  // element by element, pack by pack
    for (int g = 0; g < 4; ++g) {
      k_pack_fwd(L[g], n_out[g], vl[g], true, st);
      k_pack_bwd(L[g], n_in[g], ac[g], false, st);
    }
    return;
  }
  // enough blocks for the largest pack, at most two waves per job
  const int bx = std::min(grid_for(most / 8, 256), 148 * 2);
  pack_layer_kernel<<<dim3(bx, 8), 256, 0, st>>>(J);
  count_launches(1);
}
void k_ce_chunk_fwd(const float *z, int ldz, int v0, int vc, const int32_t *tok, int M, int S,
                    int first, float *rmax, float *rsum, float *zlab, cudaStream_t st) {
  {
    ce_chunk_fwd_kernel<<<M, 256, 0, st>>>(z, ldz, v0, vc, tok, M, S, first, rmax, rsum, zlab);
    count_launches(1);
  }
}
void k_ce_finalize(const float *rmax, const float *rsum, const float *zlab, int M, int S,
                   float *lse, float *loss, cudaStream_t st) {
  {
    ce_finalize_kernel<<<1, 1024, 0, st>>>(rmax, rsum, zlab, M, S, lse, loss);
    count_launches(1);
  }
}
void k_ce_chunk_bwd(const float *z, int ldz, int v0, int vc, const float *lse, const int32_t *tok,
                    int M, int S, float inv_n, uint16_t *dz, cudaStream_t st) {
  const int64_t n = (int64_t)M * vc;
  {
    ce_chunk_bwd_kernel<<<grid_for(n, 256), 256, 0, st>>>(z, ldz, v0, vc, lse, tok, M, S, inv_n, dz);
    count_launches(1);
  }
}
void k_cast_bf16(const float *in, uint16_t *out, int64_t n, cudaStream_t st) {
  if (n > 0) {
    cast_bf16_kernel<<<grid_for(n, 256), 256, 0, st>>>(in, out, n);
    count_launches(1);
  }
}
// Waits on an mbarrier that nothing ever arrives on, through the same bounded wait every
// pipelined kernel uses, with a limit of `limit` cycles: the wait gives up, raises
// SOUP_KERR_WAIT_TIMEOUT in *err and the kernel returns.  Exercises the error path (flag set
// on the device, read by the host) without a real stall.
__global__ void wait_probe_kernel(int *err, long long limit) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  soupk::mbar_init(&bar, 1);
  soupk::fence_mbar_init();
  abort_flag = 0;
  volatile int *ab = &abort_flag;
  soupk::mbar_wait(&bar, 0, err, ab, limit);
}
void k_wait_probe(int *err, long long limit_cycles, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(err, limit_cycles);
  count_launches(1);
}
void k_nf4_dequant(const uint8_t *codes, const float *absmax, int64_t n, float *out_f32,
                   uint16_t *out_bf16, cudaStream_t st) {
  if (n > 0)
    {
    nf4_dequant_kernel<<<grid_for(n, 256), 256, 0, st>>>(codes, absmax, n, out_f32, out_bf16,
                                                         nf4_codebook_param());
    count_launches(1);
  }
}

}  // namespace soup
