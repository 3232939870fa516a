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
template <bool F16>
__global__ void rmsnorm_fwd_kernel(const float *h, const uint16_t *w, float eps, int M, int H,
                                   uint16_t *out) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const float *x = h + (size_t)row * H;
  float ss = 0.f;
  for (int i = lane * 4; i < H; i += 128) {
    const float4 v = *reinterpret_cast<const float4 *>(x + i);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  const float r = 1.0f / sqrtf(ss / (float)H + eps);
  uint16_t *o = out + (size_t)row * H;
  for (int i = lane * 4; i < H; i += 128) {
    const float4 v = *reinterpret_cast<const float4 *>(x + i);
    const uint2 wv = *reinterpret_cast<const uint2 *>(w + i);
    uint2 res;
    res.x = pack16x2<F16>(v.x * r * bf16_lo(wv.x), v.y * r * bf16_hi(wv.x));
    res.y = pack16x2<F16>(v.z * r * bf16_lo(wv.y), v.w * r * bf16_hi(wv.y));
    *reinterpret_cast<uint2 *>(o + i) = res;
  }
}

__global__ void rmsnorm_bwd_kernel(const float *dy, const float *h, const uint16_t *w, float eps,
                                   int M, int H, const float *dres, float *out, uint16_t *out_bf16) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const float *x = h + (size_t)row * H;
  const float *g = dy + (size_t)row * H;
  float ss = 0.f, sgh = 0.f;
  for (int i = lane * 4; i < H; i += 128) {
    const float4 v = *reinterpret_cast<const float4 *>(x + i);
    const float4 d = *reinterpret_cast<const float4 *>(g + i);
    const uint2 wv = *reinterpret_cast<const uint2 *>(w + i);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    sgh += d.x * bf16_lo(wv.x) * v.x + d.y * bf16_hi(wv.x) * v.y + d.z * bf16_lo(wv.y) * v.z +
           d.w * bf16_hi(wv.y) * v.w;
  }
  ss = warp_sum(ss);
  sgh = warp_sum(sgh);
  const float r = 1.0f / sqrtf(ss / (float)H + eps);
  const float c = r * r * r * sgh / (float)H;  // dx = r*g - x * r^3 * sum(g*x) / H
  float *o = out + (size_t)row * H;
  const float *dr = dres ? dres + (size_t)row * H : nullptr;
  uint16_t *ob = out_bf16 ? out_bf16 + (size_t)row * H : nullptr;
  for (int i = lane * 4; i < H; i += 128) {
    const float4 v = *reinterpret_cast<const float4 *>(x + i);
    const float4 d = *reinterpret_cast<const float4 *>(g + i);
    const uint2 wv = *reinterpret_cast<const uint2 *>(w + i);
    float4 res = make_float4(r * d.x * bf16_lo(wv.x) - v.x * c, r * d.y * bf16_hi(wv.x) - v.y * c,
                             r * d.z * bf16_lo(wv.y) - v.z * c, r * d.w * bf16_hi(wv.y) - v.w * c);
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
template <bool F16>
__global__ void rope_fwd_kernel(uint16_t *qkv, int ld, const float *cs, const float *sn, int M,
                                int S, int nheads_rot, int d) {
  const int half = d >> 1;
  const int64_t total = (int64_t)M * nheads_rot * half;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int i = (int)(idx % half);
    const int64_t rest = idx / half;
    const int head = (int)(rest % nheads_rot);
    const int m = (int)(rest / nheads_rot);
    const int pos = m % S;
    uint16_t *p = qkv + (size_t)m * ld + (size_t)head * d;
    const float x1 = ld16<F16>(p[i]), x2 = ld16<F16>(p[i + half]);
    const float c = cs[pos * half + i], s = sn[pos * half + i];
    p[i] = st16<F16>(x1 * c - x2 * s);
    p[i + half] = st16<F16>(x2 * c + x1 * s);
  }
}

__global__ void rope_bwd_kernel(const float *dqkv, uint16_t *out, int ld, const float *cs,
                                const float *sn, int M, int S, int nheads_rot, int nheads_all,
                                int d) {
  const int half = d >> 1;
  const int64_t total = (int64_t)M * nheads_all * half;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int i = (int)(idx % half);
    const int64_t rest = idx / half;
    const int head = (int)(rest % nheads_all);
    const int m = (int)(rest / nheads_all);
    const float *g = dqkv + (size_t)m * ld + (size_t)head * d;
    uint16_t *o = out + (size_t)m * ld + (size_t)head * d;
    const float d1 = g[i], d2 = g[i + half];
    if (head < nheads_rot) {
      const int pos = m % S;
      const float c = cs[pos * half + i], s = sn[pos * half + i];
      o[i] = f_to_bf16(d1 * c + d2 * s);
      o[i + half] = f_to_bf16(d2 * c - d1 * s);
    } else {
      o[i] = f_to_bf16(d1);
      o[i + half] = f_to_bf16(d2);
    }
  }
}

// ------------------------------------------------------------------ SwiGLU
SOUP_DEV float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

template <bool F16>
__global__ void swiglu_fwd_kernel(const uint16_t *gu, int M, int I, uint16_t *act) {
  const int64_t total = (int64_t)M * I;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = idx / I, j = idx % I;
    const float g = ld16<F16>(gu[m * 2 * I + j]);
    const float u = ld16<F16>(gu[m * 2 * I + I + j]);
    act[idx] = st16<F16>(g * sigmoidf_(g) * u);
  }
}

template <bool F16>
__global__ void swiglu_bwd_kernel(const float *dact, const uint16_t *gu, int M, int I, uint16_t *dgu) {
  const int64_t total = (int64_t)M * I;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = idx / I, j = idx % I;
    const float g = ld16<F16>(gu[m * 2 * I + j]);
    const float u = ld16<F16>(gu[m * 2 * I + I + j]);
    const float da = dact[idx];
    const float sg = sigmoidf_(g);
    dgu[m * 2 * I + j] = f_to_bf16(da * u * (sg * (1.0f + g * (1.0f - sg))));
    dgu[m * 2 * I + I + j] = f_to_bf16(da * g * sg);
  }
}

// ------------------------------------------------------------------ LoRA projections
// part[split][m][o] = sum over k in the split's range of X[m, k] * W_o(k), o < 64, with
//   DOWN: X = x [M, K], W_o(k) = A_seg[j, k]                       (u = x A^T)
//   DU:   X = dY [M, Ng], W_o(k) = B_seg[k - off_seg, j] inside the segment, else 0
// Tile: 32 rows x 64 outputs per 256-thread block; blockIdx.y picks the K range.  The
// splits are then summed in split order by lora_reduce_kernel (no atomics).
template <bool DU, bool XF16>
__global__ void __launch_bounds__(256) lora_part_kernel(const uint16_t *X, int ldx, int M, int K,
                                                        int KS, const LoraSeg L, float *part) {
  __shared__ float xs[32][65];
  __shared__ float ws[64][65];
  const int t = threadIdx.x;
  const int m0 = blockIdx.x * 32;
  const int kb = blockIdx.y * KS, ke = min(K, kb + KS);
  const int nout = L.nseg * L.r;
  const int row = t >> 3, cb = t & 7;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int k0 = kb; k0 < ke; k0 += 64) {
    for (int i = t; i < 32 * 64; i += 256) {
      const int rr = i >> 6, kk = i & 63;
      const int m = m0 + rr, k = k0 + kk;
      xs[rr][kk] = (m < M && k < ke) ? ld16<XF16>(X[(size_t)m * ldx + k]) : 0.f;
    }
    for (int i = t; i < 64 * 64; i += 256) {
      const int o = i >> 6, kk = i & 63;
      const int k = k0 + kk;
      float v = 0.f;
      if (o < nout && k < ke) {
        const int seg = o / L.r, j = o % L.r;
        if (!DU) {
          v = L.A[seg][(size_t)j * K + k];
        } else if (k >= L.off[seg] && k < L.off[seg] + L.n[seg]) {
          v = L.B[seg][(size_t)(k - L.off[seg]) * L.r + j];
        }
      }
      ws[o][kk] = v;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 64; ++kk) {
      const float xv = xs[row][kk];
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[c] = fmaf(xv, ws[cb + 8 * c][kk], acc[c]);
    }
    __syncthreads();
  }
  const int m = m0 + row;
  if (m >= M) return;
  float *dst = part + ((size_t)blockIdx.y * M + m) * 64;
#pragma unroll
  for (int c = 0; c < 8; ++c) dst[cb + 8 * c] = acc[c];
}

// out_f32[m, o] = (DU ? s : 1) * sum_split part; out16[m, o] = 16-bit(s * sum), zero padded.
template <bool DU, bool OF16>
__global__ void lora_reduce_kernel(const float *part, int nsplit, int M, const LoraSeg L,
                                   float *out_f32, uint16_t *out16) {
  const int nout = L.nseg * L.r;
  const int Rp = L.Rpad();
  const int64_t total = (int64_t)M * Rp;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int m = (int)(idx / Rp), o = (int)(idx % Rp);
    if (o >= nout) {
      out16[idx] = 0;
      continue;
    }
    float acc = 0.f;
    for (int ks = 0; ks < nsplit; ++ks) acc += part[((size_t)ks * M + m) * 64 + o];
    out_f32[(size_t)m * nout + o] = DU ? L.s * acc : acc;
    out16[idx] = st16<OF16>(L.s * acc);
  }
}

// dB_seg[n - off, j] = s * sum_m dY[m, n] u[m, seg*r + j]; 64 columns per block.
template <bool F16>
__global__ void __launch_bounds__(256) lora_dB_kernel(const uint16_t *dy, int ldy, int M, int Ng,
                                                      const float *u, const LoraSeg L) {
  __shared__ float ys[32][65];
  __shared__ float us[32][65];
  const int t = threadIdx.x;
  const int n0 = blockIdx.x * 64;
  const int c = t & 63, jg = t >> 6;
  const int n = n0 + c;
  const int nout = L.nseg * L.r;
  int seg = -1;
  for (int p = 0; p < L.nseg; ++p)
    if (n >= L.off[p] && n < L.off[p] + L.n[p]) seg = p;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int mb = 0; mb < M; mb += 32) {
    for (int i = t; i < 32 * 64; i += 256) {
      const int rr = i >> 6, cc = i & 63;
      const int m = mb + rr, nn = n0 + cc;
      ys[rr][cc] = (m < M && nn < Ng) ? ld16<F16>(dy[(size_t)m * ldy + nn]) : 0.f;
    }
    for (int i = t; i < 32 * 64; i += 256) {
      const int rr = i >> 6, o = i & 63;
      const int m = mb + rr;
      us[rr][o] = (m < M && o < nout) ? u[(size_t)m * nout + o] : 0.f;
    }
    __syncthreads();
    if (seg >= 0) {
      for (int rr = 0; rr < 32; ++rr) {
        const float yv = ys[rr][c];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j = jg + 4 * i;
          if (j < L.r) acc[i] = fmaf(yv, us[rr][seg * L.r + j], acc[i]);
        }
      }
    }
    __syncthreads();
  }
  if (seg < 0) return;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int j = jg + 4 * i;
    if (j < L.r) L.dB[seg][(size_t)(n - L.off[seg]) * L.r + j] = L.s * acc[i];
  }
}

// dA_seg[j, k] = sum_m du[m, seg*r + j] x[m, k]; 64 columns per block.
template <bool F16>
__global__ void __launch_bounds__(256) lora_dA_kernel(const float *du, const uint16_t *x, int ldx,
                                                      int M, int K, const LoraSeg L) {
  __shared__ float xs[32][65];
  __shared__ float ds[32][65];
  const int t = threadIdx.x;
  const int k0 = blockIdx.x * 64;
  const int c = t & 63, og = t >> 6;
  const int k = k0 + c;
  const int nout = L.nseg * L.r;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int mb = 0; mb < M; mb += 32) {
    for (int i = t; i < 32 * 64; i += 256) {
      const int rr = i >> 6, cc = i & 63;
      const int m = mb + rr, kk = k0 + cc;
      xs[rr][cc] = (m < M && kk < K) ? ld16<F16>(x[(size_t)m * ldx + kk]) : 0.f;
      ds[rr][cc] = (m < M && cc < nout) ? du[(size_t)m * nout + cc] : 0.f;
    }
    __syncthreads();
    for (int rr = 0; rr < 32; ++rr) {
      const float xv = xs[rr][c];
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = fmaf(ds[rr][og + 4 * i], xv, acc[i]);
    }
    __syncthreads();
  }
  if (k >= K) return;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int o = og + 4 * i;
    if (o < nout) L.dA[o / L.r][(size_t)(o % L.r) * K + k] = acc[i];
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
                   bool out_f16, cudaStream_t st) {
  if (M <= 0) return;
  if (out_f16) rmsnorm_fwd_kernel<true><<<cdiv(M, 8), 256, 0, st>>>(h, w, eps, M, H, out);
  else rmsnorm_fwd_kernel<false><<<cdiv(M, 8), 256, 0, st>>>(h, w, eps, M, H, out);
  count_launches(1);
}
void k_rmsnorm_bwd(const float *dy, const float *h, const uint16_t *w, float eps, int M, int H,
                   const float *dres, float *out, uint16_t *out_bf16, cudaStream_t st) {
  if (M <= 0) return;
  rmsnorm_bwd_kernel<<<cdiv(M, 8), 256, 0, st>>>(dy, h, w, eps, M, H, dres, out, out_bf16);
  count_launches(1);
}
void k_rope_fwd(uint16_t *qkv, int ld, const float *cos, const float *sin, int M, int S, int nh,
                int nkv, int d, bool f16, cudaStream_t st) {
  const int64_t n = (int64_t)M * (nh + nkv) * (d / 2);
  if (n <= 0) return;
  if (f16) rope_fwd_kernel<true><<<grid_for(n, 256), 256, 0, st>>>(qkv, ld, cos, sin, M, S, nh + nkv, d);
  else rope_fwd_kernel<false><<<grid_for(n, 256), 256, 0, st>>>(qkv, ld, cos, sin, M, S, nh + nkv, d);
  count_launches(1);
}
void k_rope_bwd(const float *dqkv, uint16_t *out, int ld, const float *cos, const float *sin,
                int M, int S, int nh, int nkv, int d, cudaStream_t st) {
  const int64_t n = (int64_t)M * (nh + 2 * nkv) * (d / 2);
  if (n <= 0) return;
  rope_bwd_kernel<<<grid_for(n, 256), 256, 0, st>>>(dqkv, out, ld, cos, sin, M, S, nh + nkv,
                                                    nh + 2 * nkv, d);
  count_launches(1);
}
void k_swiglu_fwd(const uint16_t *gu, int M, int I, uint16_t *act, bool f16, cudaStream_t st) {
  const int64_t n = (int64_t)M * I;
  if (n <= 0) return;
  if (f16) swiglu_fwd_kernel<true><<<grid_for(n, 256), 256, 0, st>>>(gu, M, I, act);
  else swiglu_fwd_kernel<false><<<grid_for(n, 256), 256, 0, st>>>(gu, M, I, act);
  count_launches(1);
}
void k_swiglu_bwd(const float *dact, const uint16_t *gu, int M, int I, uint16_t *dgu, bool gu_f16,
                  cudaStream_t st) {
  const int64_t n = (int64_t)M * I;
  if (n <= 0) return;
  if (gu_f16) swiglu_bwd_kernel<true><<<grid_for(n, 256), 256, 0, st>>>(dact, gu, M, I, dgu);
  else swiglu_bwd_kernel<false><<<grid_for(n, 256), 256, 0, st>>>(dact, gu, M, I, dgu);
  count_launches(1);
}

int lora_splits(int M, int K, int *KS) {
  const int rb = cdiv(M, 32);
  int want = std::max(1, cdiv(296, rb));
  want = std::min(want, cdiv(K, 64));
  int ks = cdiv(cdiv(K, want), 64) * 64;
  if (KS) *KS = ks;
  return cdiv(K, ks);
}
size_t lora_partial_floats(int M, int K) { return (size_t)lora_splits(M, K, nullptr) * M * 64; }

template <bool DU>
static void lora_proj(const uint16_t *X, int ldx, int M, int K, const LoraSeg &L, float *out_f32,
                      uint16_t *out16, bool x_f16, bool o_f16, float *part, cudaStream_t st) {
  if (M <= 0) return;
  int KS;
  const int ns = lora_splits(M, K, &KS);
  dim3 grid(cdiv(M, 32), ns);
  if (x_f16) lora_part_kernel<DU, true><<<grid, 256, 0, st>>>(X, ldx, M, K, KS, L, part);
  else lora_part_kernel<DU, false><<<grid, 256, 0, st>>>(X, ldx, M, K, KS, L, part);
  const int64_t n = (int64_t)M * L.Rpad();
  if (o_f16) lora_reduce_kernel<DU, true><<<grid_for(n, 256), 256, 0, st>>>(part, ns, M, L, out_f32, out16);
  else lora_reduce_kernel<DU, false><<<grid_for(n, 256), 256, 0, st>>>(part, ns, M, L, out_f32, out16);
  count_launches(2);
}
void k_lora_down(const uint16_t *x, int lda, int M, int K, const LoraSeg &L, float *u_f32,
                 uint16_t *ul, bool x_f16, bool ul_f16, float *part, cudaStream_t st) {
  lora_proj<false>(x, lda, M, K, L, u_f32, ul, x_f16, ul_f16, part, st);
}
void k_lora_du(const uint16_t *dy, int ldy, int M, const LoraSeg &L, float *du_f32, uint16_t *dul,
               bool dy_f16, bool dul_f16, float *part, cudaStream_t st) {
  int Ng = 0;
  for (int p = 0; p < L.nseg; ++p) Ng = L.off[p] + L.n[p] > Ng ? L.off[p] + L.n[p] : Ng;
  lora_proj<true>(dy, ldy, M, Ng, L, du_f32, dul, dy_f16, dul_f16, part, st);
}
void k_lora_dB(const uint16_t *dy, int ldy, int M, const float *u_f32, const LoraSeg &L, bool dy_f16,
               cudaStream_t st) {
  int Ng = 0;
  for (int p = 0; p < L.nseg; ++p) Ng = L.off[p] + L.n[p] > Ng ? L.off[p] + L.n[p] : Ng;
  if (dy_f16) lora_dB_kernel<true><<<cdiv(Ng, 64), 256, 0, st>>>(dy, ldy, M, Ng, u_f32, L);
  else lora_dB_kernel<false><<<cdiv(Ng, 64), 256, 0, st>>>(dy, ldy, M, Ng, u_f32, L);
  count_launches(1);
}
void k_lora_dA(const float *du_f32, const uint16_t *x, int lda, int M, int K, const LoraSeg &L,
               bool x_f16, cudaStream_t st) {
  if (x_f16) lora_dA_kernel<true><<<cdiv(K, 64), 256, 0, st>>>(du_f32, x, lda, M, K, L);
  else lora_dA_kernel<false><<<cdiv(K, 64), 256, 0, st>>>(du_f32, x, lda, M, K, L);
  count_launches(1);
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
