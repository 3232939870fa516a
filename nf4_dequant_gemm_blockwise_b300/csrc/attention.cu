// Causal grouped-query attention, forward and backward, on the warp-level tensor-core MMA
// (m16n8k16): the path for the shapes the tcgen05 kernels (attention_tc.cu) do not take, a
// head dimension other than 64 or 128 or more than 8 query heads per key/value head
// ("Layer streaming: fine-tune a model that does not fit in your card", "How it works": the
// family's own decoder layer; query head h reads key/value head floor(h * n_kv / n_h);
// softmax(q k^T / sqrt(d) + causal mask) v).
//
// Flash-style tiling: the S x S score matrix is never stored.  The forward keeps a running
// row max and sum per query row and writes the base-2 log-sum-exp; the backward recomputes
// the probabilities from it.  q, k, v and the output are IEEE half (the forward's operand
// format); the backward recomputes the scores from the same half q and k, then forms every
// product with a gradient in bf16 (v, k and q are converted to bf16 when they are staged).
// Determinism: every output element is accumulated by one thread in a fixed order; the
// key/value gradients of the heads that share a key/value head are summed by a separate
// kernel in head order (no atomics).
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "util.h"

namespace soup {
namespace {
using namespace soupk;

SOUP_DEV void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
SOUP_DEV void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
SOUP_DEV float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}
SOUP_DEV float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v + __shfl_xor_sync(0xffffffffu, v, 2);
}
SOUP_DEV uint32_t ld32(const uint16_t *p) { return *reinterpret_cast<const uint32_t *>(p); }

// Copy rows [r0, r0+nrows) x D of one head (column offset col) into smem [nrows][D+8];
// rows past S are zero.  TO_BF16: the source is half and is converted to bf16.
template <int D, bool TO_BF16 = false>
SOUP_DEV void load_tile(uint16_t *dst, const uint16_t *src, int ld, size_t rowbase, int r0,
                        int nrows, int S, int col) {
  constexpr int LDS = D + 8;
  for (int i = threadIdx.x; i < nrows * (D / 8); i += blockDim.x) {
    const int r = i / (D / 8), c = (i % (D / 8)) * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r0 + r < S) v = *reinterpret_cast<const uint4 *>(src + (rowbase + r0 + r) * ld + col + c);
    if (TO_BF16) {
      v.x = pack_bf16x2(lo16<true>(v.x), hi16<true>(v.x));
      v.y = pack_bf16x2(lo16<true>(v.y), hi16<true>(v.y));
      v.z = pack_bf16x2(lo16<true>(v.z), hi16<true>(v.z));
      v.w = pack_bf16x2(lo16<true>(v.w), hi16<true>(v.w));
    }
    *reinterpret_cast<uint4 *>(dst + r * LDS + c) = v;
  }
}

// ------------------------------------------------------------------------ forward
template <int D, bool F16>
__global__ void __launch_bounds__(128) attn_fwd_kernel(const uint16_t *qkv, int ld, int S, int nh,
                                                       int nkv, uint16_t *out, float *lse,
                                                       float scale_log2) {
  constexpr int KT = 64, LDS = D + 8, NC = D / 16;
  __shared__ __align__(16) uint16_t Ks[KT * LDS];
  __shared__ __align__(16) uint16_t Vs[KT * LDS];
  const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = (h * nkv) / nh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, tq = lane & 3;
  const int q0 = qb * 64 + warp * 16;
  const size_t rowbase = (size_t)b * S;
  const uint16_t *Qg = qkv + (size_t)h * D;

  uint32_t qf[NC][4];
#pragma unroll
  for (int kc = 0; kc < NC; ++kc) {
    const int r0 = q0 + gr, r1 = r0 + 8, c = kc * 16 + 2 * tq;
    qf[kc][0] = r0 < S ? ld32(Qg + (rowbase + r0) * ld + c) : 0u;
    qf[kc][1] = r1 < S ? ld32(Qg + (rowbase + r1) * ld + c) : 0u;
    qf[kc][2] = r0 < S ? ld32(Qg + (rowbase + r0) * ld + c + 8) : 0u;
    qf[kc][3] = r1 < S ? ld32(Qg + (rowbase + r1) * ld + c + 8) : 0u;
  }
  float oacc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

  const int q_end = min(S, qb * 64 + 64);
  const int n_tiles = (q_end + KT - 1) / KT;
  for (int kt = 0; kt < n_tiles; ++kt) {
    const int k0 = kt * KT;
    __syncthreads();
    load_tile<D>(Ks, qkv, ld, rowbase, k0, KT, S, (nh + g) * D);
    load_tile<D>(Vs, qkv, ld, rowbase, k0, KT, S, (nh + nkv + g) * D);
    __syncthreads();
    if (k0 > q0 + 15) continue;  // every key of the tile is after every query of this warp
    float sacc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
      for (int kc = 0; kc < NC; ++kc) {
        const uint16_t *kp = Ks + (nt * 8 + gr) * LDS + kc * 16 + 2 * tq;
        mma16816<F16>(sacc[nt], qf[kc], ld32(kp), ld32(kp + 8));
      }
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = q0 + gr + (e >= 2 ? 8 : 0);
        const int key = k0 + nt * 8 + 2 * tq + (e & 1);
        const float v = sacc[nt][e] * scale_log2;
        sacc[nt][e] = (key > row || key >= S) ? -INFINITY : v;
      }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) mx = fmaxf(mx, fmaxf(sacc[nt][2 * r], sacc[nt][2 * r + 1]));
      mx = quad_max(mx);
      const float mnew = fmaxf(mrow[r], mx);
      const float mref = mnew == -INFINITY ? 0.f : mnew;
      const float corr = exp2f(mrow[r] - mref);
      mrow[r] = mnew;
      lrow[r] *= corr;
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        oacc[dn][2 * r] *= corr;
        oacc[dn][2 * r + 1] *= corr;
      }
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const float p0 = exp2f(sacc[nt][2 * r] - mref), p1 = exp2f(sacc[nt][2 * r + 1] - mref);
        sacc[nt][2 * r] = p0;
        sacc[nt][2 * r + 1] = p1;
        lrow[r] += p0 + p1;
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t a[4];
      a[0] = pack16x2<F16>(sacc[2 * j][0], sacc[2 * j][1]);
      a[1] = pack16x2<F16>(sacc[2 * j][2], sacc[2 * j][3]);
      a[2] = pack16x2<F16>(sacc[2 * j + 1][0], sacc[2 * j + 1][1]);
      a[3] = pack16x2<F16>(sacc[2 * j + 1][2], sacc[2 * j + 1][3]);
      const int key = j * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int dn = 0; dn < NC; ++dn) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(smem_u32(Vs + key * LDS + dn * 16 + (lane >> 4) * 8), r0, r1, r2, r3);
        mma16816<F16>(oacc[2 * dn], a, r0, r1);
        mma16816<F16>(oacc[2 * dn + 1], a, r2, r3);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float l = quad_sum(lrow[r]);
    const int row = q0 + gr + 8 * r;
    if (row >= S) continue;
    const float inv = l > 0.f ? 1.0f / l : 0.f;
    uint16_t *o = out + (rowbase + row) * (size_t)(nh * D) + (size_t)h * D;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn)
      *reinterpret_cast<uint32_t *>(o + dn * 8 + 2 * tq) =
          pack16x2<F16>(oacc[dn][2 * r] * inv, oacc[dn][2 * r + 1] * inv);
    if (tq == 0) lse[((size_t)b * nh + h) * S + row] = mrow[r] + log2f(l);
  }
}

// ------------------------------------------------------------------------ backward
// dsum[b, h, q] = sum_d dO[q, h, d] * O[q, h, d]   (one warp per (row, head))
__global__ void attn_dsum_kernel(const uint16_t *o, const uint16_t *dO, int M, int S, int nh, int D,
                                 float *dsum) {
  const int64_t wid = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (int64_t)M * nh) return;
  const int m = (int)(wid / nh), h = (int)(wid % nh);
  const uint16_t *a = o + (size_t)m * nh * D + (size_t)h * D;
  const uint16_t *g = dO + (size_t)m * nh * D + (size_t)h * D;
  float s = 0.f;
  for (int i = lane * 2; i < D; i += 64) {
    const uint32_t x = ld32(a + i), y = ld32(g + i);
    s += lo16<true>(x) * bf16_lo(y) + hi16<true>(x) * bf16_hi(y);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) {
    const int b = m / S, t = m % S;
    dsum[((size_t)b * nh + h) * S + t] = s;
  }
}

// Per query head: dK_h, dV_h for one block of 64 keys (4 warps x 16 keys), written to
// per-head partial buffers part_k/part_v [B, nh, S, D].
template <int D>
__global__ void __launch_bounds__(128) attn_bwd_dkdv_kernel(
    const uint16_t *qkv, int ld, const uint16_t *dO, const float *lse, const float *dsum, int S,
    int nh, int nkv, float *part_k, float *part_v, float scale_log2, float scale) {
  constexpr int QT = 32, LDS = D + 8, NC = D / 16;
  extern __shared__ __align__(16) uint8_t smraw[];
  uint16_t *Ks = reinterpret_cast<uint16_t *>(smraw);  // half
  uint16_t *Vs = Ks + 64 * LDS;                         // bf16
  uint16_t *Qs = Vs + 64 * LDS;                         // half
  uint16_t *Qb = Qs + QT * LDS;                         // bf16
  uint16_t *dOs = Qb + QT * LDS;                        // bf16
  float *lse_s = reinterpret_cast<float *>(dOs + QT * LDS);
  float *ds_s = lse_s + QT;

  const int kb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = (h * nkv) / nh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, tq = lane & 3;
  const int kw0 = kb * 64 + warp * 16;
  const size_t rowbase = (size_t)b * S;

  load_tile<D>(Ks, qkv, ld, rowbase, kb * 64, 64, S, (nh + g) * D);
  load_tile<D, true>(Vs, qkv, ld, rowbase, kb * 64, 64, S, (nh + nkv + g) * D);

  float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[i][e] = dv[i][e] = 0.f;

  const int arow = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix A-row
  for (int q0 = (kb * 64 / QT) * QT; q0 < S; q0 += QT) {
    __syncthreads();
    load_tile<D>(Qs, qkv, ld, rowbase, q0, QT, S, h * D);
    load_tile<D, true>(Qb, qkv, ld, rowbase, q0, QT, S, h * D);
    load_tile<D>(dOs, dO, nh * D, rowbase, q0, QT, S, h * D);
    for (int i = threadIdx.x; i < QT; i += blockDim.x) {
      const bool ok = q0 + i < S;
      lse_s[i] = ok ? lse[((size_t)b * nh + h) * S + q0 + i] : INFINITY;
      ds_s[i] = ok ? dsum[((size_t)b * nh + h) * S + q0 + i] : 0.f;
    }
    __syncthreads();
    if (q0 + QT - 1 < kw0) continue;  // every query of the tile is before every key of the warp
    float st[QT / 8][4], dpt[QT / 8][4];
#pragma unroll
    for (int nt = 0; nt < QT / 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) st[nt][e] = dpt[nt][e] = 0.f;
#pragma unroll
    for (int kc = 0; kc < NC; ++kc) {
      uint32_t ak[4], av[4];
      const int col = kc * 16 + (lane >> 4) * 8;
      ldsm_x4(smem_u32(Ks + arow * LDS + col), ak[0], ak[1], ak[2], ak[3]);
      ldsm_x4(smem_u32(Vs + arow * LDS + col), av[0], av[1], av[2], av[3]);
#pragma unroll
      for (int nt = 0; nt < QT / 8; ++nt) {
        const uint16_t *qp = Qs + (nt * 8 + gr) * LDS + kc * 16 + 2 * tq;
        mma16816<true>(st[nt], ak, ld32(qp), ld32(qp + 8));
        const uint16_t *dp = dOs + (nt * 8 + gr) * LDS + kc * 16 + 2 * tq;
        mma16816<false>(dpt[nt], av, ld32(dp), ld32(dp + 8));
      }
    }
#pragma unroll
    for (int nt = 0; nt < QT / 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kw0 + gr + (e >= 2 ? 8 : 0);
        const int ql = nt * 8 + 2 * tq + (e & 1);
        const int q = q0 + ql;
        const float p = (q >= key && q < S && key < S) ? exp2f(st[nt][e] * scale_log2 - lse_s[ql]) : 0.f;
        st[nt][e] = p;
        dpt[nt][e] = p * (dpt[nt][e] - ds_s[ql]);
      }
#pragma unroll
    for (int j = 0; j < QT / 16; ++j) {
      uint32_t ap[4], as[4];
      ap[0] = pack_bf16x2(st[2 * j][0], st[2 * j][1]);
      ap[1] = pack_bf16x2(st[2 * j][2], st[2 * j][3]);
      ap[2] = pack_bf16x2(st[2 * j + 1][0], st[2 * j + 1][1]);
      ap[3] = pack_bf16x2(st[2 * j + 1][2], st[2 * j + 1][3]);
      as[0] = pack_bf16x2(dpt[2 * j][0], dpt[2 * j][1]);
      as[1] = pack_bf16x2(dpt[2 * j][2], dpt[2 * j][3]);
      as[2] = pack_bf16x2(dpt[2 * j + 1][0], dpt[2 * j + 1][1]);
      as[3] = pack_bf16x2(dpt[2 * j + 1][2], dpt[2 * j + 1][3]);
      const int qr = j * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int dn = 0; dn < NC; ++dn) {
        uint32_t r0, r1, r2, r3;
        const int col = dn * 16 + (lane >> 4) * 8;
        ldsm_x4_t(smem_u32(dOs + qr * LDS + col), r0, r1, r2, r3);
        mma16816<false>(dv[2 * dn], ap, r0, r1);
        mma16816<false>(dv[2 * dn + 1], ap, r2, r3);
        ldsm_x4_t(smem_u32(Qb + qr * LDS + col), r0, r1, r2, r3);
        mma16816<false>(dk[2 * dn], as, r0, r1);
        mma16816<false>(dk[2 * dn + 1], as, r2, r3);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int key = kw0 + gr + 8 * r;
    if (key >= S) continue;
    const size_t base = (((size_t)b * nh + h) * S + key) * D;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      *reinterpret_cast<float2 *>(part_k + base + dn * 8 + 2 * tq) =
          make_float2(dk[dn][2 * r] * scale, dk[dn][2 * r + 1] * scale);
      *reinterpret_cast<float2 *>(part_v + base + dn * 8 + 2 * tq) =
          make_float2(dv[dn][2 * r], dv[dn][2 * r + 1]);
    }
  }
}

// dK, dV of kv head g = sum over its query heads, in head order.
__global__ void attn_kv_reduce_kernel(const float *part_k, const float *part_v, int B, int S, int nh,
                                      int nkv, int D, float *dqkv, int ld) {
  const int grp = nh / nkv;
  const int64_t total = (int64_t)B * S * nkv * D;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int dd = (int)(idx % D);
    int64_t rest = idx / D;
    const int g = (int)(rest % nkv);
    rest /= nkv;
    const int t = (int)(rest % S);
    const int b = (int)(rest / S);
    float sk = 0.f, sv = 0.f;
    for (int hh = 0; hh < grp; ++hh) {
      const size_t off = (((size_t)b * nh + g * grp + hh) * S + t) * D + dd;
      sk += part_k[off];
      sv += part_v[off];
    }
    float *row = dqkv + ((size_t)b * S + t) * ld;
    row[(size_t)(nh + g) * D + dd] = sk;
    row[(size_t)(nh + nkv + g) * D + dd] = sv;
  }
}

template <int D>
__global__ void __launch_bounds__(128) attn_bwd_dq_kernel(const uint16_t *qkv, int ld,
                                                          const uint16_t *dO, const float *lse,
                                                          const float *dsum, int S, int nh, int nkv,
                                                          float *dqkv, float scale_log2, float scale) {
  constexpr int KT = 32, LDS = D + 8, NC = D / 16;
  __shared__ __align__(16) uint16_t Ks[KT * LDS];  // half, for the scores
  __shared__ __align__(16) uint16_t Kb[KT * LDS];  // bf16, for dQ
  __shared__ __align__(16) uint16_t Vs[KT * LDS];  // bf16, for dP
  const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = (h * nkv) / nh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, tq = lane & 3;
  const int q0 = qb * 64 + warp * 16;
  const size_t rowbase = (size_t)b * S;
  const uint16_t *Qg = qkv + (size_t)h * D;
  const uint16_t *dOg = dO + (size_t)h * D;
  const int ldo = nh * D;

  uint32_t qf[NC][4], df[NC][4];
#pragma unroll
  for (int kc = 0; kc < NC; ++kc) {
    const int r0 = q0 + gr, r1 = r0 + 8, c = kc * 16 + 2 * tq;
    qf[kc][0] = r0 < S ? ld32(Qg + (rowbase + r0) * ld + c) : 0u;
    qf[kc][1] = r1 < S ? ld32(Qg + (rowbase + r1) * ld + c) : 0u;
    qf[kc][2] = r0 < S ? ld32(Qg + (rowbase + r0) * ld + c + 8) : 0u;
    qf[kc][3] = r1 < S ? ld32(Qg + (rowbase + r1) * ld + c + 8) : 0u;
    df[kc][0] = r0 < S ? ld32(dOg + (rowbase + r0) * ldo + c) : 0u;
    df[kc][1] = r1 < S ? ld32(dOg + (rowbase + r1) * ldo + c) : 0u;
    df[kc][2] = r0 < S ? ld32(dOg + (rowbase + r0) * ldo + c + 8) : 0u;
    df[kc][3] = r1 < S ? ld32(dOg + (rowbase + r1) * ldo + c + 8) : 0u;
  }
  float lrow[2], drow[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = q0 + gr + 8 * r;
    lrow[r] = row < S ? lse[((size_t)b * nh + h) * S + row] : INFINITY;
    drow[r] = row < S ? dsum[((size_t)b * nh + h) * S + row] : 0.f;
  }
  float dq[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;

  const int q_end = min(S, qb * 64 + 64);
  const int n_tiles = (q_end + KT - 1) / KT;
  for (int kt = 0; kt < n_tiles; ++kt) {
    const int k0 = kt * KT;
    __syncthreads();
    load_tile<D>(Ks, qkv, ld, rowbase, k0, KT, S, (nh + g) * D);
    load_tile<D, true>(Kb, qkv, ld, rowbase, k0, KT, S, (nh + g) * D);
    load_tile<D, true>(Vs, qkv, ld, rowbase, k0, KT, S, (nh + nkv + g) * D);
    __syncthreads();
    if (k0 > q0 + 15) continue;
    float s[KT / 8][4], dp[KT / 8][4];
#pragma unroll
    for (int nt = 0; nt < KT / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = dp[nt][e] = 0.f;
#pragma unroll
      for (int kc = 0; kc < NC; ++kc) {
        const uint16_t *kp = Ks + (nt * 8 + gr) * LDS + kc * 16 + 2 * tq;
        mma16816<true>(s[nt], qf[kc], ld32(kp), ld32(kp + 8));
        const uint16_t *vp = Vs + (nt * 8 + gr) * LDS + kc * 16 + 2 * tq;
        mma16816<false>(dp[nt], df[kc], ld32(vp), ld32(vp + 8));
      }
    }
#pragma unroll
    for (int nt = 0; nt < KT / 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = e >> 1;
        const int row = q0 + gr + 8 * r;
        const int key = k0 + nt * 8 + 2 * tq + (e & 1);
        const float p = (key <= row && key < S && row < S) ? exp2f(s[nt][e] * scale_log2 - lrow[r]) : 0.f;
        s[nt][e] = p * (dp[nt][e] - drow[r]);
      }
#pragma unroll
    for (int j = 0; j < KT / 16; ++j) {
      uint32_t a[4];
      a[0] = pack_bf16x2(s[2 * j][0], s[2 * j][1]);
      a[1] = pack_bf16x2(s[2 * j][2], s[2 * j][3]);
      a[2] = pack_bf16x2(s[2 * j + 1][0], s[2 * j + 1][1]);
      a[3] = pack_bf16x2(s[2 * j + 1][2], s[2 * j + 1][3]);
      const int key = j * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int dn = 0; dn < NC; ++dn) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(smem_u32(Kb + key * LDS + dn * 16 + (lane >> 4) * 8), r0, r1, r2, r3);
        mma16816<false>(dq[2 * dn], a, r0, r1);
        mma16816<false>(dq[2 * dn + 1], a, r2, r3);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = q0 + gr + 8 * r;
    if (row >= S) continue;
    float *o = dqkv + (rowbase + row) * ld + (size_t)h * D;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn)
      *reinterpret_cast<float2 *>(o + dn * 8 + 2 * tq) =
          make_float2(dq[dn][2 * r] * scale, dq[dn][2 * r + 1] * scale);
  }
}

template <int D>
int attn_bwd_impl(const uint16_t *qkv, int ld, const uint16_t *o, const uint16_t *dO,
                  const float *lse, int B, int S, int nh, int nkv, float *scratch, float *dqkv,
                  cudaStream_t st) {
  const float scale = 1.0f / sqrtf((float)D);
  const float scale_log2 = scale * 1.4426950408889634f;
  float *dsum = scratch;
  float *part_k = dsum + (size_t)B * nh * S;
  float *part_v = part_k + (size_t)B * nh * S * D;
  const int M = B * S;
  {
    const int64_t threads = (int64_t)M * nh * 32;
    attn_dsum_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(o, dO, M, S, nh, D, dsum);
  }
  dim3 grid((S + 63) / 64, nh, B);
  constexpr int LDS = D + 8;
  const int smem = (2 * 64 + 3 * 32) * LDS * 2 + 2 * 32 * 4;
  {
    static std::atomic<int> attr_set[MAX_DEVICES];  // per device, per head dim
    int done = 0;
    cudaError_t e = per_device_once(attr_set, &done, [&](int, int *v) {
      *v = 1;
      return cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (e != cudaSuccess) return set_error(SOUP_ECUDA, "attn smem attribute: %s", cudaGetErrorString(e));
  }
  attn_bwd_dkdv_kernel<D><<<grid, 128, smem, st>>>(qkv, ld, dO, lse, dsum, S, nh, nkv, part_k,
                                                   part_v, scale_log2, scale);
  const int64_t nred = (int64_t)B * S * nkv * D;
  attn_kv_reduce_kernel<<<(unsigned)std::min<int64_t>((nred + 255) / 256, 148 * 32), 256, 0, st>>>(
      part_k, part_v, B, S, nh, nkv, D, dqkv, ld);
  attn_bwd_dq_kernel<D><<<grid, 128, 0, st>>>(qkv, ld, dO, lse, dsum, S, nh, nkv, dqkv, scale_log2, scale);
  count_launches(4);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(SOUP_ECUDA, "attention backward launch: %s", cudaGetErrorString(e));
  return 0;
}

}  // namespace

size_t attn_bwd_scratch_floats(int B, int S, int nh, int nkv, int d) {
  const size_t mma = (size_t)B * nh * S * (1 + 2 * (size_t)d);
  return std::max(mma, attn_tc_scratch_floats(B, S, nh, nkv, d));
}

int k_attn_fwd(const uint16_t *qkv, int ld, int B, int S, int nh, int nkv, int d, uint16_t *o,
               float *lse, int *err, cudaStream_t st) {
  if (B <= 0 || S <= 0) return 0;
  if (attn_tc_eligible(d, nh, nkv)) return k_attn_fwd_tc(qkv, ld, B, S, nh, nkv, d, o, lse, err, st);
  const float scale_log2 = (1.0f / sqrtf((float)d)) * 1.4426950408889634f;
  dim3 grid((S + 63) / 64, nh, B);
  if (d == 128) attn_fwd_kernel<128, true><<<grid, 128, 0, st>>>(qkv, ld, S, nh, nkv, o, lse, scale_log2);
  else if (d == 64) attn_fwd_kernel<64, true><<<grid, 128, 0, st>>>(qkv, ld, S, nh, nkv, o, lse, scale_log2);
  else return set_error(SOUP_EINVAL, "attention: head_dim %d not supported (64 or 128)", d);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(SOUP_ECUDA, "attention forward launch: %s", cudaGetErrorString(e));
  return 0;
}

int k_attn_bwd(const uint16_t *qkv, int ld, const uint16_t *o, const uint16_t *dO,
               const float *lse, int B, int S, int nh, int nkv, int d, float *scratch, float *dqkv,
               int *err, cudaStream_t st) {
  if (B <= 0 || S <= 0) return 0;
  if (attn_tc_eligible(d, nh, nkv))
    return k_attn_bwd_tc(qkv, ld, o, dO, lse, B, S, nh, nkv, d, scratch, dqkv, err, st);
  if (d == 128) return attn_bwd_impl<128>(qkv, ld, o, dO, lse, B, S, nh, nkv, scratch, dqkv, st);
  if (d == 64) return attn_bwd_impl<64>(qkv, ld, o, dO, lse, B, S, nh, nkv, scratch, dqkv, st);
  return set_error(SOUP_EINVAL, "attention: head_dim %d not supported (64 or 128)", d);
}

}  // namespace soup
