// LoRA gradients of a whole decoder layer in one launch.
//
// What is computed ("Layer streaming: fine-tune a model that does not fit in your card",
// "Honest scope": plain LoRA; only the adapters receive gradients), for each projection p of
// each fused GEMM group, with u = x A_p^T and du = s dY_p B_p already formed:
//   dB_p = s dY_p^T u_p        [out_p, r]    (a reduction over the M tokens)
//   dA_p = du_p^T x            [r, in]       (a reduction over the M tokens)
// written over the gradient (or added to it, old + g in one float addition, when
// accumulating micro-batches).
//
// Layout of the work: every (group, product, 64-column tile) is one job, and each job is one
// thread-block cluster of CL CTAs (1, 2, 4 or 8: enough that each CTA takes at least 256
// tokens); CTA rank c takes the c-th CL-th of the tokens.  The products
// run on the tensor cores as TF32 mma.sync (the 16-bit dY and x are exact in TF32; u, du are
// rounded to TF32 where they are staged).  Each CTA leaves its partial tile in its own shared
// memory, and after a cluster barrier every CTA sums a CL-th of the tile over the CL ranks in
// rank order through distributed shared memory — a fixed order, so the result is
// bit-reproducible, with no partial buffers in global memory and no second kernel.  The eight
// products of a layer (four groups, dB and dA) share one launch.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "util.h"

namespace soup {
namespace {
using namespace soupk;
namespace cg = cooperative_groups;

constexpr int CL_MAX = 8;   // CTAs per cluster at most (the portable cluster size)
constexpr int MIN_ROWS = 256;  // tokens per CTA at least, when there are enough

struct GradJobs {
  LoraGradGroup grp[4];
  int ngroups, M, MC;       // tokens, tokens per cluster rank (a multiple of 32)
  int CL;                   // CTAs per cluster
  int first[9];             // first tile of job kind 2 g (dB) and 2 g + 1 (dA); first[2n] = total
};

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
SOUP_DEV int seg_of(const LoraSeg &L, int n) {
  int q = 0;
  for (int k = 1; k < L.nseg; ++k)
    if (n >= L.off[k] && n < L.off[k] + L.n[k]) q = k;
  return q;
}
SOUP_DEV uint4 pack8(const uint16_t *src, int e_valid) {
  uint32_t h[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) h[e] = e < e_valid ? src[e] : 0u;
  return make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
}

// Shared memory of one CTA: the staged operands of a 32-token chunk and the partial tile.
struct SmemB {              // dB job: 64 output rows n x r
  uint32_t ds[32][72];      // dY [m][n] as TF32
  uint32_t us[32][72];      // u  [m][o] as TF32
  float red[64][24];        // partial dB tile [n][j]
};
struct SmemA {              // dA job: 64 outputs o x 64 features k
  uint32_t dus[32][72];     // du [m][o] as TF32
  uint32_t xs[32][72];      // x  [m][k] as TF32
  float red[64][68];        // partial dA tile [o][k]
};
union Smem {
  SmemB b;
  SmemA a;
};

// dB tile: output rows n0 .. n0 + 63 of group G, tokens [mb, me).  Warp w takes rows
// 16w .. 16w + 15 (two per lane: na, nb); a tile that straddles a segment boundary runs once
// per segment with the other segment's rows masked.
template <bool XF16>
SOUP_DEV void db_tile(const LoraGradGroup &G, int n0, int mb, int me, SmemB &sm) {
  const LoraSeg &L = G.L;
  const int t = threadIdx.x, w = t >> 5, lane = t & 31, g = lane >> 2, q = lane & 3;
  const int nout = L.nseg * L.r, JT = (L.r + 7) / 8, Ng = G.Ng;
  const int s_lo = seg_of(L, n0), s_hi = seg_of(L, min(n0 + 63, Ng - 1));
  const int na = n0 + 16 * w + g, nb = na + 8;
  uint4 dr[2];
  float ur[16];
  auto load = [&](int m0) {
#pragma unroll
    for (int it = 0; it < 2; ++it) {  // dY: 32 m x 64 n, 8 elements per item
      const int i = t + 128 * it, rr = i >> 3, c8 = (i & 7) * 8;
      const int m = m0 + rr, n = n0 + c8;
      const uint16_t *src = G.dy + (size_t)m * G.ldy + n;
      if (m < me && n + 8 <= Ng && ((G.ldy | n) & 7) == 0) dr[it] = *reinterpret_cast<const uint4 *>(src);
      else dr[it] = m < me ? pack8(src, Ng - n) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int it = 0; it < 16; ++it) {  // u: 32 m x 64 o
      const int i = t + 128 * it, rr = i >> 6, o = i & 63;
      const int m = m0 + rr;
      ur[it] = (m < me && o < nout) ? G.u[(size_t)m * nout + o] : 0.f;
    }
  };
  float acc[3][4] = {};
  if (mb < me) load(mb);
  for (int m0 = mb; m0 < me; m0 += 32) {
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int i = t + 128 * it, rr = i >> 3, c8 = (i & 7) * 8;
      const uint32_t wv[4] = {dr[it].x, dr[it].y, dr[it].z, dr[it].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {  // the gradient is bf16
        sm.ds[rr][c8 + 2 * e] = __float_as_uint(bf16_lo(wv[e]));
        sm.ds[rr][c8 + 2 * e + 1] = __float_as_uint(bf16_hi(wv[e]));
      }
    }
#pragma unroll
    for (int it = 0; it < 16; ++it) {
      const int i = t + 128 * it;
      sm.us[i >> 6][i & 63] = to_tf32(ur[it]);
    }
    __syncthreads();
    if (m0 + 32 < me) load(m0 + 32);
    for (int sg = s_lo; sg <= s_hi; ++sg) {
      const bool ina = na < Ng && seg_of(L, na) == sg, inb = nb < Ng && seg_of(L, nb) == sg;
#pragma unroll
      for (int k8 = 0; k8 < 32; k8 += 8) {
        const uint32_t a[4] = {ina ? sm.ds[k8 + q][na - n0] : 0u, inb ? sm.ds[k8 + q][nb - n0] : 0u,
                               ina ? sm.ds[k8 + q + 4][na - n0] : 0u, inb ? sm.ds[k8 + q + 4][nb - n0] : 0u};
#pragma unroll
        for (int jt = 0; jt < 3; ++jt) {
          if (jt >= JT) break;
          const int j = 8 * jt + g;
          const uint32_t b0 = j < L.r ? sm.us[k8 + q][sg * L.r + j] : 0u;
          const uint32_t b1 = j < L.r ? sm.us[k8 + q + 4][sg * L.r + j] : 0u;
          mma_tf32(acc[jt], a, b0, b1);
        }
      }
    }
    __syncthreads();
  }
  // the partial tile [64 n][r] into this CTA's shared memory
#pragma unroll
  for (int jt = 0; jt < 3; ++jt) {
    const int j = 8 * jt + 2 * q;
    if (j < 24) {
      sm.red[na - n0][j] = acc[jt][0];
      sm.red[nb - n0][j] = acc[jt][2];
    }
    if (j + 1 < 24) {
      sm.red[na - n0][j + 1] = acc[jt][1];
      sm.red[nb - n0][j + 1] = acc[jt][3];
    }
  }
}

// dA tile: outputs o (warp w: 16w .. 16w + 15; warps past nout idle) x features k0 .. k0 + 63.
template <bool XF16>
SOUP_DEV void da_tile(const LoraGradGroup &G, int k0, int mb, int me, SmemA &sm) {
  const LoraSeg &L = G.L;
  const int t = threadIdx.x, w = t >> 5, lane = t & 31, g = lane >> 2, q = lane & 3;
  const int nout = L.nseg * L.r, K = G.K;
  const bool live = 16 * w < nout;
  float dr[16];
  uint4 xr[2];
  auto load = [&](int m0) {
#pragma unroll
    for (int it = 0; it < 16; ++it) {  // du: 32 m x 64 o
      const int i = t + 128 * it, rr = i >> 6, o = i & 63;
      const int m = m0 + rr;
      dr[it] = (m < me && o < nout) ? G.du[(size_t)m * nout + o] : 0.f;
    }
#pragma unroll
    for (int it = 0; it < 2; ++it) {  // x: 32 m x 64 k, 8 elements per item
      const int i = t + 128 * it, rr = i >> 3, c8 = (i & 7) * 8;
      const int m = m0 + rr, k = k0 + c8;
      const uint16_t *src = G.x + (size_t)m * G.ldx + k;
      if (m < me && k + 8 <= K && ((G.ldx | k) & 7) == 0) xr[it] = *reinterpret_cast<const uint4 *>(src);
      else xr[it] = m < me ? pack8(src, K - k) : make_uint4(0, 0, 0, 0);
    }
  };
  float acc[8][4] = {};
  if (mb < me) load(mb);
  for (int m0 = mb; m0 < me; m0 += 32) {
#pragma unroll
    for (int it = 0; it < 16; ++it) {
      const int i = t + 128 * it;
      sm.dus[i >> 6][i & 63] = to_tf32(dr[it]);
    }
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int i = t + 128 * it, rr = i >> 3, c8 = (i & 7) * 8;
      const uint32_t wv[4] = {xr[it].x, xr[it].y, xr[it].z, xr[it].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sm.xs[rr][c8 + 2 * e] = __float_as_uint(lo16<XF16>(wv[e]));
        sm.xs[rr][c8 + 2 * e + 1] = __float_as_uint(hi16<XF16>(wv[e]));
      }
    }
    __syncthreads();
    if (m0 + 32 < me) load(m0 + 32);
    if (live) {
#pragma unroll
      for (int k8 = 0; k8 < 32; k8 += 8) {
        const int oa = 16 * w + g;
        const uint32_t a[4] = {sm.dus[k8 + q][oa], sm.dus[k8 + q][oa + 8], sm.dus[k8 + q + 4][oa],
                               sm.dus[k8 + q + 4][oa + 8]};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const int kc = 8 * nt + g;
          mma_tf32(acc[nt], a, sm.xs[k8 + q][kc], sm.xs[k8 + q + 4][kc]);
        }
      }
    }
    __syncthreads();
  }
  const int oa = 16 * w + g;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int k = 8 * nt + 2 * q;
    sm.red[oa][k] = acc[nt][0];
    sm.red[oa][k + 1] = acc[nt][1];
    sm.red[oa + 8][k] = acc[nt][2];
    sm.red[oa + 8][k + 1] = acc[nt][3];
  }
}

template <bool XF16>
__global__ void __launch_bounds__(128) lora_grad_kernel(const GradJobs J) {
  __shared__ __align__(16) Smem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();  // this CTA's share of the tokens
  const int CL = J.CL;
  const int tile = blockIdx.x;
  int kind = 0;
  while (kind + 1 < 2 * J.ngroups && tile >= J.first[kind + 1]) ++kind;
  const LoraGradGroup &G = J.grp[kind >> 1];
  const LoraSeg &L = G.L;
  const int local = tile - J.first[kind];
  const int mb = rank * J.MC, me = min(J.M, mb + J.MC);
  const bool is_db = (kind & 1) == 0;
  if (is_db) db_tile<XF16>(G, local * 64, mb, me, sm.b);
  else da_tile<XF16>(G, local * 64, mb, me, sm.a);
  cluster.sync();  // every rank's partial tile is in its shared memory
  if (is_db) {
    // rank c sums rows c * 64 / CL .. of the tile over the CL ranks, in rank order
    const float *part[CL_MAX];
#pragma unroll
    for (int c = 0; c < CL_MAX; ++c) part[c] = cluster.map_shared_rank(&sm.b.red[0][0], c < CL ? c : 0);
    const int rows = 64 / CL;
    for (int i = threadIdx.x; i < rows * L.r; i += blockDim.x) {
      const int nl = rows * rank + i / L.r, j = i % L.r;
      const int n = local * 64 + nl;
      float pv[CL_MAX];  // every remote load in flight before the first add
#pragma unroll
      for (int c = 0; c < CL_MAX; ++c) pv[c] = c < CL ? part[c][nl * 24 + j] : 0.f;
      float acc = pv[0];
#pragma unroll
      for (int c = 1; c < CL_MAX; ++c)
        if (c < CL) acc += pv[c];
      if (n < G.Ng) {
        const int sg = seg_of(L, n);
        if (n >= L.off[sg] && n < L.off[sg] + L.n[sg]) {
          float *dst = L.dB[sg] + (size_t)(n - L.off[sg]) * L.r + j;
          const float gv = L.s * acc;
          *dst = L.accumulate ? *dst + gv : gv;
        }
      }
    }
  } else {
    // rank c sums outputs c * 64 / CL .. of the tile (x 64 features) over the CL ranks, in order
    const int nout = L.nseg * L.r;
    const float *part[CL_MAX];
#pragma unroll
    for (int c = 0; c < CL_MAX; ++c) part[c] = cluster.map_shared_rank(&sm.a.red[0][0], c < CL ? c : 0);
    const int outs = 64 / CL;
    for (int i = threadIdx.x; i < outs * 64; i += blockDim.x) {
      const int ol = outs * rank + i / 64, kl = i % 64;
      const int k = local * 64 + kl;
      float pv[CL_MAX];
#pragma unroll
      for (int c = 0; c < CL_MAX; ++c) pv[c] = c < CL ? part[c][ol * 68 + kl] : 0.f;
      float acc = pv[0];
#pragma unroll
      for (int c = 1; c < CL_MAX; ++c)
        if (c < CL) acc += pv[c];
      if (ol < nout && k < G.K) {
        float *dst = L.dA[ol / L.r] + (size_t)(ol % L.r) * G.K + k;
        *dst = L.accumulate ? *dst + acc : acc;
      }
    }
  }
  cluster.sync();  // no CTA leaves while another still reads its shared memory
}

}  // namespace

void k_lora_grads(const LoraGradGroup *groups, int ngroups, int M, bool x_f16, cudaStream_t st) {
  if (M <= 0 || ngroups <= 0) return;
  GradJobs J;
  J.ngroups = ngroups;
  J.M = M;
  int cl = 1;
  while (cl < CL_MAX && (M + 2 * cl - 1) / (2 * cl) >= MIN_ROWS) cl *= 2;
  J.CL = cl;
  J.MC = ((M + cl - 1) / cl + 31) / 32 * 32;
  int tiles = 0;
  for (int g = 0; g < ngroups; ++g) {
    J.grp[g] = groups[g];
    J.first[2 * g] = tiles;
    tiles += (groups[g].Ng + 63) / 64;
    J.first[2 * g + 1] = tiles;
    tiles += (groups[g].K + 63) / 64;
  }
  J.first[2 * ngroups] = tiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, cl);
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = cl;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (x_f16) cudaLaunchKernelEx(&cfg, lora_grad_kernel<true>, J);
  else cudaLaunchKernelEx(&cfg, lora_grad_kernel<false>, J);
  count_launches(1);
}

}  // namespace soup
