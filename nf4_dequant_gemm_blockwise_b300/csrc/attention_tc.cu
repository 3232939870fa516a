// Causal grouped-query attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA),
// forward and backward, for the decoder layer of the streamed step ("Layer streaming:
// fine-tune a model that does not fit in your card", "How it works": the family's own decoder
// layer; query head h reads key/value head floor(h * n_kv / n_h); softmax(q k^T / sqrt(d) +
// causal mask) v).
//
// The flash formulation: the S x S score matrix is never stored; the forward keeps a running
// row max and sum and writes the base-2 log-sum-exp; the backward recomputes the
// probabilities from it.  Operand formats: scores from IEEE-half q and k, the forward's p v in
// half; every product with a gradient in bf16 (a bf16 copy of q, k and v is made once per
// backward).  Accumulation in float, in TMEM.
//
// Each CTA has 6 warps: warps 0-3 are the row threads (thread t owns TMEM lane t, one row of
// every accumulator), warp 4 issues the TMA copies, warp 5 allocates TMEM and one of its lanes
// issues the tcgen05.mma instructions.
//   forward  one CTA per (128-query block, head, sequence); key/value blocks of 128 in a
//            two-stage ring.  S = Q K^T goes to TMEM; each row thread takes its row's max,
//            exponentials and sum and writes P (half) into shared memory in the swizzled
//            K-major layout; P V accumulates into the output in TMEM, rescaled lazily.
//   dQ       one CTA per (128-query block, head, sequence), key blocks of 64: S = Q K^T and
//            dP = dO V^T (double-buffered in TMEM), dS = P (dP - D) written as bf16 into one of
//            two shared buffers, dQ += dS K (K read MN-major).
//   dK, dV   one CTA per (128-key block, query head, sequence), query blocks of 64:
//            S^T = K Q^T, dP^T = V dO^T, P^T and dS^T written as bf16, dV += P^T dO and
//            dK += dS^T Q (dO and Q read MN-major).  The query heads that share a key/value
//            head form one thread-block cluster and sum their dK, dV through distributed
//            shared memory in head order: deterministic, no atomics.
// Every wait is bounded (common.cuh): on a timeout the kernel raises its error flag, lets its
// copies land, frees TMEM and returns.
#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "util.h"

namespace cg = cooperative_groups;

namespace soup {
namespace {
using namespace soupk;

constexpr int THREADS = 192;
constexpr int ROWS = 128;                 // row threads = TMEM lanes
constexpr int TMA_WARP = 4, MMA_WARP = 5;
constexpr int PANEL128 = 128 * 128;       // one 64-column panel of a 128-row 16-bit tile
constexpr int PANEL64 = 64 * 128;         // ... of a 64-row tile

struct AttnArgs {
  int S, nh, nkv, grp;     // grp = nh / nkv query heads per key/value head
  int ld;                  // row stride of qkv (and of dqkv), elements
  float scale, scale_log2;
  uint16_t *o;             // forward output, half [B*S, nh*D]
  float *lse;              // [B, nh, S]
  const float *dsum;       // [B, nh, S]
  float *dqkv;             // [B*S, ld]
  int *err;
};

SOUP_DEV uint8_t *align1k(uint8_t *p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}
SOUP_DEV uint4 u4(const uint32_t *p) { return make_uint4(p[0], p[1], p[2], p[3]); }
// A wait's outcome made the same for the whole warp: tcgen05.ld is a warp-wide (.sync.aligned)
// instruction, so no lane may go on to one while another lane of its warp has given up.
SOUP_DEV bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// ---------------------------------------------------------------------------------- forward
// The output accumulates in TMEM across the key blocks (P V with accumulate on).  A row's
// reference max is raised lazily: only when a block's max exceeds it by more than 2^8 (log2
// units) is the row's TMEM output rescaled, so P = exp2(s - ref) <= 256 stays exact in half and
// the final O / l is the same whatever reference was used.  S is read out of TMEM in one batch,
// which frees it for the next block's Q K^T while the exponentials run.
constexpr float RESCALE_LOG2 = 8.0f;

template <int D>
struct Fwd {
  static constexpr int TILE = 128 * D * 2;      // a 128-row Q, K or V tile
  static constexpr int P_BYTES = 128 * 128 * 2;
  static constexpr int SMEM = 5 * TILE + P_BYTES + 1024 + 256;
  static constexpr uint32_t TMEM_COLS = 256;    // S (128) + O (D)
};

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap map_h128, const AttnArgs a) {
  using C = Fwd<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1k(smem_raw);
  uint8_t *Qs = smem, *Ks = smem + C::TILE, *Vs = Ks + 2 * C::TILE, *Ps = Vs + 2 * C::TILE;
  uint64_t *bar = reinterpret_cast<uint64_t *>(Ps + C::P_BYTES);
  uint64_t *q_full = bar, *k_full = bar + 1, *v_full = bar + 3, *kv_empty = bar + 5;
  uint64_t *s_full = bar + 7, *s_free = bar + 8, *p_full = bar + 9, *pv_done = bar + 10;
  uint64_t *mma_done = bar + 11;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 12);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.S;
  const int qb = (int)gridDim.x - 1 - (int)blockIdx.x;  // the longest rows of keys start first
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / a.grp;
  const int nkb = qb + 1;  // key blocks 0 .. qb

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, ROWS);
    mbar_init(p_full, ROWS);
    mbar_init(pv_done, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tc_alloc(tmem_slot, C::TMEM_COLS);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_s = tmem, t_o = tmem + 128;

  if (warp == TMA_WARP) {
    if (lane == 0) {
      tma_prefetch_desc(&map_h128);
      const int cq = h * D, ck = (a.nh + g) * D, cv = (a.nh + a.nkv + g) * D;
      mbar_arrive_expect_tx(q_full, C::TILE);
#pragma unroll
      for (int p = 0; p < D / 64; ++p)
        tma_load_3d(Qs + p * PANEL128, &map_h128, cq + 64 * p, qb * 128, b, q_full);
      int issued = 0;
      for (int j = 0; j < nkb; ++j) {
        const int s = j & 1;
        if (j >= 2 && !mbar_wait(&kv_empty[s], ((j >> 1) - 1) & 1, a.err, abort_flag)) break;
        mbar_arrive_expect_tx(&k_full[s], C::TILE);
#pragma unroll
        for (int p = 0; p < D / 64; ++p)
          tma_load_3d(Ks + s * C::TILE + p * PANEL128, &map_h128, ck + 64 * p, j * 128, b, &k_full[s]);
        mbar_arrive_expect_tx(&v_full[s], C::TILE);
#pragma unroll
        for (int p = 0; p < D / 64; ++p)
          tma_load_3d(Vs + s * C::TILE + p * PANEL128, &map_h128, cv + 64 * p, j * 128, b, &v_full[s]);
        ++issued;
      }
      // never leave the CTA with copies still landing in its shared memory
      volatile int no_abort = 0;
      mbar_wait(q_full, 0, a.err, &no_abort);
      for (int j = max(0, issued - 2); j < issued; ++j) {
        mbar_wait(&k_full[j & 1], (j >> 1) & 1, a.err, &no_abort);
        mbar_wait(&v_full[j & 1], (j >> 1) & 1, a.err, &no_abort);
      }
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_16(128, 128, 0, 0, 1);  // half, both K-major
      constexpr uint32_t id_pv = idesc_16(128, D, 0, 1, 1);   // half, V MN-major
      const uint32_t qa = smem_u32(Qs), pa = smem_u32(Ps);
      auto issue_s = [&](int j) -> bool {
        const int s = j & 1;
        if (!mbar_wait(&k_full[s], (j >> 1) & 1, a.err, abort_flag)) return false;
        tc_fence_after();
        const uint32_t ka = smem_u32(Ks + s * C::TILE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * PANEL128 + (kk & 3) * 32;
          tc_mma_bf16(t_s, smem_desc(qa + off, 16, 1024), smem_desc(ka + off, 16, 1024), id_s, kk > 0);
        }
        tc_commit(s_full);
        return true;
      };
      bool ok = mbar_wait(q_full, 0, a.err, abort_flag) && issue_s(0);
      for (int j = 0; ok && j < nkb; ++j) {
        const int s = j & 1;
        // S_{j+1} as soon as the row threads hold S_j in registers
        if (j + 1 < nkb) {
          if (!mbar_wait(s_free, j & 1, a.err, abort_flag) || !issue_s(j + 1)) break;
        }
        // P_j is in shared memory (and any rescale of O for block j is done)
        if (!mbar_wait(p_full, j & 1, a.err, abort_flag)) break;
        if (!mbar_wait(&v_full[s], (j >> 1) & 1, a.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t va = smem_u32(Vs + s * C::TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_bf16(t_o, smem_desc(pa + (kk >> 2) * PANEL128 + (kk & 3) * 32, 16, 1024),
                      smem_desc(va + kk * 2048, PANEL128, 1024), id_pv, (j | kk) != 0);
        tc_commit(pv_done);
        tc_commit(&kv_empty[s]);
      }
      tc_commit(mma_done);
      volatile int no_abort = 0;
      mbar_wait(mma_done, 0, a.err, &no_abort);  // every MMA retired before TMEM is freed
    }
  } else {
    // ------------------------------------------------------------------ row threads
    const int r = threadIdx.x;
    const int row = qb * 128 + r;
    const uint32_t lq = (uint32_t)(warp * 32) << 16;
    float ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkb; ++j) {
      if (!warp_all(mbar_wait(s_full, j & 1, a.err, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v0[32], v1[32], v2[32], v3[32];
      __syncwarp();
      tc_ld_32x32b_x32(t_s + lq, v0);
      tc_ld_32x32b_x32(t_s + lq + 32, v1);
      tc_ld_32x32b_x32(t_s + lq + 64, v2);
      tc_ld_32x32b_x32(t_s + lq + 96, v3);
      tc_wait_ld();
      tc_fence_before();
      mbar_arrive(s_free);  // S_j is in registers: the next block's scores may overwrite it
      // keys j*128 .. j*128 + lim are visible to this row (the causal mask; rows of the last
      // block past S are computed and dropped)
      // keys after this row are masked to -inf; only the last (diagonal) block has any (rows of
      // that block past S are computed and dropped)
      if (j == nkb - 1) {
        auto mask = [&](uint32_t(&v)[32], int c0) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (c0 + i > r) v[i] = 0xff800000u;
        };
        mask(v0, 0);
        mask(v1, 32);
        mask(v2, 64);
        mask(v3, 96);
      }
      // independent partial maxima and sums: the row is one thread's work, so the instruction
      // stream needs the parallelism
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      auto rmax = [&](const uint32_t(&v)[32]) {
#pragma unroll
        for (int i = 0; i < 32; ++i) m4[i & 3] = fmaxf(m4[i & 3], __uint_as_float(v[i]));
      };
      rmax(v0);
      rmax(v1);
      rmax(v2);
      rmax(v3);
      const float mnew = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * a.scale_log2;
      const bool resc = mnew > ref + RESCALE_LOG2;  // always at the first block (ref = -inf)
      const float nref = resc ? mnew : ref;
      const float corr = resc ? ex2(ref - nref) : 1.f;  // 0 at the first block
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[4][16];
      auto probs = [&](const uint32_t(&v)[32], int c) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2(fmaf(__uint_as_float(v[2 * i]), a.scale_log2, -nref));
          const float p1 = ex2(fmaf(__uint_as_float(v[2 * i + 1]), a.scale_log2, -nref));
          s4[i & 3] += p0 + p1;
          pk[c][i] = pack_h2(p0, p1);
        }
      };
      probs(v0, 0);
      probs(v1, 1);
      probs(v2, 2);
      probs(v3, 3);
      const float sum = (s4[0] + s4[1]) + (s4[2] + s4[3]);
      l = l * corr + sum;
      if (j > 0) {
        // P V of the previous block has finished with P's buffer and with O
        if (!warp_all(mbar_wait(pv_done, (j - 1) & 1, a.err, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, resc)) {  // the warp rescales its 32 rows of O (corr 1: kept)
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tc_ld_32x32b_x32(t_o + lq + c * 32, o);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
            tc_st_32x32b_x32(t_o + lq + c * 32, o);
          }
          tc_wait_st();
        }
      }
      ref = nref;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint8_t *pp = Ps + (c >> 1) * PANEL128;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4 *>(pp + sw128(r, (c & 1) * 4 + q)) = u4(pk[c] + 4 * q);
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    ok = warp_all(ok && mbar_wait(pv_done, (nkb - 1) & 1, a.err, abort_flag) && !*abort_flag);
    tc_fence_after();
    if (ok) {
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      uint16_t *dst = a.o + ((size_t)b * S + row) * (size_t)(a.nh * D) + (size_t)h * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        __syncwarp();
        tc_ld_32x32b_x32(t_o + lq + c * 32, o);  // every lane of the warp; rows < S store
        tc_wait_ld();
        if (row < S) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_h2(__uint_as_float(o[8 * q + 2 * e]) * inv, __uint_as_float(o[8 * q + 2 * e + 1]) * inv);
            *reinterpret_cast<uint4 *>(dst + c * 32 + 8 * q) = u4(w);
          }
        }
      }
      if (row < S) a.lse[((size_t)b * a.nh + h) * S + row] = ref + log2f(l);
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tc_dealloc(tmem, C::TMEM_COLS);
  }
}

// --------------------------------------------------------------------------- backward prep
// dsum[b, h, t] = sum_d dO[m, h, d] O[m, h, d] (O half, dO bf16), and the bf16 copy of the
// qkv row m.  One block of 256 threads per row m = b * S + t.
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const uint16_t *qkv, int ld,
                                                            const uint16_t *o, const uint16_t *dO,
                                                            int S, int nh, int D, float *dsum,
                                                            uint16_t *qkv_b) {
  const int m = blockIdx.x;
  const uint16_t *src = qkv + (size_t)m * ld;
  uint16_t *dst = qkv_b + (size_t)m * ld;
  for (int i = threadIdx.x * 8; i < ld; i += 256 * 8) {
    uint4 v = *reinterpret_cast<const uint4 *>(src + i);
    v.x = pack_bf16x2(lo16<true>(v.x), hi16<true>(v.x));
    v.y = pack_bf16x2(lo16<true>(v.y), hi16<true>(v.y));
    v.z = pack_bf16x2(lo16<true>(v.z), hi16<true>(v.z));
    v.w = pack_bf16x2(lo16<true>(v.w), hi16<true>(v.w));
    *reinterpret_cast<uint4 *>(dst + i) = v;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = m / S, t = m % S;
  for (int hh = warp; hh < nh; hh += 8) {
    const uint16_t *x = o + ((size_t)m * nh + hh) * D;
    const uint16_t *y = dO + ((size_t)m * nh + hh) * D;
    float s = 0.f;
    for (int i = lane * 2; i < D; i += 64) {
      const uint32_t xv = *reinterpret_cast<const uint32_t *>(x + i);
      const uint32_t yv = *reinterpret_cast<const uint32_t *>(y + i);
      s += lo16<true>(xv) * bf16_lo(yv) + hi16<true>(xv) * bf16_hi(yv);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) dsum[((size_t)b * nh + hh) * S + t] = s;
  }
}

// ------------------------------------------------------------------------------------ dQ
template <int D>
struct Dq {
  static constexpr int QT = 128 * D * 2;      // Q (half) or dO (bf16) tile, 128 rows
  static constexpr int KT = 64 * D * 2;       // K or V tile, 64 rows
  static constexpr int STAGE = 3 * KT;        // K half, K bf16, V bf16
  static constexpr int DS_BYTES = 128 * 64 * 2;  // one dS buffer; two alternate
  static constexpr int SMEM = 2 * QT + 2 * STAGE + 2 * DS_BYTES + 1024 + 256;
  static constexpr uint32_t TMEM_COLS = 512;  // S, dP double-buffered (4 x 64) + dQ (D)
};

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    attn_dq_tc_kernel(const __grid_constant__ CUtensorMap map_h128,
                      const __grid_constant__ CUtensorMap map_do128,
                      const __grid_constant__ CUtensorMap map_h64,
                      const __grid_constant__ CUtensorMap map_b64, const AttnArgs a) {
  using C = Dq<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1k(smem_raw);
  uint8_t *Qs = smem, *dOs = smem + C::QT, *ring = smem + 2 * C::QT;
  uint8_t *dSs = ring + 2 * C::STAGE;  // two buffers: block j writes buffer j & 1
  uint64_t *bar = reinterpret_cast<uint64_t *>(dSs + 2 * C::DS_BYTES);
  uint64_t *qd_full = bar, *kv_full = bar + 1, *kv_empty = bar + 3, *sd_full = bar + 5;
  uint64_t *ds_full = bar + 7, *ds_free = bar + 9, *mma_done = bar + 11;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 12);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.S;
  const int qb = (int)gridDim.x - 1 - (int)blockIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / a.grp;
  const int nkb = (min(S, qb * 128 + 128) + 63) / 64;  // key blocks of 64

  if (threadIdx.x == 0) {
    mbar_init(qd_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
      mbar_init(&sd_full[s], 1);
      mbar_init(&ds_full[s], ROWS);
      mbar_init(&ds_free[s], 1);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tc_alloc(tmem_slot, C::TMEM_COLS);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_dq = tmem + 256;

  if (warp == TMA_WARP) {
    if (lane == 0) {
      tma_prefetch_desc(&map_h128);
      tma_prefetch_desc(&map_h64);
      tma_prefetch_desc(&map_b64);
      const int cq = h * D, ck = (a.nh + g) * D, cv = (a.nh + a.nkv + g) * D;
      mbar_arrive_expect_tx(qd_full, 2 * C::QT);
#pragma unroll
      for (int p = 0; p < D / 64; ++p) {
        tma_load_3d(Qs + p * PANEL128, &map_h128, cq + 64 * p, qb * 128, b, qd_full);
        tma_load_3d(dOs + p * PANEL128, &map_do128, h * D + 64 * p, qb * 128, b, qd_full);
      }
      int issued = 0;
      for (int j = 0; j < nkb; ++j) {
        const int s = j & 1;
        if (j >= 2 && !mbar_wait(&kv_empty[s], ((j >> 1) - 1) & 1, a.err, abort_flag)) break;
        uint8_t *st = ring + s * C::STAGE;
        mbar_arrive_expect_tx(&kv_full[s], C::STAGE);
#pragma unroll
        for (int p = 0; p < D / 64; ++p) {
          tma_load_3d(st + p * PANEL64, &map_h64, ck + 64 * p, j * 64, b, &kv_full[s]);
          tma_load_3d(st + C::KT + p * PANEL64, &map_b64, ck + 64 * p, j * 64, b, &kv_full[s]);
          tma_load_3d(st + 2 * C::KT + p * PANEL64, &map_b64, cv + 64 * p, j * 64, b, &kv_full[s]);
        }
        ++issued;
      }
      volatile int no_abort = 0;
      mbar_wait(qd_full, 0, a.err, &no_abort);
      for (int j = max(0, issued - 2); j < issued; ++j)
        mbar_wait(&kv_full[j & 1], (j >> 1) & 1, a.err, &no_abort);
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_16(128, 64, 0, 0, 1);   // S: half
      constexpr uint32_t id_dp = idesc_16(128, 64, 0, 0, 0);  // dP: bf16
      constexpr uint32_t id_dq = idesc_16(128, D, 0, 1, 0);   // dQ: bf16, K MN-major
      const uint32_t qa = smem_u32(Qs), da = smem_u32(dOs), dsa = smem_u32(dSs);
      auto issue_sd = [&](int j) -> bool {
        const int s = j & 1;
        if (!mbar_wait(&kv_full[s], (j >> 1) & 1, a.err, abort_flag)) return false;
        tc_fence_after();
        const uint32_t kh = smem_u32(ring + s * C::STAGE), vb = kh + 2 * C::KT;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o128 = (kk >> 2) * PANEL128 + (kk & 3) * 32;
          const uint32_t o64 = (kk >> 2) * PANEL64 + (kk & 3) * 32;
          tc_mma_bf16(tmem + s * 128, smem_desc(qa + o128, 16, 1024), smem_desc(kh + o64, 16, 1024),
                      id_s, kk > 0);
          tc_mma_bf16(tmem + s * 128 + 64, smem_desc(da + o128, 16, 1024),
                      smem_desc(vb + o64, 16, 1024), id_dp, kk > 0);
        }
        tc_commit(&sd_full[s]);
        return true;
      };
      bool ok = mbar_wait(qd_full, 0, a.err, abort_flag) && issue_sd(0);
      for (int j = 0; ok && j < nkb; ++j) {
        const int s = j & 1;
        // the TMEM buffer of block j + 1 was last read by the row threads for block j - 1
        if (j + 1 < nkb && !issue_sd(j + 1)) break;
        if (!mbar_wait(&ds_full[s], (j >> 1) & 1, a.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t kb16 = smem_u32(ring + s * C::STAGE) + C::KT;
        const uint32_t dsb = dsa + s * C::DS_BYTES;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_bf16(t_dq, smem_desc(dsb + kk * 32, 16, 1024),
                      smem_desc(kb16 + kk * 2048, PANEL64, 1024), id_dq, (j | kk) != 0);
        tc_commit(&kv_empty[s]);
        tc_commit(&ds_free[s]);
      }
      tc_commit(mma_done);
      volatile int no_abort = 0;
      mbar_wait(mma_done, 0, a.err, &no_abort);
    }
  } else {
    // ------------------------------------------------------------------ row threads
    const int r = threadIdx.x;
    const int row = qb * 128 + r;
    const uint32_t lq = (uint32_t)(warp * 32) << 16;
    const size_t lrow = ((size_t)b * a.nh + h) * S + row;
    const float lse_r = row < S ? a.lse[lrow] : INFINITY;
    const float ds_r = row < S ? a.dsum[lrow] : 0.f;
    bool ok = true;
    for (int j = 0; j < nkb; ++j) {
      const int s = j & 1;
      if (!warp_all(mbar_wait(&sd_full[s], (j >> 1) & 1, a.err, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s0[32], s1[32], d0[32], d1[32];  // S and dP of this row, one wait for all four
      __syncwarp();
      tc_ld_32x32b_x32(tmem + lq + s * 128, s0);
      tc_ld_32x32b_x32(tmem + lq + s * 128 + 32, s1);
      tc_ld_32x32b_x32(tmem + lq + s * 128 + 64, d0);
      tc_ld_32x32b_x32(tmem + lq + s * 128 + 96, d1);
      tc_wait_ld();
      uint32_t pk[2][16];
      auto dsrow = [&](const uint32_t(&sv)[32], const uint32_t(&dv)[32], int c) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int key = j * 64 + c * 32 + 2 * i;
          float d2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const bool vis = key + e <= row && key + e < S && row < S;
            const float p = vis ? ex2(__uint_as_float(sv[2 * i + e]) * a.scale_log2 - lse_r) : 0.f;
            d2[e] = p * (__uint_as_float(dv[2 * i + e]) - ds_r);
          }
          pk[c][i] = pack_bf16x2(d2[0], d2[1]);
        }
      };
      dsrow(s0, d0, 0);
      dsrow(s1, d1, 1);
      // buffer s was last read by the dQ product of block j - 2
      if (j >= 2 && !warp_all(mbar_wait(&ds_free[s], ((j >> 1) - 1) & 1, a.err, abort_flag))) {
        ok = false;
        break;
      }
      uint8_t *dsb = dSs + s * C::DS_BYTES;
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4 *>(dsb + sw128(r, c * 4 + q)) = u4(pk[c] + 4 * q);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&ds_full[s]);
    }
    volatile int no_abort = 0;
    ok = warp_all(ok && mbar_wait(mma_done, 0, a.err, &no_abort) && !*abort_flag);
    tc_fence_after();
    if (ok) {
      float *dst = a.dqkv + ((size_t)b * S + row) * a.ld + (size_t)h * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        __syncwarp();
        tc_ld_32x32b_x32(t_dq + lq + c * 32, v);  // every lane of the warp, then only rows < S store
        tc_wait_ld();
        if (row < S) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            *reinterpret_cast<float4 *>(dst + c * 32 + 4 * e) =
                make_float4(__uint_as_float(v[4 * e]) * a.scale, __uint_as_float(v[4 * e + 1]) * a.scale,
                            __uint_as_float(v[4 * e + 2]) * a.scale, __uint_as_float(v[4 * e + 3]) * a.scale);
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tc_dealloc(tmem, C::TMEM_COLS);
  }
}

// -------------------------------------------------------------------------------- dK, dV
template <int D>
struct Dkv {
  static constexpr int KT = 128 * D * 2;      // K (half) or V (bf16) tile, 128 rows
  static constexpr int QT = 64 * D * 2;       // Q or dO tile, 64 rows
  static constexpr int STAGE = 3 * QT;        // Q half, Q bf16, dO bf16
  static constexpr int PT = 128 * 64 * 2;     // P^T or dS^T tile (bf16)
  static constexpr int LDR = D + 4;           // float row stride of the reduction tiles
  static constexpr int MAIN = 2 * KT + 2 * STAGE + 2 * PT;
  static constexpr int RED = 2 * 128 * LDR * 4;
  static constexpr int BODY = MAIN > RED ? MAIN : RED;
  static constexpr int SMEM = BODY + 1024 + 256;
  static constexpr uint32_t TMEM_COLS = 512;  // S^T, dP^T double-buffered (4 x 64) + dV + dK
};

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    attn_dkdv_tc_kernel(const __grid_constant__ CUtensorMap map_h128,
                        const __grid_constant__ CUtensorMap map_b128,
                        const __grid_constant__ CUtensorMap map_h64,
                        const __grid_constant__ CUtensorMap map_b64,
                        const __grid_constant__ CUtensorMap map_do64, const AttnArgs a) {
  using C = Dkv<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1k(smem_raw);
  uint8_t *Ks = smem, *Vs = smem + C::KT, *ring = smem + 2 * C::KT;
  uint8_t *Pt = ring + 2 * C::STAGE, *dSt = Pt + C::PT;
  float *red_k = reinterpret_cast<float *>(smem);  // after the main loop: [128][LDR] each
  float *red_v = red_k + 128 * C::LDR;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::BODY);
  uint64_t *kv_full = bar, *q_full = bar + 1, *q_empty = bar + 3, *sd_full = bar + 5;
  uint64_t *pds_full = bar + 7, *pds_free = bar + 8, *mma_done = bar + 9;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 10);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  cg::cluster_group cluster = cg::this_cluster();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.S;
  const int h = blockIdx.x, kb = blockIdx.y, b = blockIdx.z;
  const int g = h / a.grp;
  const int k0 = kb * 128;
  const int qfirst = 2 * kb;                 // first query block of 64 at or after the keys
  const int nqb = (S + 63) / 64 - qfirst;    // >= 1

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
      mbar_init(&sd_full[s], 1);
    }
    mbar_init(pds_full, ROWS);
    mbar_init(pds_free, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tc_alloc(tmem_slot, C::TMEM_COLS);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_dv = tmem + 256, t_dk = tmem + 256 + D;

  if (warp == TMA_WARP) {
    if (lane == 0) {
      tma_prefetch_desc(&map_h64);
      tma_prefetch_desc(&map_b64);
      tma_prefetch_desc(&map_do64);
      const int cq = h * D, ck = (a.nh + g) * D, cv = (a.nh + a.nkv + g) * D;
      mbar_arrive_expect_tx(kv_full, 2 * C::KT);
#pragma unroll
      for (int p = 0; p < D / 64; ++p) {
        tma_load_3d(Ks + p * PANEL128, &map_h128, ck + 64 * p, k0, b, kv_full);
        tma_load_3d(Vs + p * PANEL128, &map_b128, cv + 64 * p, k0, b, kv_full);
      }
      int issued = 0;
      for (int i = 0; i < nqb; ++i) {
        const int s = i & 1;
        if (i >= 2 && !mbar_wait(&q_empty[s], ((i >> 1) - 1) & 1, a.err, abort_flag)) break;
        uint8_t *st = ring + s * C::STAGE;
        const int q0 = (qfirst + i) * 64;
        mbar_arrive_expect_tx(&q_full[s], C::STAGE);
#pragma unroll
        for (int p = 0; p < D / 64; ++p) {
          tma_load_3d(st + p * PANEL64, &map_h64, cq + 64 * p, q0, b, &q_full[s]);
          tma_load_3d(st + C::QT + p * PANEL64, &map_b64, cq + 64 * p, q0, b, &q_full[s]);
          tma_load_3d(st + 2 * C::QT + p * PANEL64, &map_do64, h * D + 64 * p, q0, b, &q_full[s]);
        }
        ++issued;
      }
      volatile int no_abort = 0;
      mbar_wait(kv_full, 0, a.err, &no_abort);
      for (int i = max(0, issued - 2); i < issued; ++i)
        mbar_wait(&q_full[i & 1], (i >> 1) & 1, a.err, &no_abort);
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_16(128, 64, 0, 0, 1);    // S^T: half
      constexpr uint32_t id_dp = idesc_16(128, 64, 0, 0, 0);   // dP^T: bf16
      constexpr uint32_t id_acc = idesc_16(128, D, 0, 1, 0);   // dV, dK: bf16, B MN-major
      const uint32_t ka = smem_u32(Ks), va = smem_u32(Vs), pa = smem_u32(Pt), dsa = smem_u32(dSt);
      auto issue_sd = [&](int i) -> bool {
        const int s = i & 1;
        if (!mbar_wait(&q_full[s], (i >> 1) & 1, a.err, abort_flag)) return false;
        tc_fence_after();
        const uint32_t qh = smem_u32(ring + s * C::STAGE), dob = qh + 2 * C::QT;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o128 = (kk >> 2) * PANEL128 + (kk & 3) * 32;
          const uint32_t o64 = (kk >> 2) * PANEL64 + (kk & 3) * 32;
          tc_mma_bf16(tmem + s * 128, smem_desc(ka + o128, 16, 1024), smem_desc(qh + o64, 16, 1024),
                      id_s, kk > 0);
          tc_mma_bf16(tmem + s * 128 + 64, smem_desc(va + o128, 16, 1024),
                      smem_desc(dob + o64, 16, 1024), id_dp, kk > 0);
        }
        tc_commit(&sd_full[s]);
        return true;
      };
      bool ok = mbar_wait(kv_full, 0, a.err, abort_flag) && issue_sd(0);
      for (int i = 0; ok && i < nqb; ++i) {
        const int s = i & 1;
        if (i + 1 < nqb && !issue_sd(i + 1)) break;
        if (!mbar_wait(pds_full, i & 1, a.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t qb16 = smem_u32(ring + s * C::STAGE) + C::QT, dob = qb16 + C::QT;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          tc_mma_bf16(t_dv, smem_desc(pa + kk * 32, 16, 1024),
                      smem_desc(dob + kk * 2048, PANEL64, 1024), id_acc, (i | kk) != 0);
          tc_mma_bf16(t_dk, smem_desc(dsa + kk * 32, 16, 1024),
                      smem_desc(qb16 + kk * 2048, PANEL64, 1024), id_acc, (i | kk) != 0);
        }
        tc_commit(&q_empty[s]);
        tc_commit(pds_free);
      }
      tc_commit(mma_done);
      volatile int no_abort = 0;
      mbar_wait(mma_done, 0, a.err, &no_abort);
    }
  } else {
    // ------------------------------------------------------------------ row threads
    const int r = threadIdx.x;
    const int key = k0 + r;
    const uint32_t lq = (uint32_t)(warp * 32) << 16;
    const size_t lbase = ((size_t)b * a.nh + h) * S;
    bool ok = true;
    for (int i = 0; i < nqb; ++i) {
      const int s = i & 1;
      const int q0 = (qfirst + i) * 64;
      if (!warp_all(mbar_wait(&sd_full[s], (i >> 1) & 1, a.err, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t ppk[2][16], dpk[2][16];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        // the chunk's 32 query log-sum-exps and row sums: the same addresses across the warp
        // (one broadcast load each), issued before the TMEM loads are waited for
        float lsv[32], dsv[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int q = q0 + c * 32 + e;
          lsv[e] = q < S ? __ldg(a.lse + lbase + q) : INFINITY;
          dsv[e] = q < S ? __ldg(a.dsum + lbase + q) : 0.f;
        }
        uint32_t sv[32], dv[32];
        __syncwarp();
        tc_ld_32x32b_x32(tmem + lq + s * 128 + c * 32, sv);
        tc_ld_32x32b_x32(tmem + lq + s * 128 + 64 + c * 32, dv);
        tc_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float p2[2], d2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int qi = c * 32 + 2 * e + u, q = q0 + qi;
            const bool vis = q >= key && q < S && key < S;
            const float p = vis ? ex2(__uint_as_float(sv[2 * e + u]) * a.scale_log2 - lsv[2 * e + u]) : 0.f;
            p2[u] = p;
            d2[u] = p * (__uint_as_float(dv[2 * e + u]) - dsv[2 * e + u]);
          }
          ppk[c][e] = pack_bf16x2(p2[0], p2[1]);
          dpk[c][e] = pack_bf16x2(d2[0], d2[1]);
        }
      }
      // the dV / dK products of the previous query block have finished with P^T and dS^T
      if (i >= 1 && !warp_all(mbar_wait(pds_free, (i - 1) & 1, a.err, abort_flag))) {
        ok = false;
        break;
      }
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          *reinterpret_cast<uint4 *>(Pt + sw128(r, c * 4 + q)) = u4(ppk[c] + 4 * q);
          *reinterpret_cast<uint4 *>(dSt + sw128(r, c * 4 + q)) = u4(dpk[c] + 4 * q);
        }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(pds_full);
    }
    volatile int no_abort = 0;
    ok = warp_all(ok && mbar_wait(mma_done, 0, a.err, &no_abort) && !*abort_flag);
    tc_fence_after();
    if (ok) {
      // this head's dK (scaled) and dV rows into the reduction tiles (the operand space is idle:
      // every MMA has retired and every copy has landed)
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t kv[32], vv[32];
        __syncwarp();
        tc_ld_32x32b_x32(t_dk + lq + c * 32, kv);
        tc_ld_32x32b_x32(t_dv + lq + c * 32, vv);
        tc_wait_ld();
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          *reinterpret_cast<float4 *>(red_k + r * C::LDR + c * 32 + 4 * e) =
              make_float4(__uint_as_float(kv[4 * e]) * a.scale, __uint_as_float(kv[4 * e + 1]) * a.scale,
                          __uint_as_float(kv[4 * e + 2]) * a.scale, __uint_as_float(kv[4 * e + 3]) * a.scale);
          *reinterpret_cast<float4 *>(red_v + r * C::LDR + c * 32 + 4 * e) =
              make_float4(__uint_as_float(vv[4 * e]), __uint_as_float(vv[4 * e + 1]),
                          __uint_as_float(vv[4 * e + 2]), __uint_as_float(vv[4 * e + 3]));
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  cluster.sync();  // every head's tiles are in its shared memory
  {
    // rank `rank` sums rows [r0, r1) of the key block over the cluster's heads, in head order
    const int grp = a.grp;
    const int rank = (int)cluster.block_rank();
    const int per = (128 + grp - 1) / grp;
    const int r0 = rank * per, r1 = min(128, r0 + per);
    const float *pk[8], *pv[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      pk[c] = cluster.map_shared_rank(red_k, c < grp ? c : 0);
      pv[c] = cluster.map_shared_rank(red_v, c < grp ? c : 0);
    }
    constexpr int C4 = D / 4;
    for (int idx = threadIdx.x; idx < (r1 - r0) * C4; idx += THREADS) {
      const int rr = r0 + idx / C4, c4 = (idx % C4) * 4;
      const int t = k0 + rr;
      if (t >= S) continue;
      // every remote load in flight before the first add; then the sum in head order
      float4 xk[8], xv[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        xk[c] = c < grp ? *reinterpret_cast<const float4 *>(pk[c] + rr * C::LDR + c4) : z;
        xv[c] = c < grp ? *reinterpret_cast<const float4 *>(pv[c] + rr * C::LDR + c4) : z;
      }
      float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sv = sk;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        if (c >= grp) break;
        sk.x += xk[c].x; sk.y += xk[c].y; sk.z += xk[c].z; sk.w += xk[c].w;
        sv.x += xv[c].x; sv.y += xv[c].y; sv.z += xv[c].z; sv.w += xv[c].w;
      }
      float *rowp = a.dqkv + ((size_t)b * S + t) * a.ld;
      *reinterpret_cast<float4 *>(rowp + (size_t)(a.nh + g) * D + c4) = sk;
      *reinterpret_cast<float4 *>(rowp + (size_t)(a.nh + a.nkv + g) * D + c4) = sv;
    }
  }
  cluster.sync();  // no CTA leaves while another still reads its shared memory
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tc_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------ host side
// Dynamic shared memory for a kernel whose CTAs each hold `tmem_cols` TMEM columns: at least
// `used` bytes, and enough that no more CTAs fit on an SM than its 512 TMEM columns hold, so a
// CTA's tcgen05.alloc never waits on another resident CTA (which, inside a cluster waiting on
// its peers, could wait forever).  Checked with the occupancy calculator; computed once per
// device and kernel.
template <typename K>
int tmem_safe_smem(std::atomic<int> (&slot)[MAX_DEVICES], K kern, int used, int tmem_cols, int *bytes) {
  cudaError_t e = per_device_once(slot, bytes, [&](int dev, int *v) {
    int per_sm = 0, reserved = 0, optin = 0;
    cudaError_t r = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (r == cudaSuccess) r = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (r == cudaSuccess) r = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (r != cudaSuccess) return r;
    const int max_ctas = 512 / tmem_cols;
    // max_ctas + 1 CTAs of (n + reserved) bytes must not fit in per_sm
    const int n = std::max(used, per_sm / (max_ctas + 1) - reserved + 16);
    if (n > optin) return cudaErrorInvalidValue;
    r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, n);
    if (r != cudaSuccess) return r;
    int occ = 0;
    r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, THREADS, n);
    if (r != cudaSuccess) return r;
    if (occ < 1 || occ > max_ctas) return cudaErrorInvalidConfiguration;
    *v = n;
    return cudaSuccess;
  });
  if (e != cudaSuccess)
    return set_error(SOUP_ECUDA, "attention: no shared-memory size keeps TMEM exclusive (%s)", cudaGetErrorString(e));
  return 0;
}

// rows of the fused buffer as a [B][S][ld] tensor, 64-column boxes of `rows` rows
int map_rows(CUtensorMap *m, CUtensorMapDataType dt, const void *base, int ld, int S, int B, int rows,
             const char *what) {
  if (reinterpret_cast<uintptr_t>(base) % 16)
    return set_error(SOUP_EINVAL, "attention: %s is not 16-byte aligned", what);
  return tmap_3d(m, dt, base, (uint64_t)ld, (uint64_t)S, (uint64_t)B, (uint64_t)ld * 2,
                 (uint64_t)S * ld * 2, 64, (uint32_t)rows, CU_TENSOR_MAP_SWIZZLE_128B, what);
}

AttnArgs make_args(int S, int nh, int nkv, int d, int ld, int *err) {
  AttnArgs a{};
  a.S = S;
  a.nh = nh;
  a.nkv = nkv;
  a.grp = nh / nkv;
  a.ld = ld;
  a.scale = 1.0f / sqrtf((float)d);
  a.scale_log2 = a.scale * 1.4426950408889634f;
  a.err = err;
  return a;
}

template <int D>
int fwd_tc(const uint16_t *qkv, int ld, int B, int S, int nh, int nkv, uint16_t *o, float *lse,
           int *err, cudaStream_t st) {
  static std::atomic<int> attr[MAX_DEVICES];
  int smem = 0;
  SOUP_TRY(tmem_safe_smem(attr, attn_fwd_tc_kernel<D>, Fwd<D>::SMEM, Fwd<D>::TMEM_COLS, &smem));
  CUtensorMap mh;
  SOUP_TRY(map_rows(&mh, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qkv, ld, S, B, 128, "qkv"));
  AttnArgs a = make_args(S, nh, nkv, D, ld, err);
  a.o = o;
  a.lse = lse;
  dim3 grid((S + 127) / 128, nh, B);
  attn_fwd_tc_kernel<D><<<grid, THREADS, smem, st>>>(mh, a);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(SOUP_ECUDA, "attention forward launch: %s", cudaGetErrorString(e));
  return 0;
}

template <int D>
int bwd_tc(const uint16_t *qkv, int ld, const uint16_t *o, const uint16_t *dO, const float *lse,
           int B, int S, int nh, int nkv, float *scratch, float *dqkv, int *err, cudaStream_t st) {
  static std::atomic<int> attr_dq[MAX_DEVICES], attr_kv[MAX_DEVICES];
  int smem_dq = 0, smem_kv = 0;
  SOUP_TRY(tmem_safe_smem(attr_dq, attn_dq_tc_kernel<D>, Dq<D>::SMEM, Dq<D>::TMEM_COLS, &smem_dq));
  SOUP_TRY(tmem_safe_smem(attr_kv, attn_dkdv_tc_kernel<D>, Dkv<D>::SMEM, Dkv<D>::TMEM_COLS, &smem_kv));
  const int M = B * S, qd = nh * D;
  float *dsum = scratch;
  uint16_t *qkv_b = reinterpret_cast<uint16_t *>(scratch + (((size_t)B * nh * S + 63) / 64) * 64);
  CUtensorMap h128, h64, b128, b64, do128, do64;
  SOUP_TRY(map_rows(&h128, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qkv, ld, S, B, 128, "qkv"));
  SOUP_TRY(map_rows(&h64, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qkv, ld, S, B, 64, "qkv"));
  SOUP_TRY(map_rows(&b128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, qkv_b, ld, S, B, 128, "qkv (bf16 copy)"));
  SOUP_TRY(map_rows(&b64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, qkv_b, ld, S, B, 64, "qkv (bf16 copy)"));
  SOUP_TRY(map_rows(&do128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dO, qd, S, B, 128, "dO"));
  SOUP_TRY(map_rows(&do64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dO, qd, S, B, 64, "dO"));
  AttnArgs a = make_args(S, nh, nkv, D, ld, err);
  a.lse = const_cast<float *>(lse);
  a.dsum = dsum;
  a.dqkv = dqkv;

  attn_bwd_prep_kernel<<<M, 256, 0, st>>>(qkv, ld, o, dO, S, nh, D, dsum, qkv_b);
  attn_dq_tc_kernel<D><<<dim3((S + 127) / 128, nh, B), THREADS, smem_dq, st>>>(h128, do128, h64, b64, a);
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nh, (S + 127) / 128, B);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem_kv;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = a.grp;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, attn_dkdv_tc_kernel<D>, h128, b128, h64, b64, do64, a);
    if (e != cudaSuccess) return set_error(SOUP_ECUDA, "attention dK/dV launch: %s", cudaGetErrorString(e));
  }
  count_launches(3);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(SOUP_ECUDA, "attention backward launch: %s", cudaGetErrorString(e));
  return 0;
}

}  // namespace

int attn_tc_eligible(int d, int nh, int nkv) {
  return (d == 64 || d == 128) && nkv > 0 && nh % nkv == 0 && nh / nkv <= 8;
}

size_t attn_tc_scratch_floats(int B, int S, int nh, int nkv, int d) {
  const size_t ld = (size_t)(nh + 2 * nkv) * d;
  return (((size_t)B * nh * S + 63) / 64) * 64 + ((size_t)B * S * ld + 1) / 2;
}

int k_attn_fwd_tc(const uint16_t *qkv, int ld, int B, int S, int nh, int nkv, int d, uint16_t *o,
                  float *lse, int *err, cudaStream_t st) {
  if (d == 128) return fwd_tc<128>(qkv, ld, B, S, nh, nkv, o, lse, err, st);
  return fwd_tc<64>(qkv, ld, B, S, nh, nkv, o, lse, err, st);
}

int k_attn_bwd_tc(const uint16_t *qkv, int ld, const uint16_t *o, const uint16_t *dO,
                  const float *lse, int B, int S, int nh, int nkv, int d, float *scratch,
                  float *dqkv, int *err, cudaStream_t st) {
  if (d == 128) return bwd_tc<128>(qkv, ld, o, dO, lse, B, S, nh, nkv, scratch, dqkv, err, st);
  return bwd_tc<64>(qkv, ld, o, dO, lse, B, S, nh, nkv, scratch, dqkv, err, st);
}

}  // namespace soup
