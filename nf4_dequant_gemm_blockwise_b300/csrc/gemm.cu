// Base-weight GEMMs of the streamed LoRA step on sm_103a.
//
// What is computed ("Layer streaming: fine-tune a model that does not fit in your card",
// "How it works": every projection of the decoder layer runs on the streamed weight bytes;
// the backward needs W^T dL/dy, so the weights are read again; "Bit-exact is two claims":
// the backward dequantises, it never caches dequantised weights):
//   forward  y  = x  deq(W)^T + s (x A^T) B^T
//   backward dx = dY deq(W)   + s (dY B)   A
// deq(W)[n,k] = round16(float(c[code] * absmax[block])), blocks of 64 along the flattened
// [out, in] matrix, where round16 rounds to nearest-even in the GEMM's 16-bit operand format:
// IEEE half for the forward (activations are half there), bf16 for dX (gradients need the
// exponent range).  The rank-r LoRA term is folded into the same tensor-core reduction as
// extra 64-wide K tiles: the caller packs s(xA^T) (or s(dY B)) as bf16 [M, R] and the
// matching B rows (or A rows) as bf16, zero-padded to R = 64 * ceil(segments * r / 64).
//
// Tensor-core kernel (tcgen05, one CTA per 128 x BN output tile, 320 threads):
//   warp 8      TMA producer: activation tile (128 x 64 bf16, 128-byte swizzle), the raw
//               4-bit codes and float absmax of the weight tile (or a bf16 weight tile)
//   warps 0..7  dequantise codes -> bf16 into the swizzled shared-memory layout the tensor
//               core reads (K-major for the forward, MN-major for dX), then run the
//               epilogue from TMEM
//   warp 9      allocates TMEM; one lane issues tcgen05.mma (M=128, N=BN, K=16) x 4 per
//               stage and commits each stage back to the producer
// Dequantisation uses a per-block table: the 16 products c_k * absmax rounded to bf16,
// then byte permutes look up four codes at a time (no shared-memory table, no divergence).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "util.h"

namespace soup {
namespace {
using namespace soupk;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int DQ_WARPS = 8;
constexpr int THREADS = (DQ_WARPS + 2) * 32;
enum BMode { B_NF4_K = 0, B_NF4_MN = 1, B_BF16_K = 2, B_BF16_MN = 3 };

template <int BN, int BMODE, bool F16>
struct TcCfg {
  static constexpr bool NF4 = (BMODE == B_NF4_K || BMODE == B_NF4_MN);
  // bf16 weights feeding a half-precision GEMM are converted in shared memory, in place
  static constexpr bool CONV = !NF4 && F16;
  static constexpr bool PRODUCE = NF4 || CONV;  // the worker warps touch the B tile
  static constexpr bool MN = (BMODE == B_NF4_MN || BMODE == B_BF16_MN);
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int RAW_BYTES = NF4 ? BN * 32 : 0;
  static constexpr int ABS_BYTES = NF4 ? ((BN * 16 + 1023) / 1024) * 1024 : 0;
  static constexpr int STAGE = A_BYTES + B_BYTES + RAW_BYTES + ABS_BYTES;
  static constexpr int NS = NF4 ? 3 : 4;
  static constexpr int SMEM = NS * STAGE + 1024 + 256;
  // expected TMA bytes per main stage
  static constexpr uint32_t TX_MAIN =
      A_BYTES + (NF4 ? (BN * 32 + (MN ? 64 * 16 : BN * 16)) : B_BYTES);
  static constexpr uint32_t TX_EXT = A_BYTES + B_BYTES;
};

struct TcParams {
  Codebook cb;
  int M, Ng, n_main, n_ext;
  void *out;
  int ldo;
  const float *add_src;
  int ld_add;
  int *err;
};

// Dequantise one 64-weight block: cw = 32 bytes of packed codes, a = the block's absmax.
// out[c] = 8 16-bit weights c*8 .. c*8+7 (half if F16, else bf16).
template <bool F16>
SOUP_DEV void dq_block64(const float *cb, const uint32_t (&cw)[8], float a, uint4 (&out)[8]) {
  uint32_t P[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) P[j] = pack16x2<F16>(cb[2 * j] * a, cb[2 * j + 1] * a);
  uint32_t LO[4], HI[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    LO[j] = prmt(P[2 * j], P[2 * j + 1], 0x6420);  // low bytes of entries 4j..4j+3
    HI[j] = prmt(P[2 * j], P[2 * j + 1], 0x7531);  // high bytes
  }
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t x = cw[w];
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      // four selectors = four codes; a byte holds (even code << 4 | odd code)
      const uint32_t s = (x >> (16 * h)) & 0xFFFFu;
      const uint32_t s7 = s & 0x7777u;
      const uint32_t pick = ((s >> 1) & 0x4444u) | 0x3210u;  // +4 for codes 8..15
      const uint32_t lo = prmt(prmt(LO[0], LO[1], s7), prmt(LO[2], LO[3], s7), pick);
      const uint32_t hi = prmt(prmt(HI[0], HI[1], s7), prmt(HI[2], HI[3], s7), pick);
      o[2 * h] = prmt(lo, hi, 0x4051);      // (even, odd) code of byte 0 -> 16x2
      o[2 * h + 1] = prmt(lo, hi, 0x6273);  // byte 1
    }
    out[w] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Offset of 16-byte chunk c of row r inside a 128-byte-swizzled tile (rows of 128 bytes,
// 8-row atoms of 1024 bytes).
SOUP_DEV uint32_t sw128(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

template <int BN, int BMODE, int EPI, bool F16>
__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_b0,
                   const __grid_constant__ CUtensorMap map_b1,
                   const __grid_constant__ CUtensorMap map_ul,
                   const __grid_constant__ CUtensorMap map_vl, const TcParams p) {
  using C = TcCfg<BN, BMODE, F16>;
  constexpr int NS = C::NS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw_base + 1023u) & ~1023u) - raw_base);
  uint8_t *stage0 = smem;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + NS * C::STAGE);
  uint64_t *full = bar;             // TMA landed
  uint64_t *bready = bar + NS;      // B operand ready (dequantised)
  uint64_t *empty = bar + 2 * NS;   // MMAs done reading the stage
  uint64_t *accf = bar + 3 * NS;    // accumulator complete
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 3 * NS + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * BM;
  const int n_total = p.n_main + p.n_ext;

  auto A_s = [&](int s) { return stage0 + s * C::STAGE; };
  auto B_s = [&](int s) { return stage0 + s * C::STAGE + C::A_BYTES; };
  auto R_s = [&](int s) { return stage0 + s * C::STAGE + C::A_BYTES + C::B_BYTES; };
  auto S_s = [&](int s) {
    return stage0 + s * C::STAGE + C::A_BYTES + C::B_BYTES + C::RAW_BYTES;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&bready[s], DQ_WARPS);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accf, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == DQ_WARPS + 1) {
    tc_alloc(tmem_slot, BN);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == DQ_WARPS) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&map_a);
      tma_prefetch_desc(&map_b0);
      int issued = 0;
      for (int kt = 0; kt < n_total; ++kt) {
        const int s = kt % NS;
        if (kt >= NS && !mbar_wait(&empty[s], ((kt / NS) - 1) & 1, p.err, abort_flag)) break;
        if (kt < p.n_main) {
          mbar_arrive_expect_tx(&full[s], C::TX_MAIN);
          tma_load_2d(A_s(s), &map_a, kt * BK, m0, &full[s]);
          if (BMODE == B_NF4_K) {
            tma_load_2d(R_s(s), &map_b0, kt * (BK / 2), n0, &full[s]);
            tma_load_2d(S_s(s), &map_b1, (kt & ~3), n0, &full[s]);
          } else if (BMODE == B_NF4_MN) {
            tma_load_2d(R_s(s), &map_b0, n0 / 2, kt * BK, &full[s]);
            tma_load_2d(S_s(s), &map_b1, n0 / 64, kt * BK, &full[s]);
          } else if (BMODE == B_BF16_K) {
            tma_load_2d(B_s(s), &map_b0, kt * BK, n0, &full[s]);
          } else {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_2d(B_s(s) + c * 8192, &map_b0, n0 + 64 * c, kt * BK, &full[s]);
          }
        } else {
          const int e = kt - p.n_main;
          mbar_arrive_expect_tx(&full[s], C::TX_EXT);
          tma_load_2d(A_s(s), &map_ul, e * BK, m0, &full[s]);
          if (!C::MN) {
            tma_load_2d(B_s(s), &map_vl, e * BK, n0, &full[s]);
          } else {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_2d(B_s(s) + c * 8192, &map_vl, n0 + 64 * c, e * BK, &full[s]);
          }
        }
        ++issued;
      }
      // never leave the CTA with copies still landing in its shared memory
      for (int kt = (issued > NS ? issued - NS : 0); kt < issued; ++kt) {
        volatile int no_abort = 0;
        mbar_wait(&full[kt % NS], (kt / NS) & 1, p.err, &no_abort);
      }
    }
  } else if (warp == DQ_WARPS + 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_16(BM, BN, 0, C::MN ? 1 : 0, F16 ? 1 : 0);
      uint64_t *wait_bar = C::PRODUCE ? bready : full;
      for (int kt = 0; kt < n_total; ++kt) {
        const int s = kt % NS;
        if (!mbar_wait(&wait_bar[s], (kt / NS) & 1, p.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(A_s(s));
        const uint32_t b_addr = smem_u32(B_s(s));
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = smem_desc(a_addr + kk * 32, 16, 1024);
          const uint64_t bd = C::MN ? smem_desc(b_addr + kk * 2048, 8192, 1024)
                                    : smem_desc(b_addr + kk * 32, 16, 1024);
          tc_mma_bf16(tmem, ad, bd, idesc, (kt | kk) != 0);
        }
        tc_commit(&empty[s]);
      }
      tc_commit(accf);
      volatile int no_abort = 0;
      mbar_wait(accf, 0, p.err, &no_abort);  // every MMA retired before TMEM is freed
    }
  } else {
    // ---------------------------------------------------------------- dequant warps
    const int t = threadIdx.x;  // 0 .. 255
    for (int kt = 0; C::PRODUCE && kt < n_total; ++kt) {
      const int s = kt % NS;
      if (!mbar_wait(&full[s], (kt / NS) & 1, p.err, abort_flag)) break;
      if (C::CONV && kt < p.n_main) {
        // bf16 -> half, element by element; the byte layout (and so the swizzle) is unchanged
        uint4 *Bs = reinterpret_cast<uint4 *>(B_s(s));
        for (int i = t; i < C::B_BYTES / 16; i += DQ_WARPS * 32) {
          uint4 v = Bs[i];
          v.x = pack_h2(bf16_lo(v.x), bf16_hi(v.x));
          v.y = pack_h2(bf16_lo(v.y), bf16_hi(v.y));
          v.z = pack_h2(bf16_lo(v.z), bf16_hi(v.z));
          v.w = pack_h2(bf16_lo(v.w), bf16_hi(v.w));
          Bs[i] = v;
        }
        fence_async_smem();
      }
      if (C::NF4 && kt < p.n_main) {
        uint8_t *Bs = B_s(s);
        const uint8_t *Rs = R_s(s);
        const uint8_t *Ss = S_s(s);
        if (BMODE == B_NF4_K) {
          for (int n = t; n < BN; n += DQ_WARPS * 32) {
            const uint4 c0 = *reinterpret_cast<const uint4 *>(Rs + n * 32);
            const uint4 c1 = *reinterpret_cast<const uint4 *>(Rs + n * 32 + 16);
            const float a = *reinterpret_cast<const float *>(Ss + n * 16 + (kt & 3) * 4);
            const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            uint4 o[8];
            dq_block64<F16>(p.cb.v, cw, a, o);
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(Bs + sw128(n, c)) = o[c];
          }
        } else {
          for (int it = t; it < 64 * (BN / 64); it += DQ_WARPS * 32) {
            const int n = it & 63, seg = it >> 6;
            const uint4 c0 = *reinterpret_cast<const uint4 *>(Rs + sw128(n, 2 * seg));
            const uint4 c1 = *reinterpret_cast<const uint4 *>(Rs + sw128(n, 2 * seg + 1));
            const float a = *reinterpret_cast<const float *>(Ss + n * 16 + seg * 4);
            const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            uint4 o[8];
            dq_block64<F16>(p.cb.v, cw, a, o);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4 *>(Bs + seg * 8192 + sw128(n, c)) = o[c];
          }
        }
        fence_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bready[s]);
    }
    // ---------------------------------------------------------------- epilogue
    volatile int no_abort = 0;
    const bool ok = !*abort_flag && mbar_wait(accf, 0, p.err, &no_abort) && !*abort_flag;
    tc_fence_after();
    if (ok) {
      const int q = warp & 3;
      const int m = m0 + q * 32 + lane;
      for (int cc = 0; cc < BN / 64; ++cc) {
        const int col = (warp >> 2) * (BN / 2) + cc * 32;
        uint32_t r[32];
        tc_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + col, r);
        tc_wait_ld();
        if (m >= p.M) continue;
        const int n = n0 + col;
        if (n >= p.Ng) continue;
        const bool full_row = (n + 32 <= p.Ng);
        if (EPI == EPI_16) {
          uint16_t *o = reinterpret_cast<uint16_t *>(p.out) + (size_t)m * p.ldo + n;
          if (full_row) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 w;
              w.x = pack16x2<F16>(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
              w.y = pack16x2<F16>(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
              w.z = pack16x2<F16>(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
              w.w = pack16x2<F16>(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
              *reinterpret_cast<uint4 *>(o + 8 * v) = w;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n + j < p.Ng) o[j] = st16<F16>(__uint_as_float(r[j]));
          }
        } else {
          float *o = reinterpret_cast<float *>(p.out) + (size_t)m * p.ldo + n;
          const float *src = (EPI == EPI_F32_ADD) ? p.add_src + (size_t)m * p.ld_add + n
                                                  : (EPI == EPI_F32_ACC ? o : nullptr);
          if (full_row) {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              float4 w = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                     __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
              if (src) {
                const float4 b = *reinterpret_cast<const float4 *>(src + 4 * v);
                w.x = b.x + w.x; w.y = b.y + w.y; w.z = b.z + w.z; w.w = b.w + w.w;
              }
              *reinterpret_cast<float4 *>(o + 4 * v) = w;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (n + j < p.Ng) {
                float w = __uint_as_float(r[j]);
                if (src) w = src[j] + w;
                o[j] = w;
              }
            }
          }
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == DQ_WARPS + 1) {
    __syncwarp();
    tc_fence_after();
    tc_dealloc(tmem, BN);
  }
}

// ---------------------------------------------------------------------------------------
// Tiled fallback for shapes the tensor-core kernel does not take (blocks that straddle rows,
// unaligned strides).  Same operand definition, float accumulation, 64x64 tiles.
struct FbParams {
  Codebook cb;
  int f16;
  int mode, M, Ng, Kg, wfmt, Nw, Kw, ldw, lda, R, epi, ldo, ld_add;
  const uint16_t *a;
  const uint8_t *codes;
  const float *absmax;
  const uint16_t *w;
  const uint16_t *ul, *vl;
  void *out;
  const float *add_src;
};

SOUP_DEV float fb_round(const FbParams &p, float v) {
  return p.f16 ? h16_to_f(f_to_h16(v)) : bf16_to_f(f_to_bf16(v));
}
SOUP_DEV float fb_ld16(const FbParams &p, uint16_t v) { return p.f16 ? h16_to_f(v) : bf16_to_f(v); }
SOUP_DEV float fb_weight(const FbParams &p, int row, int col) {  // W[row, col] as used
  if (p.wfmt == W_NF4) {
    const int64_t f = (int64_t)row * p.Kw + col;
    const uint8_t b = p.codes[f >> 1];
    const int code = (f & 1) ? (b & 15) : (b >> 4);
    const float v = p.cb.v[code] * p.absmax[f >> 6];
    return fb_round(p, v);
  }
  return fb_round(p, bf16_to_f(p.w[(int64_t)row * p.ldw + col]));
}

__global__ void __launch_bounds__(256) fallback_gemm_kernel(const FbParams p) {
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4] = {};
  const int k_main = p.Kg;
  const int k_total = k_main + p.R;
  for (int k0 = 0; k0 < k_total; k0 += 16) {
    for (int i = threadIdx.x; i < 16 * 64; i += 256) {
      const int kk = i >> 6, mm = i & 63;
      const int m = m0 + mm, k = k0 + kk;
      float v = 0.f;
      if (m < p.M && k < k_total) {
        if (k < k_main) v = fb_ld16(p, p.a[(int64_t)m * p.lda + k]);
        else v = fb_ld16(p, p.ul[(int64_t)m * p.R + (k - k_main)]);
      }
      As[kk][mm] = v;
      const int n = n0 + mm;
      float b = 0.f;
      if (n < p.Ng && k < k_total) {
        if (k < k_main) b = (p.mode == GEMM_FWD) ? fb_weight(p, n, k) : fb_weight(p, k, n);
        else {
          const int j = k - k_main;
          b = (p.mode == GEMM_FWD) ? fb_ld16(p, p.vl[(int64_t)n * p.R + j])
                                   : fb_ld16(p, p.vl[(int64_t)j * p.Ng + n]);
        }
      }
      Bs[kk][mm] = b;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= p.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= p.Ng) continue;
      const float v = acc[i][j];
      if (p.epi == EPI_16) {
        reinterpret_cast<uint16_t *>(p.out)[(int64_t)m * p.ldo + n] = p.f16 ? f_to_h16(v) : f_to_bf16(v);
      } else {
        float *o = reinterpret_cast<float *>(p.out) + (int64_t)m * p.ldo + n;
        if (p.epi == EPI_F32) *o = v;
        else if (p.epi == EPI_F32_ADD) *o = p.add_src[(int64_t)m * p.ld_add + n] + v;
        else *o = *o + v;
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_mu;
int g_force_fallback = 0;

int get_encode() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return 0;
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
    return set_error(SOUP_ECUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(e));
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return 0;
}

int make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner,
             uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
             CUtensorMapSwizzle sw, const char *what) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void *>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(SOUP_EINVAL, "tensor map for %s rejected (CUresult %d)", what, (int)r);
  return 0;
}

template <int BN, int BMODE, int EPI, bool F16>
int launch_tc(const GemmArgs &g, const CUtensorMap *maps, cudaStream_t st) {
  using C = TcCfg<BN, BMODE, F16>;
  static bool attr_done = false;  // per instantiation; set under g_mu
  auto kern = tc_gemm_kernel<BN, BMODE, EPI, F16>;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!attr_done) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
      if (e != cudaSuccess) return set_error(SOUP_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      attr_done = true;
    }
  }
  TcParams p;
  p.cb = nf4_codebook_param();
  p.M = g.M;
  p.Ng = g.Ng();
  p.n_main = (g.Kg() + BK - 1) / BK;
  p.n_ext = g.R / BK;
  p.out = g.out;
  p.ldo = g.ldo;
  p.add_src = g.add_src;
  p.ld_add = g.ld_add;
  p.err = g.err;
  dim3 grid((p.Ng + BN - 1) / BN, (g.M + BM - 1) / BM);
  kern<<<grid, THREADS, C::SMEM, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(SOUP_ECUDA, "tc_gemm launch: %s", cudaGetErrorString(e));
  return 0;
}

template <int BN, int BMODE, bool F16>
int launch_tc_epi(const GemmArgs &g, const CUtensorMap *maps, cudaStream_t st) {
  switch (g.epi) {
    case EPI_16: return launch_tc<BN, BMODE, EPI_16, F16>(g, maps, st);
    case EPI_F32: return launch_tc<BN, BMODE, EPI_F32, F16>(g, maps, st);
    case EPI_F32_ADD: return launch_tc<BN, BMODE, EPI_F32_ADD, F16>(g, maps, st);
    default: return launch_tc<BN, BMODE, EPI_F32_ACC, F16>(g, maps, st);
  }
}
template <int BN, int BMODE>
int launch_tc_op(const GemmArgs &g, const CUtensorMap *maps, cudaStream_t st) {
  return g.op_f16 ? launch_tc_epi<BN, BMODE, true>(g, maps, st)
                  : launch_tc_epi<BN, BMODE, false>(g, maps, st);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

int gemm_uses_tc(const GemmArgs &g) {
  if (g_force_fallback) return 0;
  const int Ng = g.Ng();
  if (g.M < 1 || Ng < 1 || g.Kg() < 1) return 0;
  if (g.Kw % 256 != 0) return 0;                      // absmax rows: 16-byte multiple
  if (g.lda % 8 || !aligned16(g.a)) return 0;
  if (g.R % 64) return 0;
  if (g.R && (!aligned16(g.ul) || !aligned16(g.vl))) return 0;
  if (g.mode == GEMM_DX && Ng % 64) return 0;
  if (g.mode == GEMM_DX && g.R && Ng % 8) return 0;
  if (g.wfmt == W_NF4) {
    if (!aligned16(g.codes) || !aligned16(g.absmax)) return 0;
  } else {
    const int ldw = g.ldw ? g.ldw : g.Kw;
    if (ldw % 8 || !aligned16(g.w)) return 0;
    if (g.mode == GEMM_DX && Ng % 8) return 0;
  }
  if (g.epi == EPI_16 ? (g.ldo % 8) : (g.ldo % 4)) return 0;
  if (g.epi == EPI_F32_ADD && (g.ld_add % 4 || !aligned16(g.add_src))) return 0;
  if (!aligned16(g.out)) return 0;
  return 1;
}

double gemm_flops(const GemmArgs &g) {
  return 2.0 * g.M * (double)g.Ng() * (g.Kg() + g.R);
}

double gemm_bytes(const GemmArgs &g) {
  const double nw = (double)g.Nw * g.Kw;
  const double wb = g.wfmt == W_NF4 ? nw * 0.5 + nw / 64.0 * 4.0 : nw * 2.0;
  const double out_b = g.epi == EPI_16 ? 2.0 : 4.0;
  double b = wb + 2.0 * g.M * g.Kg() + out_b * g.M * (double)g.Ng();
  if (g.epi == EPI_F32_ADD || g.epi == EPI_F32_ACC) b += 4.0 * g.M * (double)g.Ng();
  b += 2.0 * g.R * ((double)g.M + g.Ng());
  return b;
}

void gemm_force_fallback(int on) { g_force_fallback = on; }

int gemm_launch(const GemmArgs &g, cudaStream_t st) {
  if (g.M == 0) return 0;
  if (g.M < 0 || g.Nw <= 0 || g.Kw <= 0 || !g.a || !g.out)
    return set_error(SOUP_EINVAL, "gemm: bad shape or null pointer");
  if (g.wfmt == W_NF4 && (!g.codes || !g.absmax)) return set_error(SOUP_EINVAL, "gemm: NF4 weight missing");
  if (g.wfmt == W_BF16 && !g.w) return set_error(SOUP_EINVAL, "gemm: bf16 weight missing");
  if (g.R && (!g.ul || !g.vl || g.R % 64)) return set_error(SOUP_EINVAL, "gemm: bad LoRA extension");
  if ((g.epi == EPI_F32_ADD) && !g.add_src) return set_error(SOUP_EINVAL, "gemm: residual missing");

  if (!gemm_uses_tc(g)) {
    FbParams p;
    p.cb = nf4_codebook_param();
    p.f16 = g.op_f16;
    p.mode = g.mode; p.M = g.M; p.Ng = g.Ng(); p.Kg = g.Kg(); p.wfmt = g.wfmt;
    p.Nw = g.Nw; p.Kw = g.Kw; p.ldw = g.ldw ? g.ldw : g.Kw; p.lda = g.lda; p.R = g.R;
    p.epi = g.epi; p.ldo = g.ldo; p.ld_add = g.ld_add; p.a = g.a; p.codes = g.codes;
    p.absmax = g.absmax; p.w = g.w; p.ul = g.ul; p.vl = g.vl; p.out = g.out;
    p.add_src = g.add_src;
    dim3 grid((p.Ng + 63) / 64, (g.M + 63) / 64);
    fallback_gemm_kernel<<<grid, 256, 0, st>>>(p);
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(SOUP_ECUDA, "fallback gemm launch: %s", cudaGetErrorString(e));
    return 0;
  }
  int rc = get_encode();
  if (rc) return rc;
  constexpr int BN = 256;
  const int Ng = g.Ng(), Kg = g.Kg();
  CUtensorMap maps[5];
  const CUtensorMapDataType t16 = g.op_f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  rc = make_map(&maps[0], t16, g.a, (uint64_t)Kg, (uint64_t)g.M,
                (uint64_t)g.lda * 2, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B, "activations");
  if (rc) return rc;
  int bmode;
  if (g.wfmt == W_NF4) {
    const uint64_t rowb = (uint64_t)g.Kw / 2, arow = (uint64_t)g.Kw / 64;
    if (g.mode == GEMM_FWD) {
      bmode = B_NF4_K;
      rc = make_map(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, g.codes, rowb, (uint64_t)g.Nw, rowb,
                    32, BN, CU_TENSOR_MAP_SWIZZLE_NONE, "codes");
      if (!rc) rc = make_map(&maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, g.absmax, arow,
                             (uint64_t)g.Nw, arow * 4, 4, BN, CU_TENSOR_MAP_SWIZZLE_NONE, "absmax");
    } else {
      bmode = B_NF4_MN;
      rc = make_map(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, g.codes, rowb, (uint64_t)g.Nw, rowb,
                    BN / 2, BK, CU_TENSOR_MAP_SWIZZLE_128B, "codes");
      if (!rc) rc = make_map(&maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, g.absmax, arow,
                             (uint64_t)g.Nw, arow * 4, BN / 64, BK, CU_TENSOR_MAP_SWIZZLE_NONE,
                             "absmax");
    }
  } else {
    const uint64_t ldw = g.ldw ? g.ldw : g.Kw;
    if (g.mode == GEMM_FWD) {
      bmode = B_BF16_K;
      rc = make_map(&maps[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.w, (uint64_t)g.Kw,
                    (uint64_t)g.Nw, ldw * 2, 64, BN, CU_TENSOR_MAP_SWIZZLE_128B, "weights");
    } else {
      bmode = B_BF16_MN;
      rc = make_map(&maps[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.w, (uint64_t)g.Kw,
                    (uint64_t)g.Nw, ldw * 2, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B, "weights");
    }
    maps[2] = maps[1];
  }
  if (rc) return rc;
  if (g.R) {
    rc = make_map(&maps[3], t16, g.ul, (uint64_t)g.R, (uint64_t)g.M,
                  (uint64_t)g.R * 2, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B, "lora ul");
    if (rc) return rc;
    if (g.mode == GEMM_FWD)
      rc = make_map(&maps[4], t16, g.vl, (uint64_t)g.R, (uint64_t)Ng,
                    (uint64_t)g.R * 2, 64, BN, CU_TENSOR_MAP_SWIZZLE_128B, "lora vl");
    else
      rc = make_map(&maps[4], t16, g.vl, (uint64_t)Ng, (uint64_t)g.R,
                    (uint64_t)Ng * 2, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B, "lora vl");
    if (rc) return rc;
  } else {
    maps[3] = maps[0];
    maps[4] = maps[0];
  }
  switch (bmode) {
    case B_NF4_K: return launch_tc_op<BN, B_NF4_K>(g, maps, st);
    case B_NF4_MN: return launch_tc_op<BN, B_NF4_MN>(g, maps, st);
    case B_BF16_K: return launch_tc_op<BN, B_BF16_K>(g, maps, st);
    default: return launch_tc_op<BN, B_BF16_MN>(g, maps, st);
  }
}

}  // namespace soup
