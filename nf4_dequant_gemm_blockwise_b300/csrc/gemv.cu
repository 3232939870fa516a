// Small-M NF4 dequant GEMMs: decode-sized token counts (1 <= M <= 16), where the projection
// is bound by reading the 4-bit weight once from HBM.
//
// What is computed is the same as the tensor-core path ("Layer streaming: fine-tune a model
// that does not fit in your card", "How it works"):
//   forward  y  = x deq(W)^T + s (x A^T) B^T        (x half, y half or float)
//   backward dx = dY deq(W) + s (dY B) A            (dY bf16, dx float)
// with deq(W)[n, k] = c[code] * absmax[n, k / 64] and the 64-element blocks along the rows of
// W [N, K].  The rounding differs from the tensor-core path: the codebook value c is the 16-bit
// operand and the block scale is applied in float (forward: to the block's partial dot
// product; dX: to the gradient operand), and the LoRA term is added in float.
//
// Design (sm_103a, one weight read):
// * weight-stationary mma.sync m16n8k16: the dequantised weight is the 16-row A operand taken
//   straight from registers, the M <= 16 tokens are the 8-column B operand (one or two
//   column tiles), so no dequantised tile is ever written to shared memory;
// * dequantisation is one shared-memory load per code byte: a 256-entry table maps a byte
//   (two codes) to the pair of 16-bit codebook values, replicated once per lane (32 KB) so
//   that every lane reads its own bank;
// * the reduction index inside each 16-wide MMA step is permuted so that every lane's
//   fragment is a whole byte of codes, and the activation / gradient fragment is loaded with
//   the same permutation (a sum is independent of the order of its terms);
// * stream-K: the (strip, k-block) units are cut into equal contiguous ranges, one per
//   persistent CTA, so every SM streams the same number of weight bytes; a strip cut by a CTA
//   boundary leaves one partial per CTA, summed in CTA order by a fix-up kernel (no atomics,
//   so every launch is bit-reproducible).
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "util.h"

namespace soup {
namespace {
using namespace soupk;

constexpr int GV_THREADS = 256;
constexpr int GV_WARPS = GV_THREADS / 32;
constexpr int LUT_WORDS = 256 * 32;  // 256 byte values x one copy per lane
// One strip's outputs: 64 columns (forward: weight rows; dX: input features) x 16 tokens.
constexpr int VALS = 64 * 16;
// Per-warp result slots in shared memory hold only the token tiles in use: TS = 8 * NT floats
// per column, SLOT = columns * TS per slot, two slots per warp.
template <int SLOT>
struct GvSmem {
  static constexpr int BYTES = GV_WARPS * 2 * SLOT * 4;  // dynamic part (the table is static)
};

struct GvParams {
  const uint16_t *a;  // FWD: x [M, Kw] half; DX: dY [M, Nw] bf16; row stride lda
  int lda, M;
  const uint8_t *codes;
  const float *absmax;
  int Nw, Kw, kblocks;
  long long U;    // work units = strips * per_strip
  int per_strip;  // units per strip
  int sw;         // output columns per strip (64, or 32 for the forward with 9..16 tokens)
  int G;          // CTAs of the main kernel
  float *part;    // [G][2][VALS]: the CTA's first / last strip when a CTA boundary cuts it
  int epi, ldo, ld_add;
  void *out;
  const float *add_src;
  const float *lora_u;
  LoraSeg L;
  Codebook cb;
  int *err;       // device error flags (may be null)
  int wait_prev;  // launched as a dependent of the kernel that writes lora_u: wait before using it
};

SOUP_DEV long long range_begin(long long U, int parts, int i) { return (long long)i * U / parts; }
// The CTA whose range holds unit u.
SOUP_DEV int cta_of(const GvParams &p, long long u) {
  return (int)(((u + 1) * p.G + p.U - 1) / p.U) - 1;
}

// Table lookup: off = (byte << 7) | (lane << 2), the byte offset of this lane's copy of entry
// `byte`.  byte7<I>(w) = byte I of w, shifted left by 7.
SOUP_DEV uint32_t lut_at(const uint32_t *lut, uint32_t off) {
  return *reinterpret_cast<const uint32_t *>(reinterpret_cast<const char *>(lut) + off);
}
template <int I>
SOUP_DEV uint32_t byte7(uint32_t w) {
  if constexpr (I == 0) return (w << 7) & 0x7F80u;
  else return (w >> (8 * I - 7)) & 0x7F80u;
}

template <bool F16>
SOUP_DEV void build_lut(uint32_t *lut, float *s_cb, const Codebook &cb) {
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < 16; ++i) s_cb[i] = cb.v[i];  // static indices: read in place
  }
  __syncthreads();
  // entry e = (first code << 4) | second code -> (c[first], c[second]); first = lower index.
  // Each warp writes a run of entries, four per 16-byte store instruction: each group of eight
  // lanes fills one entry's 128-byte row of lane copies (no bank conflicts)
  const int nw = blockDim.x >> 5, w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int per = 256 / nw;  // 32 (8 warps) or 16 (16 warps)
  for (int j = 0; j < per / 4; ++j) {
    const int e = per * w + 4 * j + (l >> 3);
    const uint32_t v = pack16x2<F16>(s_cb[e >> 4], s_cb[e & 15]);
    reinterpret_cast<uint4 *>(lut + e * 32)[l & 7] = make_uint4(v, v, v, v);
  }
  __syncthreads();
}

SOUP_DEV uint2 ldg_nc_u2(const void *p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}
SOUP_DEV uint32_t ldg_nc_u1(const void *p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Shared memory used by the epilogue once the table is no longer needed (LUT_WORDS floats):
// the LoRA operands of one strip and the token rows of lora_u.
//   FWD: lb[o * r + j] = B_q[row - off_q, j] for the strip's row o (0 outside every segment)
//   DX:  lb[(q * r + j) * 64 + o] = A_q[j, col0 + o]
// followed by lu[m * nout + i] = lora_u[m, i].
template <int MODE>
SOUP_DEV void stage_lora(const GvParams &p, float *stage, int col0) {
  const LoraSeg &L = p.L;
  const int nout = L.nseg * L.r;
  const int nlb = MODE == GEMM_FWD ? p.sw * L.r : nout * 64;
  for (int i = threadIdx.x; i < nlb; i += blockDim.x) {
    float v = 0.f;
    if (MODE == GEMM_FWD) {
      const int o = i / L.r, j = i - o * L.r, n = col0 + o;
      for (int q = 0; q < L.nseg; ++q)
        if (n >= L.off[q] && n < L.off[q] + L.n[q]) v = L.B[q][(size_t)(n - L.off[q]) * L.r + j];
    } else {
      const int qj = i >> 6, o = i & 63, q = qj / L.r, j = qj - q * L.r;
      v = L.A[q][(size_t)j * p.Kw + col0 + o];
    }
    stage[i] = v;
  }
  for (int i = threadIdx.x; i < p.M * nout; i += blockDim.x) stage[nlb + i] = p.lora_u[i];
}
// LoRA term of (token m, strip column o; the strip starts at column col0) from the staged
// operands.
template <int MODE>
SOUP_DEV float lora_term(const GvParams &p, const float *stage, int col0, int m, int o) {
  const LoraSeg &L = p.L;
  const int nout = L.nseg * L.r;
  if (MODE == GEMM_FWD) {
    // the row's own segment (its staged B row is zero if it is in none)
    const int n = col0 + o;
    int q = 0;
    for (int k = 1; k < L.nseg; ++k)
      if (n >= L.off[k] && n < L.off[k] + L.n[k]) q = k;
    const float *lu = stage + p.sw * L.r + m * nout + q * L.r;
    const float *lb = stage + o * L.r;
    float t = 0.f;
    for (int j = 0; j < L.r; ++j) t = fmaf(lu[j], lb[j], t);
    return L.s * t;
  } else {
    const float *lu = stage + nout * 64 + m * nout;
    float v = 0.f;
    for (int i = 0; i < nout; ++i) v = fmaf(lu[i], stage[i * 64 + o], v);
    return v;
  }
}
// The epilogue for output (token m, column col).
template <int MODE>
SOUP_DEV void gv_emit(const GvParams &p, int m, int col, float v) {
  const size_t o = (size_t)m * p.ldo + col;
  switch (p.epi) {
    case EPI_16:
      if (MODE == GEMM_FWD) flag_range(half_out_of_range(v), p.err);
      reinterpret_cast<uint16_t *>(p.out)[o] = MODE == GEMM_FWD ? f_to_h16(v) : f_to_bf16(v);
      break;
    case EPI_F32: reinterpret_cast<float *>(p.out)[o] = v; break;
    case EPI_F32_ADD:
      reinterpret_cast<float *>(p.out)[o] = p.add_src[(size_t)m * p.ld_add + col] + v;
      break;
    default: reinterpret_cast<float *>(p.out)[o] += v; break;
  }
}

// After the warps have parked their strip results in red[warp][slot] (slot 0 = the warp's
// first strip, 1 = its second) and their strip ranges in wr[warp] (relative to the CTA's first
// strip; -1 = empty): add them per strip in warp order, then finish each strip the CTA holds
// whole, or park it in the CTA's partial slot for the fix-up.  Work items are the (column,
// token) pairs with token < M, so every thread has one even for a single token.
template <int MODE, int TS, int SLOT, int W>
SOUP_DEV void cta_finish(const GvParams &p, const float *red, float *stage, const int2 *wr,
                         long long u0, long long u1) {
  const int PS = p.per_strip;
  const int ncols = MODE == GEMM_FWD ? p.Nw : p.Kw;
  const long long cs0 = u0 / PS, cs1 = (u1 - 1) / PS;
  const bool lora = p.lora_u && p.L.nseg > 0;
  for (long long s = cs0; s <= cs1; ++s) {
    const int sl = (int)(s - cs0);
    const bool head = s * PS >= u0;                 // this CTA holds the strip's first unit
    const bool whole = head && (s + 1) * PS <= u1;
    const int slot = sl == 0 ? 0 : 1;
    const int col0 = (int)s * p.sw;
    // the LoRA term is added once per strip: by its only CTA, or into the partial of the CTA
    // that holds its first unit
    if (head && lora) {
      stage_lora<MODE>(p, stage, col0);
      __syncthreads();
    }
    for (int idx = threadIdx.x; idx < p.sw * p.M; idx += blockDim.x) {
      const int o = idx / p.M, tok = idx - o * p.M;
      const int e = o * 16 + tok, col = col0 + o;
      if (col >= ncols) continue;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const int2 r = wr[w];
        if (r.x >= 0 && sl >= r.x && sl <= r.y) v += red[(w * 2 + (sl - r.x)) * SLOT + o * TS + tok];
      }
      if (head && lora) v += lora_term<MODE>(p, stage, col0, tok, o);
      if (whole) gv_emit<MODE>(p, tok, col, v);
      else p.part[((size_t)blockIdx.x * 2 + slot) * VALS + e] = v;
    }
    __syncthreads();
  }
}

// Lane 0 of each warp: its strip range relative to the CTA's first strip (-1: no units).
SOUP_DEV void publish_range(int2 *wr, long long wu0, long long wu1, long long u0, int PS) {
  if ((threadIdx.x & 31) == 0) {
    const long long cs0 = u0 / PS;
    wr[threadIdx.x >> 5] = wu1 > wu0 ? make_int2((int)(wu0 / PS - cs0), (int)((wu1 - 1) / PS - cs0))
                                     : make_int2(-1, -1);
  }
}

// ------------------------------------------------------------------ forward
// Strip = RT 16-row MMA tiles of weight rows (RT = 4, or 2 with two token tiles to stay within
// the register budget), unit = one 64-wide k-block of those rows: a [16 RT rows x 32 bytes]
// tile of codes, brought into shared memory by TMA.  Each of the 16 warps walks its own range
// of units through a private ring of D stages (lane 0 issues the copies, one mbarrier per
// stage), so the bytes in flight are bounded by shared memory, not registers.  Lane (g, t)
// takes bytes [8t, 8t + 8) of rows 16j + g and 16j + g + 8 of the tile; MMA step s uses bytes
// 2s, 2s + 1 of them, i.e. the k values 16t + 4s .. 16t + 4s + 3 of the block, and the
// activation fragment holds the same four k values of token g (and g + 8), loaded once per
// unit for the RT row tiles.  Block scales and activations come through registers, one unit
// ahead.
constexpr int GVT_WARPS = 16;
constexpr int GVT_THREADS = GVT_WARPS * 32;

template <int NT, int RT>
struct FwdCfg {
  static constexpr int TS = 8 * NT, SLOT = 16 * RT * TS;  // result slot: rows x token stride
  static constexpr int UB = 16 * RT * 32;                  // bytes of one unit's code tile
  static constexpr int D = RT == 4 ? 4 : 8;                // ring stages per warp
  static constexpr int LUT_B = LUT_WORDS * 4;
  static constexpr int RED_B = GVT_WARPS * 2 * SLOT * 4;
  static constexpr int RING_B = GVT_WARPS * D * UB;
  static constexpr int BAR_B = GVT_WARPS * D * 8;
  static constexpr int SMEM = 128 + RED_B + RING_B + BAR_B;  // dynamic part (+ alignment)
};

template <int NT, int RT>
struct FwdRegs {
  float s[RT][2];
  uint4 x[NT][2];
};

template <int NT, int RT>
SOUP_DEV void fwd_prefetch(const GvParams &p, FwdRegs<NT, RT> &r, long long strip, int kb, int g,
                           int t) {
  const int n0 = (int)strip * (16 * RT);
  const int tiles = min(RT, (p.Nw - n0) / 16);
  const float *ab = p.absmax + (size_t)(n0 + g) * p.kblocks + kb;
#pragma unroll
  for (int j = 0; j < RT; ++j) {
    if (j < tiles) {  // Nw % 16 == 0: rows n and n + 8 of the tile are both inside
      r.s[j][0] = __ldg(ab + (size_t)(16 * j) * p.kblocks);
      r.s[j][1] = __ldg(ab + (size_t)(16 * j + 8) * p.kblocks);
    } else {
      r.s[j][0] = r.s[j][1] = 0.f;
    }
  }
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const int m = g + 8 * i;
    if (m < p.M) {
      const uint4 *xp = reinterpret_cast<const uint4 *>(p.a + (size_t)m * p.lda + kb * 64 + 16 * t);
      r.x[i][0] = __ldg(xp);
      r.x[i][1] = __ldg(xp + 1);
    } else {
      r.x[i][0] = r.x[i][1] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

template <int NT, int RT>
SOUP_DEV void fwd_compute(const uint32_t *lut, uint32_t lane4, const uint8_t *tile,
                          const FwdRegs<NT, RT> &r, int g, int t, float (&acc)[RT][NT][4]) {
#pragma unroll
  for (int j = 0; j < RT; ++j) {
    const uint2 c0 = *reinterpret_cast<const uint2 *>(tile + (16 * j + g) * 32 + 8 * t);
    const uint2 c1 = *reinterpret_cast<const uint2 *>(tile + (16 * j + g + 8) * 32 + 8 * t);
    float blk[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) blk[i][0] = blk[i][1] = blk[i][2] = blk[i][3] = 0.f;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint32_t w0 = s < 2 ? c0.x : c0.y, w1 = s < 2 ? c1.x : c1.y;
      uint32_t a[4];
      if ((s & 1) == 0) {
        a[0] = lut_at(lut, byte7<0>(w0) | lane4);
        a[1] = lut_at(lut, byte7<0>(w1) | lane4);
        a[2] = lut_at(lut, byte7<1>(w0) | lane4);
        a[3] = lut_at(lut, byte7<1>(w1) | lane4);
      } else {
        a[0] = lut_at(lut, byte7<2>(w0) | lane4);
        a[1] = lut_at(lut, byte7<2>(w1) | lane4);
        a[2] = lut_at(lut, byte7<3>(w0) | lane4);
        a[3] = lut_at(lut, byte7<3>(w1) | lane4);
      }
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const uint4 &xq = r.x[i][s >> 1];
        mma16816<true>(blk[i], a, (s & 1) ? xq.z : xq.x, (s & 1) ? xq.w : xq.y);
      }
    }
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      acc[j][i][0] = fmaf(r.s[j][0], blk[i][0], acc[j][i][0]);
      acc[j][i][1] = fmaf(r.s[j][0], blk[i][1], acc[j][i][1]);
      acc[j][i][2] = fmaf(r.s[j][1], blk[i][2], acc[j][i][2]);
      acc[j][i][3] = fmaf(r.s[j][1], blk[i][3], acc[j][i][3]);
    }
  }
}

template <int NT, int RT>
SOUP_DEV void fwd_park(float *slot, float (&acc)[RT][NT][4], int g, int t) {
  constexpr int TS = 8 * NT;
#pragma unroll
  for (int j = 0; j < RT; ++j)
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const int row = 16 * j + g, tok = 8 * i + 2 * t;
      slot[row * TS + tok] = acc[j][i][0];
      slot[row * TS + tok + 1] = acc[j][i][1];
      slot[(row + 8) * TS + tok] = acc[j][i][2];
      slot[(row + 8) * TS + tok + 1] = acc[j][i][3];
      acc[j][i][0] = acc[j][i][1] = acc[j][i][2] = acc[j][i][3] = 0.f;
    }
}

template <int NT, int RT>
__global__ void __launch_bounds__(GVT_THREADS, 1)
    gemv_fwd_kernel(const __grid_constant__ CUtensorMap cmap, const GvParams p) {
  using C = FwdCfg<NT, RT>;
  constexpr int D = C::D;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  uint8_t *sm = smem_raw + (((raw_base + 127u) & ~127u) - raw_base);  // TMA destinations: 128 B
  // the table is a static array, so every lookup addresses it with an immediate base
  __shared__ __align__(16) uint32_t lut[LUT_WORDS];
  float *red = reinterpret_cast<float *>(sm);
  uint8_t *ring = sm + C::RED_B;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::RED_B + C::RING_B);
  __shared__ float s_cb[16];
  __shared__ int2 s_wr[GVT_WARPS];
  __shared__ int s_abort;
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const uint32_t lane4 = (uint32_t)lane << 2;
  const long long u0 = range_begin(p.U, p.G, blockIdx.x), u1 = range_begin(p.U, p.G, blockIdx.x + 1);
  const long long wu0 = u0 + range_begin(u1 - u0, GVT_WARPS, warp);
  const long long wu1 = u0 + range_begin(u1 - u0, GVT_WARPS, warp + 1);
  const int n = (int)(wu1 - wu0);
  const int PS = p.per_strip;
  uint8_t *myring = ring + warp * D * C::UB;
  uint64_t *mybar = bars + warp * D;
  if (threadIdx.x == 0) s_abort = 0;
  // lane 0 issues the copies: unit (istrip, ikb) next
  long long istrip = wu0 / PS;
  int ikb = (int)(wu0 - istrip * PS);
  int issued = 0;
  if (lane == 0) {
    for (int i = 0; i < D; ++i) mbar_init(&mybar[i], 1);
    fence_mbar_init();
    tma_prefetch_desc(&cmap);
    for (; issued < D && issued < n; ++issued) {
      mbar_arrive_expect_tx(&mybar[issued], C::UB);
      tma_load_2d(myring + issued * C::UB, &cmap, ikb * 32, (int)istrip * (16 * RT), &mybar[issued]);
      if (++ikb == PS) { ikb = 0; ++istrip; }
    }
  }
  __syncwarp();
  long long strip = wu0 / PS;
  int kb = (int)(wu0 - strip * PS);
  const long long first_strip = strip;
  FwdRegs<NT, RT> cur, nxt;
  if (n > 0) fwd_prefetch(p, cur, strip, kb, g, t);
  build_lut<true>(lut, s_cb, p.cb);  // ends with __syncthreads (also publishes s_abort)
  float acc[RT][NT][4];
#pragma unroll
  for (int j = 0; j < RT; ++j)
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[j][i][0] = acc[j][i][1] = acc[j][i][2] = acc[j][i][3] = 0.f;
  float *myred = red + warp * 2 * C::SLOT;
  long long nstrip = strip;
  int nkb = kb;
  int done = 0;
  for (int i = 0; i < n; ++i) {
    if (++nkb == PS) { nkb = 0; ++nstrip; }
    if (i + 1 < n) fwd_prefetch(p, nxt, nstrip, nkb, g, t);
    const int st = i % D;
    const bool ok = mbar_wait(&mybar[st], (i / D) & 1, p.err, &s_abort);
    if (__any_sync(0xffffffffu, !ok)) break;
    if (strip != first_strip && kb == 0) fwd_park<NT, RT>(myred, acc, g, t);  // second strip
    fwd_compute<NT, RT>(lut, lane4, myring + st * C::UB, cur, g, t, acc);
    ++done;
    __syncwarp();  // every lane has consumed the stage before it is refilled
    if (lane == 0 && issued < n) {
      const int s2 = issued % D;
      mbar_arrive_expect_tx(&mybar[s2], C::UB);
      tma_load_2d(myring + s2 * C::UB, &cmap, ikb * 32, (int)istrip * (16 * RT), &mybar[s2]);
      if (++ikb == PS) { ikb = 0; ++istrip; }
      ++issued;
    }
    if (++kb == PS) { kb = 0; ++strip; }
    cur = nxt;
  }
  if (lane == 0) {
    // after a timeout, never leave copies landing in shared memory
    for (int i = done; i < issued; ++i) {
      volatile int no_abort = 0;
      mbar_wait(&mybar[i % D], (i / D) & 1, p.err, &no_abort);
    }
  }
  if (n > 0) {
    const long long last = (wu1 - 1) / PS;
    fwd_park<NT, RT>(myred + (last == first_strip ? 0 : C::SLOT), acc, g, t);
  }
  publish_range(s_wr, wu0, wu1, u0, PS);
  if (p.wait_prev) pdl_wait();
  __syncthreads();
  cta_finish<GEMM_FWD, C::TS, C::SLOT, GVT_WARPS>(p, red, reinterpret_cast<float *>(lut), s_wr, u0, u1);
}

// ------------------------------------------------------------------ dX
// Strip = one 64-wide block kb of the input features, unit = 32 weight rows of that block (two
// 16-row MMA tiles).  In tile h, lane (g, t) holds the 4-byte word at byte 4g of the block in
// rows n = 16h + 4t .. 16h + 4t + 3: MMA q (q = 0..3) takes byte q of each word, i.e. the
// output features 8g + 2q (high nibbles, A row g) and 8g + 2q + 1 (low nibbles, A row g + 8),
// with rows n, n + 1 as reduction columns 2t, 2t + 1 and rows n + 2, n + 3 as 2t + 8, 2t + 9.
// Byte pairs of two rows are merged nibble-wise so that one table entry gives both rows'
// values; the block scales multiply the gradient operand, which is per row.
template <int NT>
struct DxUnit {
  uint32_t w[2][4];
  float s[2][4];
  uint2 d[2][NT];
};

template <int NT>
SOUP_DEV void dx_load(const GvParams &p, DxUnit<NT> &b, int kb, long long rc, int g, int t) {
  const size_t rowb = (size_t)p.Kw / 2;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int n = (int)rc * 32 + 16 * h + 4 * t;
    if (n < p.Nw) {  // Nw % 16 == 0: the whole 16-row tile is inside
      const uint8_t *cp = p.codes + (size_t)n * rowb + kb * 32 + 4 * g;
      const float *ap = p.absmax + (size_t)n * p.kblocks + kb;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b.w[h][j] = ldg_nc_u1(cp + j * rowb);
        b.s[h][j] = __ldg(ap + j * p.kblocks);
      }
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const int m = g + 8 * i;
        b.d[h][i] = m < p.M ? __ldg(reinterpret_cast<const uint2 *>(p.a + (size_t)m * p.lda + n))
                            : make_uint2(0u, 0u);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b.w[h][j] = 0u;
        b.s[h][j] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < NT; ++i) b.d[h][i] = make_uint2(0u, 0u);
    }
  }
}

template <int NT>
SOUP_DEV void dx_compute(const uint32_t *lut, uint32_t lane4, const DxUnit<NT> &b,
                         float (&acc)[NT][4][4]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t b0[NT], b1[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      b0[i] = pack_bf16x2(bf16_lo(b.d[h][i].x) * b.s[h][0], bf16_hi(b.d[h][i].x) * b.s[h][1]);
      b1[i] = pack_bf16x2(bf16_lo(b.d[h][i].y) * b.s[h][2], bf16_hi(b.d[h][i].y) * b.s[h][3]);
    }
    const uint32_t w0 = b.w[h][0], w1 = b.w[h][1], w2 = b.w[h][2], w3 = b.w[h][3];
    // byte q of H01: (high nibble of w0's byte q, high nibble of w1's byte q); L01: low nibbles
    const uint32_t H01 = (w0 & 0xF0F0F0F0u) | ((w1 >> 4) & 0x0F0F0F0Fu);
    const uint32_t L01 = ((w0 << 4) & 0xF0F0F0F0u) | (w1 & 0x0F0F0F0Fu);
    const uint32_t H23 = (w2 & 0xF0F0F0F0u) | ((w3 >> 4) & 0x0F0F0F0Fu);
    const uint32_t L23 = ((w2 << 4) & 0xF0F0F0F0u) | (w3 & 0x0F0F0F0Fu);
    uint32_t a[4];
#define SOUP_DX_Q(Q)                                      \
    a[0] = lut_at(lut, byte7<Q>(H01) | lane4);            \
    a[1] = lut_at(lut, byte7<Q>(L01) | lane4);            \
    a[2] = lut_at(lut, byte7<Q>(H23) | lane4);            \
    a[3] = lut_at(lut, byte7<Q>(L23) | lane4);            \
    _Pragma("unroll") for (int i = 0; i < NT; ++i) mma16816<false>(acc[i][Q], a, b0[i], b1[i]);
    SOUP_DX_Q(0)
    SOUP_DX_Q(1)
    SOUP_DX_Q(2)
    SOUP_DX_Q(3)
#undef SOUP_DX_Q
  }
}

template <int NT>
SOUP_DEV void dx_park(float *slot, float (&acc)[NT][4][4], int g, int t) {
  constexpr int TS = 8 * NT;
#pragma unroll
  for (int i = 0; i < NT; ++i)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int tok = 8 * i + 2 * t, o = 8 * g + 2 * q;
      slot[o * TS + tok] = acc[i][q][0];
      slot[o * TS + tok + 1] = acc[i][q][1];
      slot[(o + 1) * TS + tok] = acc[i][q][2];
      slot[(o + 1) * TS + tok + 1] = acc[i][q][3];
      acc[i][q][0] = acc[i][q][1] = acc[i][q][2] = acc[i][q][3] = 0.f;
    }
}

template <int NT>
__global__ void __launch_bounds__(GV_THREADS, 2) gemv_dx_kernel(const GvParams p) {
  constexpr int TS = 8 * NT, SLOT = 64 * TS;
  extern __shared__ __align__(16) uint32_t gsm[];
  __shared__ __align__(16) uint32_t lut[LUT_WORDS];  // static: immediate base in every lookup
  __shared__ float s_cb[16];
  __shared__ int2 s_wr[GV_WARPS];
  float *red = reinterpret_cast<float *>(gsm);
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const uint32_t lane4 = (uint32_t)lane << 2;
  const long long u0 = range_begin(p.U, p.G, blockIdx.x), u1 = range_begin(p.U, p.G, blockIdx.x + 1);
  const long long wu0 = u0 + range_begin(u1 - u0, GV_WARPS, warp);
  const long long wu1 = u0 + range_begin(u1 - u0, GV_WARPS, warp + 1);
  const int PS = p.per_strip;
  long long strip = wu0 / PS;
  int rc = (int)(wu0 - strip * PS);
  long long nstrip = strip;
  int nrc = rc;
  DxUnit<NT> A, B;
  if (wu0 < wu1) dx_load(p, A, (int)nstrip, nrc, g, t);
  build_lut<false>(lut, s_cb, p.cb);
  float acc[NT][4][4];
#pragma unroll
  for (int i = 0; i < NT; ++i)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[i][q][0] = acc[i][q][1] = acc[i][q][2] = acc[i][q][3] = 0.f;
  float *myred = red + warp * 2 * SLOT;
  const long long first_strip = strip;
  auto advance = [&](long long &s_, int &r_) {
    if (++r_ == PS) { r_ = 0; ++s_; }
  };
  advance(nstrip, nrc);
  for (long long u = wu0; u < wu1; u += 2) {
    if (u + 1 < wu1) { dx_load(p, B, (int)nstrip, nrc, g, t); advance(nstrip, nrc); }
    if (strip != first_strip && rc == 0) dx_park<NT>(myred, acc, g, t);
    dx_compute<NT>(lut, lane4, A, acc);
    advance(strip, rc);
    if (u + 1 >= wu1) break;
    if (u + 2 < wu1) { dx_load(p, A, (int)nstrip, nrc, g, t); advance(nstrip, nrc); }
    if (strip != first_strip && rc == 0) dx_park<NT>(myred, acc, g, t);
    dx_compute<NT>(lut, lane4, B, acc);
    advance(strip, rc);
  }
  if (wu0 < wu1) {
    const long long last = (wu1 - 1) / PS;
    dx_park<NT>(myred + (last == first_strip ? 0 : SLOT), acc, g, t);
  }
  publish_range(s_wr, wu0, wu1, u0, PS);
  if (p.wait_prev) pdl_wait();
  __syncthreads();
  cta_finish<GEMM_DX, TS, SLOT, GV_WARPS>(p, red, reinterpret_cast<float *>(lut), s_wr, u0, u1);
}

// ------------------------------------------------------------------ fix-up
// Strips cut by CTA boundaries: one thread per (boundary, output) adds the CTAs' partials in
// CTA order and stores the result (the partials already hold the LoRA term).  The first
// boundary inside a strip handles it.  Launched as a programmatic dependent of the main
// kernel: waits for it before reading the partials.
template <int MODE>
__global__ void __launch_bounds__(GV_THREADS) gemv_fixup_kernel(const GvParams p) {
  pdl_wait();
  const int per_b = p.sw * p.M;
  const long long idx = (long long)blockIdx.x * GV_THREADS + threadIdx.x;
  if (idx >= (long long)(p.G - 1) * per_b) return;
  const int c = 1 + (int)(idx / per_b), rem = (int)(idx % per_b);
  const int o = rem / p.M, tok = rem - o * p.M;
  const int PS = p.per_strip;
  const long long ub = range_begin(p.U, p.G, c);
  if (ub % PS == 0) return;  // boundary on a strip edge: nothing cut
  const long long s = ub / PS;
  const long long prev = range_begin(p.U, p.G, c - 1);
  if (prev > s * PS) return;  // an earlier boundary inside this strip handles it
  const int col = (int)s * p.sw + o;
  if (col >= (MODE == GEMM_FWD ? p.Nw : p.Kw)) return;
  const int e = o * 16 + tok;
  const int c_hi = cta_of(p, (s + 1) * PS - 1);
  // CTA c - 1 holds the strip's head: slot 0 if the strip is its first one, else slot 1;
  // every later CTA starts inside the strip, so the strip is its first one
  float v = p.part[((size_t)(c - 1) * 2 + (prev == s * PS ? 0 : 1)) * VALS + e];
#pragma unroll 4
  for (int k = c; k <= c_hi; ++k) v += p.part[(size_t)k * 2 * VALS + e];
  gv_emit<MODE>(p, tok, col, v);
}

// ------------------------------------------------------------------ host
int sm_count() {
  static std::atomic<int> sms[MAX_DEVICES];
  int n = 0;
  if (per_device_once(sms, &n, [](int dev, int *v) {
        return cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
      }) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

template <int MODE, int NT, typename K>
int resident_ctas(K kern, int threads, int smem, int *out) {
  static std::atomic<int> cached[MAX_DEVICES];  // per device, per (MODE, NT) instantiation
  cudaError_t e = per_device_once(cached, out, [&](int, int *v) {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (r == cudaSuccess) r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(v, kern, threads, smem);
    return r;
  });
  if (e != cudaSuccess) return set_error(SOUP_ECUDA, "small-M GEMM setup: %s", cudaGetErrorString(e));
  return 0;
}

bool al(const void *p, int b) { return (reinterpret_cast<uintptr_t>(p) % b) == 0; }

template <int MODE, int NT, int RT, int THREADS, int SMEM, typename K, typename... Pre>
int launch_mode(const GemmArgs &g, K kern, cudaStream_t st, const Pre &...pre) {
  constexpr int W = THREADS / 32;
  int per_sm = 0;
  SOUP_TRY((resident_ctas<MODE, NT * 8 + RT>(kern, THREADS, SMEM, &per_sm)));
  const int sms = sm_count();
  if (per_sm < 1 || sms < 1) return set_error(SOUP_ECUDA, "small-M GEMM: no resident CTA");
  GvParams p;
  p.a = g.a;
  p.lda = g.lda;
  p.M = g.M;
  p.codes = g.codes;
  p.absmax = g.absmax;
  p.Nw = g.Nw;
  p.Kw = g.Kw;
  p.kblocks = g.Kw / 64;
  // forward: strips of 16 * RT weight rows x k-blocks; dX: strips of 64 features x 32-row chunks
  p.sw = MODE == GEMM_FWD ? 16 * RT : 64;
  const long long nstrips = MODE == GEMM_FWD ? (g.Nw + p.sw - 1) / p.sw : g.Kw / 64;
  p.per_strip = MODE == GEMM_FWD ? g.Kw / 64 : (g.Nw + 31) / 32;
  p.U = nstrips * p.per_strip;
  long long G = std::min<long long>((long long)per_sm * sms, GV_MAX_CTAS);
  G = std::min<long long>(G, (long long)(g.part_floats / (2 * VALS)));
  // every warp's range must touch at most two strips (its two result slots)
  const long long need = (p.U + (long long)W * p.per_strip - 1) / ((long long)W * p.per_strip) + 1;
  G = std::max(G, need);
  G = std::min<long long>(G, p.U);
  if (G < 1 || (size_t)G * 2 * VALS > g.part_floats)
    return set_error(SOUP_EINVAL, "small-M GEMM: partial buffer too small");
  p.G = (int)G;
  p.part = g.part;
  p.epi = g.epi;
  p.ldo = g.ldo;
  p.ld_add = g.ld_add;
  p.out = g.out;
  p.add_src = g.add_src;
  p.lora_u = g.lora_u;
  p.L = g.lseg;
  p.cb = nf4_codebook_param();
  p.err = g.err;
  // after the LoRA projection that produced lora_u, the weight stream starts at once and the
  // kernel waits for lora_u only before its epilogue
  p.wait_prev = (g.after_lora && g.lora_u && g.lseg.nseg > 0) ? 1 : 0;
  if (p.wait_prev) {
    cudaError_t e = launch_pdl(kern, dim3(p.G), dim3(THREADS), SMEM, st, pre..., p);
    if (e != cudaSuccess) return set_error(SOUP_ECUDA, "small-M GEMM launch: %s", cudaGetErrorString(e));
  } else {
    kern<<<p.G, THREADS, SMEM, st>>>(pre..., p);
  }
  int launches = 1;
  // the fix-up has work only if some CTA boundary cuts a strip
  bool cut = false;
  for (long long c = 1; c < G && !cut; ++c) cut = (c * p.U / G) % p.per_strip != 0;
  if (cut) {
    const long long n = (G - 1) * (long long)p.sw * p.M;
    cudaError_t e = launch_pdl(gemv_fixup_kernel<MODE>, dim3((unsigned)((n + GV_THREADS - 1) / GV_THREADS)),
                               dim3(GV_THREADS), 0, st, p);
    if (e != cudaSuccess) return set_error(SOUP_ECUDA, "small-M fix-up launch: %s", cudaGetErrorString(e));
    ++launches;
  }
  count_launches(launches);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(SOUP_ECUDA, "small-M GEMM launch: %s", cudaGetErrorString(e));
  return 0;
}

template <int NT, int RT>
int launch_fwd(const GemmArgs &g, cudaStream_t st) {
  using C = FwdCfg<NT, RT>;
  CUtensorMap cmap;
  SOUP_TRY(tmap_2d(&cmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.codes, (uint64_t)g.Kw / 2, (uint64_t)g.Nw,
                   (uint64_t)g.Kw / 2, 32, 16 * RT, CU_TENSOR_MAP_SWIZZLE_NONE, "codes (small-M)"));
  return launch_mode<GEMM_FWD, NT, RT, GVT_THREADS, C::SMEM>(g, gemv_fwd_kernel<NT, RT>, st, cmap);
}

}  // namespace

size_t gemv_part_floats(int) { return (size_t)GV_MAX_CTAS * 2 * VALS; }

int gemv_eligible(const GemmArgs &g) {
  if (g.wfmt != W_NF4 || g.M < 1 || g.M > 16) return 0;
  if (g.Nw % 16 || g.Kw % 64) return 0;
  if (g.mode == GEMM_FWD ? !g.op_f16 : g.op_f16) return 0;
  if (g.R && !(g.lora_u && g.lseg.nseg > 0)) return 0;  // the float LoRA operands are needed
  if (g.lseg.nseg > 0 && !g.lora_u) return 0;
  if (!g.part || g.part_floats < 2 * (size_t)VALS) return 0;
  if (!al(g.codes, 16) || !al(g.absmax, 4)) return 0;
  if (g.mode == GEMM_FWD ? (g.lda % 8 || !al(g.a, 16)) : (g.lda % 4 || !al(g.a, 8))) return 0;
  if (g.epi == EPI_F32_ADD && !g.add_src) return 0;
  return 1;
}

int gemv_launch(const GemmArgs &g, cudaStream_t st) {
  if (!gemv_eligible(g)) return set_error(SOUP_EINVAL, "small-M GEMM: arguments not eligible");
  if (g.mode == GEMM_FWD) return g.M <= 8 ? launch_fwd<1, 4>(g, st) : launch_fwd<2, 2>(g, st);
  return g.M <= 8 ? launch_mode<GEMM_DX, 1, 0, GV_THREADS, GvSmem<64 * 8>::BYTES>(g, gemv_dx_kernel<1>, st)
                  : launch_mode<GEMM_DX, 2, 0, GV_THREADS, GvSmem<64 * 16>::BYTES>(g, gemv_dx_kernel<2>, st);
}

}  // namespace soup
