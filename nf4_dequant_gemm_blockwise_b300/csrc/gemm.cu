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
// Tensor-core kernel (tcgen05, one CTA per 128 x BN output tile, 576 threads):
//   warp 16      TMA producer: activation tile (128 x 64, 128-byte swizzle), the raw 4-bit
//                codes and float absmax of the weight tile (or a bf16 weight tile)
//   warps 0..15  two groups of 8 worker warps taking alternate k-tiles: dequantise codes into
//                the swizzled 16-bit layout the tensor core reads (K-major for the forward,
//                MN-major for dX); afterwards all 16 run the epilogue from TMEM
//   warp 17      allocates TMEM; one lane issues tcgen05.mma (M=128, N=BN, K=16) x 4 per
//                k-tile and commits each stage back to the producer and the workers
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
constexpr int DQ_WARPS = 8;            // warps per worker group (one row-block per thread)
constexpr int NGROUPS = 2;             // worker groups take alternate k-tiles
constexpr int WORKERS = DQ_WARPS * NGROUPS;
constexpr int THREADS = (WORKERS + 2) * 32;
enum BMode { B_NF4_K = 0, B_NF4_MN = 1, B_BF16_K = 2, B_BF16_MN = 3 };

template <int BN, int BMODE, bool F16, int MT>
struct TcCfg {
  static constexpr bool NF4 = (BMODE == B_NF4_K || BMODE == B_NF4_MN);
  // bf16 weights feeding a half-precision GEMM are converted in shared memory, in place
  static constexpr bool CONV = !NF4 && F16;
  static constexpr bool PRODUCE = NF4 || CONV;  // the worker warps touch the B tile
  static constexpr bool MN = (BMODE == B_NF4_MN || BMODE == B_BF16_MN);
  // Two rings.  The load ring (NL stages) receives the activation tile and, for NF4, the raw
  // codes; the B ring (NB stages) holds the 16-bit weight operand the tensor core reads
  // (dequantised by the worker warps, or loaded directly for bf16 weights).  The float block
  // scales are read by the workers straight from global memory (L1-cached, one k-tile ahead).
  // MT m-tiles of 128 rows per CTA share every B tile (MT accumulators of BN TMEM columns)
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int RAW_BYTES = NF4 ? BN * 32 : 0;
  static constexpr int LSTAGE = MT * A_BYTES + RAW_BYTES;
  // Both ring depths are multiples of the number of worker groups: the groups take alternate
  // k-tiles, so every stage then belongs to one group, which waits on each of its phases in
  // turn.  (With an odd depth a group could meet a stage two phases on and its parity wait
  // would pass on the stale phase.)
  static constexpr int NL = 4;
  static constexpr int NB = MT == 1 ? 4 : 2;
  static_assert(NL % NGROUPS == 0 && NB % NGROUPS == 0, "ring depths must split between groups");
  static constexpr int SMEM = NL * LSTAGE + NB * B_BYTES + 1024 + 1024;
  static_assert(SMEM <= 232448, "over the 227 KB shared-memory limit per CTA");
  static constexpr int TMEM_COLS = MT * BN;
  // expected TMA bytes per main / LoRA-extension k-tile (block scales are read by the workers)
  static constexpr uint32_t TX_MAIN = MT * A_BYTES + (NF4 ? BN * 32 : B_BYTES);
  static constexpr uint32_t TX_EXT = MT * A_BYTES + B_BYTES;
};

struct TcParams {
  Codebook cb;
  const float *absmax;  // NF4 block scales of W [Nw, Kw]: absmax[row * kblocks + col / 64]
  int kblocks, Nw;
  int M, Ng, n_main, n_ext;
  int splits, per_split;  // split-K: blockIdx.z takes k-tiles [z * per_split, ...); >1 -> partials
  float *part;            // split-K partial tiles [splits, M, Ng] (float)
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
    // selectors of the eight codes of this word (a byte holds even code << 4 | odd code):
    // the low three bits pick a byte of a register pair, bit 3 picks the pair (+4); byte
    // permutes read the low 16 bits of a selector, so the upper half is shifted down
    const uint32_t x7 = x & 0x77777777u;
    const uint32_t pk = ((x >> 1) & 0x44444444u) | 0x32103210u;
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t s7 = h ? x7 >> 16 : x7;
      const uint32_t pick = h ? pk >> 16 : pk;
      const uint32_t lo = prmt(prmt(LO[0], LO[1], s7), prmt(LO[2], LO[3], s7), pick);
      const uint32_t hi = prmt(prmt(HI[0], HI[1], s7), prmt(HI[2], HI[3], s7), pick);
      o[2 * h] = prmt(lo, hi, 0x4051);      // (even, odd) code of byte 0 -> 16x2
      o[2 * h + 1] = prmt(lo, hi, 0x6273);  // byte 1
    }
    out[w] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

template <int BN, int BMODE, int EPI, bool F16, int MT>
__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_b0,
                   const __grid_constant__ CUtensorMap map_b1,
                   const __grid_constant__ CUtensorMap map_ul,
                   const __grid_constant__ CUtensorMap map_vl, const TcParams p) {
  using C = TcCfg<BN, BMODE, F16, MT>;
  constexpr int NL = C::NL, NB = C::NB;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw_base + 1023u) & ~1023u) - raw_base);
  uint8_t *lring = smem;                                   // NL x LSTAGE
  uint8_t *bring = smem + NL * C::LSTAGE;                  // NB x B_BYTES
  uint64_t *bar = reinterpret_cast<uint64_t *>(bring + NB * C::B_BYTES);
  uint64_t *lfull = bar;              // load stage landed (TMA)
  uint64_t *lempty = bar + NL;        // MMAs done with the load stage
  uint64_t *bready = bar + 2 * NL;    // B stage written (dequantised / converted)
  uint64_t *bempty = bar + 2 * NL + NB;  // MMAs done with the B stage
  uint64_t *accf = bar + 2 * NL + 2 * NB;  // accumulator complete
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accf + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  pdl_trigger();  // a dependent split-K reduction may be scheduled now; it waits for this grid
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // m-tiles vary fastest in the launch order, so the CTAs that share a weight tile run
  // together and the tile is read from DRAM once (the others hit L2)
  const int n0 = blockIdx.y * BN;
  const int m0 = blockIdx.x * BM * MT;
  // this split's k-tiles, renumbered from 0: main tiles [kb, ke), then the LoRA extension
  // tiles on the last split only
  const int z = blockIdx.z;
  const int kb = z * p.per_split;
  const int ke = min(p.n_main, kb + p.per_split);
  const int n_my_main = max(0, ke - kb);
  const int n_total = n_my_main + (z == p.splits - 1 ? p.n_ext : 0);

  auto A_s = [&](int s) { return lring + s * C::LSTAGE; };
  auto R_s = [&](int s) { return lring + s * C::LSTAGE + MT * C::A_BYTES; };
  auto B_s = [&](int s) { return bring + s * C::B_BYTES; };

  // the codebook goes through shared memory: indexing the parameter block with a run-time
  // index would force a local copy of it
  __shared__ float s_cb[16];
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < 16; ++i) s_cb[i] = p.cb.v[i];  // static indices: read in place
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int s = 0; s < NL; ++s) {
      mbar_init(&lfull[s], 1);
      mbar_init(&lempty[s], 1);
    }
    for (int s = 0; s < NB; ++s) {
      mbar_init(&bready[s], DQ_WARPS);
      mbar_init(&bempty[s], 1);
    }
    mbar_init(accf, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == WORKERS + 1) {
    tc_alloc(tmem_slot, C::TMEM_COLS);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == WORKERS) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&map_a);
      tma_prefetch_desc(&map_b0);
      int issued = 0;
      for (int kt = 0; kt < n_total; ++kt) {
        const int sl = kt % NL, sb = kt % NB;
        if (kt >= NL && !mbar_wait(&lempty[sl], ((kt / NL) - 1) & 1, p.err, abort_flag)) break;
        const bool b_direct = !C::NF4 || kt >= n_my_main;  // B arrives by TMA into the B ring
        if (b_direct && kt >= NB && !mbar_wait(&bempty[sb], ((kt / NB) - 1) & 1, p.err, abort_flag)) break;
        if (kt < n_my_main) {
          const int g = kb + kt;  // global k-tile
          mbar_arrive_expect_tx(&lfull[sl], C::TX_MAIN);
#pragma unroll
          for (int i = 0; i < MT; ++i)
            tma_load_2d(A_s(sl) + i * C::A_BYTES, &map_a, g * BK, m0 + i * BM, &lfull[sl]);
          if (BMODE == B_NF4_K) {
            tma_load_2d(R_s(sl), &map_b0, g * (BK / 2), n0, &lfull[sl]);
          } else if (BMODE == B_NF4_MN) {
            tma_load_2d(R_s(sl), &map_b0, n0 / 2, g * BK, &lfull[sl]);
          } else if (BMODE == B_BF16_K) {
            tma_load_2d(B_s(sb), &map_b0, g * BK, n0, &lfull[sl]);
          } else {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_2d(B_s(sb) + c * 8192, &map_b0, n0 + 64 * c, g * BK, &lfull[sl]);
          }
        } else {
          const int e = kt - n_my_main;
          mbar_arrive_expect_tx(&lfull[sl], C::TX_EXT);
#pragma unroll
          for (int i = 0; i < MT; ++i)
            tma_load_2d(A_s(sl) + i * C::A_BYTES, &map_ul, e * BK, m0 + i * BM, &lfull[sl]);
          if (!C::MN) {
            tma_load_2d(B_s(sb), &map_vl, e * BK, n0, &lfull[sl]);
          } else {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_2d(B_s(sb) + c * 8192, &map_vl, n0 + 64 * c, e * BK, &lfull[sl]);
          }
        }
        ++issued;
      }
      // never leave the CTA with copies still landing in its shared memory
      for (int kt = (issued > NL ? issued - NL : 0); kt < issued; ++kt) {
        volatile int no_abort = 0;
        mbar_wait(&lfull[kt % NL], (kt / NL) & 1, p.err, &no_abort);
      }
    }
  } else if (warp == WORKERS + 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_16(BM, BN, 0, C::MN ? 1 : 0, F16 ? 1 : 0);
      for (int kt = 0; kt < n_total; ++kt) {
        const int sl = kt % NL, sb = kt % NB;
        // produce modes: the workers waited for the load stage before marking the B stage
        // ready; direct modes: the load-stage barrier also counts the B tile's bytes
        const bool ok = C::PRODUCE ? mbar_wait(&bready[sb], (kt / NB) & 1, p.err, abort_flag)
                                   : mbar_wait(&lfull[sl], (kt / NL) & 1, p.err, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(A_s(sl));
        const uint32_t b_addr = smem_u32(B_s(sb));
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t bd = C::MN ? smem_desc(b_addr + kk * 2048, 8192, 1024)
                                    : smem_desc(b_addr + kk * 32, 16, 1024);
#pragma unroll
          for (int i = 0; i < MT; ++i) {
            const uint64_t ad = smem_desc(a_addr + i * C::A_BYTES + kk * 32, 16, 1024);
            tc_mma_bf16(tmem + i * BN, ad, bd, idesc, (kt | kk) != 0);
          }
        }
        tc_commit(&lempty[sl]);
        tc_commit(&bempty[sb]);
      }
      tc_commit(accf);
      volatile int no_abort = 0;
      mbar_wait(accf, 0, p.err, &no_abort);  // every MMA retired before TMEM is freed
    }
  } else {
    // ---------------------------------------------------------------- worker warps
    const int grp = warp / DQ_WARPS;
    const int t = threadIdx.x - grp * DQ_WARPS * 32;  // 0 .. 255 within the group
    float cbr[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) cbr[i] = s_cb[i];
    // this thread's block scale for k-tile kt: forward = (row n0 + t, block kt); dX = (row
    // kt * 64 + (t & 63), block n0 / 64 + (t >> 6)); rows past the weight read as 0
    auto absmax_of = [&](int kt) -> float {
      if (!C::NF4 || kt >= n_my_main) return 0.f;
      const int g = kb + kt;
      const int row = (BMODE == B_NF4_K) ? n0 + t : g * BK + (t & 63);
      const int col = (BMODE == B_NF4_K) ? g : n0 / 64 + (t >> 6);
      if (row >= p.Nw || col >= p.kblocks) return 0.f;
      return __ldg(p.absmax + (size_t)row * p.kblocks + col);
    };
    float a_next = absmax_of(grp);
    for (int kt = grp; C::PRODUCE && kt < n_total; kt += NGROUPS) {
      const int sl = kt % NL, sb = kt % NB;
      const float a = a_next;
      a_next = absmax_of(kt + NGROUPS);  // in flight while this tile is waited for and dequantised
      if (!mbar_wait(&lfull[sl], (kt / NL) & 1, p.err, abort_flag)) break;
      if (C::NF4 && kt < n_my_main) {
        // dequantise into registers first, then wait for the B stage (the MMAs of this
        // group's previous tile in it) and store
        uint8_t *Bs = B_s(sb);
        const uint8_t *Rs = R_s(sl);
        uint4 o[8];
        if (BMODE == B_NF4_K) {
          // BN == 256 rows: one row-block per thread
          const int n = t;
          const uint4 c0 = *reinterpret_cast<const uint4 *>(Rs + n * 32);
          const uint4 c1 = *reinterpret_cast<const uint4 *>(Rs + n * 32 + 16);
          const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          dq_block64<F16>(cbr, cw, a, o);
        } else {
          // 64 reduction rows x (BN / 64) column segments: one row-block per thread
          const int n = t & 63, seg = t >> 6;
          const uint4 c0 = *reinterpret_cast<const uint4 *>(Rs + sw128(n, 2 * seg));
          const uint4 c1 = *reinterpret_cast<const uint4 *>(Rs + sw128(n, 2 * seg + 1));
          const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          dq_block64<F16>(cbr, cw, a, o);
        }
        if (kt >= NB && !mbar_wait(&bempty[sb], ((kt / NB) - 1) & 1, p.err, abort_flag)) break;
        if (BMODE == B_NF4_K) {
#pragma unroll
          for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(Bs + sw128(t, c)) = o[c];
        } else {
          const int n = t & 63, seg = t >> 6;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4 *>(Bs + seg * 8192 + sw128(n, c)) = o[c];
        }
        fence_async_smem();
      } else if (C::CONV && kt < n_my_main) {
        // bf16 -> half, element by element; the byte layout (and so the swizzle) is unchanged
        uint4 *Bs = reinterpret_cast<uint4 *>(B_s(sb));
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
      __syncwarp();
      if (lane == 0) mbar_arrive(&bready[sb]);
    }
    // ---------------------------------------------------------------- epilogue
    volatile int no_abort = 0;
    const bool ok = !*abort_flag && mbar_wait(accf, 0, p.err, &no_abort) && !*abort_flag;
    tc_fence_after();
    if (ok) {
      // Each warp owns 32 rows (its TMEM lane quarter) x COLS columns of every m-tile.  The
      // block goes through shared memory — the rings are idle now: every MMA has retired and
      // every TMA copy has landed — so that the global stores cover whole row segments: lane l
      // takes columns 2l, 2l + 1 of one row per store, 128 or 256 contiguous bytes per
      // instruction instead of 32 scattered rows.
      const int q = warp & 3;
      constexpr int COLS = BN / (WORKERS / 4);  // columns per warp
      constexpr int LDSW = COLS + 4;            // staged row stride in floats (conflict-free)
      static_assert(WORKERS * 32 * LDSW * 4 <= NL * C::LSTAGE + NB * C::B_BYTES, "staging space");
      float *stage = reinterpret_cast<float *>(smem) + (size_t)warp * 32 * LDSW;
      const int c0 = (warp >> 2) * COLS;         // first column of this warp inside the tile
      const int ncol = n0 + c0 + 2 * lane;       // this lane's first output column
      const bool pair_ok = ((p.splits > 1 ? p.Ng : p.ldo) & 1) == 0 &&
                           (EPI != EPI_F32_ADD || p.splits > 1 || (p.ld_add & 1) == 0);
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int cc = 0; cc < COLS / 32; ++cc) {
          uint32_t r[32];
          tc_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + mt * BN + c0 + cc * 32, r);
          tc_wait_ld();
          float *row = stage + lane * LDSW + cc * 32;
#pragma unroll
          for (int v = 0; v < 8; ++v)
            *reinterpret_cast<float4 *>(row + 4 * v) =
                make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                            __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
        }
        __syncwarp();
        bool bad = false;
        const int mrow0 = m0 + mt * BM + q * 32;
        for (int rr = 0; rr < 32; ++rr) {
          const int m = mrow0 + rr;
          if (m >= p.M) break;
          const float2 v = *reinterpret_cast<const float2 *>(stage + rr * LDSW + 2 * lane);
          const bool in0 = ncol < p.Ng, in1 = ncol + 1 < p.Ng;
          if (!in0) continue;
          if (p.splits > 1) {
            float *o = p.part + ((size_t)z * p.M + m) * p.Ng + ncol;
            if (in1 && pair_ok) *reinterpret_cast<float2 *>(o) = v;
            else {
              o[0] = v.x;
              if (in1) o[1] = v.y;
            }
          } else if (EPI == EPI_16) {
            if (F16) bad |= half_out_of_range(v.x) || (in1 && half_out_of_range(v.y));
            uint16_t *o = reinterpret_cast<uint16_t *>(p.out) + (size_t)m * p.ldo + ncol;
            if (in1 && pair_ok) *reinterpret_cast<uint32_t *>(o) = pack16x2<F16>(v.x, v.y);
            else {
              o[0] = st16<F16>(v.x);
              if (in1) o[1] = st16<F16>(v.y);
            }
          } else {
            float *o = reinterpret_cast<float *>(p.out) + (size_t)m * p.ldo + ncol;
            float2 w = v;
            if (EPI == EPI_F32_ADD || EPI == EPI_F32_ACC) {
              const float *src = EPI == EPI_F32_ADD ? p.add_src + (size_t)m * p.ld_add + ncol : o;
              if (in1 && pair_ok) {
                const float2 b = *reinterpret_cast<const float2 *>(src);
                w.x = b.x + w.x;
                w.y = b.y + w.y;
              } else {
                w.x = src[0] + w.x;
                if (in1) w.y = src[1] + w.y;
              }
            }
            if (in1 && pair_ok) *reinterpret_cast<float2 *>(o) = w;
            else {
              o[0] = w.x;
              if (in1) o[1] = w.y;
            }
          }
        }
        if (F16 && EPI == EPI_16) flag_range(bad, p.err);
        __syncwarp();  // the staged block is read before the next m-tile overwrites it
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == WORKERS + 1) {
    __syncwarp();
    tc_fence_after();
    tc_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------------------
// Tiled fallback for shapes the tensor-core kernel does not take (blocks that straddle rows,
// unaligned strides).  Same operand definition, float accumulation, 64x64 tiles.
struct FbParams {
  Codebook cb;
  int f16;
  int *err;
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
        if (p.f16) flag_range(half_out_of_range(v), p.err);
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
// Split-K reduction: out = epilogue(sum over splits, in split order) — deterministic.
struct RedParams {
  const float *part;
  int splits, M, Ng, epi, f16, ldo, ld_add;
  void *out;
  const float *add_src;
  int *err;
};
// Sum of the split partial planes in split order, then the epilogue.  Launched as a
// programmatic dependent of the GEMM: waits for it before reading the partials.  V = 4: four
// consecutive columns per item (Ng, ldo, ld_add multiples of 4, 16-byte aligned buffers).
template <int V>
__global__ void splitk_reduce_kernel(const RedParams p) {
  pdl_wait();
  const int nv = p.Ng / V;
  const int64_t total = (int64_t)p.M * nv;
  const int64_t plane = (int64_t)p.M * p.Ng;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int m = (int)(idx / nv), n = (int)(idx - (int64_t)m * nv) * V;
    const size_t e = (size_t)m * p.Ng + n;
    float v[V];
    if constexpr (V == 4) {
      // every split's load in flight before the first add (splits <= 4); added in split order
      float4 b[4];
#pragma unroll
      for (int z = 0; z < 4; ++z)
        b[z] = z < p.splits ? *reinterpret_cast<const float4 *>(p.part + (size_t)z * plane + e)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      float4 a = b[0];
#pragma unroll
      for (int z = 1; z < 4; ++z)
        if (z < p.splits) {
          a.x += b[z].x; a.y += b[z].y; a.z += b[z].z; a.w += b[z].w;
        }
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else {
      v[0] = p.part[e];
      for (int z = 1; z < p.splits; ++z) v[0] += p.part[(size_t)z * plane + e];
    }
    if (p.epi == EPI_16) {
      uint16_t *o = reinterpret_cast<uint16_t *>(p.out) + (size_t)m * p.ldo + n;
      if (p.f16) {
        bool bad = false;
#pragma unroll
        for (int j = 0; j < V; ++j) bad |= half_out_of_range(v[j]);
        flag_range(bad, p.err);
      }
      if constexpr (V == 4) {  // one 8-byte store (n, ldo multiples of 4, 16-byte aligned base)
        *reinterpret_cast<uint2 *>(o) = p.f16 ? make_uint2(pack_h2(v[0], v[1]), pack_h2(v[2], v[3]))
                                              : make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
      } else {
        o[0] = p.f16 ? f_to_h16(v[0]) : f_to_bf16(v[0]);
      }
    } else {
      float *o = reinterpret_cast<float *>(p.out) + (size_t)m * p.ldo + n;
      if constexpr (V == 4) {
        float4 r = make_float4(v[0], v[1], v[2], v[3]);
        if (p.epi != EPI_F32) {
          const float4 c = p.epi == EPI_F32_ADD
                               ? *reinterpret_cast<const float4 *>(p.add_src + (size_t)m * p.ld_add + n)
                               : *reinterpret_cast<const float4 *>(o);
          r = make_float4(c.x + v[0], c.y + v[1], c.z + v[2], c.w + v[3]);
        }
        *reinterpret_cast<float4 *>(o) = r;
      } else {
        if (p.epi == EPI_F32) o[0] = v[0];
        else if (p.epi == EPI_F32_ADD) o[0] = p.add_src[(size_t)m * p.ld_add + n] + v[0];
        else o[0] = o[0] + v[0];
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

template <int BN, int BMODE, int EPI, bool F16, int MT>
int launch_tc(const GemmArgs &g, const CUtensorMap *maps, cudaStream_t st) {
  using C = TcCfg<BN, BMODE, F16, MT>;
  static bool attr_done = false;  // per instantiation; set under g_mu
  auto kern = tc_gemm_kernel<BN, BMODE, EPI, F16, MT>;
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
  p.absmax = g.absmax;
  p.kblocks = g.Kw / 64;
  p.Nw = g.Nw;
  p.M = g.M;
  p.Ng = g.Ng();
  p.n_main = (g.Kg() + BK - 1) / BK;
  p.n_ext = g.R / BK;
  p.splits = g.splits > 1 ? g.splits : 1;
  p.per_split = (p.n_main + p.splits - 1) / p.splits;
  p.part = g.part;
  p.out = g.out;
  p.ldo = g.ldo;
  p.add_src = g.add_src;
  p.ld_add = g.ld_add;
  p.err = g.err;
  dim3 grid((g.M + BM * MT - 1) / (BM * MT), (p.Ng + BN - 1) / BN, p.splits);
  kern<<<grid, THREADS, C::SMEM, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
  count_launches(1);
  if (p.splits > 1) {
    RedParams rp;
    rp.part = g.part; rp.splits = p.splits; rp.M = g.M; rp.Ng = p.Ng; rp.epi = g.epi;
    rp.f16 = g.op_f16; rp.ldo = g.ldo; rp.ld_add = g.ld_add; rp.out = g.out; rp.add_src = g.add_src;
    rp.err = g.err;
    const bool vec = p.Ng % 4 == 0 && g.ldo % 4 == 0 && (g.epi != EPI_F32_ADD || g.ld_add % 4 == 0) &&
                     (reinterpret_cast<uintptr_t>(g.part) & 15) == 0 && p.splits <= 4;
    const int64_t n = (int64_t)g.M * p.Ng / (vec ? 4 : 1);
    const int blocks = (int)std::min<int64_t>((n + 255) / 256, 148 * 16);
    cudaError_t le = vec ? launch_pdl(splitk_reduce_kernel<4>, dim3(blocks), dim3(256), 0, st, rp)
                         : launch_pdl(splitk_reduce_kernel<1>, dim3(blocks), dim3(256), 0, st, rp);
    if (le != cudaSuccess) return set_error(SOUP_ECUDA, "split-K reduce launch: %s", cudaGetErrorString(le));
    count_launches(1);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(SOUP_ECUDA, "tc_gemm launch: %s", cudaGetErrorString(e));
  return 0;
}

template <int BN, int BMODE, bool F16, int MT>
int launch_tc_epi(const GemmArgs &g, const CUtensorMap *maps, cudaStream_t st) {
  switch (g.epi) {
    case EPI_16: return launch_tc<BN, BMODE, EPI_16, F16, MT>(g, maps, st);
    case EPI_F32: return launch_tc<BN, BMODE, EPI_F32, F16, MT>(g, maps, st);
    case EPI_F32_ADD: return launch_tc<BN, BMODE, EPI_F32_ADD, F16, MT>(g, maps, st);
    default: return launch_tc<BN, BMODE, EPI_F32_ACC, F16, MT>(g, maps, st);
  }
}
template <int BN, int BMODE>
int launch_tc_op(const GemmArgs &g, const CUtensorMap *maps, cudaStream_t st) {
  if (g.mtiles == 2)
    return g.op_f16 ? launch_tc_epi<BN, BMODE, true, 2>(g, maps, st)
                    : launch_tc_epi<BN, BMODE, false, 2>(g, maps, st);
  return g.op_f16 ? launch_tc_epi<BN, BMODE, true, 1>(g, maps, st)
                  : launch_tc_epi<BN, BMODE, false, 1>(g, maps, st);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

int tmap_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
            uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw,
            const char *what) {
  SOUP_TRY(get_encode());
  return make_map(m, dt, base, inner, outer, row_bytes, box_inner, box_outer, sw, what);
}

int tmap_3d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t d0, uint64_t d1,
            uint64_t d2, uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1,
            CUtensorMapSwizzle sw, const char *what) {
  SOUP_TRY(get_encode());
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1, stride2};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, dt, 3, const_cast<void *>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(SOUP_EINVAL, "tensor map for %s rejected (CUresult %d)", what, (int)r);
  return 0;
}

// Tiling of one call: m-tiles per CTA (1 or 2) and split-K factor (1..4), minimising a model
// of waves x k-tiles per CTA x time per k-tile, plus the cost of writing and re-reading the
// float partial planes.  Two m-tiles halve the dequantisation per flop: an NF4 k-tile costs
// max(512 x MT tensor cycles, ~900 cycles of byte-permute work for the 256 x 64 B tile);
// bf16 weights have no dequantisation.  Split-K needs the caller's partial buffer.
struct Tiling {
  int mt, s;
};
Tiling choose_tiling(const GemmArgs &g, int bn) {
  const int64_t ntile = (g.Ng() + bn - 1) / bn;
  const int kt = (g.Kg() + 63) / 64;
  const bool nf4 = g.wfmt == W_NF4;
  const bool can_split = g.part && g.part_floats > 0 && g.splits_allowed;
  const double cyc_per_s = 1.9e9, bw = 6.0e12;  // partial traffic (mostly L2-resident), bytes / s
  Tiling best{1, 1};
  double best_t = 1e300;
  for (int mt = 1; mt <= 2; ++mt) {
    if (mt == 2 && g.M <= 128) break;
    const double per_ktile = nf4 ? std::max(512.0 * mt, 900.0) : 512.0 * mt;
    const int64_t tiles = (int64_t)((g.M + 128 * mt - 1) / (128 * mt)) * ntile;
    for (int s = 1; s <= 4; ++s) {
      if (s > 1 && (!can_split || kt / s < 4 || (double)s * g.M * g.Ng() > (double)g.part_floats)) break;
      const int64_t waves = (tiles * s + 147) / 148;
      const double t = (double)waves * ((kt + s - 1) / s) * per_ktile +
                       (s > 1 ? 2.0 * s * g.M * (double)g.Ng() * 4.0 / bw * cyc_per_s : 0.0);
      if (t < best_t * 0.97) {  // a clear gain only: fewer CTAs, fewer partial planes first
        best_t = t;
        best = {mt, s};
      }
    }
  }
  return best;
}

int choose_splits(const GemmArgs &g, int bn) { return choose_tiling(g, bn).s; }
int choose_mtiles(const GemmArgs &g, int bn) { return choose_tiling(g, bn).mt; }

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

  if (!g_force_fallback && gemv_eligible(g)) return gemv_launch(g, st);
  if (!gemm_uses_tc(g)) {
    FbParams p;
    p.cb = nf4_codebook_param();
    p.f16 = g.op_f16;
    p.err = g.err;
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
  GemmArgs g2 = g;
  const Tiling tl = choose_tiling(g, BN);
  g2.mtiles = tl.mt;
  g2.splits = tl.s;
  return gemm_launch_tc(g2, st);
}

int gemm_launch_tc(const GemmArgs &g, cudaStream_t st) {
  int rc = 0;
  constexpr int BN = 256;
  const int Ng = g.Ng(), Kg = g.Kg();
  CUtensorMap maps[5];
  const CUtensorMapDataType t16 = g.op_f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  rc = make_map(&maps[0], t16, g.a, (uint64_t)Kg, (uint64_t)g.M,
                (uint64_t)g.lda * 2, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B, "activations");
  if (rc) return rc;
  int bmode;
  maps[2] = maps[0];
  if (g.wfmt == W_NF4) {
    const uint64_t rowb = (uint64_t)g.Kw / 2;
    if (g.mode == GEMM_FWD) {
      bmode = B_NF4_K;
      rc = make_map(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, g.codes, rowb, (uint64_t)g.Nw, rowb,
                    32, BN, CU_TENSOR_MAP_SWIZZLE_NONE, "codes");
    } else {
      bmode = B_NF4_MN;
      rc = make_map(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, g.codes, rowb, (uint64_t)g.Nw, rowb,
                    BN / 2, BK, CU_TENSOR_MAP_SWIZZLE_128B, "codes");
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
