// The LoRA down-projection u = x A^T of every fused GEMM group (forward), and its backward
// counterpart du = s dY B, each in one launch.
//
// What is computed ("Layer streaming: fine-tune a model that does not fit in your card",
// "Honest scope": plain LoRA, y = x W^T + s (x A^T) B^T): for the fused group's segments p
// (q|k|v, gate|up, or a single projection), with r the rank and s = alpha / r,
//   DOWN  u[m, p r + j]  = sum_k x[m, k] A_p[j, k]                  (all segments share x)
//   DU    du[m, p r + j] = s sum_n dY[m, off_p + n] B_p[n, j]        (segment p's columns)
// written as float [M, nseg r] and as a 16-bit copy scaled by s, [M, Rpad] zero-padded, that
// the GEMM's LoRA extension tiles read.
//
// Layout of the work: one CTA per (64-token tile, cluster rank, job); a job is the whole DOWN
// product, or one segment of the DU product.  A job's reduction range is cut into CL equal
// slices, one per rank of a thread-block cluster (CL a power of two up to 16).  Each CTA streams its
// slice through a six-stage cp.async ring (32 reduction steps per stage; the 8 warps split the
// steps of a stage by parity, each then holding a partial tile) and multiplies on the
// tensor cores as TF32 mma.sync (the 16-bit x and dY are exact in TF32; A and B are rounded to
// TF32, nearest with ties away, when they are read).  The CTAs of a cluster leave their partial
// tiles in shared memory and, after a cluster barrier, each sums a CL-th of the rows over the
// ranks in rank order through distributed shared memory: a fixed order, no partial buffers in
// global memory, no second kernel.
#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "util.h"

namespace soup {
namespace {
using namespace soupk;
namespace cg = cooperative_groups;

constexpr int ROWS = 64;         // tokens per CTA
constexpr int THREADS = 256;     // 8 warps: warp w takes rows 16 (w & 3) .. and k-steps of parity w >> 2
constexpr int KC = 32;           // reduction steps per stage
constexpr int NST = 6;           // stages in flight
constexpr int CL_CAP = 16;       // CTAs per cluster at most (16 where the device schedules it)
constexpr int XS_LD = 40;        // 16-bit elements per staged token row (80 bytes: conflict-free)
constexpr int XS_BYTES = ROWS * XS_LD * 2;
constexpr int WD_LD = 40;        // DOWN: floats per staged A row (160 bytes: conflict-free pairs)
constexpr int WS_FLOATS = 2560;  // DOWN: [64 outputs][40]; DU: [32 steps][r + 8], r <= 64
constexpr int STAGE = XS_BYTES + WS_FLOATS * 4;
constexpr int RED_LD = 68;       // float row stride of a partial tile
constexpr int SMEM = NST * STAGE + 128;
static_assert(2 * ROWS * RED_LD * 4 <= NST * STAGE, "both partial tiles fit in the ring");

struct SkJob {
  int k0, k1;            // reduction range: columns of X (DOWN: [0, K); DU: the segment's)
  int o0, no;            // fused outputs [o0, o0 + no), no a multiple of 8, <= 64
  const float *w[MAX_SEG];  // DOWN: A_p [r, K] of each segment; DU: w[0] = B_p [n_p, r]
};
struct SkArgs {
  const uint16_t *X;
  int ldx, M, r, nout, Rpad, njobs, CL;
  float s;
  SkJob job[MAX_SEG];
  float *out_f32;
  uint16_t *out16;
  int *err;
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
// 16-byte asynchronous copy global -> shared; `valid` false writes zeros (no bytes are read).
SOUP_DEV void cp16(void *dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
SOUP_DEV void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
SOUP_DEV void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Inside each group of 8 reduction steps, thread quad q holds steps 2q and 2q + 1 where the
// MMA's fragment layout names steps q and q + 4: the same relabelling on both operands, so the
// product is unchanged and each operand pair is one 32- or 64-bit shared load.
template <bool DU, bool XF16, bool OF16>
__global__ void __launch_bounds__(THREADS) lora_skinny_kernel(const SkArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int t = threadIdx.x, w = t >> 5, lane = t & 31, g = lane >> 2, q = lane & 3;
  const int rg = w & 3, par = w >> 2;
  const int m0 = blockIdx.x * ROWS;
  const int rank = (int)cluster.block_rank();
  const SkJob &J = a.job[blockIdx.z];
  const int len = J.k1 - J.k0;
  const int slice = ((len + a.CL - 1) / a.CL + KC - 1) / KC * KC;
  const int kb = J.k0 + min(len, rank * slice), ke = J.k0 + min(len, (rank + 1) * slice);
  const int nchunks = (ke - kb + KC - 1) / KC;
  const int NT = J.no / 8;
  const int wld = DU ? a.r + 8 : WD_LD;  // float stride of the staged W rows

  auto xs_of = [&](int st) { return reinterpret_cast<uint16_t *>(smem + st * STAGE); };
  auto ws_of = [&](int st) { return reinterpret_cast<float *>(smem + st * STAGE + XS_BYTES); };

  // this thread's copies, fixed for every stage but for the reduction offset
  const int xr = t >> 2, xc = (t & 3) * 8;  // X: token row, first step
  const bool x_row_ok = m0 + xr < a.M;
  const uint16_t *x_src = a.X + (size_t)(x_row_ok ? m0 + xr : 0) * a.ldx + xc;
  const float *w_src[2] = {nullptr, nullptr};
  int w_dst[2] = {-1, -1}, w_k[2] = {0, 0};
  if (!DU) {  // W[o][k] = A_seg[j][k] for o = seg r + j: 8 copies per output row
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int i = t + THREADS * it, o = i >> 3, c4 = (i & 7) * 4;
      if (o < J.no) {
        w_src[it] = J.w[o / a.r] + (size_t)(o % a.r) * len + c4;
        w_dst[it] = o * WD_LD + c4;
        w_k[it] = c4;
      }
    }
  } else {  // W[k][j] = B_p[k - off_p][j]: r / 4 copies per reduction step
    const int per = a.r / 4;
    if (t < KC * per) {
      const int kk = t / per, c4 = (t % per) * 4;
      w_src[0] = J.w[0] + (size_t)kk * a.r + c4;
      w_dst[0] = kk * wld + c4;
      w_k[0] = kk;
    }
  }

  auto issue = [&](int c) {
    const int st = c % NST, k0 = kb + c * KC;
    uint16_t *xs = xs_of(st);
    float *ws = ws_of(st);
    {
      const bool ok = x_row_ok && k0 + xc < ke;
      cp16(xs + xr * XS_LD + xc, ok ? x_src + k0 : a.X, ok);
    }
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      if (w_dst[it] < 0) continue;
      const bool ok = k0 + w_k[it] < ke;
      // DOWN: A rows are read at column k0; DU: B rows at step k0 - off_p
      const float *src = DU ? w_src[it] + (size_t)(k0 - J.k0) * a.r : w_src[it] + k0;
      cp16(ws + w_dst[it], ok ? src : J.w[0], ok);
    }
  };

  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
  for (int c = 0; c < NST - 1; ++c) {
    if (c < nchunks) issue(c);
    cp_commit();
  }
  for (int c = 0; c < nchunks; ++c) {
    cp_wait<NST - 2>();
    __syncthreads();  // chunk c landed for every thread; chunk c - 1 is no longer read
    if (c + NST - 1 < nchunks) issue(c + NST - 1);
    cp_commit();
    const uint16_t *xs = xs_of(c % NST);
    const float *ws = ws_of(c % NST);
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const int k8 = (2 * ks + par) * 8;
      const uint16_t *xp = xs + (16 * rg + g) * XS_LD + k8 + 2 * q;
      const uint32_t lo = *reinterpret_cast<const uint32_t *>(xp);
      const uint32_t hi = *reinterpret_cast<const uint32_t *>(xp + 8 * XS_LD);
      const uint32_t af[4] = {__float_as_uint(lo16<XF16>(lo)), __float_as_uint(lo16<XF16>(hi)),
                              __float_as_uint(hi16<XF16>(lo)), __float_as_uint(hi16<XF16>(hi))};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        if (nt >= NT) break;
        const int o = 8 * nt + g;
        float b0, b1;
        if (DU) {
          b0 = ws[(k8 + 2 * q) * wld + o];
          b1 = ws[(k8 + 2 * q + 1) * wld + o];
        } else {
          const float2 bb = *reinterpret_cast<const float2 *>(ws + o * WD_LD + k8 + 2 * q);
          b0 = bb.x;
          b1 = bb.y;
        }
        mma_tf32(acc[nt], af, to_tf32(b0), to_tf32(b1));
      }
    }
  }
  cp_wait<0>();
  __syncthreads();  // the ring is idle: it now holds the two partial tiles (k-step parities)

  float *red = reinterpret_cast<float *>(smem) + par * ROWS * RED_LD;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    if (nt >= NT) break;
    const int row = 16 * rg + g, o = 8 * nt + 2 * q;
    red[row * RED_LD + o] = acc[nt][0];
    red[row * RED_LD + o + 1] = acc[nt][1];
    red[(row + 8) * RED_LD + o] = acc[nt][2];
    red[(row + 8) * RED_LD + o + 1] = acc[nt][3];
  }
  cluster.sync();  // every rank's partial tiles are in its shared memory
  {
    const int CL = a.CL, per = ROWS / CL;
    const float *red0 = reinterpret_cast<const float *>(smem);
    bool bad = false;
    for (int i = t; i < per * J.no; i += THREADS) {
      const int row = rank * per + i / J.no, o = i % J.no;
      const int m = m0 + row;
      if (m >= a.M) continue;
      // ranks in order; within a rank, parity 0 then parity 1.  Every remote load is issued
      // before the first add, so the distributed-shared-memory latency is paid once.
      float p0[CL_CAP], p1[CL_CAP];
#pragma unroll
      for (int c = 0; c < CL_CAP; ++c) {
        const float *pc = cluster.map_shared_rank(red0, c < CL ? c : 0);
        p0[c] = c < CL ? pc[row * RED_LD + o] : 0.f;
        p1[c] = c < CL ? pc[(ROWS + row) * RED_LD + o] : 0.f;
      }
      float v = 0.f;
#pragma unroll
      for (int c = 0; c < CL_CAP; ++c)
        if (c < CL) v += p0[c] + p1[c];
      const float sv = a.s * v;
      a.out_f32[(size_t)m * a.nout + J.o0 + o] = DU ? sv : v;
      if (OF16) bad |= half_out_of_range(sv);
      a.out16[(size_t)m * a.Rpad + J.o0 + o] = st16<OF16>(sv);
    }
    if (blockIdx.z == 0) {  // the 16-bit copy's zero padding
      const int padw = a.Rpad - a.nout;
      for (int i = t; i < per * padw; i += THREADS) {
        const int m = m0 + rank * per + i / padw;
        if (m < a.M) a.out16[(size_t)m * a.Rpad + a.nout + i % padw] = 0;
      }
    }
    if (OF16) flag_range(bad, a.err);
  }
  cluster.sync();  // no CTA leaves while another still reads its shared memory
}

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

template <bool DU, bool XF16, bool OF16>
int launch_skinny(const SkArgs &a, int mtiles, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(mtiles, a.CL, a.njobs);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = a.CL;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, lora_skinny_kernel<DU, XF16, OF16>, a);
  if (e != cudaSuccess) return set_error(SOUP_ECUDA, "LoRA projection launch: %s", cudaGetErrorString(e));
  count_launches(1);
  return 0;
}

// Largest cluster the device schedules for these kernels (16 where it can, else 8), set up
// once per device: the shared-memory and cluster-size attributes of every instantiation.
int cluster_cap() {
  static std::atomic<int> cap[MAX_DEVICES];
  int v = 0;
  cudaError_t e = per_device_once(cap, &v, [](int, int *out) {
    void (*ks[8])(SkArgs) = {lora_skinny_kernel<false, false, false>, lora_skinny_kernel<false, false, true>,
                             lora_skinny_kernel<false, true, false>,  lora_skinny_kernel<false, true, true>,
                             lora_skinny_kernel<true, false, false>,  lora_skinny_kernel<true, false, true>,
                             lora_skinny_kernel<true, true, false>,   lora_skinny_kernel<true, true, true>};
    bool big = true;
    for (auto k : ks) {
      cudaError_t r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
      if (r != cudaSuccess) return r;
      if (cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) big = false;
    }
    cudaGetLastError();  // a refused non-portable size is not an error here
    if (big) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(1, CL_CAP, 1);
      cfg.blockDim = dim3(THREADS);
      cfg.dynamicSmemBytes = SMEM;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 1;
      at[0].val.clusterDim.y = CL_CAP;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, ks[0], &cfg) != cudaSuccess || n < 1) big = false;
      cudaGetLastError();
    }
    *out = big ? CL_CAP : 8;
    return cudaSuccess;
  });
  if (e != cudaSuccess) {
    set_error(SOUP_ECUDA, "LoRA projection setup: %s", cudaGetErrorString(e));
    return -1;
  }
  return v;
}

// CTAs per cluster: enough for about 1.5 CTAs per SM over the grid, while every slice keeps at
// least 4 stages.
int pick_cl(int longest, int ctas_per_rank, int cap) {
  int cl = 1;
  while (cl < cap && ctas_per_rank * cl < 222 && longest / (2 * cl) >= 4 * KC) cl *= 2;
  return cl;
}
}  // namespace

int lora_skinny(bool du, const uint16_t *X, int ldx, int M, int K, const LoraSeg &L, float *out_f32,
                uint16_t *out16, bool x_f16, bool o_f16, int *err, cudaStream_t st) {
  if (M <= 0) return 0;
  const int nout = L.nseg * L.r;
  if (L.nseg < 1 || L.r < 8 || L.r % 8 || nout > 64 || ldx % 8 || !al16(X) || !al16(out_f32) ||
      !al16(out16))
    return 1;  // not this kernel's shape: the caller takes the two-kernel path
  SkArgs a{};
  a.X = X;
  a.ldx = ldx;
  a.M = M;
  a.r = L.r;
  a.nout = nout;
  a.Rpad = L.Rpad();
  a.s = L.s;
  a.out_f32 = out_f32;
  a.out16 = out16;
  a.err = err;
  int longest = 0;
  if (!du) {
    if (K % 8) return 1;
    a.njobs = 1;
    SkJob &J = a.job[0];
    J.k0 = 0;
    J.k1 = K;
    J.o0 = 0;
    J.no = nout;
    for (int p = 0; p < L.nseg; ++p) {
      if (!al16(L.A[p])) return 1;
      J.w[p] = L.A[p];
    }
    longest = K;
  } else {
    a.njobs = L.nseg;
    for (int p = 0; p < L.nseg; ++p) {
      if (L.off[p] % 8 || L.n[p] % 8 || L.n[p] <= 0 || !al16(L.B[p])) return 1;
      SkJob &J = a.job[p];
      J.k0 = L.off[p];
      J.k1 = L.off[p] + L.n[p];
      J.o0 = p * L.r;
      J.no = L.r;
      J.w[0] = L.B[p];
      longest = std::max(longest, L.n[p]);
    }
  }
  const int cap = cluster_cap();
  if (cap < 0) return SOUP_ECUDA;
  const int mtiles = (M + ROWS - 1) / ROWS;
  a.CL = pick_cl(longest, mtiles * a.njobs, cap);
  if (!du) {
    if (x_f16) return o_f16 ? launch_skinny<false, true, true>(a, mtiles, st) : launch_skinny<false, true, false>(a, mtiles, st);
    return o_f16 ? launch_skinny<false, false, true>(a, mtiles, st) : launch_skinny<false, false, false>(a, mtiles, st);
  }
  if (x_f16) return o_f16 ? launch_skinny<true, true, true>(a, mtiles, st) : launch_skinny<true, true, false>(a, mtiles, st);
  return o_f16 ? launch_skinny<true, false, true>(a, mtiles, st) : launch_skinny<true, false, false>(a, mtiles, st);
}

}  // namespace soup
