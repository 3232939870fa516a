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
// slices, one per rank of a thread-block cluster (CL a power of two up to 16).  Each CTA streams
// its slice through a six-stage ring of 64 reduction steps: one thread issues the TMA copies of
// the token tile (and, for DOWN, of the A rows), 128-byte swizzled, completing on the stage's
// mbarrier; the B rows of DU come by cp.async.  The 8 warps split a stage's steps by parity and
// multiply on the tensor cores as TF32 mma.sync (the 16-bit x and dY are exact in TF32; A and B
// are rounded to TF32, nearest with ties away, when they are read).  Each CTA adds its two parity
// tiles, and after a cluster barrier each CTA sums a CL-th of the rows over the ranks in rank
// order through distributed shared memory: a fixed order, no partial buffers in global memory,
// no second kernel.
#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "util.h"

namespace soup {
namespace {
using namespace soupk;
namespace cg = cooperative_groups;

constexpr int ROWS = 64;         // tokens per CTA
constexpr int THREADS = 256;     // 8 warps: warp w takes rows 16 (w & 3) .. and k-steps of parity w >> 2
constexpr int KC = 64;           // reduction steps per stage
constexpr int NST = 6;           // stages in flight
constexpr int CL_CAP = 16;       // CTAs per cluster at most (16 where the device schedules it)
constexpr int X_BYTES = ROWS * 128;  // token tile: 64 rows x 64 16-bit steps, 128-byte swizzle
constexpr int RED_LD = 68;       // float row stride of a partial tile
constexpr int RED_BYTES = 2 * ROWS * RED_LD * 4;
// W part of a stage: DOWN two 32-step panels of the no A rows (128-byte swizzle); DU KC rows of
// B (r floats, padded to r + 4: conflict-free column reads); rounded up to 1 KB (the swizzle atom)
__host__ __device__ constexpr int w_bytes(bool du, int no, int r) {
  return ((du ? KC * (r + 4) * 4 : 2 * no * 128) + 1023) / 1024 * 1024;
}
__host__ __device__ constexpr int stage_bytes(bool du, int no, int r) { return X_BYTES + w_bytes(du, no, r); }
constexpr int SMEM_MAX =
    NST * (stage_bytes(false, 64, 64) > stage_bytes(true, 64, 64) ? stage_bytes(false, 64, 64) : stage_bytes(true, 64, 64)) +
    1024 + 128;

struct SkJob {
  int k0, k1;            // reduction range: columns of X (DOWN: [0, K); DU: the segment's)
  int o0, no;            // fused outputs [o0, o0 + no), no a multiple of 8, <= 64
  const float *w[MAX_SEG];  // DOWN: A_p [r, K] of each segment; DU: w[0] = B_p [n_p, r]
};
struct SkArgs {
  int M, r, nout, Rpad, njobs, nseg, CL;
  int stage;             // bytes per ring stage (stage_bytes of the jobs' shape)
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
__global__ void __launch_bounds__(THREADS)
    lora_skinny_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_a0,
                       const __grid_constant__ CUtensorMap map_a1, const __grid_constant__ CUtensorMap map_a2,
                       const SkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((base + 1023u) & ~1023u) - base);
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
  const int wld = a.r + 4;  // DU: float stride of the staged B rows
  const int STAGE = a.stage;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NST * STAGE);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(full + NST);
  auto xs_of = [&](int st) { return smem + st * STAGE; };
  auto ws_of = [&](int st) { return smem + st * STAGE + X_BYTES; };
  if (t == 0) {
    for (int i = 0; i < NST; ++i) mbar_init(&full[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // DU: this thread's copies of B rows (r / 4 of 16 bytes per reduction step)
  const float *w_src[4];
  int w_dst[4], w_k[4];
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int i = t + THREADS * it, per = a.r / 4;
    w_src[it] = nullptr;
    w_dst[it] = -1;
    w_k[it] = 0;
    if (DU && i < KC * per) {
      const int kk = i / per, c4 = (i % per) * 4;
      w_src[it] = J.w[0] + (size_t)kk * a.r + c4;
      w_dst[it] = kk * wld + c4;
      w_k[it] = kk;
    }
  }
  const CUtensorMap *amap[3] = {&map_a0, &map_a1, &map_a2};
  const uint32_t tx = X_BYTES + (DU ? 0 : 2 * J.no * 128);
  auto issue = [&](int c) {
    const int st = c % NST, k0 = kb + c * KC;
    if (t == 0) {
      fence_async_smem();  // the stage's previous contents were read through the generic proxy
      mbar_arrive_expect_tx(&full[st], tx);
      tma_load_2d(xs_of(st), &map_x, k0, m0, &full[st]);
      if (!DU)
        for (int p = 0; p < a.nseg; ++p)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            tma_load_2d(ws_of(st) + hh * J.no * 128 + p * a.r * 128, amap[p], k0 + 32 * hh, 0, &full[st]);
    }
    if (DU) {
      float *ws = reinterpret_cast<float *>(ws_of(st));
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        if (w_dst[it] < 0) continue;
        const bool ok = k0 + w_k[it] < ke;
        cp16(ws + w_dst[it], ok ? w_src[it] + (size_t)(k0 - J.k0) * a.r : J.w[0], ok);
      }
    }
  };

  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
  for (int c = 0; c < NST - 1; ++c) {
    if (c < nchunks) issue(c);
    if (DU) cp_commit();
  }
  for (int c = 0; c < nchunks; ++c) {
    const int st = c % NST;
    if (DU) cp_wait<NST - 2>();
    mbar_wait(&full[st], (c / NST) & 1, a.err, abort_flag);
    __syncthreads();  // chunk c landed for every thread; chunk c - 1 is no longer read
    if (c + NST - 1 < nchunks) issue(c + NST - 1);
    if (DU) cp_commit();
    const uint8_t *xs = xs_of(st);
    const uint8_t *wsb = ws_of(st);
#pragma unroll
    for (int ks = 0; ks < KC / 16; ++ks) {
      const int k8 = (2 * ks + par) * 8;
      // token rows 16 rg + g and + 8 (both have g as their row mod 8); the 128-byte swizzle
      // moves the 16-byte chunk k8 / 8 of a row to chunk (k8 / 8) ^ (row mod 8)
      const uint8_t *xp = xs + (16 * rg + g) * 128 + ((((k8 >> 3) ^ g)) << 4) + 4 * q;
      const uint32_t lo = *reinterpret_cast<const uint32_t *>(xp);
      const uint32_t hi = *reinterpret_cast<const uint32_t *>(xp + 8 * 128);
      const uint32_t af[4] = {__float_as_uint(lo16<XF16>(lo)), __float_as_uint(lo16<XF16>(hi)),
                              __float_as_uint(hi16<XF16>(lo)), __float_as_uint(hi16<XF16>(hi))};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        if (nt >= NT) break;
        const int o = 8 * nt + g;
        float b0, b1;
        if (DU) {
          const float *ws = reinterpret_cast<const float *>(wsb);
          b0 = ws[(k8 + 2 * q) * wld + o];
          b1 = ws[(k8 + 2 * q + 1) * wld + o];
        } else {
          // A row o, steps k8 + 2q, + 1: panel k8 / 32, 16-byte chunk ((k8 % 32) / 4 + q / 2)
          // swizzled with o mod 8 (= g), 8-byte half q % 2
          const int chunk = ((k8 & 31) >> 2) + (q >> 1);
          const float2 bb = *reinterpret_cast<const float2 *>(
              wsb + (k8 >> 5) * J.no * 128 + o * 128 + ((chunk ^ g) << 4) + (q & 1) * 8);
          b0 = bb.x;
          b1 = bb.y;
        }
        mma_tf32(acc[nt], af, to_tf32(b0), to_tf32(b1));
      }
    }
  }
  if (DU) cp_wait<0>();
  __syncthreads();  // every chunk consumed: the ring now holds the two partial tiles
  if (*abort_flag && t == 0) {  // a wait gave up: let every issued copy land before reuse
    volatile int no_abort = 0;
    for (int c = max(0, nchunks - NST); c < nchunks; ++c)
      mbar_wait(&full[c % NST], (c / NST) & 1, a.err, &no_abort);
  }
  __syncthreads();

  float *red = reinterpret_cast<float *>(smem);
  {
    float *mine = red + par * ROWS * RED_LD;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      if (nt >= NT) break;
      const int row = 16 * rg + g, o = 8 * nt + 2 * q;
      mine[row * RED_LD + o] = acc[nt][0];
      mine[row * RED_LD + o + 1] = acc[nt][1];
      mine[(row + 8) * RED_LD + o] = acc[nt][2];
      mine[(row + 8) * RED_LD + o + 1] = acc[nt][3];
    }
  }
  __syncthreads();
  for (int i = t; i < ROWS * J.no; i += THREADS) {  // this rank's tile: parity 0 + parity 1
    const int row = i / J.no, o = i % J.no;
    red[row * RED_LD + o] += red[(ROWS + row) * RED_LD + o];
  }
  cluster.sync();  // every rank's tile is in its shared memory
  {
    // rank `rank` sums rows rank * per .. over the ranks in rank order, four outputs per thread;
    // every remote load is issued before the first add
    const int CL = a.CL, per = ROWS / CL, nq = J.no / 4;
    bool bad = false;
    for (int i = t; i < per * nq; i += THREADS) {
      const int row = rank * per + i / nq, o = (i % nq) * 4;
      const int m = m0 + row;
      if (m >= a.M) continue;
      float4 pv[CL_CAP];
#pragma unroll
      for (int c = 0; c < CL_CAP; ++c) {
        const float *pc = cluster.map_shared_rank(red, c < CL ? c : 0);
        pv[c] = c < CL ? *reinterpret_cast<const float4 *>(pc + row * RED_LD + o) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int c = 0; c < CL_CAP; ++c)
        if (c < CL) {
          v.x += pv[c].x;
          v.y += pv[c].y;
          v.z += pv[c].z;
          v.w += pv[c].w;
        }
      const float4 sv = make_float4(a.s * v.x, a.s * v.y, a.s * v.z, a.s * v.w);
      *reinterpret_cast<float4 *>(a.out_f32 + (size_t)m * a.nout + J.o0 + o) = DU ? sv : v;
      if (OF16)
        bad |= half_out_of_range(sv.x) || half_out_of_range(sv.y) || half_out_of_range(sv.z) ||
               half_out_of_range(sv.w);
      *reinterpret_cast<uint2 *>(a.out16 + (size_t)m * a.Rpad + J.o0 + o) =
          make_uint2(pack16x2<OF16>(sv.x, sv.y), pack16x2<OF16>(sv.z, sv.w));
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
int launch_skinny(const CUtensorMap *maps, const SkArgs &a, int mtiles, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(mtiles, a.CL, a.njobs);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = std::max(NST * a.stage, RED_BYTES) + 1024 + 128;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = a.CL;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, lora_skinny_kernel<DU, XF16, OF16>, maps[0], maps[1], maps[2],
                                     maps[3], a);
  if (e != cudaSuccess) {
    cudaGetLastError();  // not sticky: the caller falls back to the two-kernel path
    return set_error(SOUP_ECUDA, "LoRA projection launch: %s", cudaGetErrorString(e));
  }
  count_launches(1);
  return 0;
}

// Largest cluster the device schedules for these kernels (16 where it can, else 8), set up
// once per device: the shared-memory and cluster-size attributes of every instantiation.
int cluster_cap() {
  static std::atomic<int> cap[MAX_DEVICES];
  int v = 0;
  cudaError_t e = per_device_once(cap, &v, [](int, int *out) {
    using K = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, SkArgs);
    K ks[8] = {lora_skinny_kernel<false, false, false>, lora_skinny_kernel<false, false, true>,
               lora_skinny_kernel<false, true, false>,  lora_skinny_kernel<false, true, true>,
               lora_skinny_kernel<true, false, false>,  lora_skinny_kernel<true, false, true>,
               lora_skinny_kernel<true, true, false>,   lora_skinny_kernel<true, true, true>};
    bool big = true;
    for (auto k : ks) {
      cudaError_t r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
      if (r != cudaSuccess) return r;
      if (cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) big = false;
    }
    cudaGetLastError();  // a refused non-portable size is not an error here
    if (big) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(1, CL_CAP, 1);
      cfg.blockDim = dim3(THREADS);
      cfg.dynamicSmemBytes = SMEM_MAX;
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
// least 2 stages.
int pick_cl(int longest, int ctas_per_rank, int cap) {
  int cl = 1;
  while (cl < cap && ctas_per_rank * cl < 222 && longest / (2 * cl) >= 2 * KC) cl *= 2;
  return cl;
}
}  // namespace

int lora_skinny(bool du, const uint16_t *X, int ldx, int M, int K, const LoraSeg &L, float *out_f32,
                uint16_t *out16, bool x_f16, bool o_f16, int *err, cudaStream_t st) {
  if (M <= 0) return 0;
  const int nout = L.nseg * L.r;
  if (L.nseg < 1 || L.nseg > 3 || L.r < 8 || L.r % 8 || nout > 64 || ldx % 8 || !al16(X) ||
      !al16(out_f32) || !al16(out16))
    return 1;  // not this kernel's shape: the caller takes the two-kernel path
  SkArgs a{};
  a.M = M;
  a.r = L.r;
  a.nout = nout;
  a.Rpad = L.Rpad();
  a.nseg = L.nseg;
  a.s = L.s;
  a.out_f32 = out_f32;
  a.out16 = out16;
  a.err = err;
  int longest = 0, ncols = 0;
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
    longest = ncols = K;
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
      ncols = std::max(ncols, J.k1);
    }
  }
  if (ncols > ldx) return 1;
  // the token tile (64 x 64 16-bit, 128-byte swizzle) and, for DOWN, each segment's A rows in
  // 32-step panels; unused maps repeat the token map
  CUtensorMap maps[4];
  SOUP_TRY(tmap_2d(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT16, X, (uint64_t)ncols, (uint64_t)M,
                   (uint64_t)ldx * 2, KC, ROWS, CU_TENSOR_MAP_SWIZZLE_128B, "LoRA projection input"));
  for (int p = 0; p < 3; ++p) {
    if (!du && p < L.nseg)
      SOUP_TRY(tmap_2d(&maps[1 + p], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, L.A[p], (uint64_t)K, (uint64_t)L.r,
                       (uint64_t)K * 4, 32, L.r, CU_TENSOR_MAP_SWIZZLE_128B, "LoRA A"));
    else
      maps[1 + p] = maps[0];
  }
  a.stage = stage_bytes(du, du ? L.r : nout, L.r);
  const int cap = cluster_cap();
  if (cap < 0) return SOUP_ECUDA;
  const int mtiles = (M + ROWS - 1) / ROWS;
  a.CL = pick_cl(longest, mtiles * a.njobs, cap);
  if (!du) {
    if (x_f16) return o_f16 ? launch_skinny<false, true, true>(maps, a, mtiles, st) : launch_skinny<false, true, false>(maps, a, mtiles, st);
    return o_f16 ? launch_skinny<false, false, true>(maps, a, mtiles, st) : launch_skinny<false, false, false>(maps, a, mtiles, st);
  }
  if (x_f16) return o_f16 ? launch_skinny<true, true, true>(maps, a, mtiles, st) : launch_skinny<true, true, false>(maps, a, mtiles, st);
  return o_f16 ? launch_skinny<true, false, true>(maps, a, mtiles, st) : launch_skinny<true, false, false>(maps, a, mtiles, st);
}

}  // namespace soup
