// Device-side helpers shared by the sm_103a kernels: bf16 packing, mbarriers with bounded
// waits, TMA tiled loads, and the tcgen05 (5th-generation tensor core) instructions, all as
// inline PTX.  Every spin-wait here gives up after a wall-clock budget and raises a flag
// that the host reads, so a logic error cannot hang the device.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#define SOUP_DEV __device__ __forceinline__

// Error flags written by kernels into a device int (bitwise OR).
// RANGE: a value stored as an IEEE-half operand was NaN or beyond +-65504.
enum : int { SOUP_KERR_WAIT_TIMEOUT = 1, SOUP_KERR_BAD_ARG = 2, SOUP_KERR_RANGE = 4 };

// ~0.2 s at 2 GHz: far beyond any legitimate wait in these kernels (the longest, a CTA's
// whole main loop before its epilogue, is well under a millisecond).
#define SOUP_WAIT_CYCLES (400000000ll)

namespace soupk {

SOUP_DEV uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

SOUP_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
SOUP_DEV float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
SOUP_DEV float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
SOUP_DEV float bf16_to_f(uint16_t v) { return __uint_as_float(((uint32_t)v) << 16); }
SOUP_DEV uint16_t f_to_bf16(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t *>(&b);
}

// IEEE half helpers (the forward path's tensor-core operand format).
SOUP_DEV uint32_t pack_h2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
SOUP_DEV float h16_to_f(uint16_t v) { return __half2float(__ushort_as_half(v)); }
SOUP_DEV uint16_t f_to_h16(float f) { return __half_as_ushort(__float2half_rn(f)); }

// 2^x on the special-function unit (PTX ex2.approx.ftz.f32): a relative error of a few ulp,
// far below the 16-bit rounding of the probabilities it produces; 2^-inf = +0.
SOUP_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// True when v does not survive a store as IEEE half: NaN, or |v| >= 65520 (which rounds to
// infinity).  Kernels that store the forward's half operands OR SOUP_KERR_RANGE into their
// error flag when any value fails; the compare is one instruction, the atomic runs only then.
SOUP_DEV bool half_out_of_range(float v) { return !(fabsf(v) < 65520.f); }
SOUP_DEV void flag_range(bool bad, int *err) {
  if (bad && err) atomicOr(err, SOUP_KERR_RANGE);
}

// 16-bit operand format chosen at compile time: F16 = IEEE half, else bf16.
template <bool F16>
SOUP_DEV float ld16(uint16_t v) { return F16 ? h16_to_f(v) : bf16_to_f(v); }
template <bool F16>
SOUP_DEV uint16_t st16(float f) { return F16 ? f_to_h16(f) : f_to_bf16(f); }
template <bool F16>
SOUP_DEV uint32_t pack16x2(float lo, float hi) { return F16 ? pack_h2(lo, hi) : pack_bf16x2(lo, hi); }
template <bool F16>
SOUP_DEV float lo16(uint32_t v) { return ld16<F16>((uint16_t)(v & 0xffffu)); }
template <bool F16>
SOUP_DEV float hi16(uint32_t v) { return ld16<F16>((uint16_t)(v >> 16)); }

SOUP_DEV uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm volatile("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// ------------------------------------------------------------------ mbarrier
SOUP_DEV void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
SOUP_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
SOUP_DEV void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

SOUP_DEV void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
SOUP_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
SOUP_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: returns false (and sets *err) if the phase did not complete within `limit`
// cycles, or if another role already gave up (*abort != 0).
SOUP_DEV bool mbar_wait(uint64_t *bar, uint32_t parity, int *err, volatile int *abort,
                        long long limit = SOUP_WAIT_CYCLES) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort) return false;
      if (clock64() - t0 > limit) {
        *abort = 1;
        if (err) atomicOr(err, SOUP_KERR_WAIT_TIMEOUT);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------ TMA
SOUP_DEV void tma_prefetch_desc(const CUtensorMap *m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
// 2-D tiled load: c0 is the innermost coordinate (elements), c1 the row.
SOUP_DEV void tma_load_2d(void *smem_dst, const CUtensorMap *m, int c0, int c1, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// 3-D tiled load: c0 innermost (elements), c1 row, c2 outermost (e.g. the sequence of a batch).
SOUP_DEV void tma_load_3d(void *smem_dst, const CUtensorMap *m, int c0, int c1, int c2, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ tcgen05
SOUP_DEV void tc_alloc(uint32_t *smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_slot)),
               "r"(ncols)
               : "memory");
}
SOUP_DEV void tc_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
SOUP_DEV void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
SOUP_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
SOUP_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, f32 accumulate (kind::f16).
SOUP_DEV void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on an mbarrier once every previously issued tcgen05.mma of this thread completes.
SOUP_DEV void tc_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// Load 32 consecutive f32 columns of this warp's 32 TMEM lanes (one lane per thread).
SOUP_DEV void tc_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// Load 8 consecutive f32 columns of this warp's 32 TMEM lanes (one lane per thread).
SOUP_DEV void tc_ld_32x32b_x8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
SOUP_DEV void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Store 32 consecutive f32 columns of this warp's 32 TMEM lanes (one lane per thread).
SOUP_DEV void tc_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
SOUP_DEV void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Offset of 16-byte chunk c of row r inside a 128-byte-swizzled tile (rows of 128 bytes,
// 8-row atoms of 1024 bytes): the layout a SWIZZLE_128B TMA copy writes into a 1024-byte
// aligned destination and the tensor core reads through smem_desc.
SOUP_DEV uint32_t sw128(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Shared-memory matrix descriptor (tcgen05): start address, leading/stride byte offsets,
// fixed version field 1 at bit 46, swizzle mode in bits 61-63 (2 = 128-byte swizzle).
SOUP_DEV uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// Instruction descriptor for kind::f16, f32 D, M x N tile; A and B both f16 (f16 = 1) or
// both bf16.  b_mn_major: B operand stored with its N (output) dimension contiguous.
__host__ __device__ constexpr uint32_t idesc_16(int M, int N, int a_mn_major, int b_mn_major,
                                                int f16) {
  return (1u << 4)                                // D format: f32
         | ((uint32_t)(f16 ? 0 : 1) << 7)         // A format: f16 (0) or bf16 (1)
         | ((uint32_t)(f16 ? 0 : 1) << 10)        // B format: same as A
         | ((uint32_t)a_mn_major << 15)  // A major-ness
         | ((uint32_t)b_mn_major << 16)  // B major-ness
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// ------------------------------------------------------------------ mma.sync (warp level)
// D (16x8, f32) += A (16x16, row) * B (16x8, col); F16: half operands, else bf16.
template <bool F16>
SOUP_DEV void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if (F16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ programmatic dependent launch
// A kernel launched with launch_pdl may start while the previous kernel on its stream is still
// running; it must call pdl_wait() before it touches anything that kernel writes (the wait
// returns once that kernel has completed and its writes are visible).  pdl_trigger() lets the
// next kernel be scheduled early.
SOUP_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
SOUP_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace soupk

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
