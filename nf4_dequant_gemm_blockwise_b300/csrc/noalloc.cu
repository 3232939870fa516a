// soup_proj_fwd_noalloc: the single-projection forward (x W^T + s (x A^T) B^T) for callers
// that cannot allocate device memory themselves — for example code embedded in a host
// application that owns the whole device-memory budget and forbids allocations outside it, or
// latency-critical callers that cannot afford cudaMalloc's implicit device synchronisation.
//
// Its working memory (the LoRA down-projection, its 16-bit pack, the packed LoRA B rows, the
// reduction partials and an error flag) lives in one file-scope device array of fixed size,
// reserved on every GPU that loads this library and kept until the process exits.  Nothing
// here calls cudaMalloc, cudaFree or any allocating routine.
//
// Rules for callers:
//   - The first call on a device looks up the array's device address with
//     cudaGetSymbolAddress (once per device, with that device current) and caches it; make
//     that first call before any stream capture on the device.
//   - All calls share the one array and it keeps the previous call's contents.  Calls whose
//     GPU work overlaps (different streams, or different host threads) race on it: order them
//     on one stream or synchronise between them.
//   - A call whose working memory would exceed the array is rejected with SOUP_EINVAL before
//     anything is enqueued.
//   - Kernels OR their error bits (a bounded wait that gave up, a half-precision overflow) into
//     a flag at the start of the array.  The flag is zero when the library loads and is read
//     and cleared only by soup_proj_noalloc_status, so it collects every call's errors since
//     the last read.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "gemm.h"
#include "kernels.h"
#include "soup.h"
#include "util.h"

namespace soup {
namespace {

constexpr size_t kScratchBytes = 16ull << 20;  // 16 MiB per device
static __device__ __align__(256) unsigned char g_proj_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of the static scratch on the current device (looked up once per device).
int scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(SOUP_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return set_error(SOUP_EINVAL, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_proj_scratch);
    if (e != cudaSuccess || !p)
      return set_error(SOUP_ECUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return 0;
}

// The error flag sits at a fixed place (the first 256 bytes) so that soup_proj_noalloc_status
// can find it without knowing the calls' shapes; the working buffers follow it.
constexpr uint64_t kErrOffset = 0;
struct Layout {
  uint64_t u_f32, ul, vl, part, gpart, gpart_floats, total;
};
Layout layout(int M, int N, int K) {
  Layout s;
  uint64_t off = 256;  // past the error flag
  auto take = [&](uint64_t b) {
    const uint64_t o = off;
    off = (off + b + 255) / 256 * 256;
    return o;
  };
  s.u_f32 = take(4ull * M * 64);
  s.ul = take(2ull * M * 64);
  s.vl = take(2ull * N * 64);
  s.part = take(4ull * lora_splits(M, K, nullptr) * M * 64);  // the down-projection's partials
  // small-M path: per-CTA partial strips (no split-K buffer for the tensor-core path)
  s.gpart_floats = M <= 16 ? gemv_part_floats(GEMM_FWD) : 0;
  s.gpart = take(4 * s.gpart_floats);
  s.total = off;
  return s;
}

}  // namespace
}  // namespace soup

using namespace soup;

extern "C" int soup_proj_fwd_noalloc(const uint16_t *x, int M, int N, int K, const uint8_t *codes,
                                     const float *absmax, const uint16_t *w_bf16, const float *A,
                                     const float *B, int r, float s, int x_f16, uint16_t *y,
                                     uintptr_t stream) {
  if (M < 0 || N < 1 || K < 1 || r < 0 || r > 64)
    return set_error(SOUP_EINVAL, "bad shape M=%d N=%d K=%d r=%d", M, N, K, r);
  if (r > 0 && (!A || !B)) return set_error(SOUP_EINVAL, "NULL LoRA pointer with r > 0");
  if (!(codes && absmax) && !w_bf16) return set_error(SOUP_EINVAL, "no weight given");
  if (codes && (int64_t)N * K % 64) return set_error(SOUP_EINVAL, "N*K must be a multiple of 64");
  if (M == 0) return 0;
  if (!x || !y) return set_error(SOUP_EINVAL, "NULL x or y");
  const Layout L = layout(M, N, K);
  if (L.total > kScratchBytes)
    return set_error(SOUP_EINVAL,
                     "soup_proj_fwd_noalloc: M=%d N=%d K=%d needs %llu bytes of working memory; the "
                     "static scratch holds %llu",
                     M, N, K, (unsigned long long)L.total, (unsigned long long)kScratchBytes);
  void *base_v = nullptr;
  SOUP_TRY(scratch_address(&base_v));
  uint8_t *base = static_cast<uint8_t *>(base_v);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool f16 = x_f16 != 0;
  LoraSeg seg;
  seg.nseg = 1;
  seg.r = r;
  seg.s = s;
  seg.off[0] = 0;
  seg.n[0] = N;
  seg.A[0] = A;
  seg.B[0] = B;
  GemmArgs g;
  g.mode = GEMM_FWD;
  g.Nw = N;
  g.Kw = K;
  if (codes) {
    g.wfmt = W_NF4;
    g.codes = codes;
    g.absmax = absmax;
  } else {
    g.wfmt = W_BF16;
    g.w = w_bf16;
  }
  g.op_f16 = f16 ? 1 : 0;
  g.M = M;
  g.a = x;
  g.lda = K;
  g.epi = EPI_16;
  g.out = y;
  g.ldo = N;
  g.err = reinterpret_cast<int *>(base + kErrOffset);
  // partial strips of the small-M path only; the tensor-core path runs without split-K here
  g.part = L.gpart_floats ? reinterpret_cast<float *>(base + L.gpart) : nullptr;
  g.part_floats = L.gpart_floats;
  g.splits_allowed = 0;
  if (r > 0) {
    k_lora_down(x, K, M, K, seg, reinterpret_cast<float *>(base + L.u_f32),
                reinterpret_cast<uint16_t *>(base + L.ul), f16, f16,
                reinterpret_cast<float *>(base + L.part), g.err, st);
    g.lora_u = reinterpret_cast<float *>(base + L.u_f32);
    g.lseg = seg;
    g.after_lora = 1;
    if (!gemv_eligible(g)) {
      k_pack_fwd(seg, N, reinterpret_cast<uint16_t *>(base + L.vl), f16, st);
      g.ul = reinterpret_cast<uint16_t *>(base + L.ul);
      g.vl = reinterpret_cast<uint16_t *>(base + L.vl);
      g.R = seg.Rpad();
    }
  }
  return gemm_launch(g, st);
}

extern "C" int soup_proj_noalloc_status(uintptr_t stream) {
  void *base_v = nullptr;
  SOUP_TRY(scratch_address(&base_v));
  int *err = reinterpret_cast<int *>(static_cast<uint8_t *>(base_v) + kErrOffset);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int flags = 0;
  SOUP_CUDA_TRY(cudaMemcpyAsync(&flags, err, sizeof(int), cudaMemcpyDeviceToHost, st));
  SOUP_CUDA_TRY(cudaStreamSynchronize(st));
  if (flags) SOUP_CUDA_TRY(cudaMemsetAsync(err, 0, sizeof(int), st));
  return kernel_flags_status(flags, "soup_proj_fwd_noalloc");
}
