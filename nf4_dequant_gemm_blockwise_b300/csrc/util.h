// Host-side error reporting shared by the library's translation units.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "soup.h"

namespace soup {
constexpr int MAX_DEVICES = 64;

// A per-device value computed once (kernel attributes, occupancy, SM counts): slot[dev] holds
// it after the first call on device dev; fn(dev, &value) computes it.  Thread-safe: racing
// first calls may both run fn, which must therefore be idempotent.  A value of 0 is not
// cached.  Declare the slot array with static storage (zero-initialised).
template <typename Fn>
cudaError_t per_device_once(std::atomic<int> (&slot)[MAX_DEVICES], int *out, Fn fn) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  int v = slot[dev].load(std::memory_order_acquire);
  if (v == 0) {
    e = fn(dev, &v);
    if (e != cudaSuccess) return e;
    slot[dev].store(v, std::memory_order_release);
  }
  *out = v;
  return cudaSuccess;
}

// Record a formatted message as this thread's last error and return `code`.
int set_error(int code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
// Status of the error bits kernels OR into a device flag (SOUP_KERR_* in common.cuh):
// 0 when no bit is set, else SOUP_ETIMEDOUT (a bounded wait gave up) or SOUP_ERANGE (a value
// left the 16-bit operand range), with the message set.  `who` names the flag's owner.
int kernel_flags_status(int flags, const char *who);
void clear_error();
// Process-wide count of kernels this library has launched (for launch accounting).
void count_launches(int n);
uint64_t launches_so_far();
}  // namespace soup

#define SOUP_CUDA_TRY(call)                                                              \
  do {                                                                                   \
    cudaError_t _e = (call);                                                             \
    if (_e != cudaSuccess)                                                               \
      return ::soup::set_error(SOUP_ECUDA, "%s: %s", #call, cudaGetErrorString(_e));    \
  } while (0)
#define SOUP_TRY(call)        \
  do {                        \
    int _rc = (call);         \
    if (_rc < 0) return _rc;  \
  } while (0)
