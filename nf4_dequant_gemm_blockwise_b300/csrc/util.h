// Host-side error reporting shared by the library's translation units.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "soup.h"

namespace soup {
// Record a formatted message as this thread's last error and return `code`.
int set_error(int code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
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
