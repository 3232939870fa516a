// Host side of the layer store: the NF4 codebook, the blockwise quantiser, the shard layout
// and the page-locked arena ("About Soup": the checkpoint is rewritten once into one shard
// per decoder layer and held in host RAM; "Layer streaming: fine-tune a model that does not
// fit in your card", "How it works": page-locked when the machine allows it; "Measured
// numbers": pinned copies overlap compute, pageable ones do not, and a power-of-two pinned
// allocator cost 1.73x at 14B — so the store here is ONE exact-size page-locked arena).
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <thread>
#include <vector>

#include "kernels.h"
#include "store.h"
#include "util.h"

namespace soup {

// ------------------------------------------------------------------ codebook
// NormalFloat-4: eight positive values at the standard-normal quantiles of eight evenly
// spaced probabilities from delta towards 1/2, seven negative ones mirrored from seven
// evenly spaced probabilities over the same range, and zero; divided by the largest.
// delta = (1 - 1/32 + 1 - 1/30) / 2.  The quantile is found by bisection on the normal
// CDF, Phi(z) = erfc(-z / sqrt 2) / 2, carried to full double precision.
static double normal_cdf(double z) { return 0.5 * std::erfc(-z / std::sqrt(2.0)); }

static double normal_quantile_upper(double p) {  // p in [1/2, 1): z >= 0 with Phi(z) = p
  double lo = 0.0, hi = 40.0;
  for (int i = 0; i < 200; ++i) {
    const double mid = 0.5 * (lo + hi);
    if (normal_cdf(mid) < p) lo = mid;
    else hi = mid;
  }
  return 0.5 * (lo + hi);
}

static const Codebook &build_codebook() {
  static Codebook cb;
  static std::once_flag once;
  std::call_once(once, [] {
    const double delta = 0.5 * ((1.0 - 1.0 / 32.0) + (1.0 - 1.0 / 30.0));
    double v[16];
    for (int i = 0; i < 7; ++i) v[i] = -normal_quantile_upper(delta + i * ((0.5 - delta) / 7.0));
    v[7] = 0.0;
    for (int j = 0; j < 8; ++j) v[8 + j] = normal_quantile_upper(delta + (7 - j) * ((0.5 - delta) / 8.0));
    const double zmax = v[15];
    for (int i = 0; i < 16; ++i) cb.v[i] = (float)(v[i] / zmax);
  });
  return cb;
}

const Codebook &nf4_codebook_param() { return build_codebook(); }

const float *nf4_midpoints() {
  static float mid[15];
  static std::once_flag once;
  std::call_once(once, [] {
    const Codebook &c = build_codebook();
    for (int k = 0; k < 15; ++k) mid[k] = (float)(((double)c.v[k] + (double)c.v[k + 1]) * 0.5);
  });
  return mid;
}

// ------------------------------------------------------------------ quantiser
static inline float bf16_bits_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Quantise blocks [b0, b1) of a tensor of n elements.
static void quantize_blocks(const uint16_t *src, int64_t n, uint8_t *codes, float *absmax,
                            int64_t b0, int64_t b1) {
  const float *mid = nf4_midpoints();
  for (int64_t b = b0; b < b1; ++b) {
    const int64_t e0 = b * 64;
    const int cnt = (int)std::min<int64_t>(64, n - e0);
    float x[64];
    float amax = 0.f;
    for (int i = 0; i < cnt; ++i) {
      x[i] = bf16_bits_to_float(src[e0 + i]);
      const float a = std::fabs(x[i]);
      if (a > amax) amax = a;
    }
    absmax[b] = amax;
    uint8_t c[64];
    for (int i = 0; i < 64; ++i) {
      if (i >= cnt || amax == 0.f) {
        c[i] = 7;
        continue;
      }
      const float q = x[i] / amax;  // IEEE single-precision divide
      int k = 0;
      for (int j = 0; j < 15; ++j) k += (q > mid[j]);
      c[i] = (uint8_t)k;
    }
    const int nbytes = (cnt + 1) / 2;
    for (int j = 0; j < nbytes; ++j) codes[e0 / 2 + j] = (uint8_t)((c[2 * j] << 4) | c[2 * j + 1]);
  }
}

void nf4_quantize_host(const uint16_t *src, int64_t n, uint8_t *codes, float *absmax, int n_threads) {
  const int64_t nb = (n + 63) / 64;
  if (n_threads <= 0) n_threads = (int)std::max(1u, std::thread::hardware_concurrency());
  const int64_t per = std::max<int64_t>(1024, (nb + n_threads - 1) / n_threads);
  if (nb <= per) {
    quantize_blocks(src, n, codes, absmax, 0, nb);
    return;
  }
  std::vector<std::thread> th;
  for (int64_t b = 0; b < nb; b += per)
    th.emplace_back(quantize_blocks, src, n, codes, absmax, b, std::min(nb, b + per));
  for (auto &t : th) t.join();
}

// ------------------------------------------------------------------ layout
static uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

int validate_cfg(const soup_cfg *c) {
  if (!c) return set_error(SOUP_EINVAL, "cfg is NULL");
  if (c->n_layers < 1 || c->hidden < 64 || c->inter < 1 || c->n_heads < 1 || c->n_kv_heads < 1 ||
      c->head_dim < 2 || c->vocab < 2)
    return set_error(SOUP_EINVAL, "cfg: non-positive size");
  if (c->n_heads % c->n_kv_heads)
    return set_error(SOUP_EINVAL, "cfg: n_heads %d not a multiple of n_kv_heads %d", c->n_heads, c->n_kv_heads);
  if (c->head_dim != 64 && c->head_dim != 128)
    return set_error(SOUP_EINVAL, "cfg: head_dim must be 64 or 128");
  if (c->hidden % 64 || c->inter % 8)
    return set_error(SOUP_EINVAL, "cfg: hidden must be a multiple of 64 and inter of 8");
  if (c->hidden > 8192)
    return set_error(SOUP_EINVAL, "cfg: hidden must be at most 8192 (one row per norm block)");
  if (c->lora_r < 1 || 3 * c->lora_r > 64)
    return set_error(SOUP_EINVAL, "cfg: lora_r must be in [1, 21]");
  if (c->base_fmt != SOUP_FMT_BF16 && c->base_fmt != SOUP_FMT_NF4)
    return set_error(SOUP_EINVAL, "cfg: base_fmt must be SOUP_FMT_BF16 or SOUP_FMT_NF4");
  if (!(c->rms_eps > 0.f) || !(c->rope_theta > 0.f) || !(c->lora_alpha > 0.f))
    return set_error(SOUP_EINVAL, "cfg: eps, theta and alpha must be positive");
  if (c->base_fmt == SOUP_FMT_NF4) {
    const int64_t H = c->hidden, I = c->inter, qd = (int64_t)c->n_heads * c->head_dim,
                  kvd = (int64_t)c->n_kv_heads * c->head_dim;
    const int64_t numel[7] = {qd * H, kvd * H, kvd * H, H * qd, I * H, I * H, H * I};
    for (int p = 0; p < 7; ++p)
      if (numel[p] % 64)
        return set_error(SOUP_EINVAL, "cfg: projection %d has %lld weights, not a multiple of 64", p,
                         (long long)numel[p]);
  }
  return 0;
}

void group_shapes(const soup_cfg *c, int n_out[4], int n_in[4]) {
  const int qd = c->n_heads * c->head_dim, kvd = c->n_kv_heads * c->head_dim;
  n_out[SOUP_G_QKV] = qd + 2 * kvd; n_in[SOUP_G_QKV] = c->hidden;
  n_out[SOUP_G_O] = c->hidden;      n_in[SOUP_G_O] = qd;
  n_out[SOUP_G_GU] = 2 * c->inter;  n_in[SOUP_G_GU] = c->hidden;
  n_out[SOUP_G_DOWN] = c->hidden;   n_in[SOUP_G_DOWN] = c->inter;
}

int shard_layout(const soup_cfg *c, soup_shard_layout *L) {
  SOUP_TRY(validate_cfg(c));
  std::memset(L, 0, sizeof(*L));
  group_shapes(c, L->n_out, L->n_in);
  uint64_t off = 0, end = 0;
  for (int g = 0; g < SOUP_NGROUP; ++g) {
    const uint64_t numel = (uint64_t)L->n_out[g] * L->n_in[g];
    L->w_off[g] = off;
    L->w_bytes[g] = c->base_fmt == SOUP_FMT_NF4 ? (numel + 1) / 2 : numel * 2;
    end = off + L->w_bytes[g];
    off = align_up(end, 1024);
    if (c->base_fmt == SOUP_FMT_NF4) {
      L->a_off[g] = off;
      L->a_bytes[g] = (numel + 63) / 64 * 4;
      end = off + L->a_bytes[g];
      off = align_up(end, 1024);
    }
  }
  L->ln1_off = off;
  end = off + 2ull * c->hidden;
  off = align_up(end, 1024);
  L->ln2_off = off;
  end = off + 2ull * c->hidden;
  L->payload = 0;
  for (int g = 0; g < SOUP_NGROUP; ++g) L->payload += L->w_bytes[g] + L->a_bytes[g];
  L->payload += 4ull * c->hidden;
  L->stride = align_up(end, 4096);
  return 0;
}

// ------------------------------------------------------------------ store
int store_create(const soup_cfg *c, int allow_pageable, soup_store **out) {
  if (!out) return set_error(SOUP_EINVAL, "out is NULL");
  *out = nullptr;
  soup_shard_layout L;
  SOUP_TRY(shard_layout(c, &L));
  soup_store *st = new (std::nothrow) soup_store();
  if (!st) return set_error(SOUP_ENOMEM, "store: host allocation failed");
  st->cfg = *c;
  st->lay = L;
  st->bytes = L.stride * (uint64_t)c->n_layers;
  void *p = nullptr;
  const bool force_pageable = allow_pageable == SOUP_STORE_PAGEABLE;
  cudaError_t e = force_pageable ? cudaErrorNotPermitted : cudaHostAlloc(&p, st->bytes, cudaHostAllocDefault);
  int rc = 0;
  if (e == cudaSuccess) {
    st->pinned = 1;
  } else {
    // A failed page-lock leaves a sticky runtime error; clear it before falling back.
    (void)cudaGetLastError();
    if (!allow_pageable) {
      delete st;
      return set_error(SOUP_ENOMEM, "store: page-locking %llu bytes failed (%s)",
                       (unsigned long long)(L.stride * (uint64_t)c->n_layers), cudaGetErrorString(e));
    }
    p = std::aligned_alloc(4096, st->bytes);
    if (!p) {
      delete st;
      return set_error(SOUP_ENOMEM, "store: host allocation of %llu bytes failed",
                       (unsigned long long)(L.stride * (uint64_t)c->n_layers));
    }
    st->pinned = 0;
    if (!force_pageable)
      rc = set_error(SOUP_EPAGEABLE, "store: page-locking failed (%s); using pageable memory",
                     cudaGetErrorString(e));
  }
  st->base = static_cast<uint8_t *>(p);
  st->filled.assign(c->n_layers, 0);
  *out = st;
  return rc;
}

int store_put_shard(soup_store *st, int layer, const void *shard, uint64_t bytes) {
  if (!st || !shard) return set_error(SOUP_EINVAL, "store_put_shard: NULL argument");
  if (layer < 0 || layer >= st->cfg.n_layers) return set_error(SOUP_EINVAL, "layer %d out of range", layer);
  if (bytes != st->lay.stride)
    return set_error(SOUP_EINVAL, "store_put_shard: %llu bytes, the shard stride is %llu",
                     (unsigned long long)bytes, (unsigned long long)st->lay.stride);
  std::memcpy(st->base + (uint64_t)layer * st->lay.stride, shard, bytes);
  st->filled[layer] = 1;
  return 0;
}

int store_put_layer(soup_store *st, int layer, const uint16_t *const *src, int n_threads) {
  if (!st || !src) return set_error(SOUP_EINVAL, "store_put_layer: NULL argument");
  const soup_cfg &c = st->cfg;
  if (layer < 0 || layer >= c.n_layers) return set_error(SOUP_EINVAL, "layer %d out of range", layer);
  for (int i = 0; i < 9; ++i)
    if (!src[i]) return set_error(SOUP_EINVAL, "source tensor %d is NULL", i);
  const soup_shard_layout &L = st->lay;
  uint8_t *sh = st->base + (uint64_t)layer * L.stride;
  const int qd = c.n_heads * c.head_dim, kvd = c.n_kv_heads * c.head_dim;
  // (group, row offset inside the group, rows, cols) of each projection
  const int grp[7] = {SOUP_G_QKV, SOUP_G_QKV, SOUP_G_QKV, SOUP_G_O, SOUP_G_GU, SOUP_G_GU, SOUP_G_DOWN};
  const int roff[7] = {0, qd, qd + kvd, 0, 0, c.inter, 0};
  const int rows[7] = {qd, kvd, kvd, c.hidden, c.inter, c.inter, c.hidden};
  for (int p = 0; p < 7; ++p) {
    const int g = grp[p];
    const int cols = L.n_in[g];
    const int64_t n = (int64_t)rows[p] * cols;
    const int64_t first = (int64_t)roff[p] * cols;
    if (c.base_fmt == SOUP_FMT_NF4) {
      nf4_quantize_host(src[p], n, sh + L.w_off[g] + first / 2,
                        reinterpret_cast<float *>(sh + L.a_off[g]) + first / 64, n_threads);
    } else {
      std::memcpy(sh + L.w_off[g] + first * 2, src[p], n * 2);
    }
  }
  std::memcpy(sh + L.ln1_off, src[7], 2ull * c.hidden);
  std::memcpy(sh + L.ln2_off, src[8], 2ull * c.hidden);
  st->filled[layer] = 1;
  return 0;
}

// The head tables go into one mapped page-locked allocation: the embedding gather reads its
// rows straight from it, and the output head is copied from it into the device buffer.
int store_put_head(soup_store *st, const uint16_t *embed, const uint16_t *lm_head) {
  if (!st || !embed) return set_error(SOUP_EINVAL, "store_put_head: NULL argument");
  const soup_cfg &c = st->cfg;
  if (c.tied && lm_head) return set_error(SOUP_EINVAL, "store_put_head: a tied stack has no separate head");
  if (!c.tied && !lm_head) return set_error(SOUP_EINVAL, "store_put_head: an untied stack needs lm_head");
  const uint64_t table = 2ull * c.vocab * c.hidden;
  const uint64_t bytes = c.tied ? table : 2 * table;
  if (!st->head) {
    void *p = nullptr;
    cudaError_t e = cudaHostAlloc(&p, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return set_error(SOUP_ENOMEM, "store_put_head: page-locking %llu bytes failed (%s); the streamed "
                       "head needs page-locked memory", (unsigned long long)bytes, cudaGetErrorString(e));
    }
    void *d = nullptr;
    e = cudaHostGetDevicePointer(&d, p, 0);
    if (e != cudaSuccess || !d) {
      (void)cudaGetLastError();
      cudaFreeHost(p);
      return set_error(SOUP_ECUDA, "store_put_head: no device address for the head tables (%s)",
                       cudaGetErrorString(e));
    }
    st->head = static_cast<uint8_t *>(p);
    st->head_dev = static_cast<uint8_t *>(d);
    st->head_bytes = bytes;
  }
  std::memcpy(st->head, embed, table);
  if (!c.tied) std::memcpy(st->head + table, lm_head, table);
  return 0;
}

void store_free(soup_store *st) {
  if (!st) return;
  if (st->head) cudaFreeHost(st->head);
  if (st->base) {
    if (st->pinned) cudaFreeHost(st->base);
    else std::free(st->base);
  }
  delete st;
}

}  // namespace soup
