// The C ABI declared in include/soup.h: argument checks, error strings, and thin wrappers
// over the store, the step orchestrator and the single-projection kernels.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "gemm.h"
#include "kernels.h"
#include "soup.h"
#include "step.h"
#include "store.h"
#include "util.h"

namespace soup {
namespace {
thread_local std::string g_err;
}
int set_error(int code, const char *fmt, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}
void clear_error() { g_err.clear(); }
int kernel_flags_status(int flags, const char *who) {
  if (!flags) return 0;
  if (flags & 1)  // SOUP_KERR_WAIT_TIMEOUT
    return set_error(SOUP_ETIMEDOUT, "%s: a kernel's bounded wait gave up (flags 0x%x); its outputs are unusable",
                     who, flags);
  if (flags & 4)  // SOUP_KERR_RANGE
    return set_error(SOUP_ERANGE,
                     "%s: a value left the range of IEEE half (|x| > 65504 or NaN) where the forward stores "
                     "its 16-bit operands (flags 0x%x)", who, flags);
  return set_error(SOUP_ECUDA, "%s: kernel error flags 0x%x", who, flags);
}
namespace {
std::atomic<uint64_t> g_launches{0};
}
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
uint64_t launches_so_far() { return g_launches.load(std::memory_order_relaxed); }
}  // namespace soup

using namespace soup;

extern "C" {

const char *soup_last_error(void) { return g_err.c_str(); }
const char *soup_version(void) { return "soup-b300 0.1 (sm_103a)"; }
uint64_t soup_kernel_launches(void) { return launches_so_far(); }


int soup_nf4_codebook(float *out) {
  if (!out) return set_error(SOUP_EINVAL, "out is NULL");
  std::memcpy(out, nf4_codebook_param().v, 16 * sizeof(float));
  return 0;
}

int soup_shard_layout_of(const soup_cfg *cfg, soup_shard_layout *out) {
  if (!out) return set_error(SOUP_EINVAL, "out is NULL");
  return shard_layout(cfg, out);
}

int soup_nf4_quantize_host(const uint16_t *src, int64_t n, uint8_t *codes, float *absmax,
                           int n_threads) {
  if (n < 0 || (n > 0 && (!src || !codes || !absmax))) return set_error(SOUP_EINVAL, "NULL argument");
  nf4_quantize_host(src, n, codes, absmax, n_threads);
  return 0;
}

int soup_store_create(const soup_cfg *cfg, int allow_pageable, soup_store **out) {
  return store_create(cfg, allow_pageable, out);
}
int soup_store_put_layer(soup_store *st, int layer, const uint16_t *const *src, int n_threads) {
  return store_put_layer(st, layer, src, n_threads);
}
int soup_store_put_shard(soup_store *st, int layer, const void *shard, uint64_t bytes) {
  return store_put_shard(st, layer, shard, bytes);
}
int soup_store_put_head(soup_store *st, const uint16_t *embed, const uint16_t *lm_head) {
  return store_put_head(st, embed, lm_head);
}
int soup_store_build(const soup_cfg *cfg, const uint16_t *const *src, int allow_pageable,
                     soup_store **out) {
  if (!src) return set_error(SOUP_EINVAL, "src is NULL");
  int rc = store_create(cfg, allow_pageable, out);
  if (rc < 0 && rc != SOUP_EPAGEABLE) return rc;
  for (int l = 0; l < cfg->n_layers; ++l) {
    int r2 = store_put_layer(*out, l, src + (size_t)l * 9, 0);
    if (r2 < 0) {
      store_free(*out);
      *out = nullptr;
      return r2;
    }
  }
  return rc;
}
int soup_store_info(const soup_store *st, void **base, uint64_t *bytes, int *pinned) {
  if (!st) return set_error(SOUP_EINVAL, "store is NULL");
  if (base) *base = st->base;
  if (bytes) *bytes = st->bytes;
  if (pinned) *pinned = st->pinned;
  return 0;
}
void soup_store_free(soup_store *st) { store_free(st); }

int soup_workspace_bytes(const soup_cfg *cfg, int max_batch, int max_seq, int n_slots, int mode,
                         uint64_t *ws_bytes) {
  if (!ws_bytes) return set_error(SOUP_EINVAL, "ws_bytes is NULL");
  Plan P;
  SOUP_TRY(make_plan(cfg, max_batch, max_seq, n_slots, mode, &P));
  *ws_bytes = P.total;
  return 0;
}

uint64_t soup_peak_bytes(const soup_cfg *cfg, int batch, int seq, int n_slots, int mode,
                         uint64_t *workspace_bytes) {
  Plan P;
  if (make_plan(cfg, batch, seq, n_slots, mode, &P) < 0) return 0;
  if (workspace_bytes) *workspace_bytes = P.total;
  const uint64_t V = cfg->vocab, H = cfg->hidden, r = cfg->lora_r;
  uint64_t lora = 0;
  int n_out[4], n_in[4];
  group_shapes(cfg, n_out, n_in);
  const int qd = cfg->n_heads * cfg->head_dim, kvd = cfg->n_kv_heads * cfg->head_dim;
  const uint64_t outs[7] = {(uint64_t)qd, (uint64_t)kvd, (uint64_t)kvd, H, (uint64_t)cfg->inter,
                            (uint64_t)cfg->inter, H};
  const uint64_t ins[7] = {H, H, H, (uint64_t)qd, H, H, (uint64_t)cfg->inter};
  for (int p = 0; p < 7; ++p) lora += r * (outs[p] + ins[p]);
  lora *= (uint64_t)cfg->n_layers;
  // float32 adapters, their gradients and the two AdamW moments
  const uint64_t tables = (mode & SOUP_MODE_STREAM_HEAD) ? 0 : 2 * V * H + (cfg->tied ? 0 : 2 * V * H);
  const uint64_t resident_t = tables + 2 * H + 4 * 4 * lora;
  return P.total + resident_t;
}

int soup_stream_init(soup_store *st, const soup_cfg *cfg, int max_batch, int max_seq, void *dev_ws,
                     uint64_t ws_bytes, const void *embed, const void *lm_head, const void *final_norm,
                     uintptr_t compute_stream, uintptr_t copy_stream, int n_slots, int mode,
                     soup_stream **out) {
  return stream_init(st, cfg, max_batch, max_seq, dev_ws, ws_bytes, embed, lm_head, final_norm,
                     compute_stream, copy_stream, n_slots, mode, out);
}
int soup_step_fwd(soup_stream *h, const int32_t *tokens_dev, int B, int S, const float *const *lora_A,
                  const float *const *lora_B, float *loss_dev, float *logits_dev, float *layer_out_dev) {
  return step_fwd(h, tokens_dev, B, S, lora_A, lora_B, loss_dev, logits_dev, layer_out_dev);
}
int soup_step_bwd(soup_stream *h, float *const *dA, float *const *dB, float *dh_out_dev) {
  return step_bwd(h, dA, dB, dh_out_dev, 0);
}
int soup_step_bwd_ex(soup_stream *h, float *const *dA, float *const *dB, float *dh_out_dev,
                     int flags) {
  return step_bwd(h, dA, dB, dh_out_dev, flags);
}
int soup_sync(soup_stream *h, int timeout_ms) { return stream_sync(h, timeout_ms); }
int soup_stream_stats(soup_stream *h, soup_stats *out, int reset) { return stream_stats(h, out, reset); }
int soup_stream_debug(soup_stream *h, int what, int value) {
  if (!h) return set_error(SOUP_EINVAL, "handle is NULL");
  if (what == SOUP_DBG_PROFILE) h->dbg_profile = value;
  else if (what == SOUP_DBG_STALE_SLOT) h->dbg_stale = value;
  else if (what == SOUP_DBG_COPY_DELAY_US) {
    if (value < 0 || value > 1000000) return set_error(SOUP_EINVAL, "copy delay %d us outside [0, 1 s]", value);
    h->dbg_copy_delay_us = value;
  } else if (what == SOUP_DBG_WAIT_PROBE) {
    if (value < 1 || value > 1000000) return set_error(SOUP_EINVAL, "probe limit %d us outside [1, 1 s]", value);
    k_wait_probe(h->err_dev, 2000ll * value, h->cs);  // ~2000 SM cycles per microsecond
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(SOUP_ECUDA, "wait probe launch: %s", cudaGetErrorString(e));
    SOUP_CUDA_TRY(cudaEventRecord(h->done, h->cs));
  } else return set_error(SOUP_EINVAL, "unknown debug switch %d", what);
  return 0;
}
void soup_stream_free(soup_stream *h) { soup_stream_free_impl(h); }
int soup_stream_kernel_stats(soup_stream *h, soup_kernel_stat *out, int max, int *n, int reset) {
  return stream_kernel_stats(h, out, max, n, reset);
}

// ------------------------------------------------------------------ single projection
namespace {
struct ProjScratch {
  uint64_t u_f32, ul, vl, ac, du_f32, dul, part, gpart, gpart_floats, err, total;
};
ProjScratch proj_plan(int M, int N, int K) {
  ProjScratch s;
  uint64_t off = 0;
  auto take = [&](uint64_t b) {
    const uint64_t o = off;
    off = (off + b + 1023) / 1024 * 1024;
    return o;
  };
  s.u_f32 = take(4ull * M * 64);
  s.ul = take(2ull * M * 64);
  s.vl = take(2ull * N * 64);
  s.ac = take(2ull * 64 * K);
  s.du_f32 = take(4ull * M * 64);
  s.dul = take(2ull * M * 64);
  s.part = take(4ull * std::max(lora_scratch_floats(std::max(M, 1), K, 64),
                                 lora_scratch_floats(std::max(M, 1), N, 64)));
  s.gpart_floats = std::min<uint64_t>(4ull * M * std::max(N, K), 1ull << 26);
  if (M <= 16)  // the small-M path's per-CTA partial strips
    s.gpart_floats = std::max<uint64_t>(s.gpart_floats, std::max(gemv_part_floats(GEMM_FWD),
                                                                 gemv_part_floats(GEMM_DX)));
  s.gpart = take(4 * s.gpart_floats);
  s.err = take(64);
  s.total = off;
  return s;
}
int proj_check(int M, int N, int K, const uint8_t *codes, const float *absmax, const uint16_t *w,
               const float *A, const float *B, int r, void *scratch, uint64_t bytes) {
  if (M < 0 || N < 1 || K < 1 || r < 0 || r > 64)
    return set_error(SOUP_EINVAL, "bad shape M=%d N=%d K=%d r=%d", M, N, K, r);
  if (r > 0 && (!A || !B)) return set_error(SOUP_EINVAL, "NULL LoRA pointer with r > 0");
  if (!scratch) return set_error(SOUP_EINVAL, "NULL scratch pointer");
  if (!(codes && absmax) && !w) return set_error(SOUP_EINVAL, "no weight given");
  if ((int64_t)N * K % 64 && codes) return set_error(SOUP_EINVAL, "N*K must be a multiple of 64");
  if (bytes < proj_plan(M, N, K).total) return set_error(SOUP_ENOMEM, "scratch too small");
  if (reinterpret_cast<uintptr_t>(scratch) % 256) return set_error(SOUP_EINVAL, "scratch must be 256-byte aligned");
  return 0;
}
LoraSeg one_seg(int N, const float *A, const float *B, int r, float s, float *dA, float *dB) {
  LoraSeg L;
  L.nseg = 1;
  L.r = r;
  L.s = s;
  L.off[0] = 0;
  L.n[0] = N;
  L.A[0] = A;
  L.B[0] = B;
  L.dA[0] = dA;
  L.dB[0] = dB;
  return L;
}
GemmArgs proj_weight(int mode, int N, int K, const uint8_t *codes, const float *absmax, const uint16_t *w) {
  GemmArgs g;
  g.mode = mode;
  g.Nw = N;
  g.Kw = K;
  if (codes) {
    g.wfmt = W_NF4;
    g.codes = codes;
    g.absmax = absmax;
  } else {
    g.wfmt = W_BF16;
    g.w = w;
  }
  return g;
}
}  // namespace

int soup_proj_scratch_bytes(int M, int N, int K, int r, uint64_t *bytes) {
  if (!bytes || M < 0 || N < 1 || K < 1 || r < 0 || r > 64) return set_error(SOUP_EINVAL, "bad argument");
  *bytes = proj_plan(M, N, K).total;
  return 0;
}

int soup_proj_fwd(const uint16_t *x, int M, int N, int K, const uint8_t *codes, const float *absmax,
                  const uint16_t *w_bf16, const float *A, const float *B, int r, float s, int x_f16,
                  uint16_t *y, void *scratch, uint64_t scratch_bytes, uintptr_t stream) {
  SOUP_TRY(proj_check(M, N, K, codes, absmax, w_bf16, A, B, r, scratch, scratch_bytes));
  if (M == 0) return 0;
  if (!x || !y) return set_error(SOUP_EINVAL, "NULL x or y");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const ProjScratch P = proj_plan(M, N, K);
  uint8_t *base = static_cast<uint8_t *>(scratch);
  LoraSeg L = one_seg(N, A, B, r, s, nullptr, nullptr);
  const bool f16 = x_f16 != 0;
  GemmArgs g = proj_weight(GEMM_FWD, N, K, codes, absmax, w_bf16);
  g.op_f16 = f16 ? 1 : 0;
  g.M = M; g.a = x; g.lda = K;
  g.epi = EPI_16; g.out = y; g.ldo = N;
  g.err = reinterpret_cast<int *>(base + P.err);
  g.part = reinterpret_cast<float *>(base + P.gpart);
  g.part_floats = P.gpart_floats;
  if (r > 0) {
    k_lora_down(x, K, M, K, L, reinterpret_cast<float *>(base + P.u_f32),
                reinterpret_cast<uint16_t *>(base + P.ul), f16, f16,
                reinterpret_cast<float *>(base + P.part), reinterpret_cast<int *>(base + P.err), st);
    g.lora_u = reinterpret_cast<float *>(base + P.u_f32);
    g.lseg = L;
    g.after_lora = 1;
    if (!gemv_eligible(g)) {  // the tensor-core path takes the LoRA term as 16-bit K tiles
      k_pack_fwd(L, N, reinterpret_cast<uint16_t *>(base + P.vl), f16, st);
      g.ul = reinterpret_cast<uint16_t *>(base + P.ul);
      g.vl = reinterpret_cast<uint16_t *>(base + P.vl);
      g.R = L.Rpad();
    }
  }
  return gemm_launch(g, st);
}

int soup_proj_dx(const uint16_t *dy, int M, int N, int K, const uint8_t *codes, const float *absmax,
                 const uint16_t *w_bf16, const float *A, const float *B, int r, float s, float *dx,
                 void *scratch, uint64_t scratch_bytes, uintptr_t stream) {
  SOUP_TRY(proj_check(M, N, K, codes, absmax, w_bf16, A, B, r, scratch, scratch_bytes));
  if (M == 0) return 0;
  if (!dy || !dx) return set_error(SOUP_EINVAL, "NULL dy or dx");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const ProjScratch P = proj_plan(M, N, K);
  uint8_t *base = static_cast<uint8_t *>(scratch);
  LoraSeg L = one_seg(N, A, B, r, s, nullptr, nullptr);
  GemmArgs g = proj_weight(GEMM_DX, N, K, codes, absmax, w_bf16);
  g.M = M; g.a = dy; g.lda = N;
  g.epi = EPI_F32; g.out = dx; g.ldo = K;
  g.err = reinterpret_cast<int *>(base + P.err);
  g.part = reinterpret_cast<float *>(base + P.gpart);
  g.part_floats = P.gpart_floats;
  if (r > 0) {
    k_lora_du(dy, N, M, L, reinterpret_cast<float *>(base + P.du_f32),
              reinterpret_cast<uint16_t *>(base + P.dul), false, false,
              reinterpret_cast<float *>(base + P.part), st);
    g.lora_u = reinterpret_cast<float *>(base + P.du_f32);
    g.lseg = L;
    g.after_lora = 1;
    if (!gemv_eligible(g)) {
      k_pack_bwd(L, K, reinterpret_cast<uint16_t *>(base + P.ac), false, st);
      g.ul = reinterpret_cast<uint16_t *>(base + P.dul);
      g.vl = reinterpret_cast<uint16_t *>(base + P.ac);
      g.R = L.Rpad();
    }
  }
  return gemm_launch(g, st);
}

int soup_proj_lora_grad(const uint16_t *x, const uint16_t *dy, int M, int N, int K, const float *A,
                        const float *B, int r, float s, int x_f16, float *dA, float *dB, void *scratch,
                        uint64_t scratch_bytes, uintptr_t stream) {
  if (!dA || !dB || !x || !dy) return set_error(SOUP_EINVAL, "NULL argument");
  if (M < 1 || N < 1 || K < 1 || r < 1 || r > 64 || !A || !B || !scratch)
    return set_error(SOUP_EINVAL, "bad argument");
  if (scratch_bytes < proj_plan(M, N, K).total) return set_error(SOUP_ENOMEM, "scratch too small");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const ProjScratch P = proj_plan(M, N, K);
  uint8_t *base = static_cast<uint8_t *>(scratch);
  LoraSeg L = one_seg(N, A, B, r, s, dA, dB);
  float *part = reinterpret_cast<float *>(base + P.part);
  const bool f16 = x_f16 != 0;
  k_lora_down(x, K, M, K, L, reinterpret_cast<float *>(base + P.u_f32),
              reinterpret_cast<uint16_t *>(base + P.ul), f16, f16, part,
              reinterpret_cast<int *>(base + P.err), st);
  k_lora_du(dy, N, M, L, reinterpret_cast<float *>(base + P.du_f32),
            reinterpret_cast<uint16_t *>(base + P.dul), false, false, part, st);
  LoraGradGroup G;
  G.L = L;
  G.dy = dy;
  G.ldy = N;
  G.Ng = N;
  G.u = reinterpret_cast<float *>(base + P.u_f32);
  G.du = reinterpret_cast<float *>(base + P.du_f32);
  G.x = x;
  G.ldx = K;
  G.K = K;
  k_lora_grads(&G, 1, M, f16, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(SOUP_ECUDA, "lora grad launch: %s", cudaGetErrorString(e));
  return 0;
}

int soup_proj_status(void *scratch, int M, int N, int K, uintptr_t stream) {
  if (!scratch || M < 0 || N < 1 || K < 1) return set_error(SOUP_EINVAL, "bad argument");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int *err = reinterpret_cast<int *>(static_cast<uint8_t *>(scratch) + proj_plan(M, N, K).err);
  int flags = 0;
  SOUP_CUDA_TRY(cudaMemcpyAsync(&flags, err, sizeof(int), cudaMemcpyDeviceToHost, st));
  SOUP_CUDA_TRY(cudaStreamSynchronize(st));
  SOUP_CUDA_TRY(cudaMemsetAsync(err, 0, sizeof(int), st));
  return kernel_flags_status(flags, "soup_proj_status");
}

namespace {
int attn_check(int B, int S, int nh, int nkv, int d) {
  if (B < 0 || S < 0 || nh < 1 || nkv < 1 || nh % nkv != 0)
    return set_error(SOUP_EINVAL, "attention: bad shape (B %d, S %d, heads %d / %d)", B, S, nh, nkv);
  if (d != 64 && d != 128) return set_error(SOUP_EINVAL, "attention: head_dim %d not supported (64 or 128)", d);
  return 0;
}
}  // namespace

uint64_t soup_attn_bwd_scratch_bytes(int B, int S, int n_heads, int n_kv_heads, int head_dim) {
  if (attn_check(B, S, n_heads, n_kv_heads, head_dim) < 0) return 0;
  return 4ull * attn_bwd_scratch_floats(B, S, n_heads, n_kv_heads, head_dim);
}

int soup_attn_fwd(const uint16_t *qkv, int B, int S, int n_heads, int n_kv_heads, int head_dim,
                  uint16_t *o, float *lse, int *err, uintptr_t stream) {
  SOUP_TRY(attn_check(B, S, n_heads, n_kv_heads, head_dim));
  if (B == 0 || S == 0) return 0;
  if (!qkv || !o || !lse) return set_error(SOUP_EINVAL, "attention: NULL buffer");
  const int ld = (n_heads + 2 * n_kv_heads) * head_dim;
  return k_attn_fwd(qkv, ld, B, S, n_heads, n_kv_heads, head_dim, o, lse, err,
                    reinterpret_cast<cudaStream_t>(stream));
}

int soup_attn_bwd(const uint16_t *qkv, const uint16_t *o, const uint16_t *dO, const float *lse, int B,
                  int S, int n_heads, int n_kv_heads, int head_dim, void *scratch,
                  uint64_t scratch_bytes, float *dqkv, int *err, uintptr_t stream) {
  SOUP_TRY(attn_check(B, S, n_heads, n_kv_heads, head_dim));
  if (B == 0 || S == 0) return 0;
  if (!qkv || !o || !dO || !lse || !dqkv || !scratch) return set_error(SOUP_EINVAL, "attention: NULL buffer");
  if (reinterpret_cast<uintptr_t>(scratch) % 256) return set_error(SOUP_EINVAL, "attention: scratch must be 256-byte aligned");
  const uint64_t need = 4ull * attn_bwd_scratch_floats(B, S, n_heads, n_kv_heads, head_dim);
  if (scratch_bytes < need)
    return set_error(SOUP_EINVAL, "attention: scratch %llu bytes < %llu", (unsigned long long)scratch_bytes,
                     (unsigned long long)need);
  const int ld = (n_heads + 2 * n_kv_heads) * head_dim;
  return k_attn_bwd(qkv, ld, o, dO, lse, B, S, n_heads, n_kv_heads, head_dim, static_cast<float *>(scratch),
                    dqkv, err, reinterpret_cast<cudaStream_t>(stream));
}

int soup_nf4_dequant(const uint8_t *codes, const float *absmax, int64_t n, float *out_f32,
                     uint16_t *out_bf16, uintptr_t stream) {
  if (n < 0 || (n > 0 && (!codes || !absmax))) return set_error(SOUP_EINVAL, "NULL argument");
  k_nf4_dequant(codes, absmax, n, out_f32, out_bf16, reinterpret_cast<cudaStream_t>(stream));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(SOUP_ECUDA, "dequant launch: %s", cudaGetErrorString(e));
  return 0;
}

int soup_adamw_step(float *param, const float *grad, float *m, float *v, int64_t n,
                    const soup_adamw *hp, int64_t step, uintptr_t stream) {
  if (!hp || n < 0) return set_error(SOUP_EINVAL, "adamw: NULL hyper-parameters or n < 0");
  if (n > 0 && (!param || !grad || !m || !v)) return set_error(SOUP_EINVAL, "adamw: NULL buffer");
  if (step < 1) return set_error(SOUP_EINVAL, "adamw: step numbers start at 1 (got %lld)", (long long)step);
  if (!(hp->beta1 >= 0.f && hp->beta1 < 1.f && hp->beta2 >= 0.f && hp->beta2 < 1.f))
    return set_error(SOUP_EINVAL, "adamw: betas must lie in [0, 1)");
  const uintptr_t lo[4] = {(uintptr_t)param, (uintptr_t)grad, (uintptr_t)m, (uintptr_t)v};
  for (int i = 0; i < 4 && n > 0; ++i)
    for (int j = i + 1; j < 4; ++j)
      if (lo[i] < lo[j] + 4ull * n && lo[j] < lo[i] + 4ull * n)
        return set_error(SOUP_EINVAL, "adamw: buffers %d and %d overlap", i, j);
  k_adamw(param, grad, m, v, n, hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay,
          hp->grad_scale, step, reinterpret_cast<cudaStream_t>(stream));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(SOUP_ECUDA, "adamw launch: %s", cudaGetErrorString(e));
  return 0;
}

}  // extern "C"
