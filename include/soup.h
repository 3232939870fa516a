/*
 * soup.h — C ABI of libsoup: one LoRA fine-tuning step over a frozen decoder stack that is
 * streamed layer by layer from a pinned host store through a small pool of device slots.
 *
 * Sources (page title, section):
 *   "About Soup"                                   — the frozen base is never loaded whole;
 *       one shard per layer, copied into a small pool of pre-allocated buffers on a
 *       dedicated stream so the next layer's load overlaps the current layer's compute;
 *       NF4 shrinks the store about fourfold.
 *   "Layer streaming: fine-tune a model that does not fit in your card" (the docs page),
 *       "Turn it on"     — quantization none (bf16) or 4bit (NF4); stream_buffers in [2, 8].
 *       "How it works"   — resident embeddings, final norm, untied head, LoRA adapters and
 *                          their gradients; page-locked store; each layer read twice per
 *                          step because the backward needs W^T dL/dy.
 *       "Read this first" / "Bit-exact is two claims, not one" — the streamed run must equal
 *                          the resident run bit for bit, forward and every LoRA gradient,
 *                          including layers above ~165 MiB.
 *       "Measured numbers" — pinned copies overlap compute, pageable ones do not.
 *
 * Conventions for every entry point:
 *   - Return value: SOUP_OK (0) or a negative SOUP_E* code; soup_last_error() then holds a
 *     one-line message (thread-local, valid until the next call on the same thread).
 *     SOUP_EPAGEABLE is a warning: the object was created and is usable.
 *   - "dev" pointers are CUDA device pointers owned by the caller; "host" pointers are
 *     ordinary host memory owned by the caller.  The library never frees caller memory.
 *   - Streams are raw cudaStream_t values passed as uintptr_t (0 = legacy default stream).
 *     Work is enqueued asynchronously; the host returns before the GPU finishes.
 *   - bf16 values travel as uint16_t bit patterns; float is IEEE binary32.
 *   - Matrices are row-major and densely packed unless a leading dimension is given.
 *   - Nothing in a step allocates device memory: the caller passes one workspace sized by
 *     soup_workspace_bytes().
 */
#ifndef SOUP_H
#define SOUP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  SOUP_OK = 0,
  SOUP_EINVAL = -1,     /* bad argument or unsupported shape; nothing was enqueued      */
  SOUP_ENOMEM = -2,     /* a host allocation failed, or the workspace is too small      */
  SOUP_ECUDA = -3,      /* a CUDA runtime call failed (message names it)                */
  SOUP_ESTATE = -4,     /* call out of order (e.g. backward without a forward)          */
  SOUP_ETIMEDOUT = -5,  /* soup_sync gave up, or a kernel's bounded wait ran out        */
  SOUP_EPAGEABLE = -6,  /* warning: page-locking failed, the store is pageable          */
  SOUP_ERANGE = -7      /* a forward value stored as an IEEE-half operand was NaN or
                           beyond +-65504 (the half range); the results are unusable     */
};

enum { SOUP_FMT_BF16 = 0, SOUP_FMT_NF4 = 1 };

/* Projection order used by every per-projection array: index p in [0, 7). */
enum { SOUP_Q = 0, SOUP_K, SOUP_V, SOUP_O, SOUP_GATE, SOUP_UP, SOUP_DOWN, SOUP_NPROJ };
/* The four GEMM groups of a layer: projections that share an input are fused along N. */
enum { SOUP_G_QKV = 0, SOUP_G_O, SOUP_G_GU, SOUP_G_DOWN, SOUP_NGROUP };

/* Shape of a Llama-shaped decoder stack. */
typedef struct soup_cfg {
  int32_t n_layers, hidden, inter, n_heads, n_kv_heads, head_dim, vocab;
  int32_t tied;          /* 1: the output head is the embedding matrix                  */
  float rope_theta, rms_eps;
  int32_t base_fmt;      /* SOUP_FMT_BF16 or SOUP_FMT_NF4 for the streamed projections   */
  int32_t lora_r;        /* LoRA rank r, 1..64                                           */
  float lora_alpha;      /* LoRA scale s = lora_alpha / lora_r                            */
} soup_cfg;

/* Byte layout of one layer shard.  All offsets are multiples of 1024 and relative to the
 * shard's start; shards sit at multiples of `stride` in the store, in a slot and in the
 * resident array alike, so kernels see identical alignment in every mode.
 * Group g's weight section holds the group's projections stacked along the output
 * dimension (q,k,v / o / gate,up / down):
 *   NF4:  codes  uint8 [n_out[g] * n_in[g] / 2], byte j = code[2j] << 4 | code[2j+1],
 *         absmax float [n_out[g] * n_in[g] / 64], blocks of 64 over the flattened
 *         row-major [n_out, n_in] matrix (stacking keeps each projection's own blocks
 *         because every projection's element count is a multiple of 64);
 *   bf16: weights uint16 [n_out[g], n_in[g]] and no absmax section (a_bytes = 0).
 * ln1/ln2: the two RMSNorm weight vectors, bf16 [hidden]. */
typedef struct soup_shard_layout {
  uint64_t stride, payload;
  uint64_t w_off[SOUP_NGROUP], w_bytes[SOUP_NGROUP];
  uint64_t a_off[SOUP_NGROUP], a_bytes[SOUP_NGROUP];
  uint64_t ln1_off, ln2_off;
  int32_t n_out[SOUP_NGROUP], n_in[SOUP_NGROUP];
} soup_shard_layout;

typedef struct soup_store soup_store;
typedef struct soup_stream soup_stream;

/* Per-handle counters since soup_stream_init (or the last reset). Times in ms, from CUDA
 * events on the stream that ran the work; a field is 0 when its events were not enabled. */
typedef struct soup_stats {
  uint64_t steps_fwd, steps_bwd;
  uint64_t copies, copy_bytes;    /* shard copies host -> slot                              */
  double copy_ms;                 /* sum of per-copy durations on the copy stream           */
  uint64_t gemm_launches;         /* NF4/bf16 base-weight GEMM launches (profiling on)       */
  double gemm_ms;                 /* their summed durations                                 */
  double gemm_flops, gemm_bytes;  /* their algorithmic flops and bytes                      */
} soup_stats;

/* ------------------------------------------------------------------ diagnostics */

/* Message of the last failing call on this thread ("" if none). Never NULL. */
const char *soup_last_error(void);
/* Library version string. */
const char *soup_version(void);
/* Number of kernels this library has launched in this process so far (all devices). */
uint64_t soup_kernel_launches(void);

/* The 16 NF4 code values, ascending, as this library derives them (float64 construction
 * from normal quantiles, rounded once to float): "Turn it on" names NF4 without printing
 * it, so the construction follows the NormalFloat definition.  out: host float[16]. */
int soup_nf4_codebook(float *out);

/* ------------------------------------------------------------------ store (host) */

/* Fill `out` with the shard layout for cfg.  Returns SOUP_EINVAL for an invalid cfg. */
int soup_shard_layout_of(const soup_cfg *cfg, soup_shard_layout *out);

/* Quantise one tensor on the host ("How it works": the checkpoint is rewritten once into
 * one shard per layer, quantising as it goes).
 *   src:    host uint16 [n] bf16 source values (row-major flattened)
 *   codes:  host uint8  [(n + 1) / 2] out; absmax: host float [(n + 63) / 64] out.
 *   n_threads <= 0 uses all host cores.  Bit-exact with the plain definition: IEEE float
 *   divide, code = number of midpoints strictly below x / absmax, zero blocks -> code 7. */
int soup_nf4_quantize_host(const uint16_t *src, int64_t n, uint8_t *codes, float *absmax,
                           int n_threads);

/* Create an empty store of cfg.n_layers shards in ONE page-locked host arena (exact size,
 * no power-of-two rounding: the pages report rounding cost 1.73x at 14B).  If page-locking
 * fails and allow_pageable != 0, a pageable arena is used and SOUP_EPAGEABLE is returned
 * ("Measured numbers": pageable copies are synchronous and lose the overlap).
 * allow_pageable == SOUP_STORE_PAGEABLE skips page-locking altogether (returns SOUP_OK), to
 * measure what the pageable fallback costs. */
enum { SOUP_STORE_PAGEABLE = 2 };
int soup_store_create(const soup_cfg *cfg, int allow_pageable, soup_store **out);
/* Quantise (NF4) or copy (bf16) one layer into its shard.  src: host pointers to the nine
 * bf16 tensors of the layer in order q,k,v,o,gate,up,down ([out,in] each), ln1, ln2 [hidden].
 * May be called from several host threads for different layers. */
int soup_store_put_layer(soup_store *st, int layer, const uint16_t *const *src, int n_threads);
/* Fill one shard from its bytes as laid out by soup_shard_layout_of (a shard read back from
 * another store of the same cfg, or from a cache of built shards).  bytes must equal the
 * layout's stride; the store keeps its own copy.  Thread-safe for different layers. */
int soup_store_put_shard(soup_store *st, int layer, const void *shard, uint64_t bytes);
/* Put the embedding and the output head into the store, for streams in SOUP_MODE_STREAM_HEAD
 * ("Layer streaming: fine-tune a model that does not fit in your card", "Measured numbers":
 * the untied embed_tokens and lm_head move into the store and reuse one device buffer).
 *   embed: host bf16 [vocab, hidden]; lm_head: host bf16 [vocab, hidden], NULL when cfg.tied
 *   (the embedding is then the head).  The store keeps its own page-locked, device-mapped copy
 *   (SOUP_ENOMEM if page-locking fails).  May be called again to replace the tables. */
int soup_store_put_head(soup_store *st, const uint16_t *embed, const uint16_t *lm_head);
/* soup_store_create + put_layer for every layer: src is [n_layers * 9] host pointers. */
int soup_store_build(const soup_cfg *cfg, const uint16_t *const *src, int allow_pageable,
                     soup_store **out);
/* Arena base (host pointer), total bytes, and whether it is page-locked. */
int soup_store_info(const soup_store *st, void **base, uint64_t *bytes, int *pinned);
void soup_store_free(soup_store *st);

/* ------------------------------------------------------------------ memory plan */

/* Stream modes: the `mode` argument of soup_workspace_bytes, soup_peak_bytes and
 * soup_stream_init is a bit set (0 = the streamed default).
 *   SOUP_MODE_RESIDENT: every shard lives in the workspace, copied once at init; no streaming.
 *   SOUP_MODE_KEEP_ACTIVATIONS: the forward keeps every layer's activations for the backward,
 *     which then skips re-running each layer's forward but still reads every layer's weights
 *     again ("Layer streaming: fine-tune a model that does not fit in your card", "How it
 *     works": training.stream_recompute: off).  Costs one activation set per layer.
 *   SOUP_MODE_STREAM_HEAD: the embedding and the untied output head live in the store
 *     (soup_store_put_head), not in caller memory.  The device holds one vocabulary-sized
 *     buffer [vocab, hidden] bf16 inside the workspace, which the output head occupies (copied
 *     from the store at soup_stream_init); the embedding gather reads each step's rows straight
 *     from the page-locked store, so only B*S rows cross the bus ("Layer streaming: fine-tune a
 *     model that does not fit in your card", "Measured numbers": embed_tokens and lm_head move
 *     into the store and reuse one device buffer).  Results are bitwise those of a stream with
 *     resident tables (same kernels on the same bytes).
 * Other bits: SOUP_EINVAL. */
enum { SOUP_MODE_RESIDENT = 1, SOUP_MODE_KEEP_ACTIVATIONS = 2, SOUP_MODE_STREAM_HEAD = 4 };

/* Device bytes of the workspace a stream handle needs for batches up to max_batch x max_seq:
 * n_slots shard slots (or every layer in SOUP_MODE_RESIDENT), saved activations (one layer's
 * set, or every layer's in SOUP_MODE_KEEP_ACTIVATIONS), per-layer scratch, LoRA operand packs
 * and the vocabulary chunk of the loss. Writes *ws_bytes. */
int soup_workspace_bytes(const soup_cfg *cfg, int max_batch, int max_seq, int n_slots,
                         int mode, uint64_t *ws_bytes);
/* Device bytes of a whole training run: workspace + caller-side resident tensors (embedding,
 * untied head — neither in SOUP_MODE_STREAM_HEAD, where the workspace holds the one vocabulary
 * buffer — final norm, float32 LoRA A/B, their gradients and the two AdamW moments).
 * The pages bound peak VRAM by a single layer plus the resident parts ("About Soup"); this
 * is that bound made exact.  Not counted: the library's static 16 MiB array behind
 * soup_proj_fwd_noalloc, module memory resident on every device that loads the library.
 * Returns 0 for an invalid cfg or mode.  workspace_bytes (optional) receives the workspace
 * part. */
uint64_t soup_peak_bytes(const soup_cfg *cfg, int batch, int seq, int n_slots, int mode,
                         uint64_t *workspace_bytes);

/* ------------------------------------------------------------------ streamed step */

/* Bind a store to a device workspace.
 *   dev_ws / ws_bytes: caller device buffer, >= soup_workspace_bytes(), 256-B aligned.
 *   embed: dev bf16 [vocab, hidden]; lm_head: dev bf16 [vocab, hidden] or NULL when tied;
 *   both ignored (may be NULL) in SOUP_MODE_STREAM_HEAD, where the store's tables are used
 *   (SOUP_ESTATE if soup_store_put_head was never called);  final_norm: dev bf16 [hidden].
 *   compute_stream / copy_stream: distinct streams ("How it works": a dedicated copy stream).
 *   n_slots in [2, 8] ("Turn it on": stream_buffers).
 *   mode (bits above): SOUP_MODE_RESIDENT copies every shard to the workspace once here
 *   (synchronously) and then runs the same kernels with no copies — the reference the
 *   streamed run must match bit for bit.  SOUP_MODE_KEEP_ACTIVATIONS skips the backward's
 *   recompute; results are bitwise those of the recomputing stream (same kernels, same
 *   inputs).
 * Kernel paths follow from the shapes alone (so streamed and resident runs always take the
 * same ones): a projection whose reduction length (hidden, inter, n_heads * head_dim) is a
 * multiple of 256 runs on the tcgen05 GEMM, otherwise on a plain tiled CUDA-core kernel (the
 * 2-layer test stack's inter = 688 does); NF4 projections over at most 16 tokens take the
 * small-M path;
 * attention runs on tcgen05 for head_dim 64 / 128 with at most 8 query heads per kv head,
 * otherwise on the warp-level MMA kernels. */
int soup_stream_init(soup_store *st, const soup_cfg *cfg, int max_batch, int max_seq,
                     void *dev_ws, uint64_t ws_bytes, const void *embed, const void *lm_head,
                     const void *final_norm, uintptr_t compute_stream, uintptr_t copy_stream,
                     int n_slots, int mode, soup_stream **out);

/* Forward over all layers plus the vocabulary-chunked loss.
 *   tokens_dev: dev int32 [B, S], ids in [0, vocab) (ids out of range are clamped).
 *   lora_A: host array [n_layers * 7] of dev float [r, in_p]; lora_B: [n_layers * 7] of dev
 *   float [out_p, r]; p in SOUP_Q..SOUP_DOWN order.  They must stay valid until the matching
 *   soup_step_bwd has been enqueued.  Both NULL switches the adapters off: the frozen base
 *   alone over the same stream, the reference model of preference losses ("Layer streaming:
 *   fine-tune a model that does not fit in your card", opening version notes: DPO's
 *   reference model is the streamed base with its adapters switched off); soup_step_bwd then
 *   returns SOUP_ESTATE until a forward with adapters.  One NULL and one not: SOUP_EINVAL.
 *   loss_dev: dev float [1], mean next-token cross-entropy over B*(S-1) positions.
 *   logits_dev (optional, NULL in timed runs): dev float [B*S, vocab].
 *   layer_out_dev (optional): dev float [(n_layers + 1), B*S, hidden] — the residual stream
 *   entering each layer and leaving the last.
 * B*S must be <= max_batch*max_seq, S <= max_seq, S >= 2. */
int soup_step_fwd(soup_stream *h, const int32_t *tokens_dev, int B, int S,
                  const float *const *lora_A, const float *const *lora_B, float *loss_dev,
                  float *logits_dev, float *layer_out_dev);

/* Backward of the last forward: re-streams the layers in reverse, recomputes each layer's
 * forward, and writes every LoRA gradient (overwritten, not accumulated).
 *   dA: host array [n_layers * 7] of dev float [r, in_p]; dB: [n_layers * 7] of dev float
 *   [out_p, r].  dh_out_dev (optional): dev float [(n_layers + 1), B*S, hidden], dL/dh of the
 *   residual stream at each layer boundary.  SOUP_ESTATE without a preceding forward. */
int soup_step_bwd(soup_stream *h, float *const *dA, float *const *dB, float *dh_out_dev);

/* soup_step_bwd with flags.  SOUP_BWD_ACCUMULATE adds this step's LoRA gradients to the ones
 * already in dA/dB instead of overwriting them (gradient accumulation over micro-batches,
 * "Layer streaming: fine-tune a model that does not fit in your card", "Full config":
 * gradient_accumulation_steps).  Each element becomes old + g in one float addition, where g
 * is exactly the value soup_step_bwd would have written, so accumulating k micro-batches
 * equals summing k separately computed gradients in float, left to right, bit for bit.
 * flags = 0 is soup_step_bwd.  Unknown flag bits: SOUP_EINVAL. */
enum { SOUP_BWD_ACCUMULATE = 1 };
int soup_step_bwd_ex(soup_stream *h, float *const *dA, float *const *dB, float *dh_out_dev,
                     int flags);

/* Host-side bounded wait for all work enqueued on the handle: polls, never spins on the
 * device.  Returns SOUP_ETIMEDOUT after timeout_ms (timeout_ms = 0: only asks whether the work
 * is done; < 0: no limit), or the error the kernels reported since the last soup_sync that
 * returned: SOUP_ETIMEDOUT if a kernel's bounded wait gave up, SOUP_ERANGE if a forward
 * operand left the half range ("Layer streaming: fine-tune a model that does not fit in
 * your card", "Troubleshooting": a read that wedges is given up after a bounded wait and
 * reported, not waited on forever).  Reading the kernels' error flag clears it. */
int soup_sync(soup_stream *h, int timeout_ms);
int soup_stream_stats(soup_stream *h, soup_stats *out, int reset);

/* Time spent per kernel family of the step, measured with CUDA events around each group of
 * launches on the compute stream while SOUP_DBG_PROFILE is 2 (events add a little overhead, so
 * time a run with it off for throughput).  flops / bytes: the family's algorithmic work over
 * those launches (the operands and results each kernel must read and write once, not the
 * traffic it causes); tensor_bound: 1 where the family is a tensor-core contraction (its
 * roofline is the tensor pipe), 0 where it is bound by memory bandwidth. */
typedef struct soup_kernel_stat {
  char name[32];
  int32_t tensor_bound;
  uint64_t launches;   /* launch groups timed (one event pair each) */
  double ms, flops, bytes;
} soup_kernel_stat;
/* Writes up to `max` families that ran since the last reset (in a fixed order) and sets *n to
 * how many there are; reset != 0 clears the counters.  Waits for the timed work. */
int soup_stream_kernel_stats(soup_stream *h, soup_kernel_stat *out, int max, int *n, int reset);
/* Debug switches: what =
 *   SOUP_DBG_PROFILE        1: time every base GEMM with events (soup_stream_stats);
 *                           2: also time every kernel family (soup_stream_kernel_stats); 0: off;
 *   SOUP_DBG_STALE_SLOT     backward reads the slot of a neighbouring layer: a deliberately
 *                           broken control that the exactness tests must catch; reads valid
 *                           memory only (value 0/1);
 *   SOUP_DBG_COPY_DELAY_US  the host sleeps `value` microseconds (0..1e6) before enqueueing
 *                           each shard copy: changes timing only, never results;
 *   SOUP_DBG_WAIT_PROBE     enqueues, on the compute stream, one kernel whose bounded wait
 *                           on a barrier that nothing signals gives up after about `value`
 *                           microseconds (1..1e6) and raises the kernels' error flag, so the
 *                           next soup_sync returns SOUP_ETIMEDOUT — the failure path of
 *                           "Troubleshooting" (a wedged read is given up and reported),
 *                           exercised without a real stall; the stream stays usable. */
enum { SOUP_DBG_PROFILE = 1, SOUP_DBG_STALE_SLOT = 2, SOUP_DBG_COPY_DELAY_US = 3,
       SOUP_DBG_WAIT_PROBE = 4 };
int soup_stream_debug(soup_stream *h, int what, int value);
void soup_stream_free(soup_stream *h);

/* ------------------------------------------------------------------ single projection */

/* One projection of the step, for the microbench and the kernel tests.  W is a weight
 * [N, K] (out x in) given as NF4 (codes dev uint8 [N*K/2] + absmax dev float [N*K/64]) or
 * bf16 (w_bf16 dev uint16 [N, K]; codes/absmax NULL).  LoRA: A dev float [r, K],
 * B dev float [N, r], s = alpha / r, 0 <= r <= 64 (r = 0: no adapter, A and B may be NULL;
 * the plain dequant GEMM, used to time the kernel alone).  scratch: dev buffer of
 * soup_proj_scratch_bytes() bytes, 256-byte aligned, owned by the caller; its contents are
 * overwritten.  Shapes: any M >= 1; the tensor-core path needs K % 256 == 0 (both
 * directions) and N % 64 == 0 for dX; other shapes use a plain tiled kernel.
 * 16-bit operand format: x_f16 != 0 means x (and y) are IEEE half and the GEMM runs on half
 * operands (the step's forward); 0 means bf16.  dY and dx of the backward are bf16 / float. */
int soup_proj_scratch_bytes(int M, int N, int K, int r, uint64_t *bytes);

/* y[M, N] (16-bit out, dev uint16) = x W^T + s (x A^T) B^T,  x: dev 16-bit [M, K].
 * "Layer streaming: fine-tune a model that does not fit in your card", "How it works": the
 * projection runs on the streamed weight bytes; the weights are dequantised in the kernel. */
int soup_proj_fwd(const uint16_t *x, int M, int N, int K, const uint8_t *codes,
                  const float *absmax, const uint16_t *w_bf16, const float *A, const float *B,
                  int r, float s, int x_f16, uint16_t *y, void *scratch, uint64_t scratch_bytes,
                  uintptr_t stream);
/* dx[M, K] (float out) = dY W + s (dY B) A,  dY: dev bf16 [M, N].  "How it works": the
 * backward needs W^T dL/dy; the dequantisation is redone inside the GEMM, never cached. */
int soup_proj_dx(const uint16_t *dy, int M, int N, int K, const uint8_t *codes,
                 const float *absmax, const uint16_t *w_bf16, const float *A, const float *B,
                 int r, float s, float *dx, void *scratch, uint64_t scratch_bytes,
                 uintptr_t stream);
/* dA[r, K] = s (dY B)^T x,  dB[N, r] = s dY^T (x A^T); float outputs, fixed summation order.
 * x: dev 16-bit [M, K] (half if x_f16), dY: dev bf16 [M, N]. */
int soup_proj_lora_grad(const uint16_t *x, const uint16_t *dy, int M, int N, int K,
                        const float *A, const float *B, int r, float s, int x_f16, float *dA,
                        float *dB, void *scratch, uint64_t scratch_bytes, uintptr_t stream);

/* Status of the projections that used `scratch` (same M, N, K as those calls): waits for
 * `stream`, reads the scratch's device error flag, clears it, and returns SOUP_OK,
 * SOUP_ETIMEDOUT if a kernel's bounded wait gave up, or SOUP_ERANGE if a half-precision
 * forward value overflowed (the outputs are unusable in both cases).  The flag lives in the
 * scratch: zero-fill a new scratch buffer (or pass it here once) before relying on the
 * result. */
int soup_proj_status(void *scratch, int M, int N, int K, uintptr_t stream);

/* soup_proj_fwd without caller-provided scratch, for callers that cannot allocate device
 * memory (a host application that owns the whole device-memory budget, or a latency-critical
 * caller that cannot take cudaMalloc's implicit synchronisation).  The pages have no
 * counterpart: this is a deployment convenience, same arguments and result as soup_proj_fwd
 * minus the scratch pair.
 *   Working memory comes from one static 16 MiB device array inside the library, reserved on
 *   every GPU that loads it until the process exits.  A call needing more (large M or N) is
 *   rejected with SOUP_EINVAL before anything is enqueued.  The first call on a device looks up
 *   the array's address (cudaGetSymbolAddress); make it before any stream capture there.
 *   Every call shares the array and it keeps the last call's contents: calls whose GPU work
 *   overlaps race on it, so issue them in order on one stream.  No split-K partials are used,
 *   so results can differ from soup_proj_fwd by float summation order.
 *   Allocates nothing (no cudaMalloc / cudaFree). */
int soup_proj_fwd_noalloc(const uint16_t *x, int M, int N, int K, const uint8_t *codes,
                          const float *absmax, const uint16_t *w_bf16, const float *A,
                          const float *B, int r, float s, int x_f16, uint16_t *y,
                          uintptr_t stream);
/* Status of the soup_proj_fwd_noalloc calls on the current device: waits for `stream`, reads
 * the error flag those calls share (it sits at a fixed place in the static array and collects
 * the error bits of every call since it was last read), clears it, and returns SOUP_OK,
 * SOUP_ETIMEDOUT (a kernel's bounded wait gave up) or SOUP_ERANGE (a half-precision value
 * overflowed); the outputs of the calls since the last read are then unusable.  Call it on
 * the stream the calls ran on, after them.  The pages have no counterpart.  Allocates
 * nothing; like the first call, its first use on a device looks up the array's address. */
int soup_proj_noalloc_status(uintptr_t stream);

/* ------------------------------------------------------------------ attention, on its own */

/* Causal grouped-query attention of one decoder layer, the kernels the step runs ("Layer
 * streaming: fine-tune a model that does not fit in your card", "How it works": the family's
 * own decoder layer, run unchanged): query head h reads key/value head floor(h * n_kv / n_h),
 *   o = softmax(q k^T / sqrt(d) + causal mask) v,
 * per sequence b of B and head, over S positions.
 *   qkv: dev IEEE half [B * S, (n_heads + 2 n_kv_heads) * head_dim], row b * S + t holds the
 *        q heads, then the k heads, then the v heads of position t (rotary embedding already
 *        applied), 16-byte aligned.
 *   o:   dev half [B * S, n_heads * head_dim] (written);
 *   lse: dev float [B, n_heads, S] (written): log2 of the row's sum of exp2(score * log2(e)
 *        / sqrt(d) - max) plus the max, in base-2 units of the scaled score.
 *   err: dev int the kernels OR error bits into (1: a bounded wait gave up; 4 is not used
 *        here), or NULL.  head_dim 64 or 128; n_heads a multiple of n_kv_heads.  With
 *        head_dim 64 or 128 and at most 8 query heads per key/value head the tcgen05 kernels
 *        run; otherwise the warp-level MMA kernels.  B == 0 or S == 0 does nothing.
 * Asynchronous on `stream`; SOUP_EINVAL for bad shapes or NULL buffers. */
int soup_attn_fwd(const uint16_t *qkv, int B, int S, int n_heads, int n_kv_heads, int head_dim,
                  uint16_t *o, float *lse, int *err, uintptr_t stream);
/* Scratch soup_attn_bwd needs for this shape (0 for a bad shape). */
uint64_t soup_attn_bwd_scratch_bytes(int B, int S, int n_heads, int n_kv_heads, int head_dim);
/* Backward of soup_attn_fwd: dqkv (dev float [B * S, (n_heads + 2 n_kv_heads) * head_dim],
 * written completely) = dL/dq, dL/dk, dL/dv in qkv's layout, from the forward's qkv, o and lse
 * and dO = dL/do (dev bf16 [B * S, n_heads * head_dim]).  The probabilities are recomputed from
 * half q, k and lse; every product with a gradient is formed from bf16 operands with float
 * accumulation.  Deterministic: the key/value gradients of the query heads that share a
 * key/value head are summed in head order.  scratch: dev, 256-byte aligned, at least
 * soup_attn_bwd_scratch_bytes; err as for soup_attn_fwd.  Asynchronous on `stream`. */
int soup_attn_bwd(const uint16_t *qkv, const uint16_t *o, const uint16_t *dO, const float *lse, int B,
                  int S, int n_heads, int n_kv_heads, int head_dim, void *scratch,
                  uint64_t scratch_bytes, float *dqkv, int *err, uintptr_t stream);

/* ------------------------------------------------------------------ optimizer */

/* AdamW hyper-parameters.  grad_scale multiplies the gradient before it enters the moments
 * (1/k after accumulating k micro-batches). */
typedef struct soup_adamw {
  float lr, beta1, beta2, eps, weight_decay, grad_scale;
} soup_adamw;

/* One AdamW step over n float parameters in place (the pages' runs train the adapters with
 * an AdamW, "Layer streaming: fine-tune a model that does not fit in your card", "Measured
 * numbers"; here with float32 state).  With g = grad_scale * grad[i] and step number t >= 1:
 *   m = beta1 m + (1 - beta1) g;  v = beta2 v + (1 - beta2) g^2
 *   p = p - lr weight_decay p - lr (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps)
 * (Adam's bias-corrected moments, Kingma & Ba; decay decoupled from the gradient, Loshchilov
 * & Hutter).  param, m, v: dev float [n], updated in place; grad: dev float [n], read only.
 * The four buffers must not overlap; any alignment is accepted (16-byte aligned buffers take
 * the vectorised path).  m and v start at zero for t = 1.  One kernel launch on `stream`;
 * n = 0 enqueues nothing.  SOUP_EINVAL for NULL pointers, n < 0, t < 1 or beta outside
 * [0, 1). */
int soup_adamw_step(float *param, const float *grad, float *m, float *v, int64_t n,
                    const soup_adamw *hp, int64_t step, uintptr_t stream);

/* Dequantise n NF4 weights on the device: out_f32[i] = float(c[code_i] * absmax[i / 64])
 * and out_bf16[i] = that value rounded to nearest-even bf16 (either output may be NULL). */
int soup_nf4_dequant(const uint8_t *codes, const float *absmax, int64_t n, float *out_f32,
                     uint16_t *out_bf16, uintptr_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SOUP_H */
