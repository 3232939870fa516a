// Internal state of a stream handle and the workspace plan (opaque to C callers).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "soup.h"

namespace soup {

// Byte offsets of every buffer inside the caller's device workspace.
struct Plan {
  uint64_t total = 0;
  int n_slots = 0, vc = 0;
  uint64_t slots = 0, h_all = 0, hm = 0, x1 = 0, x2 = 0, qkv = 0, att = 0, lse = 0, gu = 0, act = 0;
  uint64_t u_f32[4] = {0, 0, 0, 0}, u_b[4] = {0, 0, 0, 0};
  uint64_t dh = 0, dhm = 0, dh_b = 0, dhm_b = 0, dact = 0, dgu = 0, dx = 0, datt = 0, datt_b = 0;
  uint64_t dqkv = 0, dqkv_b = 0, attn_scratch = 0, du_b = 0, lora_part = 0;
  uint64_t du_f32[4] = {0, 0, 0, 0};  // s dY B per group, kept for the layer's gradient launch
  uint64_t hn = 0, z = 0, dz = 0, dhn = 0, ce_max = 0, ce_sum = 0, ce_lab = 0, ce_lse = 0;
  std::vector<uint64_t> vl, ac;  // per (layer, group) LoRA operand packs
  uint64_t rope_cos = 0, rope_sin = 0, err = 0;
  uint64_t vocab_buf = 0;  // SOUP_MODE_STREAM_HEAD: the one vocabulary-sized table buffer
  uint64_t gemm_part = 0, gemm_part_floats = 0;
  // keep-activations mode: hm .. u_b[3] repeat once per layer at this stride (0 otherwise)
  uint64_t act_stride = 0;
};

// A shard moves between the store and a slot in four chunks, one per GEMM group (its weight
// section and, for q|k|v and gate|up, the norm vector read just before it), each with its own
// events: a chunk's copy waits only for the last kernel that read that chunk of the slot's
// previous layer, and a kernel waits only for the chunk it reads.
constexpr int NCHUNK = SOUP_NGROUP;

struct Slot {
  uint8_t *dev = nullptr;
  int layer = -1;                // layer held (or being copied in); -1 = empty
  int pending[NCHUNK] = {};      // a chunk copy was issued and compute has not waited on it yet
  uint64_t tick = 0;             // release order, for least-recently-used tie breaks
  int has_events = 0;
  cudaEvent_t ready[NCHUNK] = {};  // RAW: recorded on the copy stream after the chunk's copy
  cudaEvent_t freed[NCHUNK] = {};  // WAR: recorded on the compute stream after its last reader
};

// Kernel families of the step, each timed as a group of launches in profiling mode 2.
enum Fam : int {
  FAM_EMBED, FAM_RMSNORM_FWD, FAM_RMSNORM_BWD, FAM_ROPE_FWD, FAM_ROPE_BWD, FAM_SWIGLU_FWD,
  FAM_SWIGLU_BWD, FAM_ATTN_FWD, FAM_ATTN_BWD, FAM_CAST, FAM_LORA_PACK, FAM_LORA_DOWN, FAM_LORA_DU,
  FAM_LORA_GRAD, FAM_GEMM_FWD_QKV, FAM_GEMM_FWD_O, FAM_GEMM_FWD_GU, FAM_GEMM_FWD_DOWN,
  FAM_GEMM_DX_QKV, FAM_GEMM_DX_O, FAM_GEMM_DX_GU, FAM_GEMM_DX_DOWN, FAM_HEAD_GEMM, FAM_HEAD_DX,
  FAM_CE_FWD, FAM_CE_BWD, FAM_COUNT
};
extern const char *const kFamName[FAM_COUNT];
extern const int kFamTensor[FAM_COUNT];  // 1: tensor-pipe bound, 0: memory bound

struct TimedEv {
  cudaEvent_t start = nullptr, end = nullptr;
  double flops = 0, bytes = 0;
  int fam = -1;  // kernel family (-1: a shard copy)
};
struct FamStat {
  uint64_t launches = 0;
  double ms = 0, flops = 0, bytes = 0;
};

// mode: SOUP_MODE_RESIDENT | SOUP_MODE_KEEP_ACTIVATIONS bits (soup.h)
int make_plan(const soup_cfg *c, int maxB, int maxS, int n_slots, int mode, Plan *P);
int ce_chunk_cols(int M, int V);

}  // namespace soup

struct soup_stream {
  soup_cfg cfg;
  soup_shard_layout lay;
  soup_store *store = nullptr;
  soup::Plan plan;
  int maxB = 0, maxS = 0, resident = 0;
  int keep_act = 0;  // every layer's activations stay from the forward; no recompute
  int stream_head = 0;  // embedding gathered from the store; head table in the workspace buffer
  cudaStream_t cs = nullptr, xs = nullptr;
  uint8_t *ws = nullptr;
  const uint16_t *embed = nullptr, *lm_head = nullptr, *final_norm = nullptr;
  int *err_dev = nullptr;
  std::vector<soup::Slot> slot;
  uint64_t tick = 0;
  cudaEvent_t done = nullptr;
  // per-step state
  int B = 0, S = 0, fwd_ready = 0, in_bwd = 0;
  int last_layer_fresh = 0;  // set by step_fwd: the last layer's activations are intact
  const int32_t *tokens = nullptr;
  std::vector<const float *> lora_A, lora_B;
  std::vector<float *> grad_A, grad_B;
  int grad_accumulate = 0;  // this backward adds to grad_A/grad_B (SOUP_BWD_ACCUMULATE)
  int adapters_off = 0;     // the last forward ran without adapters (lora_A = lora_B = NULL)
  // measurement
  soup_stats stats{};
  std::vector<soup::TimedEv> copy_ev, gemm_ev, fam_ev;
  soup::FamStat fam[soup::FAM_COUNT];
  std::vector<cudaEvent_t> ev_pool;  // timing events whose measurement was harvested, for reuse
  int dbg_profile = 0, dbg_stale = 0;
  int dbg_copy_delay_us = 0;  // host sleep before each shard copy is enqueued (timing only)
};

namespace soup {
int stream_init(soup_store *st, const soup_cfg *c, int maxB, int maxS, void *ws, uint64_t ws_bytes,
                const void *embed, const void *lm_head, const void *final_norm, uintptr_t cs,
                uintptr_t xs, int n_slots, int mode, soup_stream **out);
int step_fwd(soup_stream *h, const int32_t *tokens, int B, int S, const float *const *lA,
             const float *const *lB, float *loss, float *logits, float *layer_out);
int step_bwd(soup_stream *h, float *const *dA, float *const *dB, float *dh_out, int flags);
int stream_sync(soup_stream *h, int timeout_ms);
int stream_stats(soup_stream *h, soup_stats *out, int reset);
int stream_kernel_stats(soup_stream *h, soup_kernel_stat *out, int max, int *n, int reset);
void soup_stream_free_impl(soup_stream *h);
}  // namespace soup
