// The streamed LoRA step: workspace plan, slot scheduling on a dedicated copy stream, and
// the per-layer forward / recompute / backward built from the library's kernels.
//
// "About Soup" and "Layer streaming: fine-tune a model that does not fit in your card",
// "How it works": each decoder layer is copied into one of N pre-allocated device buffers
// on a dedicated stream so the load of the next layer overlaps the compute of the current
// one; the same kernels run on the same weight bytes as a resident run; each layer is read
// twice per step because the backward recomputes the layer and needs W^T dL/dy.
// "Read this first": above ~165 MiB per layer the pages' stack read a buffer that had
// already been refilled with another layer.  Here every use of a slot is ordered by two
// events: `ready` (copy -> compute, recorded after the copy) and `freed` (compute -> copy,
// recorded after the last kernel that reads the slot); a copy into a slot waits on that
// slot's `freed`, and no kernel keeps a weight pointer beyond its own launch.
#include "step.h"

#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <thread>

#include "gemm.h"
#include "kernels.h"
#include "store.h"
#include "util.h"

namespace soup {

const char *const kFamName[FAM_COUNT] = {
    "embed", "rmsnorm_fwd", "rmsnorm_bwd", "rope_fwd", "rope_bwd", "swiglu_fwd", "swiglu_bwd",
    "attn_fwd", "attn_bwd", "cast_bf16", "lora_pack", "lora_down", "lora_du", "lora_grad",
    "gemm_fwd_qkv", "gemm_fwd_o", "gemm_fwd_gate_up", "gemm_fwd_down", "gemm_dx_qkv", "gemm_dx_o",
    "gemm_dx_gate_up", "gemm_dx_down", "head_gemm", "head_dx", "ce_fwd", "ce_bwd"};
const int kFamTensor[FAM_COUNT] = {0, 0, 0, 0, 0, 0, 0, 1, 1, 0, 0, 0, 0, 0,
                                   1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 0, 0};

static uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

// A named host-side range on a profiler's timeline (NVTX); costs nothing without a profiler.
struct TraceRange {
  explicit TraceRange(const char *name, int index = -1) {
    char buf[48];
    if (index >= 0) std::snprintf(buf, sizeof buf, "%s %d", name, index);
    else std::snprintf(buf, sizeof buf, "%s", name);
    nvtxRangePushA(buf);
  }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange &) = delete;
  TraceRange &operator=(const TraceRange &) = delete;
};

int ce_chunk_cols(int M, int V) {
  int vc = (int)((1ull << 24) / (uint64_t)std::max(M, 1) / 256ull) * 256;
  vc = std::max(256, std::min(vc, 32768));
  if (vc >= V) vc = (int)align_up((uint64_t)(V + 1) / 2, 256);  // at least two chunks
  return std::max(vc, 256);
}

int make_plan(const soup_cfg *c, int maxB, int maxS, int n_slots, int mode, Plan *P) {
  SOUP_TRY(validate_cfg(c));
  if (mode & ~(SOUP_MODE_RESIDENT | SOUP_MODE_KEEP_ACTIVATIONS | SOUP_MODE_STREAM_HEAD))
    return set_error(SOUP_EINVAL, "unknown stream mode bits 0x%x", mode);
  const bool resident = (mode & SOUP_MODE_RESIDENT) != 0;
  if (maxB < 1 || maxS < 2) return set_error(SOUP_EINVAL, "max_batch >= 1 and max_seq >= 2 required");
  if (!resident && (n_slots < 2 || n_slots > 8)) return set_error(SOUP_EINVAL, "n_slots must be in [2, 8]");
  soup_shard_layout L;
  SOUP_TRY(shard_layout(c, &L));
  *P = Plan();
  const uint64_t M = (uint64_t)maxB * maxS, H = c->hidden, I = c->inter;
  const uint64_t qd = (uint64_t)c->n_heads * c->head_dim, kvd = (uint64_t)c->n_kv_heads * c->head_dim;
  const uint64_t nqkv = qd + 2 * kvd;
  uint64_t off = 0;
  auto take = [&](uint64_t bytes) {
    const uint64_t o = off;
    off = align_up(off + std::max<uint64_t>(bytes, 1), 1024);
    return o;
  };
  P->n_slots = resident ? c->n_layers : n_slots;
  P->slots = take(L.stride * (uint64_t)P->n_slots);
  P->h_all = take(4 * (c->n_layers + 1ull) * M * H);
  P->hm = take(4 * M * H);
  P->x1 = take(2 * M * H);
  P->x2 = take(2 * M * H);
  P->qkv = take(2 * M * nqkv);
  P->att = take(2 * M * qd);
  P->lse = take(4 * M * c->n_heads);
  P->gu = take(4 * M * I);
  P->act = take(2 * M * I);
  for (int g = 0; g < 4; ++g) {
    P->u_f32[g] = take(4 * M * 64);
    P->u_b[g] = take(2 * M * 64);
  }
  if (mode & SOUP_MODE_KEEP_ACTIVATIONS) {  // layers 1 .. L-1 get their own copies
    P->act_stride = off - P->hm;
    take(P->act_stride * (uint64_t)(c->n_layers - 1));
  }
  P->dh = take(4 * M * H);
  P->dhm = take(4 * M * H);
  P->dh_b = take(2 * M * H);
  P->dhm_b = take(2 * M * H);
  P->dact = take(4 * M * I);
  P->dgu = take(4 * M * I);
  P->dx = take(4 * M * H);
  P->datt = take(4 * M * qd);
  P->datt_b = take(2 * M * qd);
  P->dqkv = take(4 * M * nqkv);
  P->dqkv_b = take(2 * M * nqkv);
  P->attn_scratch = take(4 * attn_bwd_scratch_floats(maxB, maxS, c->n_heads, c->n_kv_heads, c->head_dim));
  for (int g = 0; g < 4; ++g) P->du_f32[g] = take(4 * M * 64);
  P->du_b = take(2 * M * 64);
  {
    const int dims[5] = {(int)H, (int)qd, (int)I, (int)nqkv, (int)(2 * I)};
    size_t mx = 0;
    for (int k : dims) mx = std::max(mx, lora_scratch_floats((int)M, k, 3 * c->lora_r));
    P->lora_part = take(4 * mx);
  }
  // split-K partial tiles for the base GEMMs whose output grid under-fills the GPU (and the
  // small-M path's partial strips)
  P->gemm_part_floats = 4ull * M * std::max<uint64_t>(std::max(nqkv, H), std::max(qd, (uint64_t)I));
  P->gemm_part = take(4 * P->gemm_part_floats);
  P->hn = take(2 * M * H);
  P->vc = ce_chunk_cols((int)M, c->vocab);
  P->z = take(4 * M * (uint64_t)P->vc);
  P->dz = take(2 * M * (uint64_t)P->vc);
  P->dhn = take(4 * M * H);
  P->ce_max = take(4 * M);
  P->ce_sum = take(4 * M);
  P->ce_lab = take(4 * M);
  P->ce_lse = take(4 * M);
  const int r = c->lora_r;
  const int nseg[4] = {3, 1, 2, 1};
  P->vl.resize((size_t)c->n_layers * 4);
  P->ac.resize((size_t)c->n_layers * 4);
  for (int l = 0; l < c->n_layers; ++l)
    for (int g = 0; g < 4; ++g) {
      const uint64_t rp = align_up((uint64_t)nseg[g] * r, 64);
      P->vl[(size_t)l * 4 + g] = take(2 * (uint64_t)L.n_out[g] * rp);
      P->ac[(size_t)l * 4 + g] = take(2 * rp * (uint64_t)L.n_in[g]);
    }
  P->rope_cos = take(4ull * maxS * (c->head_dim / 2));
  P->rope_sin = take(4ull * maxS * (c->head_dim / 2));
  P->err = take(64);
  if (mode & SOUP_MODE_STREAM_HEAD) P->vocab_buf = take(2ull * c->vocab * H);
  P->total = off;
  return 0;
}

// ------------------------------------------------------------------------------------------
namespace {

inline float *F(soup_stream *h, uint64_t off) { return reinterpret_cast<float *>(h->ws + off); }
inline uint16_t *B16(soup_stream *h, uint64_t off) { return reinterpret_cast<uint16_t *>(h->ws + off); }

int check_cuda(const char *what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(SOUP_ECUDA, "%s: %s", what, cudaGetErrorString(e));
  return 0;
}

void harvest(soup_stream *h, bool block) {
  auto run = [&](std::vector<TimedEv> &v, double *ms_sum, uint64_t *count, double *flops,
                 double *bytes) {
    size_t keep = 0;
    for (size_t i = 0; i < v.size(); ++i) {
      TimedEv &e = v[i];
      cudaError_t q = block ? cudaEventSynchronize(e.end) : cudaEventQuery(e.end);
      if (q == cudaSuccess) {
        float ms = 0.f;
        cudaEventElapsedTime(&ms, e.start, e.end);
        if (ms_sum) *ms_sum += ms;
        if (count) ++*count;
        if (flops) *flops += e.flops;
        if (bytes) *bytes += e.bytes;
        if (e.fam >= 0) {
          FamStat &f = h->fam[e.fam];
          f.launches += 1;
          f.ms += ms;
          f.flops += e.flops;
          f.bytes += e.bytes;
        }
        h->ev_pool.push_back(e.start);  // reused by the next timed launch or copy
        h->ev_pool.push_back(e.end);
      } else {
        if (q != cudaErrorNotReady) (void)cudaGetLastError();
        v[keep++] = e;
      }
    }
    v.resize(keep);
  };
  run(h->copy_ev, &h->stats.copy_ms, nullptr, nullptr, nullptr);
  run(h->gemm_ev, &h->stats.gemm_ms, &h->stats.gemm_launches, &h->stats.gemm_flops,
      &h->stats.gemm_bytes);
  run(h->fam_ev, nullptr, nullptr, nullptr, nullptr);
}

// A pair of timing events for one launch or copy: from the pool of harvested ones when it has
// any (no event creation on the hot path after the first step), else new ones.
int take_events(soup_stream *h, TimedEv *e) {
  for (cudaEvent_t *ev : {&e->start, &e->end}) {
    if (!h->ev_pool.empty()) {
      *ev = h->ev_pool.back();
      h->ev_pool.pop_back();
    } else {
      SOUP_CUDA_TRY(cudaEventCreate(ev));
    }
  }
  return 0;
}

// Profiling mode 2: one event pair around a group of launches of one kernel family, with the
// group's algorithmic flops and bytes.  Costs nothing when profiling is off.
template <class Fn>
int prof(soup_stream *h, int fam, double flops, double bytes, Fn &&fn) {
  if (h->dbg_profile < 2) {
    fn();
    return 0;
  }
  TimedEv e;
  e.flops = flops;
  e.bytes = bytes;
  e.fam = fam;
  SOUP_TRY(take_events(h, &e));
  SOUP_CUDA_TRY(cudaEventRecord(e.start, h->cs));
  fn();
  SOUP_CUDA_TRY(cudaEventRecord(e.end, h->cs));
  h->fam_ev.push_back(e);
  return 0;
}

// The step's split-K scratch for a GEMM (partial tiles) and its error flag.
void gemm_scratch(soup_stream *h, GemmArgs &g) {
  g.err = h->err_dev;
  g.part = F(h, h->plan.gemm_part);
  g.part_floats = h->plan.gemm_part_floats;
}

// A base-weight GEMM of group `grp` (forward or dX), timed in profiling modes 1 and 2.
int timed_gemm(soup_stream *h, GemmArgs &g, int grp) {
  gemm_scratch(h, g);
  if (!h->dbg_profile) return gemm_launch(g, h->cs);
  TimedEv e;
  e.flops = gemm_flops(g);
  e.bytes = gemm_bytes(g);
  e.fam = (g.mode == GEMM_FWD ? FAM_GEMM_FWD_QKV : FAM_GEMM_DX_QKV) + grp;
  SOUP_TRY(take_events(h, &e));
  SOUP_CUDA_TRY(cudaEventRecord(e.start, h->cs));
  int rc = gemm_launch(g, h->cs);
  SOUP_CUDA_TRY(cudaEventRecord(e.end, h->cs));
  h->gemm_ev.push_back(e);
  return rc;
}

// Weight operand of group g inside a shard (slot, resident array, or any device copy).
GemmArgs weight_args(soup_stream *h, const uint8_t *shard, int g, int mode) {
  GemmArgs a;
  a.mode = mode;
  const soup_shard_layout &L = h->lay;
  a.Nw = L.n_out[g];
  a.Kw = L.n_in[g];
  if (h->cfg.base_fmt == SOUP_FMT_NF4) {
    a.wfmt = W_NF4;
    a.codes = shard + L.w_off[g];
    a.absmax = reinterpret_cast<const float *>(shard + L.a_off[g]);
  } else {
    a.wfmt = W_BF16;
    a.w = reinterpret_cast<const uint16_t *>(shard + L.w_off[g]);
  }
  return a;
}

LoraSeg make_seg(soup_stream *h, int layer, int g, bool grads) {
  const soup_cfg &c = h->cfg;
  LoraSeg L;
  L.r = c.lora_r;
  L.s = c.lora_alpha / (float)c.lora_r;
  static const int first[4] = {SOUP_Q, SOUP_O, SOUP_GATE, SOUP_DOWN};
  static const int nseg[4] = {3, 1, 2, 1};
  L.nseg = nseg[g];
  const int qd = c.n_heads * c.head_dim, kvd = c.n_kv_heads * c.head_dim;
  int sizes[7] = {qd, kvd, kvd, c.hidden, c.inter, c.inter, c.hidden};
  int off = 0;
  for (int p = 0; p < L.nseg; ++p) {
    const int proj = first[g] + p;
    const size_t idx = (size_t)layer * 7 + proj;
    L.off[p] = off;
    L.n[p] = sizes[proj];
    off += sizes[proj];
    if (!h->adapters_off) {
      L.A[p] = h->lora_A[idx];
      L.B[p] = h->lora_B[idx];
    }
    if (grads) {
      L.dA[p] = h->grad_A[idx];
      L.dB[p] = h->grad_B[idx];
    }
  }
  L.accumulate = grads && h->grad_accumulate;
  return L;
}

// ---------------------------------------------------------------- slot scheduling
// Next position >= from at which `layer` is used in seq (INT32_MAX if never).
int next_use(const std::vector<int> &seq, size_t from, int layer) {
  for (size_t j = from; j < seq.size(); ++j)
    if (seq[j] == layer) return (int)j;
  return INT32_MAX;
}

// Byte ranges of chunk g inside a shard: the group's weight section (codes and absmax are
// adjacent) and, for q|k|v and gate|up, the norm vector the layer reads just before that GEMM.
int chunk_ranges(const soup_shard_layout &L, int hidden, int g, uint64_t off[2], uint64_t len[2]) {
  const uint64_t end = L.a_bytes[g] ? L.a_off[g] + L.a_bytes[g] : L.w_off[g] + L.w_bytes[g];
  off[0] = L.w_off[g];
  len[0] = end - L.w_off[g];
  if (g == SOUP_G_QKV || g == SOUP_G_GU) {
    off[1] = g == SOUP_G_QKV ? L.ln1_off : L.ln2_off;
    len[1] = 2ull * hidden;
    return 2;
  }
  return 1;
}

// Copy `layer` into `slot`, chunk by chunk in the order the layer reads them (q|k|v, o,
// gate|up, down: the forward's order, and the backward's recompute's).
int issue_copy(soup_stream *h, int slot, int layer) {
  Slot &s = h->slot[slot];
  // an injected host-side delay before the copy is enqueued may change timing, never results
  if (h->dbg_copy_delay_us) std::this_thread::sleep_for(std::chrono::microseconds(h->dbg_copy_delay_us));
  const uint8_t *src = h->store->base + (uint64_t)layer * h->lay.stride;
  for (int g = 0; g < NCHUNK; ++g) {
    uint64_t off[2], len[2];
    const int n = chunk_ranges(h->lay, h->cfg.hidden, g, off, len);
    SOUP_CUDA_TRY(cudaStreamWaitEvent(h->xs, s.freed[g], 0));  // WAR: last reader of the chunk done
    TimedEv e;
    for (int k = 0; k < n; ++k) e.bytes += (double)len[k];
    SOUP_TRY(take_events(h, &e));
    SOUP_CUDA_TRY(cudaEventRecord(e.start, h->xs));
    for (int k = 0; k < n; ++k)
      SOUP_CUDA_TRY(cudaMemcpyAsync(s.dev + off[k], src + off[k], len[k], cudaMemcpyHostToDevice, h->xs));
    SOUP_CUDA_TRY(cudaEventRecord(e.end, h->xs));
    SOUP_CUDA_TRY(cudaEventRecord(s.ready[g], h->xs));         // RAW: the chunk landed
    h->copy_ev.push_back(e);
    s.pending[g] = 1;
    h->stats.copy_bytes += (uint64_t)e.bytes;
  }
  s.layer = layer;
  h->stats.copies += 1;
  return 0;
}

// Make sure seq[pos..pos+look] are resident or in flight; Belady choice of the victim among
// slots: evict the one whose content is needed furthest in the future (never one needed
// before the layer being fetched).
int prefetch(soup_stream *h, const std::vector<int> &seq, size_t pos, int look) {
  for (size_t j = pos; j < seq.size() && j <= pos + (size_t)look; ++j) {
    const int layer = seq[j];
    bool have = false;
    for (auto &s : h->slot) have |= (s.layer == layer);
    if (have) continue;
    int victim = -1, far = -1;
    uint64_t oldest = UINT64_MAX;
    for (int k = 0; k < (int)h->slot.size(); ++k) {
      const int nu = h->slot[k].layer < 0 ? INT32_MAX : next_use(seq, pos, h->slot[k].layer);
      const uint64_t t = h->slot[k].layer < 0 ? 0 : h->slot[k].tick;
      if (nu > far || (nu == far && t < oldest)) {  // ties: least recently released
        far = nu;
        oldest = t;
        victim = k;
      }
    }
    if (victim < 0 || far <= (int)j) break;  // every slot is needed before this layer
    SOUP_TRY(issue_copy(h, victim, layer));
  }
  return 0;
}

// The slot holding `layer` for the use at position pos (a copy is issued if none does).  No
// wait here: each kernel group waits for its own chunk (use_chunk).
int acquire(soup_stream *h, const std::vector<int> &seq, size_t pos, const uint8_t **shard,
            int *slot_out) {
  const int layer = seq[pos];
  if (h->resident) {
    *shard = h->ws + h->plan.slots + (uint64_t)layer * h->lay.stride;
    *slot_out = -1;
    return 0;
  }
  SOUP_TRY(prefetch(h, seq, pos, 0));
  int s = -1;
  for (int k = 0; k < (int)h->slot.size(); ++k)
    if (h->slot[k].layer == layer) s = k;
  if (s < 0) return set_error(SOUP_ESTATE, "internal: layer %d has no slot", layer);
  int use = s;
  if (h->dbg_stale && h->in_bwd) use = (s + 1) % (int)h->slot.size();  // deliberately wrong
  *shard = h->slot[use].dev;
  *slot_out = s;
  return 0;
}

// Before the first kernel that reads chunk g of the slot: wait for its copy (RAW).
int use_chunk(soup_stream *h, int slot, int g) {
  if (slot < 0) return 0;
  Slot &s = h->slot[slot];
  if (s.pending[g]) {
    SOUP_CUDA_TRY(cudaStreamWaitEvent(h->cs, s.ready[g], 0));
    s.pending[g] = 0;
  }
  return 0;
}

// After the last kernel of this use that reads chunk g: a later copy into it may start (WAR).
int release_chunk(soup_stream *h, int slot, int g) {
  if (slot < 0) return 0;
  SOUP_CUDA_TRY(cudaEventRecord(h->slot[slot].freed[g], h->cs));
  h->slot[slot].tick = ++h->tick;
  return 0;
}

// ---------------------------------------------------------------- layer maths
// Activation buffers of layer li: one set reused by every layer (the backward recomputes
// them), or one set per layer when the stream keeps activations (no recompute).
struct LayerBufs {
  uint64_t hm, x1, x2, qkv, att, lse, gu, act, u_f32[4], u_b[4];
};
LayerBufs bufs_of(const soup_stream *h, int li) {
  const Plan &P = h->plan;
  const uint64_t o = h->keep_act ? (uint64_t)li * P.act_stride : 0;
  LayerBufs b;
  b.hm = P.hm + o; b.x1 = P.x1 + o; b.x2 = P.x2 + o; b.qkv = P.qkv + o; b.att = P.att + o;
  b.lse = P.lse + o; b.gu = P.gu + o; b.act = P.act + o;
  for (int g = 0; g < 4; ++g) {
    b.u_f32[g] = P.u_f32[g] + o;
    b.u_b[g] = P.u_b[g] + o;
  }
  return b;
}

// Algorithmic work of the LoRA down-projection u = x A^T (x [M, K] 16-bit, nseg * r outputs):
// flops of the product; bytes of x, A, u (float) and its 16-bit pack.
double lora_down_flops(const LoraSeg &L, int M, int K) { return 2.0 * M * K * L.nseg * L.r; }
double lora_down_bytes(const LoraSeg &L, int M, int K) {
  const double nr = (double)L.nseg * L.r;
  return 2.0 * M * K + 4.0 * nr * K + 4.0 * M * nr + 2.0 * M * L.Rpad();
}
// Causal attention products: `mats` S x S x d products per head (2 forward: q k^T and p v; 5
// backward: the score recompute, dP, dV, dQ, dK), each over the S (S + 1) / 2 causal pairs.
double attn_flops(const soup_cfg &c, int B, int S, int mats) {
  return (double)mats * B * c.n_heads * (double)S * (S + 1) * c.head_dim;
}

// Forward of layer li on its shard (held in `slot`, -1 when resident).  In the forward proper
// each chunk is released after its GEMM; the backward's recompute (recompute = true) releases
// nothing, since the backward reads every chunk again.
int layer_forward(soup_stream *h, int li, const uint8_t *shard, int slot, bool recompute) {
  const soup_cfg &c = h->cfg;
  const Plan &P = h->plan;
  const LayerBufs Lb = bufs_of(h, li);
  const soup_shard_layout &SL = h->lay;
  cudaStream_t st = h->cs;
  const int B = h->B, S = h->S, M = B * S, H = c.hidden, I = c.inter;
  const int qd = c.n_heads * c.head_dim, nqkv = SL.n_out[SOUP_G_QKV];
  const float *hin = F(h, P.h_all) + (size_t)li * M * H;
  const uint16_t *ln1 = reinterpret_cast<const uint16_t *>(shard + SL.ln1_off);
  const uint16_t *ln2 = reinterpret_cast<const uint16_t *>(shard + SL.ln2_off);
  LoraSeg Lq = make_seg(h, li, SOUP_G_QKV, false), Lo = make_seg(h, li, SOUP_G_O, false),
          Lg = make_seg(h, li, SOUP_G_GU, false), Ld = make_seg(h, li, SOUP_G_DOWN, false);

  float *part = F(h, P.lora_part);
  // the forward's tensor-core operands are IEEE half (x1, qkv, att, x2, gu, act, LoRA packs)
  // adapters switched off (the reference forward of preference losses): no LoRA kernels and
  // no LoRA extension tiles, the plain dequant GEMMs
  const bool ad = !h->adapters_off;
  const bool rel = !recompute;
  SOUP_TRY(use_chunk(h, slot, SOUP_G_QKV));  // ln1 travels with the q|k|v chunk
  const double dM = M, dH = H, dI = I;
  SOUP_TRY(prof(h, FAM_RMSNORM_FWD, 0, 6.0 * dM * dH + 2.0 * dH,
                [&] { k_rmsnorm_fwd(hin, ln1, c.rms_eps, M, H, B16(h, Lb.x1), true, h->err_dev, st); }));
  if (ad)
    SOUP_TRY(prof(h, FAM_LORA_DOWN, lora_down_flops(Lq, M, H), lora_down_bytes(Lq, M, H), [&] {
      k_lora_down(B16(h, Lb.x1), H, M, H, Lq, F(h, Lb.u_f32[0]), B16(h, Lb.u_b[0]), true, true, part, h->err_dev, st);
    }));
  {
    GemmArgs g = weight_args(h, shard, SOUP_G_QKV, GEMM_FWD);
    g.op_f16 = 1; g.M = M; g.a = B16(h, Lb.x1); g.lda = H;
    if (ad) {
      g.ul = B16(h, Lb.u_b[0]); g.vl = B16(h, P.vl[(size_t)li * 4 + 0]); g.R = Lq.Rpad();
      g.lora_u = F(h, Lb.u_f32[0]); g.lseg = Lq; g.after_lora = 1;
    }
    g.epi = EPI_16; g.out = B16(h, Lb.qkv); g.ldo = nqkv;
    SOUP_TRY(timed_gemm(h, g, SOUP_G_QKV));
  }
  if (rel) SOUP_TRY(release_chunk(h, slot, SOUP_G_QKV));
  const double rot = (double)(c.n_heads + c.n_kv_heads) * c.head_dim;
  SOUP_TRY(prof(h, FAM_ROPE_FWD, 0, 4.0 * dM * rot, [&] {
    k_rope_fwd(B16(h, Lb.qkv), nqkv, F(h, P.rope_cos), F(h, P.rope_sin), M, S, c.n_heads,
               c.n_kv_heads, c.head_dim, true, h->err_dev, st);
  }));
  int arc = 0;
  SOUP_TRY(prof(h, FAM_ATTN_FWD, attn_flops(c, B, S, 2), 2.0 * dM * (nqkv + qd) + 4.0 * dM * c.n_heads, [&] {
    arc = k_attn_fwd(B16(h, Lb.qkv), nqkv, B, S, c.n_heads, c.n_kv_heads, c.head_dim, B16(h, Lb.att),
                     F(h, Lb.lse), h->err_dev, st);
  }));
  SOUP_TRY(arc);
  if (ad)
    SOUP_TRY(prof(h, FAM_LORA_DOWN, lora_down_flops(Lo, M, qd), lora_down_bytes(Lo, M, qd), [&] {
      k_lora_down(B16(h, Lb.att), qd, M, qd, Lo, F(h, Lb.u_f32[1]), B16(h, Lb.u_b[1]), true, true, part, h->err_dev, st);
    }));
  SOUP_TRY(use_chunk(h, slot, SOUP_G_O));
  {
    GemmArgs g = weight_args(h, shard, SOUP_G_O, GEMM_FWD);
    g.op_f16 = 1; g.M = M; g.a = B16(h, Lb.att); g.lda = qd;
    if (ad) {
      g.ul = B16(h, Lb.u_b[1]); g.vl = B16(h, P.vl[(size_t)li * 4 + 1]); g.R = Lo.Rpad();
      g.lora_u = F(h, Lb.u_f32[1]); g.lseg = Lo; g.after_lora = 1;
    }
    g.epi = EPI_F32_ADD; g.add_src = hin; g.ld_add = H; g.out = F(h, Lb.hm); g.ldo = H;
    SOUP_TRY(timed_gemm(h, g, SOUP_G_O));
  }
  if (rel) SOUP_TRY(release_chunk(h, slot, SOUP_G_O));
  SOUP_TRY(use_chunk(h, slot, SOUP_G_GU));  // ln2 travels with the gate|up chunk
  SOUP_TRY(prof(h, FAM_RMSNORM_FWD, 0, 6.0 * dM * dH + 2.0 * dH,
                [&] { k_rmsnorm_fwd(F(h, Lb.hm), ln2, c.rms_eps, M, H, B16(h, Lb.x2), true, h->err_dev, st); }));
  if (ad)
    SOUP_TRY(prof(h, FAM_LORA_DOWN, lora_down_flops(Lg, M, H), lora_down_bytes(Lg, M, H), [&] {
      k_lora_down(B16(h, Lb.x2), H, M, H, Lg, F(h, Lb.u_f32[2]), B16(h, Lb.u_b[2]), true, true, part, h->err_dev, st);
    }));
  {
    GemmArgs g = weight_args(h, shard, SOUP_G_GU, GEMM_FWD);
    g.op_f16 = 1; g.M = M; g.a = B16(h, Lb.x2); g.lda = H;
    if (ad) {
      g.ul = B16(h, Lb.u_b[2]); g.vl = B16(h, P.vl[(size_t)li * 4 + 2]); g.R = Lg.Rpad();
      g.lora_u = F(h, Lb.u_f32[2]); g.lseg = Lg; g.after_lora = 1;
    }
    g.epi = EPI_16; g.out = B16(h, Lb.gu); g.ldo = 2 * I;
    SOUP_TRY(timed_gemm(h, g, SOUP_G_GU));
  }
  if (rel) SOUP_TRY(release_chunk(h, slot, SOUP_G_GU));
  SOUP_TRY(prof(h, FAM_SWIGLU_FWD, 0, 6.0 * dM * dI,
                [&] { k_swiglu_fwd(B16(h, Lb.gu), M, I, B16(h, Lb.act), true, h->err_dev, st); }));
  if (ad)
    SOUP_TRY(prof(h, FAM_LORA_DOWN, lora_down_flops(Ld, M, I), lora_down_bytes(Ld, M, I), [&] {
      k_lora_down(B16(h, Lb.act), I, M, I, Ld, F(h, Lb.u_f32[3]), B16(h, Lb.u_b[3]), true, true, part, h->err_dev, st);
    }));
  if (!recompute) {
    SOUP_TRY(use_chunk(h, slot, SOUP_G_DOWN));
    GemmArgs g = weight_args(h, shard, SOUP_G_DOWN, GEMM_FWD);
    g.op_f16 = 1; g.M = M; g.a = B16(h, Lb.act); g.lda = I;
    if (ad) {
      g.ul = B16(h, Lb.u_b[3]); g.vl = B16(h, P.vl[(size_t)li * 4 + 3]); g.R = Ld.Rpad();
      g.lora_u = F(h, Lb.u_f32[3]); g.lseg = Ld; g.after_lora = 1;
    }
    g.epi = EPI_F32_ADD; g.add_src = F(h, Lb.hm); g.ld_add = H;
    g.out = F(h, P.h_all) + (size_t)(li + 1) * M * H; g.ldo = H;
    SOUP_TRY(timed_gemm(h, g, SOUP_G_DOWN));
    SOUP_TRY(release_chunk(h, slot, SOUP_G_DOWN));
  }
  return check_cuda("layer forward");
}

// Backward of one projection group: du = s dY B (kept per group for the layer's gradient
// launch) and dX = dY W + s (dY B) A (float out).
int group_backward(soup_stream *h, int li, const uint8_t *shard, int grp, const uint16_t *dy,
                   int ldy, float *dx_out) {
  const Plan &P = h->plan;
  cudaStream_t st = h->cs;
  const int M = h->B * h->S;
  LoraSeg L = make_seg(h, li, grp, true);
  const int K = h->lay.n_in[grp];
  // gradients travel in bf16
  const int Ng = h->lay.n_out[grp];
  const double nr = (double)L.nseg * L.r, dM = M;
  SOUP_TRY(prof(h, FAM_LORA_DU, 2.0 * dM * Ng * L.r,
                2.0 * dM * Ng + 4.0 * Ng * L.r + 4.0 * dM * nr + 2.0 * dM * L.Rpad(), [&] {
                  k_lora_du(dy, ldy, M, L, F(h, P.du_f32[grp]), B16(h, P.du_b), false, false, F(h, P.lora_part), st);
                }));
  GemmArgs g = weight_args(h, shard, grp, GEMM_DX);
  g.M = M; g.a = dy; g.lda = ldy;
  g.ul = B16(h, P.du_b); g.vl = B16(h, P.ac[(size_t)li * 4 + grp]); g.R = L.Rpad();
  g.lora_u = F(h, P.du_f32[grp]); g.lseg = L; g.after_lora = 1;
  g.epi = EPI_F32; g.out = dx_out; g.ldo = K;
  SOUP_TRY(timed_gemm(h, g, grp));
  return 0;
}

// The LoRA gradients (dB and dA) of all four groups of layer li in one launch, from the
// groups' upstream gradients, inputs, u and du, all still intact at the end of the layer.
int layer_lora_grads(soup_stream *h, int li) {
  const Plan &P = h->plan;
  const LayerBufs Lb = bufs_of(h, li);
  const soup_cfg &c = h->cfg;
  const int M = h->B * h->S, H = c.hidden, I = c.inter, qd = c.n_heads * c.head_dim;
  const int nqkv = h->lay.n_out[SOUP_G_QKV];
  const uint16_t *dy[4] = {B16(h, P.dqkv_b), B16(h, P.dhm_b), B16(h, P.dgu), B16(h, P.dh_b)};
  const int ldy[4] = {nqkv, H, 2 * I, H};
  const uint16_t *x[4] = {B16(h, Lb.x1), B16(h, Lb.att), B16(h, Lb.x2), B16(h, Lb.act)};
  const int ldx[4] = {H, qd, H, I};
  LoraGradGroup G[4];
  double flops = 0, bytes = 0;
  for (int g = 0; g < 4; ++g) {
    G[g].L = make_seg(h, li, g, true);
    G[g].dy = dy[g];
    G[g].ldy = ldy[g];
    G[g].Ng = h->lay.n_out[g];
    G[g].u = F(h, Lb.u_f32[g]);
    G[g].du = F(h, P.du_f32[g]);
    G[g].x = x[g];
    G[g].ldx = ldx[g];
    G[g].K = h->lay.n_in[g];
    const double nr = (double)G[g].L.nseg * G[g].L.r;
    flops += 2.0 * M * G[g].Ng * G[g].L.r + 2.0 * M * G[g].K * nr;
    bytes += 2.0 * M * G[g].Ng + 4.0 * M * nr + 4.0 * G[g].Ng * G[g].L.r +  // dB: dY, u, dB
             4.0 * M * nr + 2.0 * M * G[g].K + 4.0 * nr * G[g].K;             // dA: du, x, dA
  }
  return prof(h, FAM_LORA_GRAD, flops, bytes, [&] { k_lora_grads(G, 4, M, true, h->cs); });
}

// Backward of layer li; releases each chunk after its last reader (the dX GEMM of its group,
// and for q|k|v and gate|up the RMSNorm backward that reads the chunk's norm vector).
int layer_backward(soup_stream *h, int li, const uint8_t *shard, int slot) {
  const soup_cfg &c = h->cfg;
  const Plan &P = h->plan;
  const LayerBufs Lb = bufs_of(h, li);
  const soup_shard_layout &SL = h->lay;
  cudaStream_t st = h->cs;
  const int B = h->B, S = h->S, M = B * S, H = c.hidden, I = c.inter;
  const int qd = c.n_heads * c.head_dim, nqkv = SL.n_out[SOUP_G_QKV];
  const float *hin = F(h, P.h_all) + (size_t)li * M * H;
  const uint16_t *ln1 = reinterpret_cast<const uint16_t *>(shard + SL.ln1_off);
  const uint16_t *ln2 = reinterpret_cast<const uint16_t *>(shard + SL.ln2_off);

  // dh / dh_b hold dL/dh_{li+1}
  SOUP_TRY(use_chunk(h, slot, SOUP_G_DOWN));
  SOUP_TRY(group_backward(h, li, shard, SOUP_G_DOWN, B16(h, P.dh_b), H, F(h, P.dact)));
  SOUP_TRY(release_chunk(h, slot, SOUP_G_DOWN));
  const double dM = M, dH = H, dI = I;
  SOUP_TRY(prof(h, FAM_SWIGLU_BWD, 0, 12.0 * dM * dI,
                [&] { k_swiglu_bwd(F(h, P.dact), B16(h, Lb.gu), M, I, B16(h, P.dgu), true, st); }));
  SOUP_TRY(use_chunk(h, slot, SOUP_G_GU));
  SOUP_TRY(group_backward(h, li, shard, SOUP_G_GU, B16(h, P.dgu), 2 * I, F(h, P.dx)));
  SOUP_TRY(prof(h, FAM_RMSNORM_BWD, 0, 18.0 * dM * dH + 2.0 * dH, [&] {
    k_rmsnorm_bwd(F(h, P.dx), F(h, Lb.hm), ln2, c.rms_eps, M, H, F(h, P.dh), F(h, P.dhm), B16(h, P.dhm_b), st);
  }));
  SOUP_TRY(release_chunk(h, slot, SOUP_G_GU));
  SOUP_TRY(use_chunk(h, slot, SOUP_G_O));
  SOUP_TRY(group_backward(h, li, shard, SOUP_G_O, B16(h, P.dhm_b), H, F(h, P.datt)));
  SOUP_TRY(release_chunk(h, slot, SOUP_G_O));
  SOUP_TRY(prof(h, FAM_CAST, 0, 6.0 * dM * qd,
                [&] { k_cast_bf16(F(h, P.datt), B16(h, P.datt_b), (int64_t)M * qd, st); }));
  int arc = 0;
  SOUP_TRY(prof(h, FAM_ATTN_BWD, attn_flops(c, B, S, 5),
                2.0 * dM * nqkv + 4.0 * dM * qd + 4.0 * dM * c.n_heads + 4.0 * dM * nqkv, [&] {
                  arc = k_attn_bwd(B16(h, Lb.qkv), nqkv, B16(h, Lb.att), B16(h, P.datt_b), F(h, Lb.lse), B, S,
                                   c.n_heads, c.n_kv_heads, c.head_dim, F(h, P.attn_scratch), F(h, P.dqkv),
                                   h->err_dev, st);
                }));
  SOUP_TRY(arc);
  SOUP_TRY(prof(h, FAM_ROPE_BWD, 0, 6.0 * dM * nqkv, [&] {
    k_rope_bwd(F(h, P.dqkv), B16(h, P.dqkv_b), nqkv, F(h, P.rope_cos), F(h, P.rope_sin), M, S,
               c.n_heads, c.n_kv_heads, c.head_dim, st);
  }));
  SOUP_TRY(use_chunk(h, slot, SOUP_G_QKV));
  SOUP_TRY(group_backward(h, li, shard, SOUP_G_QKV, B16(h, P.dqkv_b), nqkv, F(h, P.dx)));
  // every group's dY, x, u and du are still intact here (the RMSNorm backward below is the
  // first to overwrite one: dh_b, the down projection's dY)
  SOUP_TRY(layer_lora_grads(h, li));
  SOUP_TRY(prof(h, FAM_RMSNORM_BWD, 0, 18.0 * dM * dH + 2.0 * dH, [&] {
    k_rmsnorm_bwd(F(h, P.dx), hin, ln1, c.rms_eps, M, H, F(h, P.dhm), F(h, P.dh), B16(h, P.dh_b), st);
  }));
  SOUP_TRY(release_chunk(h, slot, SOUP_G_QKV));
  return check_cuda("layer backward");
}

const uint16_t *lm_weight(soup_stream *h) { return h->lm_head ? h->lm_head : h->embed; }

}  // namespace

// ------------------------------------------------------------------------------------------
int stream_init(soup_store *st, const soup_cfg *c, int maxB, int maxS, void *ws, uint64_t ws_bytes,
                const void *embed, const void *lm_head, const void *final_norm, uintptr_t cs,
                uintptr_t xs, int n_slots, int mode, soup_stream **out) {
  if (!out) return set_error(SOUP_EINVAL, "out is NULL");
  *out = nullptr;
  const bool stream_head = (mode & SOUP_MODE_STREAM_HEAD) != 0;
  if (!st || !c || !ws || (!embed && !stream_head) || !final_norm)
    return set_error(SOUP_EINVAL, "stream_init: NULL argument");
  if (!c->tied && !lm_head && !stream_head) return set_error(SOUP_EINVAL, "untied config needs lm_head");
  if (stream_head && !st->head)
    return set_error(SOUP_ESTATE, "stream_init: SOUP_MODE_STREAM_HEAD needs soup_store_put_head first");
  if (std::memcmp(&st->cfg, c, sizeof(soup_cfg)) != 0)
    return set_error(SOUP_EINVAL, "stream_init: cfg differs from the store's");
  for (int l = 0; l < c->n_layers; ++l)
    if (!st->filled[l]) return set_error(SOUP_ESTATE, "store layer %d was never filled", l);
  const int resident = (mode & SOUP_MODE_RESIDENT) != 0;
  if (cs == xs && !resident) return set_error(SOUP_EINVAL, "compute and copy streams must differ");
  if (reinterpret_cast<uintptr_t>(ws) % 256) return set_error(SOUP_EINVAL, "workspace must be 256-byte aligned");
  Plan P;
  SOUP_TRY(make_plan(c, maxB, maxS, n_slots, mode, &P));
  if (ws_bytes < P.total)
    return set_error(SOUP_ENOMEM, "workspace %llu bytes < required %llu",
                     (unsigned long long)ws_bytes, (unsigned long long)P.total);
  soup_stream *h = new (std::nothrow) soup_stream();
  if (!h) return set_error(SOUP_ENOMEM, "host allocation failed");
  h->cfg = *c;
  h->store = st;
  h->plan = P;
  h->lay = st->lay;
  h->maxB = maxB;
  h->maxS = maxS;
  h->resident = resident;
  h->keep_act = (mode & SOUP_MODE_KEEP_ACTIVATIONS) != 0;
  h->cs = reinterpret_cast<cudaStream_t>(cs);
  h->xs = reinterpret_cast<cudaStream_t>(xs);
  h->ws = static_cast<uint8_t *>(ws);
  h->stream_head = stream_head ? 1 : 0;
  if (stream_head) {
    // the gather reads the embedding rows from the mapped page-locked store; the head table
    // (the embedding itself when tied) occupies the workspace's vocabulary buffer
    h->embed = reinterpret_cast<const uint16_t *>(st->head_dev);
    h->lm_head = reinterpret_cast<const uint16_t *>(h->ws + P.vocab_buf);
  } else {
    h->embed = static_cast<const uint16_t *>(embed);
    h->lm_head = c->tied ? nullptr : static_cast<const uint16_t *>(lm_head);
  }
  h->final_norm = static_cast<const uint16_t *>(final_norm);
  h->err_dev = reinterpret_cast<int *>(h->ws + P.err);
  auto fail = [&](int rc) {
    soup_stream_free_impl(h);
    return rc;
  };
  if (cudaMemsetAsync(h->err_dev, 0, 64, h->cs) != cudaSuccess)
    return fail(set_error(SOUP_ECUDA, "workspace memset failed"));
  // RoPE tables: angle pos * theta^(-2i/d) formed in double, cos/sin rounded to float.
  {
    const int half = c->head_dim / 2;
    std::vector<float> cs_h((size_t)maxS * half), sn_h((size_t)maxS * half);
    for (int p = 0; p < maxS; ++p)
      for (int i = 0; i < half; ++i) {
        const double inv = std::pow((double)c->rope_theta, -(2.0 * i) / c->head_dim);
        const double a = p * inv;
        cs_h[(size_t)p * half + i] = (float)std::cos(a);
        sn_h[(size_t)p * half + i] = (float)std::sin(a);
      }
    if (cudaMemcpy(h->ws + P.rope_cos, cs_h.data(), cs_h.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(h->ws + P.rope_sin, sn_h.data(), sn_h.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
      return fail(set_error(SOUP_ECUDA, "rope table upload failed"));
  }
  if (stream_head) {
    const uint64_t table = 2ull * c->vocab * c->hidden;
    if (cudaMemcpy(h->ws + P.vocab_buf, st->head + (c->tied ? 0 : table), table, cudaMemcpyHostToDevice) !=
        cudaSuccess)
      return fail(set_error(SOUP_ECUDA, "head table upload failed"));
  }
  if (h->resident) {
    for (int l = 0; l < c->n_layers; ++l) {
      if (cudaMemcpy(h->ws + P.slots + (uint64_t)l * h->lay.stride, st->base + (uint64_t)l * h->lay.stride,
                     h->lay.stride, cudaMemcpyHostToDevice) != cudaSuccess)
        return fail(set_error(SOUP_ECUDA, "resident upload of layer %d failed", l));
    }
  } else {
    h->slot.resize(n_slots);
    for (int k = 0; k < n_slots; ++k) {
      Slot &s = h->slot[k];
      s.dev = h->ws + P.slots + (uint64_t)k * h->lay.stride;
      s.has_events = 1;
      for (int g = 0; g < NCHUNK; ++g)
        if (cudaEventCreateWithFlags(&s.ready[g], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&s.freed[g], cudaEventDisableTiming) != cudaSuccess)
          return fail(set_error(SOUP_ECUDA, "event creation failed"));
      // an unrecorded event counts as complete for cudaStreamWaitEvent
    }
  }
  if (cudaEventCreateWithFlags(&h->done, cudaEventDisableTiming) != cudaSuccess)
    return fail(set_error(SOUP_ECUDA, "event creation failed"));
  SOUP_TRY(check_cuda("stream_init"));
  *out = h;
  return 0;
}

int step_fwd(soup_stream *h, const int32_t *tokens, int B, int S, const float *const *lA,
             const float *const *lB, float *loss, float *logits, float *layer_out) {
  if (!h || !tokens || !loss) return set_error(SOUP_EINVAL, "step_fwd: NULL argument");
  if (!lA != !lB) return set_error(SOUP_EINVAL, "step_fwd: lora_A and lora_B must both be given or both NULL");
  const bool adapters_off = !lA;
  const soup_cfg &c = h->cfg;
  if (B < 1 || S < 2 || S > h->maxS || (int64_t)B * S > (int64_t)h->maxB * h->maxS)
    return set_error(SOUP_EINVAL, "step_fwd: B=%d S=%d outside the workspace (max %d x %d)", B, S,
                     h->maxB, h->maxS);
  const int L = c.n_layers;
  for (int i = 0; i < L * 7 && !adapters_off; ++i)
    if (!lA[i] || !lB[i]) return set_error(SOUP_EINVAL, "step_fwd: LoRA pointer %d is NULL", i);
  h->B = B;
  h->S = S;
  h->tokens = tokens;
  h->adapters_off = adapters_off ? 1 : 0;
  if (adapters_off) {
    h->lora_A.clear();
    h->lora_B.clear();
  } else {
    h->lora_A.assign(lA, lA + (size_t)L * 7);
    h->lora_B.assign(lB, lB + (size_t)L * 7);
  }
  h->in_bwd = 0;
  harvest(h, false);
  const Plan &P = h->plan;
  cudaStream_t st = h->cs;
  const int M = B * S, H = c.hidden;
  SOUP_TRY(prof(h, FAM_EMBED, 0, 6.0 * M * H, [&] { k_embed(tokens, h->embed, c.vocab, H, M, F(h, P.h_all), st); }));
  std::vector<int> seq(L);
  for (int i = 0; i < L; ++i) seq[i] = i;
  const int look = std::max(0, (int)h->slot.size() - 1);
  for (int i = 0; i < L; ++i) {
    const uint8_t *shard;
    int s;
    // 16-bit LoRA operands of this layer's tensor-core GEMMs (forward: half B rows; dX:
    // bf16 A rows), packed just before first use so that the first layer's kernels, and so
    // the first slot release, are not queued behind every layer's packing
    if (!adapters_off) {  // one launch packs the layer's four groups, both directions
      LoraSeg Ls[4];
      uint16_t *vl[4], *ac[4];
      for (int g = 0; g < 4; ++g) {
        Ls[g] = make_seg(h, i, g, false);
        vl[g] = B16(h, P.vl[(size_t)i * 4 + g]);
        ac[g] = B16(h, P.ac[(size_t)i * 4 + g]);
      }
      double pb = 0;
      for (int g = 0; g < 4; ++g)
        pb += 4.0 * Ls[g].r * (h->lay.n_out[g] + (double)Ls[g].nseg * h->lay.n_in[g]) +
              2.0 * Ls[g].Rpad() * ((double)h->lay.n_out[g] + h->lay.n_in[g]);
      SOUP_TRY(prof(h, FAM_LORA_PACK, 0, pb, [&] { k_pack_layer(Ls, h->lay.n_out, h->lay.n_in, vl, ac, st); }));
    }
    TraceRange tr("fwd layer", i);
    SOUP_TRY(acquire(h, seq, (size_t)i, &shard, &s));
    SOUP_TRY(layer_forward(h, i, shard, s, false));
    if (!h->resident) SOUP_TRY(prefetch(h, seq, (size_t)i + 1, look - 1));
  }
  // final norm + vocabulary-chunked loss
  TraceRange tr_head("loss head fwd");
  k_rmsnorm_fwd(F(h, P.h_all) + (size_t)L * M * H, h->final_norm, c.rms_eps, M, H, B16(h, P.hn), false, nullptr, st);
  const int vc = P.vc;
  for (int v0 = 0, ci = 0; v0 < c.vocab; v0 += vc, ++ci) {
    const int n = std::min(vc, c.vocab - v0);
    GemmArgs g;
    g.mode = GEMM_FWD; g.wfmt = W_BF16; g.w = lm_weight(h) + (size_t)v0 * H; g.Nw = n; g.Kw = H;
    g.M = M; g.a = B16(h, P.hn); g.lda = H; g.epi = EPI_F32;
    float *z = logits ? logits + v0 : F(h, P.z);
    const int ldz = logits ? c.vocab : vc;
    g.out = z; g.ldo = ldz;
    gemm_scratch(h, g);
    int grc = 0;
    SOUP_TRY(prof(h, FAM_HEAD_GEMM, gemm_flops(g), gemm_bytes(g), [&] { grc = gemm_launch(g, st); }));
    SOUP_TRY(grc);
    SOUP_TRY(prof(h, FAM_CE_FWD, 0, 4.0 * M * n, [&] {
      k_ce_chunk_fwd(z, ldz, v0, n, tokens, M, S, ci == 0, F(h, P.ce_max), F(h, P.ce_sum), F(h, P.ce_lab), st);
    }));
  }
  k_ce_finalize(F(h, P.ce_max), F(h, P.ce_sum), F(h, P.ce_lab), M, S, F(h, P.ce_lse), loss, st);
  if (layer_out)
    SOUP_CUDA_TRY(cudaMemcpyAsync(layer_out, F(h, P.h_all), 4ull * (L + 1) * M * H,
                                  cudaMemcpyDeviceToDevice, st));
  SOUP_CUDA_TRY(cudaEventRecord(h->done, st));
  // a backward follows a forward with adapters only; an adapters-off forward leaves none
  h->fwd_ready = adapters_off ? 0 : 1;
  h->last_layer_fresh = 1;  // the last layer's activations are still in the scratch buffers
  h->stats.steps_fwd += 1;
  return check_cuda("step_fwd");
}

int step_bwd(soup_stream *h, float *const *dA, float *const *dB, float *dh_out, int flags) {
  if (!h || !dA || !dB) return set_error(SOUP_EINVAL, "step_bwd: NULL argument");
  if (flags & ~SOUP_BWD_ACCUMULATE) return set_error(SOUP_EINVAL, "step_bwd: unknown flags 0x%x", flags);
  if (!h->fwd_ready)
    return set_error(SOUP_ESTATE, h->adapters_off ? "step_bwd after an adapters-off forward"
                                                  : "step_bwd without a preceding step_fwd");
  const soup_cfg &c = h->cfg;
  const int L = c.n_layers;
  for (int i = 0; i < L * 7; ++i)
    if (!dA[i] || !dB[i]) return set_error(SOUP_EINVAL, "step_bwd: gradient pointer %d is NULL", i);
  h->grad_A.assign(dA, dA + (size_t)L * 7);
  h->grad_B.assign(dB, dB + (size_t)L * 7);
  h->grad_accumulate = (flags & SOUP_BWD_ACCUMULATE) != 0;
  h->in_bwd = 1;
  harvest(h, false);
  const Plan &P = h->plan;
  cudaStream_t st = h->cs;
  const int B = h->B, S = h->S, M = B * S, H = c.hidden;
  // loss backward, chunk by chunk: recompute logits, dz = (softmax - onehot) / N, dhn += dz W
  const int vc = P.vc;
  const float inv_n = 1.0f / (float)((int64_t)B * (S - 1));
  {
    TraceRange tr_head("loss head bwd");
    for (int v0 = 0, ci = 0; v0 < c.vocab; v0 += vc, ++ci) {
      const int n = std::min(vc, c.vocab - v0);
      const uint16_t *w = lm_weight(h) + (size_t)v0 * H;
      GemmArgs g;
      g.mode = GEMM_FWD; g.wfmt = W_BF16; g.w = w; g.Nw = n; g.Kw = H;
      g.M = M; g.a = B16(h, P.hn); g.lda = H; g.epi = EPI_F32; g.out = F(h, P.z); g.ldo = vc;
      gemm_scratch(h, g);
      int grc = 0;
      SOUP_TRY(prof(h, FAM_HEAD_GEMM, gemm_flops(g), gemm_bytes(g), [&] { grc = gemm_launch(g, st); }));
      SOUP_TRY(grc);
      SOUP_TRY(prof(h, FAM_CE_BWD, 0, 6.0 * M * n, [&] {
        k_ce_chunk_bwd(F(h, P.z), vc, v0, n, F(h, P.ce_lse), h->tokens, M, S, inv_n, B16(h, P.dz), st);
      }));
      GemmArgs d;
      d.mode = GEMM_DX; d.wfmt = W_BF16; d.w = w; d.Nw = n; d.Kw = H;
      d.M = M; d.a = B16(h, P.dz); d.lda = vc; d.epi = ci == 0 ? EPI_F32 : EPI_F32_ACC;
      d.out = F(h, P.dhn); d.ldo = H;
      gemm_scratch(h, d);
      SOUP_TRY(prof(h, FAM_HEAD_DX, gemm_flops(d), gemm_bytes(d), [&] { grc = gemm_launch(d, st); }));
      SOUP_TRY(grc);
    }
    k_rmsnorm_bwd(F(h, P.dhn), F(h, P.h_all) + (size_t)L * M * H, h->final_norm, c.rms_eps, M, H,
                  nullptr, F(h, P.dh), B16(h, P.dh_b), st);
  }
  if (dh_out)
    SOUP_CUDA_TRY(cudaMemcpyAsync(dh_out + (size_t)L * M * H, F(h, P.dh), 4ull * M * H,
                                  cudaMemcpyDeviceToDevice, st));
  std::vector<int> seq(L);
  for (int i = 0; i < L; ++i) seq[i] = L - 1 - i;
  const int look = std::max(0, (int)h->slot.size() - 1);
  for (int j = 0; j < L; ++j) {
    const int li = seq[j];
    const uint8_t *shard;
    int s;
    TraceRange tr("bwd layer", li);
    SOUP_TRY(acquire(h, seq, (size_t)j, &shard, &s));
    // the forward's last layer left its activations in the scratch buffers (the loss head
    // between uses separate ones): its backward reuses them instead of recomputing them, which
    // would reproduce the same values with the same kernels.  With kept activations every
    // layer's are still there ("stream_recompute: off"); only the weights are read again.
    if (!h->keep_act && !(j == 0 && h->last_layer_fresh)) SOUP_TRY(layer_forward(h, li, shard, s, true));
    h->last_layer_fresh = 0;
    SOUP_TRY(layer_backward(h, li, shard, s));
    if (!h->resident) SOUP_TRY(prefetch(h, seq, (size_t)j + 1, look - 1));
    if (dh_out)
      SOUP_CUDA_TRY(cudaMemcpyAsync(dh_out + (size_t)li * M * H, F(h, P.dh), 4ull * M * H,
                                    cudaMemcpyDeviceToDevice, st));
  }
  SOUP_CUDA_TRY(cudaEventRecord(h->done, st));
  h->in_bwd = 0;
  h->stats.steps_bwd += 1;
  return check_cuda("step_bwd");
}

int stream_sync(soup_stream *h, int timeout_ms) {
  if (!h) return set_error(SOUP_EINVAL, "handle is NULL");
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    cudaError_t q = cudaEventQuery(h->done);
    if (q == cudaSuccess) break;
    if (q != cudaErrorNotReady) return set_error(SOUP_ECUDA, "step failed: %s", cudaGetErrorString(q));
    const auto dt = std::chrono::duration_cast<std::chrono::milliseconds>(std::chrono::steady_clock::now() - t0);
    if (timeout_ms >= 0 && dt.count() > timeout_ms)
      return set_error(SOUP_ETIMEDOUT, "soup_sync: not done after %d ms", timeout_ms);
    std::this_thread::sleep_for(std::chrono::microseconds(100));
  }
  int err = 0;
  SOUP_CUDA_TRY(cudaMemcpy(&err, h->err_dev, sizeof(int), cudaMemcpyDeviceToHost));
  harvest(h, false);
  if (err) {  // reported once: the next step starts with a clear flag
    SOUP_CUDA_TRY(cudaMemset(h->err_dev, 0, sizeof(int)));
    return kernel_flags_status(err, "soup_sync");
  }
  return 0;
}

int stream_kernel_stats(soup_stream *h, soup_kernel_stat *out, int max, int *n, int reset) {
  if (!h || !n || (max > 0 && !out)) return set_error(SOUP_EINVAL, "NULL argument");
  harvest(h, true);
  int k = 0;
  for (int f = 0; f < FAM_COUNT; ++f) {
    if (!h->fam[f].launches) continue;
    if (k < max) {
      soup_kernel_stat &o = out[k];
      std::memset(&o, 0, sizeof(o));
      std::snprintf(o.name, sizeof(o.name), "%s", kFamName[f]);
      o.tensor_bound = kFamTensor[f];
      o.launches = h->fam[f].launches;
      o.ms = h->fam[f].ms;
      o.flops = h->fam[f].flops;
      o.bytes = h->fam[f].bytes;
    }
    ++k;
  }
  *n = k;
  if (reset)
    for (auto &f : h->fam) f = FamStat();
  return 0;
}

int stream_stats(soup_stream *h, soup_stats *out, int reset) {
  if (!h || !out) return set_error(SOUP_EINVAL, "NULL argument");
  harvest(h, true);
  *out = h->stats;
  if (reset) h->stats = soup_stats();
  return 0;
}

void soup_stream_free_impl(soup_stream *h) {
  if (!h) return;
  cudaStreamSynchronize(h->cs);
  if (h->xs) cudaStreamSynchronize(h->xs);
  harvest(h, true);
  for (auto &s : h->slot)
    if (s.has_events)
      for (int g = 0; g < NCHUNK; ++g) {
        if (s.ready[g]) cudaEventDestroy(s.ready[g]);
        if (s.freed[g]) cudaEventDestroy(s.freed[g]);
      }
  for (cudaEvent_t e : h->ev_pool) cudaEventDestroy(e);
  if (h->done) cudaEventDestroy(h->done);
  delete h;
}

}  // namespace soup
