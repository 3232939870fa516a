// Launchers of the memory-bound kernels of the step (row norms, RoPE, SwiGLU, LoRA
// projections and gradients, loss) and of attention.  All reductions run in a fixed order:
// no floating-point atomics, so every launch is bit-reproducible.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace soup {

constexpr int MAX_SEG = 3;  // projections fused in one GEMM group (q,k,v)

// The 16 NF4 values, passed to kernels by value (they live in the parameter bank).
struct Codebook {
  float v[16];
};
// The library's codebook (derived once on the host).
const Codebook &nf4_codebook_param();

// A group of LoRA segments that share one input x: segment p covers output columns
// [off[p], off[p] + n[p]) of the fused GEMM, with A_p [r, K] and B_p [n[p], r].
struct LoraSeg {
  int nseg = 0, r = 0;
  int off[MAX_SEG] = {0, 0, 0}, n[MAX_SEG] = {0, 0, 0};
  const float *A[MAX_SEG] = {nullptr, nullptr, nullptr};
  const float *B[MAX_SEG] = {nullptr, nullptr, nullptr};
  float *dA[MAX_SEG] = {nullptr, nullptr, nullptr};
  float *dB[MAX_SEG] = {nullptr, nullptr, nullptr};
  float s = 1.f;
  bool accumulate = false;  // dA/dB reductions add to the existing gradient (old + g)
  __host__ __device__ int Rpad() const { return ((nseg * r + 63) / 64) * 64; }
};

void k_embed(const int32_t *tok, const uint16_t *E, int V, int H, int M, float *out, cudaStream_t st);
// Tensors in 16-bit are either IEEE half (the forward's tensor-core operands: normalised
// inputs, qkv, attention output, gate/up, SwiGLU output, the forward LoRA packs) or bf16
// (gradients, the loss head); each launcher takes a flag saying which.
// Forward kernels that store half operands take `err`: a device int into which they OR
// SOUP_KERR_RANGE if a stored value was NaN or beyond the half range (may be null).
void k_rmsnorm_fwd(const float *h, const uint16_t *w, float eps, int M, int H, uint16_t *out,
                   bool out_f16, int *err, cudaStream_t st);
// out = dres + rmsnorm_backward(dy); dres may be null (treated as 0) or alias out.
void k_rmsnorm_bwd(const float *dy, const float *h, const uint16_t *w, float eps, int M, int H,
                   const float *dres, float *out, uint16_t *out_bf16, cudaStream_t st);
void k_rope_fwd(uint16_t *qkv, int ld, const float *cos, const float *sin, int M, int S, int nh,
                int nkv, int d, bool f16, int *err, cudaStream_t st);
// in: dqkv float [M, ld]; out bf16 [M, ld]: q/k heads rotated back, v heads cast.
void k_rope_bwd(const float *dqkv, uint16_t *out, int ld, const float *cos, const float *sin,
                int M, int S, int nh, int nkv, int d, cudaStream_t st);
void k_swiglu_fwd(const uint16_t *gu, int M, int I, uint16_t *act, bool f16, int *err, cudaStream_t st);
void k_swiglu_bwd(const float *dact, const uint16_t *gu, int M, int I, uint16_t *dgu, bool gu_f16,
                  cudaStream_t st);

// The LoRA projections are split over K and the partial sums are added in a fixed order by a
// second kernel.  Scratch they need, in floats, for M rows, a reduction width `dim` and
// nout = segments * r outputs:
int lora_splits(int M, int K, int *KS);
size_t lora_scratch_floats(int M, int dim, int nout);
// u = x A^T per segment -> u_f32 [M, nseg*r]; ul = 16-bit(s * u) [M, Rpad] (zero padded)
// The clustered single-launch LoRA projection (lora_proj.cu): 0 when launched (or a negative
// SOUP_E* code), 1 when the shape is not one it takes (16-byte alignment, rank a multiple of 8,
// at most 64 fused outputs, segment boundaries on 8-element multiples).
int lora_skinny(bool du, const uint16_t *X, int ldx, int M, int K, const LoraSeg &L, float *out_f32,
                uint16_t *out16, bool x_f16, bool o_f16, int *err, cudaStream_t st);
void k_lora_down(const uint16_t *x, int lda, int M, int K, const LoraSeg &L, float *u_f32,
                 uint16_t *ul, bool x_f16, bool ul_f16, float *part, int *err, cudaStream_t st);
// du_p = s dY_p B_p -> du_f32 [M, nseg*r]; dul = 16-bit(du) [M, Rpad]
void k_lora_du(const uint16_t *dy, int ldy, int M, const LoraSeg &L, float *du_f32, uint16_t *dul,
               bool dy_f16, bool dul_f16, float *part, cudaStream_t st);
// The LoRA gradients of one fused group: dB_p = s dY_p^T u_p and dA_p = du_p^T x for its
// segments, written into (or, with L.accumulate, added to) L.dB / L.dA.
struct LoraGradGroup {
  LoraSeg L;
  const uint16_t *dy = nullptr;  // bf16 dY [M, Ng], row stride ldy
  int ldy = 0, Ng = 0;
  const float *u = nullptr;      // [M, nseg r]: x A^T
  const float *du = nullptr;     // [M, nseg r]: s dY B
  const uint16_t *x = nullptr;   // 16-bit x [M, K] (half if x_f16), row stride ldx
  int ldx = 0, K = 0;
};
// Gradients of up to four groups in one launch (lora_grad.cu): per 64-column tile of each
// product a cluster of 8 CTAs splits the tokens and sums its partial tiles in rank order
// through distributed shared memory (no global scratch, fixed summation order).
void k_lora_grads(const LoraGradGroup *groups, int ngroups, int M, bool x_f16, cudaStream_t st);
// Vl [Ng, Rpad]: row n of segment p holds 16-bit(B_p[n - off_p, :]) at columns p*r .. p*r+r-1
void k_pack_fwd(const LoraSeg &L, int Ng, uint16_t *vl, bool f16, cudaStream_t st);
// Acat [Rpad, K]: row p*r + j holds 16-bit(A_p[j, :]); rows past nseg*r are zero
void k_pack_bwd(const LoraSeg &L, int K, uint16_t *acat, bool f16, cudaStream_t st);
// One launch for a layer's four groups: vl[g] as k_pack_fwd in half, ac[g] as k_pack_bwd in bf16.
void k_pack_layer(const LoraSeg (&L)[4], const int n_out[4], const int n_in[4], uint16_t *const vl[4],
                  uint16_t *const ac[4], cudaStream_t st);

// Vocabulary-chunked cross-entropy.  Rows are tokens b*S + t; row t has label tok[b*S+t+1]
// for t < S-1 and none for t = S-1.
void k_ce_chunk_fwd(const float *z, int ldz, int v0, int vc, const int32_t *tok, int M, int S,
                    int first, float *rmax, float *rsum, float *zlab, cudaStream_t st);
void k_ce_finalize(const float *rmax, const float *rsum, const float *zlab, int M, int S,
                   float *lse, float *loss, cudaStream_t st);
void k_ce_chunk_bwd(const float *z, int ldz, int v0, int vc, const float *lse, const int32_t *tok,
                    int M, int S, float inv_n, uint16_t *dz, cudaStream_t st);

void k_cast_bf16(const float *in, uint16_t *out, int64_t n, cudaStream_t st);
// One AdamW step in place over n floats (optim.cu); step >= 1, betas in [0, 1).
void k_adamw(float *p, const float *g, float *m, float *v, int64_t n, float lr, float beta1,
             float beta2, float eps, float weight_decay, float grad_scale, int64_t step,
             cudaStream_t st);
// One block that waits on an mbarrier nothing arrives on, bounded by limit_cycles, and raises
// the wait-timeout bit in *err (a test of the error path).
void k_wait_probe(int *err, long long limit_cycles, cudaStream_t st);
void k_nf4_dequant(const uint8_t *codes, const float *absmax, int64_t n, float *out_f32,
                   uint16_t *out_bf16, cudaStream_t st);

// Causal GQA attention on the fused half-precision qkv buffer [M, ld] (q heads, then k heads,
// then v heads, each head_dim wide), rows b*S + t.  o: half [M, nh*d]; lse: float [B*nh*S]
// (base-2 log-sum of exp2(scale*log2e*score)).  head_dim 64 or 128.  The tcgen05 kernels
// (attention_tc.cu) take head_dim 64 / 128 with at most 8 query heads per key/value head; other
// shapes run the warp-level MMA kernels (attention.cu).  err: device int for error bits, or NULL.
int k_attn_fwd(const uint16_t *qkv, int ld, int B, int S, int nh, int nkv, int d, uint16_t *o,
               float *lse, int *err, cudaStream_t st);
// o: half [M, nh*d] (the forward output); dO: bf16 [M, nh*d]; dqkv: float [M, ld] written
// completely (dq, dk, dv); scratch: float [attn_bwd_scratch_floats()], 256-byte aligned.
size_t attn_bwd_scratch_floats(int B, int S, int nh, int nkv, int d);
int k_attn_bwd(const uint16_t *qkv, int ld, const uint16_t *o, const uint16_t *dO,
               const float *lse, int B, int S, int nh, int nkv, int d, float *scratch, float *dqkv,
               int *err, cudaStream_t st);
// the tcgen05 path (attention_tc.cu)
int attn_tc_eligible(int d, int nh, int nkv);
size_t attn_tc_scratch_floats(int B, int S, int nh, int nkv, int d);
int k_attn_fwd_tc(const uint16_t *qkv, int ld, int B, int S, int nh, int nkv, int d, uint16_t *o,
                  float *lse, int *err, cudaStream_t st);
int k_attn_bwd_tc(const uint16_t *qkv, int ld, const uint16_t *o, const uint16_t *dO,
                  const float *lse, int B, int S, int nh, int nkv, int d, float *scratch,
                  float *dqkv, int *err, cudaStream_t st);

}  // namespace soup
