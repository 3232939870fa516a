// Internal interface of the base-weight GEMMs (NF4-dequant or bf16 weights, with the rank-r
// LoRA term folded in as extra reduction tiles).  Not part of the C ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace soup {

enum GemmMode { GEMM_FWD = 0, GEMM_DX = 1 };   // FWD: y = a W^T ; DX: y = a W
enum WFmt { W_BF16 = 0, W_NF4 = 1 };
enum Epi {
  EPI_16 = 0,       // out 16-bit (half if op_f16, else bf16) = acc
  EPI_F32 = 1,      // out f32 = acc
  EPI_F32_ADD = 2,  // out f32 = add_src + acc   (residual; add_src may alias out)
  EPI_F32_ACC = 3   // out f32 += acc
};

struct GemmArgs {
  int mode = GEMM_FWD;
  int op_f16 = 0;               // 16-bit operands (a, ul, vl, 16-bit out) are half, else bf16
  int M = 0;
  const uint16_t *a = nullptr;  // [M, Kg], row stride lda elements
  int lda = 0;
  // base weight W [Nw, Kw] (out x in)
  int wfmt = W_NF4;
  const uint8_t *codes = nullptr;   // NF4: [Nw*Kw/2]
  const float *absmax = nullptr;    // NF4: [Nw*Kw/64]
  const uint16_t *w = nullptr;      // bf16: [Nw, Kw], row stride ldw (0 = Kw)
  int ldw = 0;
  int Nw = 0, Kw = 0;
  // LoRA extension: y += ul[M, R] . vl, R a multiple of 64 (0 = none).
  // FWD: vl is [Ng, R] (row n holds the LoRA "B" row of output n, zero-padded);
  // DX:  vl is [R, Ng] (row j holds A's row j).
  const uint16_t *ul = nullptr;
  const uint16_t *vl = nullptr;
  int R = 0;
  int epi = EPI_16;
  void *out = nullptr;
  int ldo = 0;
  const float *add_src = nullptr;
  int ld_add = 0;
  int *err = nullptr;              // device int: kernels OR error bits into it
  // split-K scratch (optional): float buffer the kernel may use for partial tiles when the
  // output grid under-fills the GPU; splits is chosen by gemm_launch
  float *part = nullptr;
  size_t part_floats = 0;
  int splits_allowed = 1;
  int splits = 1;
  int mtiles = 1;                  // 128-row m-tiles per CTA (1 or 2), chosen by gemm_launch
  // LoRA term in float for the small-M path (which ignores ul / vl / R):
  //   FWD y[m, n]  += s * sum_j lora_u[m, p r + j] * B_p[n - off_p, j]   (lora_u = x A^T)
  //   DX  dx[m, k] += sum_p sum_j lora_u[m, p r + j] * A_p[j, k]          (lora_u = s dY B)
  // lseg.nseg == 0: no LoRA term on that path.
  const float *lora_u = nullptr;   // [M, nseg * r]
  LoraSeg lseg;
  // set when the kernel enqueued just before this GEMM is the LoRA projection that writes
  // lora_u (k_lora_down / k_lora_du): the small-M path then overlaps with it
  int after_lora = 0;
  // derived: Ng = output columns, Kg = reduction length
  int Ng() const { return mode == GEMM_FWD ? Nw : Kw; }
  int Kg() const { return mode == GEMM_FWD ? Kw : Nw; }
};

// Algorithmic work of one call (for the roofline): flops and compulsory bytes.
double gemm_flops(const GemmArgs &g);
double gemm_bytes(const GemmArgs &g);

// Enqueue one GEMM on `stream`.  Chooses the tcgen05 kernel when the shape allows it and the
// tiled fallback otherwise.  Returns 0 or a negative SOUP_E* code (message set).
int gemm_launch(const GemmArgs &g, cudaStream_t stream);
// 1 if gemm_launch would take the tensor-core path for this shape.
int gemm_uses_tc(const GemmArgs &g);
// Split-K factor gemm_launch picks for this call (1 = none).
int choose_splits(const GemmArgs &g, int bn);
// 128-row m-tiles per CTA (1 or 2) gemm_launch picks for this call.
int choose_mtiles(const GemmArgs &g, int bn);
int gemm_launch_tc(const GemmArgs &g, cudaStream_t stream);
// Force the fallback path (tests compare the two).
void gemm_force_fallback(int on);

// 2-D tiled TMA tensor map of a row-major [outer, inner] array (element type dt, rows
// row_bytes apart), box [box_outer, box_inner]; 0 or SOUP_E* with the message set.
int tmap_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
            uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw,
            const char *what);

// 3-D tiled TMA tensor map of a row-major [d2, d1, d0] array (rows of d0 elements stride1
// bytes apart, d1 rows per outer index, outer indices stride2 bytes apart), box
// [1, box1, box0]; rows past d1 read as zero.  0 or SOUP_E* with the message set.
int tmap_3d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t d0, uint64_t d1,
            uint64_t d2, uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1,
            CUtensorMapSwizzle sw, const char *what);

// Small-M path (1 <= M <= 16, NF4 weights; forward on half activations, dX on bf16
// gradients): weight-stationary mma.sync kernels, stream-K over the weight.  gemm_launch takes
// it whenever gemv_eligible() holds.
constexpr int GV_MAX_CTAS = 8 * 160;
// Float scratch the small-M path needs in GemmArgs::part (upper bound over devices).
size_t gemv_part_floats(int mode);
int gemv_eligible(const GemmArgs &g);
int gemv_launch(const GemmArgs &g, cudaStream_t stream);

}  // namespace soup
