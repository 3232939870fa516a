// Internal view of the host layer store (opaque to C callers).
#pragma once
#include <stdint.h>

#include <vector>

#include "soup.h"

struct soup_store {
  soup_cfg cfg;
  soup_shard_layout lay;
  uint8_t *base = nullptr;  // one arena of n_layers * lay.stride bytes
  uint64_t bytes = 0;
  int pinned = 0;
  std::vector<char> filled;
  // the embedding and (untied) output head, bf16 [vocab, hidden] each, in their own
  // page-locked allocation (soup_store_put_head); head_dev is its device-side address
  uint8_t *head = nullptr;
  uint8_t *head_dev = nullptr;
  uint64_t head_bytes = 0;
};

namespace soup {
int validate_cfg(const soup_cfg *c);
void group_shapes(const soup_cfg *c, int n_out[4], int n_in[4]);
int shard_layout(const soup_cfg *c, soup_shard_layout *L);
int store_create(const soup_cfg *c, int allow_pageable, soup_store **out);
int store_put_layer(soup_store *st, int layer, const uint16_t *const *src, int n_threads);
int store_put_shard(soup_store *st, int layer, const void *shard, uint64_t bytes);
int store_put_head(soup_store *st, const uint16_t *embed, const uint16_t *lm_head);
void store_free(soup_store *st);
void nf4_quantize_host(const uint16_t *src, int64_t n, uint8_t *codes, float *absmax, int n_threads);
const float *nf4_midpoints();
}  // namespace soup
