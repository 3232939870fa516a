/* The C ABI used from plain C99 through include/soup.h alone, on a machine without a GPU:
 * every call here runs on the host (codebook, host quantiser, layouts, memory plan, a
 * pageable store, argument checks).  Prints "key value" lines that tests/test_lib_cpu.py
 * compares with the oracle. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "soup.h"

static uint16_t bf16_bits(float x) { /* round to nearest even */
  uint32_t u;
  memcpy(&u, &x, 4);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

int main(void) {
  printf("version %s\n", soup_version());
  float cb[16];
  if (soup_nf4_codebook(cb) != SOUP_OK) return 1;
  printf("codebook");
  for (int i = 0; i < 16; ++i) {
    uint32_t u;
    memcpy(&u, &cb[i], 4);
    printf(" %08x", u);
  }
  printf("\n");

  /* 130 values: two full 64-blocks and a padded tail */
  enum { N = 130 };
  uint16_t src[N];
  for (int i = 0; i < N; ++i) src[i] = bf16_bits((float)((i * 37) % 101 - 50) / 17.0f);
  uint8_t codes[(N + 1) / 2];
  float absmax[(N + 63) / 64];
  if (soup_nf4_quantize_host(src, N, codes, absmax, 1) != SOUP_OK) return 2;
  printf("codes");
  for (int i = 0; i < (N + 1) / 2; ++i) printf(" %02x", codes[i]);
  printf("\nabsmax");
  for (int i = 0; i < (N + 63) / 64; ++i) {
    uint32_t u;
    memcpy(&u, &absmax[i], 4);
    printf(" %08x", u);
  }
  printf("\n");

  soup_cfg cfg = {2, 256, 688, 4, 2, 64, 1024, 0, 10000.0f, 1e-5f, SOUP_FMT_NF4, 8, 16.0f};
  soup_shard_layout lay;
  if (soup_shard_layout_of(&cfg, &lay) != SOUP_OK) return 3;
  printf("stride %llu\n", (unsigned long long)lay.stride);

  uint64_t ws0 = 0, ws2 = 0, ws_bad = 0;
  if (soup_workspace_bytes(&cfg, 1, 64, 2, 0, &ws0) != SOUP_OK) return 4;
  if (soup_workspace_bytes(&cfg, 1, 64, 2, SOUP_MODE_KEEP_ACTIVATIONS, &ws2) != SOUP_OK) return 5;
  printf("workspace %llu %llu\n", (unsigned long long)ws0, (unsigned long long)ws2);
  printf("bad_mode %d\n", soup_workspace_bytes(&cfg, 1, 64, 2, 8, &ws_bad));
  uint64_t ws_part = 0;
  printf("peak %llu\n", (unsigned long long)soup_peak_bytes(&cfg, 1, 64, 2, 0, &ws_part));

  soup_store *st = NULL;
  if (soup_store_create(&cfg, SOUP_STORE_PAGEABLE, &st) != SOUP_OK) return 6;
  uint8_t *shard = calloc(1, lay.stride);
  if (!shard) return 7;
  shard[0] = 0x5a;
  for (int l = 0; l < cfg.n_layers; ++l)
    if (soup_store_put_shard(st, l, shard, lay.stride) != SOUP_OK) return 8;
  printf("short_shard %d\n", soup_store_put_shard(st, 0, shard, lay.stride - 16));
  void *base = NULL;
  uint64_t bytes = 0;
  int pinned = -1;
  if (soup_store_info(st, &base, &bytes, &pinned) != SOUP_OK) return 9;
  printf("store %llu %d %02x\n", (unsigned long long)bytes, pinned, ((uint8_t *)base)[lay.stride]);
  soup_store_free(st);
  free(shard);

  soup_adamw hp = {1e-3f, 0.9f, 0.999f, 1e-8f, 0.0f, 1.0f};
  printf("adamw_step0 %d\n", soup_adamw_step((float *)16, (const float *)32, (float *)48,
                                              (float *)64, 0, &hp, 0, 0));
  printf("last_error %s\n", soup_last_error());
  return 0;
}
