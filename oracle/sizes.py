"""Byte counts the pages' memory claims rest on.

Pages: "About Soup" (only the LoRA adapters stay resident, so peak VRAM is bounded by a
single layer instead of the whole model; NF4 shrinks the store about fourfold) and
"Layer streaming: fine-tune a model that does not fit in your card", "How it works"
(embeddings, final norm, an untied head and the adapters with their gradients are the
resident tensors; N pre-allocated layer buffers).  These functions count payload bytes
from the format definition alone, with no alignment or workspace of any implementation.
"""
from __future__ import annotations

PROJ = ("q", "k", "v", "o", "gate", "up", "down")


def proj_numel(cfg) -> dict:
    return {p: cfg.proj_shape(p)[0] * cfg.proj_shape(p)[1] for p in PROJ}


def shard_payload_bytes(cfg) -> int:
    """One decoder layer in the store: NF4 = half a byte per weight plus one float32
    absmax per 64 weights; bf16 = two bytes per weight; plus the two bf16 norm vectors."""
    total = 0
    for n in proj_numel(cfg).values():
        if cfg.base_fmt == "nf4":
            total += (n + 1) // 2 + 4 * ((n + 63) // 64)
        else:
            total += 2 * n
    return total + 2 * 2 * cfg.hidden


def store_payload_bytes(cfg) -> int:
    return cfg.n_layers * shard_payload_bytes(cfg)


def lora_param_count(cfg) -> int:
    r = cfg.lora_r
    return cfg.n_layers * sum(r * (o + i) for o, i in (cfg.proj_shape(p) for p in PROJ))


def resident_bytes(cfg) -> int:
    """Embedding, untied head, final norm (bf16); LoRA A/B, their gradients and the two
    AdamW moments (float32) — everything of a training run but the streamed base."""
    emb = 2 * cfg.vocab * cfg.hidden
    head = 0 if cfg.tied else 2 * cfg.vocab * cfg.hidden
    return emb + head + 2 * cfg.hidden + 4 * 4 * lora_param_count(cfg)
