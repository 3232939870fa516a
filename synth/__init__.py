"""Seeded synthetic inputs shared by the oracle-side tests, the GPU tests and the bench.

This module draws random numbers and nothing else: it holds none of the method's
arithmetic (no quantisation, no layer maths).  Every tensor has its own stream,
keyed by (kind, layer, tensor) through ``numpy.random.SeedSequence(seed,
spawn_key=...)``, so any one tensor can be regenerated alone, in any order.

Shapes and distributions follow the workloads described for the streamed LoRA step:
frozen base weights N(0, 0.02) rounded once to bf16 (the "source checkpoint"),
norm weights 1.0, LoRA A ~ U(-1/sqrt(in), 1/sqrt(in)), LoRA B ~ N(0, 1e-3),
tokens uniform in [0, vocab).
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

# Projection order used everywhere (host pointer tables, gradients, shards).
PROJ = ("q", "k", "v", "o", "gate", "up", "down")
# Source tensors of one decoder layer, in store order.
LAYER_TENSORS = PROJ + ("ln1", "ln2")

_KIND = {"layer": 1, "embed": 2, "lm_head": 3, "lora_a": 4, "lora_b": 5, "tokens": 6,
         "act": 7, "grad": 8}


@dataclasses.dataclass(frozen=True)
class Config:
    """Shape of a Llama-shaped decoder stack (all sizes in elements)."""
    name: str
    n_layers: int
    hidden: int
    inter: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    vocab: int
    tied: bool
    rope_theta: float
    rms_eps: float
    base_fmt: str          # "nf4" or "bf16"
    lora_r: int
    lora_alpha: float
    batch: int
    seq: int

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    def proj_shape(self, p: str) -> tuple[int, int]:
        """[out, in] of projection p."""
        H, I, d = self.hidden, self.inter, self.head_dim
        return {"q": (self.n_heads * d, H), "k": (self.n_kv_heads * d, H),
                "v": (self.n_kv_heads * d, H), "o": (H, self.n_heads * d),
                "gate": (I, H), "up": (I, H), "down": (H, I)}[p]

    def with_(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


# The five workloads.  Open points (eps, theta for the Qwen-shaped stacks, alpha where it
# is not given) take the readings recorded in the design notes.
TINY = Config("tiny-llama", 2, 256, 688, 4, 2, 64, 1024, False, 10000.0, 1e-5, "nf4",
              8, 16.0, 1, 64)
QWEN3B_BF16 = Config("qwen2.5-3b-bf16", 36, 2048, 11008, 16, 2, 128, 151936, True,
                     1_000_000.0, 1e-6, "bf16", 16, 32.0, 1, 512)
LLAMA8B = Config("llama3.1-8b-nf4", 32, 4096, 14336, 32, 8, 128, 128256, False, 500000.0,
                 1e-5, "nf4", 16, 32.0, 1, 512)
QWEN32B = Config("qwen-32b-nf4", 64, 5120, 27648, 40, 8, 128, 152064, False, 1_000_000.0,
                 1e-6, "nf4", 16, 32.0, 1, 1024)
CONFIGS = {c.name: c for c in (TINY, QWEN3B_BF16, LLAMA8B, QWEN32B)}

# Single-projection microbench: weights [N, K] and token counts M.
MICRO_SHAPES = ((14336, 4096), (4096, 14336))
MICRO_M = (1, 16, 128, 512, 2048, 8192)
MICRO_R = 16


def _rng(seed: int, kind: str, *key: int) -> np.random.Generator:
    ss = np.random.SeedSequence(seed, spawn_key=(_KIND[kind],) + tuple(int(k) for k in key))
    return np.random.Generator(np.random.PCG64(ss))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round-to-nearest-even, via torch's own cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact widening)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(seed: int, kind: str, key: tuple, shape, std: float) -> np.ndarray:
    g = _rng(seed, kind, *key)
    x = g.standard_normal(size=shape, dtype=np.float32)
    x *= np.float32(std)
    return to_bf16_bits(x)


def layer_source(cfg: Config, layer: int, seed: int = 0) -> dict:
    """bf16 bit patterns of one decoder layer's frozen tensors: 7 projections [out, in]
    drawn N(0, 0.02), and two RMSNorm weight vectors of ones."""
    out = {}
    for ti, p in enumerate(PROJ):
        out[p] = normal_bf16(seed, "layer", (layer, ti), cfg.proj_shape(p), 0.02)
    one = to_bf16_bits(np.ones(cfg.hidden, np.float32))
    out["ln1"] = one.copy()
    out["ln2"] = one.copy()
    return out


def layer_sources(cfg: Config, layers, seed: int = 0, threads: int | None = None) -> list:
    """Generate several layers in parallel threads (numpy releases the GIL while filling)."""
    layers = list(layers)
    threads = threads or min(len(layers), os.cpu_count() or 1)
    with _cf.ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
        return list(ex.map(lambda i: layer_source(cfg, i, seed), layers))


def embedding(cfg: Config, seed: int = 0) -> np.ndarray:
    return normal_bf16(seed, "embed", (0,), (cfg.vocab, cfg.hidden), 0.02)


def lm_head(cfg: Config, seed: int = 0) -> np.ndarray:
    """Untied output head [vocab, hidden]; a tied stack reuses the embedding."""
    if cfg.tied:
        return embedding(cfg, seed)
    return normal_bf16(seed, "lm_head", (0,), (cfg.vocab, cfg.hidden), 0.02)


def final_norm(cfg: Config) -> np.ndarray:
    return to_bf16_bits(np.ones(cfg.hidden, np.float32))


def lora_params(cfg: Config, seed: int = 0, b_zero: bool = False) -> list:
    """Per layer, per projection: (A [r, in] fp32 ~ U(+-1/sqrt(in)), B [out, r] fp32 ~ N(0,1e-3))."""
    out = []
    r = cfg.lora_r
    for layer in range(cfg.n_layers):
        row = []
        for ti, p in enumerate(PROJ):
            n_out, n_in = cfg.proj_shape(p)
            bound = 1.0 / np.sqrt(n_in)
            a = _rng(seed, "lora_a", layer, ti).uniform(-bound, bound, size=(r, n_in)).astype(np.float32)
            if b_zero:
                b = np.zeros((n_out, r), np.float32)
            else:
                b = (_rng(seed, "lora_b", layer, ti).standard_normal(size=(n_out, r), dtype=np.float32)
                     * np.float32(1e-3))
            row.append((a, b))
        out.append(row)
    return out


def tokens(cfg: Config, seed: int = 0) -> np.ndarray:
    """Token ids [batch, seq] int32, uniform in [0, vocab)."""
    g = _rng(seed, "tokens", cfg.batch, cfg.seq)
    return g.integers(0, cfg.vocab, size=(cfg.batch, cfg.seq), dtype=np.int64).astype(np.int32)


def activations_bf16(m: int, k: int, seed: int = 0, key: int = 0) -> np.ndarray:
    """bf16 bits of an [m, k] activation block ~ N(0, 1) (the microbench's x and dY)."""
    return normal_bf16(seed, "act", (m, k, key), (m, k), 1.0)


def micro_weight(n: int, k: int, seed: int = 0) -> np.ndarray:
    """bf16 bits of one [n, k] microbench projection weight ~ N(0, 0.02)."""
    return normal_bf16(seed, "layer", (1000 + n, k), (n, k), 0.02)


def micro_lora(n: int, k: int, r: int = MICRO_R, seed: int = 0):
    bound = 1.0 / np.sqrt(k)
    a = _rng(seed, "lora_a", 1000 + n, k).uniform(-bound, bound, size=(r, k)).astype(np.float32)
    b = (_rng(seed, "lora_b", 1000 + n, k).standard_normal(size=(n, r), dtype=np.float32)
         * np.float32(1e-3))
    return a, b
