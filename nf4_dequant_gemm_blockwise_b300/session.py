"""A streamed LoRA training step as a user drives it: build the host store once, keep the
resident tensors (embedding, head, final norm, LoRA A/B and their gradients) in device
memory, and run forward + backward through the C ABI.

"About Soup": only the adapters (plus embeddings, final norm and an untied head, per
"Layer streaming: fine-tune a model that does not fit in your card", "How it works") live
on the device; the frozen decoder layers stream from a page-locked host store.
"""
from __future__ import annotations

import numpy as np
import torch

from . import api

LAYER_TENSORS = ("q", "k", "v", "o", "gate", "up", "down", "ln1", "ln2")


def _bits_to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).cuda()


class StreamedLoRA:
    """cfg: any object with the stack's fields (see api.make_cfg).
    layer_source(i) -> dict of the nine bf16-bit host arrays of layer i.
    lora: list over layers of 7 (A [r, in], B [out, r]) float32 host arrays.
    keep_activations: keep every layer's activations for the backward instead of re-running
    each layer's forward ("How it works": stream_recompute: off); weights are still re-read.
    stream_head: the embedding and the untied head go into the store instead of device memory
    ("Measured numbers": they move into the store and reuse one device buffer); the embedding
    rows are gathered straight from the page-locked store."""

    def __init__(self, cfg, layer_source, embed_bits, lm_head_bits, final_bits, lora, max_batch,
                 max_seq, n_slots=2, resident=False, store=None, threads=0, keep_activations=False,
                 stream_head=False):
        self.cfg = cfg
        self.own_store = store is None
        if store is None:
            store = api.Store(cfg, allow_pageable=True)
            for i in range(cfg.n_layers):
                src = layer_source(i)
                store.put_layer(i, [src[t] for t in LAYER_TENSORS], n_threads=threads)
        self.store = store
        if stream_head:
            store.put_head(embed_bits, None if cfg.tied else lm_head_bits)
            self.embed = self.lm_head = None
        else:
            self.embed = _bits_to_dev(embed_bits)
            self.lm_head = None if cfg.tied else _bits_to_dev(lm_head_bits)
        self.final = _bits_to_dev(final_bits)
        # adapters, gradients and AdamW moments each live in one flat float buffer (tensors
        # at 256-byte aligned offsets), so the optimizer is a single launch over all of them
        shapes = [t.shape for layer in lora for pair in layer for t in pair]
        offs, n = [], 0
        for sh in shapes:
            offs.append(n)
            n += -(-int(np.prod(sh)) // 64) * 64
        self.n_params = n
        host = np.zeros(n, np.float32)
        flat = [t for layer in lora for pair in layer for t in pair]
        for o, t in zip(offs, flat):
            host[o:o + t.size] = np.asarray(t, np.float32).ravel()
        self.params = torch.from_numpy(host).cuda()
        self.grad_flat = torch.zeros(n, dtype=torch.float32, device="cuda")
        self.exp_avg = torch.zeros(n, dtype=torch.float32, device="cuda")
        self.exp_avg_sq = torch.zeros(n, dtype=torch.float32, device="cuda")
        self.opt_step = 0

        def views(buf):
            return [buf[o:o + int(np.prod(sh))].view(*sh) for o, sh in zip(offs, shapes)]
        pv, gv = views(self.params), views(self.grad_flat)
        self.lora_A, self.lora_B = pv[0::2], pv[1::2]
        self.dA, self.dB = gv[0::2], gv[1::2]
        nbytes = api.workspace_bytes(cfg, max_batch, max_seq, n_slots, resident, keep_activations,
                                     stream_head)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.compute = torch.cuda.Stream()
        self.copy = torch.cuda.Stream()
        self.loss = torch.zeros(1, dtype=torch.float32, device="cuda")
        self.stream = api.Stream(store, max_batch, max_seq, self.workspace, self.embed, self.lm_head,
                                 self.final, self.compute, self.copy, n_slots=n_slots,
                                 resident=resident, keep_activations=keep_activations,
                                 stream_head=stream_head)
        torch.cuda.synchronize()

    def fwd(self, tokens: torch.Tensor, logits=None, layer_out=None):
        B, S = tokens.shape
        self.compute.wait_stream(torch.cuda.current_stream())
        self.stream.fwd(tokens, B, S, self.lora_A, self.lora_B, self.loss, logits, layer_out)

    def reference_fwd(self, tokens: torch.Tensor, loss: torch.Tensor, logits=None, layer_out=None):
        """Forward of the frozen base with the adapters switched off, over the same stream (the
        reference model of preference losses); no backward may follow it."""
        B, S = tokens.shape
        self.compute.wait_stream(torch.cuda.current_stream())
        self.stream.fwd(tokens, B, S, None, None, loss, logits, layer_out)

    def bwd(self, dh_out=None, accumulate=False):
        """accumulate: add this backward's LoRA gradients to the ones held (micro-batches)."""
        self.stream.bwd(self.dA, self.dB, dh_out, accumulate=accumulate)

    def step(self, tokens: torch.Tensor, logits=None, layer_out=None, dh_out=None):
        self.fwd(tokens, logits, layer_out)
        self.bwd(dh_out)

    def optimizer_step(self, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
                       grad_scale=1.0):
        """One AdamW step of every adapter on the compute stream, after the backward."""
        self.opt_step += 1
        api.adamw_step(self.params, self.grad_flat, self.exp_avg, self.exp_avg_sq, self.n_params,
                       self.opt_step, lr, beta1, beta2, eps, weight_decay, grad_scale,
                       stream=self.compute)

    def train_step(self, micro_batches, losses: torch.Tensor, lr, **adamw):
        """One optimizer step over k micro-batches ("Layer streaming: fine-tune a model that
        does not fit in your card", "Full config": gradient_accumulation_steps): forward and
        backward of each, gradients summed, AdamW with the sum scaled by 1/k.  losses: device
        float [>= k], micro-batch i's loss lands in losses[i]."""
        k = len(micro_batches)
        for i, tok in enumerate(micro_batches):
            B, S = tok.shape
            self.compute.wait_stream(torch.cuda.current_stream())
            self.stream.fwd(tok, B, S, self.lora_A, self.lora_B, losses[i:i + 1])
            self.bwd(accumulate=i > 0)
        self.optimizer_step(lr, grad_scale=1.0 / k, **adamw)

    def adapters(self):
        """Host copies of the adapters: list over layers of 7 (A, B)."""
        L = self.cfg.n_layers
        A = [t.cpu().numpy() for t in self.lora_A]
        Bm = [t.cpu().numpy() for t in self.lora_B]
        return [[(A[i * 7 + p], Bm[i * 7 + p]) for p in range(7)] for i in range(L)]

    def sync(self, timeout_ms: int = 600000):
        self.stream.sync(timeout_ms)
        torch.cuda.current_stream().wait_stream(self.compute)

    def grads(self):
        """Host copies: list over layers of 7 (dA, dB)."""
        L = self.cfg.n_layers
        dA = [t.cpu().numpy() for t in self.dA]
        dB = [t.cpu().numpy() for t in self.dB]
        return [[(dA[i * 7 + p], dB[i * 7 + p]) for p in range(7)] for i in range(L)]

    def close(self):
        self.stream.free()
        if self.own_store:
            self.store.free()
