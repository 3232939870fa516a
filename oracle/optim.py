"""AdamW on the LoRA parameters, and gradient accumulation over micro-batches.

TEST INFRASTRUCTURE ONLY (see the package header).

Pages: "Layer streaming: fine-tune a model that does not fit in your card" — "Measured
numbers" (the runs train the adapters with bitsandbytes' paged 8-bit AdamW), "Turn it on"
(at the same effective batch a real batch is preferred to accumulation) and "Full config"
(gradient_accumulation_steps above 1 is allowed).  "About Soup": only the LoRA adapters are trained.

Readings (the pages fix neither the optimizer's arithmetic nor its state format):

* The update is plain AdamW with full-precision state — Adam's bias-corrected moments
  (Kingma & Ba, "Adam: A Method for Stochastic Optimization", Algorithm 1) with the weight
  decay decoupled from the gradient (Loshchilov & Hutter, "Decoupled Weight Decay
  Regularization", Algorithm 2), the decay scaled by the learning rate.  The 8-bit paged
  state of the pages' optimizer is a memory format for small cards, not a different update.
  With step t counted from 1 and g the (scaled) gradient:

      m_t = b1 m_{t-1} + (1 - b1) g
      v_t = b2 v_{t-1} + (1 - b2) g^2
      p_t = p_{t-1} - lr * ( (m_t / (1 - b1^t)) / (sqrt(v_t / (1 - b2^t)) + eps)
                             + weight_decay * p_{t-1} )

* Gradient accumulation sums the micro-batches' gradients (each the gradient of that
  micro-batch's own mean loss); ``grad_scale`` (for example 1/steps) multiplies the sum
  before it enters the moments.

Arithmetic in float64.
"""
from __future__ import annotations

import numpy as np


def adamw_step(p, g, m, v, t, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
               grad_scale=1.0):
    """One AdamW step at step number t >= 1 (readings above).  Returns (p, m, v) as new
    float64 arrays; the inputs are not modified."""
    if t < 1:
        raise ValueError("AdamW step numbers start at 1")
    p = np.asarray(p, np.float64)
    g = np.asarray(g, np.float64) * grad_scale
    m = beta1 * np.asarray(m, np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, np.float64) + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    p_new = p - lr * (m_hat / (np.sqrt(v_hat) + eps) + weight_decay * p)
    return p_new, m, v


def accumulate(grads):
    """Sum of the micro-batches' gradients, in the order given ("Full config":
    gradient_accumulation_steps)."""
    out = np.zeros_like(np.asarray(grads[0], np.float64))
    for g in grads:
        out = out + np.asarray(g, np.float64)
    return out


def train(cfg, W, steps, lora, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
          dtype=np.float32):
    """Several optimizer steps of the LoRA adapters ("About Soup": only the adapters train).

    steps: list over optimizer steps of a list of micro-batch token arrays [B, S]; each
    micro-batch runs the forward and backward of ``model``, their gradients are summed
    (``accumulate``) and scaled by 1 / (number of micro-batches) before one ``adamw_step``
    per tensor.  The parameters are kept in ``dtype`` between steps (the library's float32
    master weights); the moments stay in float64.
    Returns (losses: list over micro-batches in order, final lora in ``dtype``)."""
    from . import model
    lora = [[(np.asarray(a, dtype).copy(), np.asarray(b, dtype).copy()) for a, b in layer]
            for layer in lora]
    state = [[[np.zeros(t.shape), np.zeros(t.shape)] for pair in layer for t in pair]
             for layer in lora]
    losses = []
    for t, micro in enumerate(steps, start=1):
        per_batch = []
        for tokens in micro:
            fwd = model.forward(cfg, W, tokens, lora, dtype=dtype)
            losses.append(float(fwd["loss"]))
            grads, _ = model.backward(cfg, W, tokens, lora, fwd, dtype=dtype)
            per_batch.append(grads)
        for li, layer in enumerate(lora):
            new_layer = []
            for pi, pair in enumerate(layer):
                new_pair = []
                for which, p in enumerate(pair):
                    g = accumulate([gb[li][pi][which] for gb in per_batch])
                    m, v = state[li][2 * pi + which]
                    p64, m, v = adamw_step(p, g, m, v, t, lr, beta1, beta2, eps, weight_decay,
                                           grad_scale=1.0 / len(micro))
                    state[li][2 * pi + which] = [m, v]
                    new_pair.append(p64.astype(dtype))
                new_layer.append(tuple(new_pair))
            lora[li] = new_layer
    return losses, lora
