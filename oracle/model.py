"""Llama-shaped decoder stack with LoRA: forward, loss and hand-derived backward.

Pages: "Layer streaming: fine-tune a model that does not fit in your card" —
"How it works" (embeddings, final norm, untied head and the LoRA adapters are the only
resident tensors; each decoder layer is the model family's own layer, run unchanged on
the streamed weights; the backward needs W^T dL/dy, so each layer is read again),
"Honest scope" (plain LoRA on the decoder layers only), and "About Soup" (only the
LoRA adapters are trained).  The pages print no equations; the layer is the standard
pre-norm Llama block, and these readings fill what they leave open:

* h' = h + o(attn(rope(q(n1)), rope(k(n1)), v(n1))),  n1 = rmsnorm(h) * w1
  h'' = h' + down(silu(gate(n2)) * up(n2)),            n2 = rmsnorm(h') * w2
* every projection p: y = x W_p^T + s (x A_p^T) B_p^T with s = alpha / r, no bias,
  no dropout
* RMSNorm x / sqrt(mean(x^2) + eps) * w; RoPE rotates the pairs (i, i + d/2) by
  pos * theta^(-2i/d) (no frequency scaling); causal softmax attention with scale
  1/sqrt(d); query head h reads key/value head floor(h * n_kv / n_h)
* loss = mean over the B*(S-1) positions that have a next token of
  -log softmax(logits)[next token]
* only LoRA A and B receive gradients.

Everything runs in the dtype of the inputs (float32 for parity, float64 for the
finite-difference pins).  Nothing is fused, blocked or reordered.
"""
from __future__ import annotations

import numpy as np

PROJ = ("q", "k", "v", "o", "gate", "up", "down")


# --------------------------------------------------------------------------- pieces

def rmsnorm(x, w, eps):
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x * r * w, r


def rmsnorm_backward(dy, x, w, r):
    """x: input, r: 1/rms per row.  dx = r * (g - xh * mean(g * xh)), g = dy * w."""
    g = dy * w
    xh = x * r
    return r * (g - xh * np.mean(g * xh, axis=-1, keepdims=True))


def rope_tables(seq, head_dim, theta, dtype):
    """cos/sin [seq, d/2] of pos * theta^(-2i/d), angles formed in float64."""
    half = head_dim // 2
    inv = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / head_dim)
    ang = np.arange(seq, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(dtype), np.sin(ang).astype(dtype)


def rope(x, cos, sin):
    """x [B, S, nh, d]: rotate the pairs (i, i + d/2)."""
    half = x.shape[-1] // 2
    x1, x2 = x[..., :half], x[..., half:]
    c, s = cos[None, :, None, :], sin[None, :, None, :]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_backward(dy, cos, sin):
    """Transpose of the rotation: rotate by the negative angle."""
    half = dy.shape[-1] // 2
    d1, d2 = dy[..., :half], dy[..., half:]
    c, s = cos[None, :, None, :], sin[None, :, None, :]
    return np.concatenate([d1 * c + d2 * s, d2 * c - d1 * s], axis=-1)


def kv_head_of(h, n_heads, n_kv):
    return (h * n_kv) // n_heads


def attention(q, k, v):
    """Causal GQA attention.  q [B,S,nh,d], k/v [B,S,nkv,d] -> (o [B,S,nh,d], p [B,nh,S,S])."""
    B, S, nh, d = q.shape
    nkv = k.shape[2]
    scale = 1.0 / np.sqrt(d)
    mask = np.triu(np.ones((S, S), bool), 1)
    o = np.zeros_like(q)
    p_all = np.zeros((B, nh, S, S), q.dtype)
    for b in range(B):
        for h in range(nh):
            g = kv_head_of(h, nh, nkv)
            s = (q[b, :, h, :] @ k[b, :, g, :].T) * scale
            s = np.where(mask, -np.inf, s)
            s = s - s.max(axis=-1, keepdims=True)
            e = np.exp(s)
            p = e / e.sum(axis=-1, keepdims=True)
            p_all[b, h] = p
            o[b, :, h, :] = p @ v[b, :, g, :]
    return o, p_all


def attention_backward(do, q, k, v, p):
    B, S, nh, d = q.shape
    nkv = k.shape[2]
    scale = 1.0 / np.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(nh):
            g = kv_head_of(h, nh, nkv)
            P = p[b, h]
            dO = do[b, :, h, :]
            dv[b, :, g, :] += P.T @ dO
            dP = dO @ v[b, :, g, :].T
            dS = P * (dP - (dP * P).sum(axis=-1, keepdims=True))
            dq[b, :, h, :] = (dS @ k[b, :, g, :]) * scale
            dk[b, :, g, :] += (dS.T @ q[b, :, h, :]) * scale
    return dq, dk, dv


def silu(x):
    return x / (1.0 + np.exp(-x))


def silu_grad(x):
    sg = 1.0 / (1.0 + np.exp(-x))
    return sg * (1.0 + x * (1.0 - sg))


def lora_linear(x, W, A, B, s):
    """y = x W^T + s (x A^T) B^T; returns (y, u = x A^T)."""
    y = x @ W.T
    if A is None:
        return y, None
    u = x @ A.T
    return y + s * (u @ B.T), u


def lora_linear_backward(dy, x, u, W, A, B, s):
    """dx = dy W + s (dy B) A;  dB = s dy^T u;  dA = s (dy B)^T x."""
    dx = dy @ W
    if A is None:
        return dx, None, None
    du = s * (dy @ B)
    dx = dx + du @ A
    dB = s * (dy.T @ u)
    dA = du.T @ x
    return dx, dA, dB


# --------------------------------------------------------------------------- layer

def layer_forward(h, W, lora, cfg, cos, sin):
    """One decoder layer.  h [B,S,H]; W: dict of projection weights [out,in] and ln1/ln2;
    lora: dict p -> (A, B) or None.  Returns (h_out, cache)."""
    Bsz, S, H = h.shape
    nh, nkv, d = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    s = cfg.lora_alpha / cfg.lora_r
    M = Bsz * S
    lo = (lambda p: (None, None)) if lora is None else (lambda p: lora[p])
    c = {"h": h}
    x1, r1 = rmsnorm(h.reshape(M, H), W["ln1"], cfg.rms_eps)
    c["x1"], c["r1"] = x1, r1
    q, c["uq"] = lora_linear(x1, W["q"], *lo("q"), s)
    k, c["uk"] = lora_linear(x1, W["k"], *lo("k"), s)
    v, c["uv"] = lora_linear(x1, W["v"], *lo("v"), s)
    q = rope(q.reshape(Bsz, S, nh, d), cos, sin)
    k = rope(k.reshape(Bsz, S, nkv, d), cos, sin)
    v = v.reshape(Bsz, S, nkv, d)
    att, p = attention(q, k, v)
    c["q"], c["k"], c["v"], c["p"] = q, k, v, p
    att = att.reshape(M, nh * d)
    c["att"] = att
    o, c["uo"] = lora_linear(att, W["o"], *lo("o"), s)
    hm = h.reshape(M, H) + o
    c["hm"] = hm
    x2, r2 = rmsnorm(hm, W["ln2"], cfg.rms_eps)
    c["x2"], c["r2"] = x2, r2
    g, c["ug"] = lora_linear(x2, W["gate"], *lo("gate"), s)
    u, c["uu"] = lora_linear(x2, W["up"], *lo("up"), s)
    a = silu(g) * u
    c["g"], c["u"], c["a"] = g, u, a
    dn, c["ud"] = lora_linear(a, W["down"], *lo("down"), s)
    out = hm + dn
    return out.reshape(Bsz, S, H), c


def layer_backward(dh_out, c, W, lora, cfg, cos, sin):
    """Backward of layer_forward.  Returns (dh_in, grads: dict p -> (dA, dB))."""
    Bsz, S, H = dh_out.shape
    nh, nkv, d = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    s = cfg.lora_alpha / cfg.lora_r
    M = Bsz * S
    lo = (lambda p: (None, None)) if lora is None else (lambda p: lora[p])
    grads = {}
    dhm = dh_out.reshape(M, H)
    # down
    da, dA, dB = lora_linear_backward(dhm, c["a"], c["ud"], W["down"], *lo("down"), s)
    grads["down"] = (dA, dB)
    # SwiGLU
    dg = da * c["u"] * silu_grad(c["g"])
    du = da * silu(c["g"])
    dx2g, dA, dB = lora_linear_backward(dg, c["x2"], c["ug"], W["gate"], *lo("gate"), s)
    grads["gate"] = (dA, dB)
    dx2u, dA, dB = lora_linear_backward(du, c["x2"], c["uu"], W["up"], *lo("up"), s)
    grads["up"] = (dA, dB)
    dhm = dhm + rmsnorm_backward(dx2g + dx2u, c["hm"], W["ln2"], c["r2"])
    # o
    datt, dA, dB = lora_linear_backward(dhm, c["att"], c["uo"], W["o"], *lo("o"), s)
    grads["o"] = (dA, dB)
    dq, dk, dv = attention_backward(datt.reshape(Bsz, S, nh, d), c["q"], c["k"], c["v"], c["p"])
    dq = rope_backward(dq, cos, sin).reshape(M, nh * d)
    dk = rope_backward(dk, cos, sin).reshape(M, nkv * d)
    dv = dv.reshape(M, nkv * d)
    dx1 = 0
    for p, dy in (("q", dq), ("k", dk), ("v", dv)):
        dxp, dA, dB = lora_linear_backward(dy, c["x1"], c["u" + p], W[p], *lo(p), s)
        grads[p] = (dA, dB)
        dx1 = dx1 + dxp
    dh = dhm + rmsnorm_backward(dx1, c["h"].reshape(M, H), W["ln1"], c["r1"])
    return dh.reshape(Bsz, S, H), grads


# --------------------------------------------------------------------------- head and loss

def logits_of(hL, w_final, w_lm, eps):
    """logits = rmsnorm(h_L) * w_f @ W_lm^T; hL [M, H]."""
    xn, r = rmsnorm(hL, w_final, eps)
    return xn @ w_lm.T, (xn, r)


def loss_of(logits, tokens):
    """Mean next-token cross-entropy over the positions that have a label.
    logits [B, S, V]; tokens [B, S]."""
    Bsz, S, V = logits.shape
    z = logits[:, :-1, :]
    y = tokens[:, 1:]
    m = z.max(axis=-1, keepdims=True)
    lse = (m + np.log(np.exp(z - m).sum(axis=-1, keepdims=True)))[..., 0]
    zy = np.take_along_axis(z, y[..., None].astype(np.int64), axis=-1)[..., 0]
    return float(np.mean(lse - zy)), lse


def loss_backward(logits, tokens):
    """dL/dlogits: (softmax - onehot) / N on labelled positions, 0 on the last one."""
    Bsz, S, V = logits.shape
    n = Bsz * (S - 1)
    z = logits[:, :-1, :]
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    p = e / e.sum(axis=-1, keepdims=True)
    y = tokens[:, 1:].astype(np.int64)
    np.put_along_axis(p, y[..., None], np.take_along_axis(p, y[..., None], axis=-1) - 1.0, axis=-1)
    dz = np.zeros_like(logits)
    dz[:, :-1, :] = p / n
    return dz


# --------------------------------------------------------------------------- whole stack

class Weights:
    """Dense per-layer weights for the oracle, in a chosen dtype.

    layers[i] is a dict p -> [out, in] array plus ln1/ln2 [H]; embed, lm_head [V, H];
    final [H].  Built by the caller from the bf16 source (NF4-dequantised for an NF4
    base); see ``weights_from_source``.
    """

    def __init__(self, layers, embed, lm_head, final):
        self.layers, self.embed, self.lm_head, self.final = layers, embed, lm_head, final


def weights_from_source(cfg, sources, embed_bits, lm_bits, final_bits, dtype=np.float32):
    """Turn bf16 source tensors into the oracle's dense weights.  NF4 base: each
    projection is quantised and dequantised by oracle.nf4 (float32 values); bf16 base:
    the bf16 values themselves."""
    from . import nf4
    layers = []
    for src in sources:
        L = {}
        for p in PROJ:
            w = src[p]
            if cfg.base_fmt == "nf4":
                packed, absmax = nf4.quantize_tensor(w)
                L[p] = nf4.dequantize_tensor(packed, absmax, w.shape).astype(dtype)
            else:
                L[p] = nf4.bf16_to_f32(w).astype(dtype)
        L["ln1"] = nf4.bf16_to_f32(src["ln1"]).astype(dtype)
        L["ln2"] = nf4.bf16_to_f32(src["ln2"]).astype(dtype)
        layers.append(L)
    return Weights(layers, nf4.bf16_to_f32(embed_bits).astype(dtype),
                   nf4.bf16_to_f32(lm_bits).astype(dtype), nf4.bf16_to_f32(final_bits).astype(dtype))


def lora_dict(lora_layer, dtype):
    if lora_layer is None:
        return None
    return {p: (np.asarray(a, dtype), np.asarray(b, dtype)) for p, (a, b) in zip(PROJ, lora_layer)}


def forward(cfg, W, tokens, lora, dtype=np.float32, keep_cache=True):
    """Full forward.  tokens [B,S] int; lora: list over layers of 7 (A,B) pairs or None.
    Returns dict with loss, logits [B,S,V], hs (list of L+1 layer inputs/outputs), caches."""
    Bsz, S = tokens.shape
    cos, sin = rope_tables(S, cfg.head_dim, cfg.rope_theta, dtype)
    h = W.embed[tokens.astype(np.int64)].astype(dtype)
    hs, caches = [h], []
    for i in range(cfg.n_layers):
        h, c = layer_forward(h, W.layers[i], lora_dict(None if lora is None else lora[i], dtype),
                             cfg, cos, sin)
        hs.append(h)
        caches.append(c if keep_cache else None)
    M = Bsz * S
    logits, head_cache = logits_of(hs[-1].reshape(M, cfg.hidden), W.final, W.lm_head, cfg.rms_eps)
    logits = logits.reshape(Bsz, S, cfg.vocab)
    loss, _ = loss_of(logits, tokens)
    return {"loss": loss, "logits": logits, "hs": hs, "caches": caches, "head": head_cache,
            "cos": cos, "sin": sin}


def backward(cfg, W, tokens, lora, fwd, dtype=np.float32):
    """Full backward from the loss.  Returns (grads: list over layers of 7 (dA, dB)),
    dhs: list of dL/dh_i for i = 0..L (same indexing as fwd['hs']))."""
    Bsz, S = tokens.shape
    M = Bsz * S
    dz = loss_backward(fwd["logits"], tokens).reshape(M, cfg.vocab)
    xn, r = fwd["head"]
    dxn = dz @ W.lm_head
    dh = rmsnorm_backward(dxn, fwd["hs"][-1].reshape(M, cfg.hidden), W.final, r)
    dh = dh.reshape(Bsz, S, cfg.hidden)
    dhs = [None] * (cfg.n_layers + 1)
    dhs[-1] = dh
    grads = [None] * cfg.n_layers
    for i in reversed(range(cfg.n_layers)):
        ld = lora_dict(None if lora is None else lora[i], dtype)
        dh, g = layer_backward(dh, fwd["caches"][i], W.layers[i], ld, cfg, fwd["cos"], fwd["sin"])
        dhs[i] = dh
        grads[i] = None if g is None else [g[p] for p in PROJ]
    return grads, dhs
