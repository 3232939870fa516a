"""NF4 blockwise quantisation, written from its definition.

Pages: "Layer streaming: fine-tune a model that does not fit in your card", sections
"Turn it on" (quantization 4bit = NF4, about 4x smaller store) and "How it works"
(the checkpoint is rewritten once into one shard per layer); "About Soup" (quantising
the streamed base to NF4 shrinks the store about fourfold).  The pages name the format
but print neither the codebook nor the block layout.  Readings taken here:

* codebook: the NormalFloat-4 construction of QLoRA (Dettmers et al. 2023): sixteen
  sorted values, eight positive ones at the standard-normal quantiles of eight evenly
  spaced probabilities running from delta down towards 1/2, seven negative ones mirrored
  from seven evenly spaced probabilities over the same range, and an exact zero; all
  divided by the largest, so the ends are -1 and +1.  delta = (1 - 1/32 + 1 - 1/30) / 2.
  Built in float64 and rounded once to float32.
* blocks of 64 consecutive elements of the row-major flattened tensor (blocks may
  straddle rows); one float32 absmax per block, not itself quantised.
* code of an element = number of codebook midpoints strictly below x / absmax, the
  quotient an IEEE float32 division; a value exactly on a midpoint takes the lower code.
  An all-zero block gets code 7 (zero) everywhere; a trailing partial block is padded
  with code 7.
* packing: byte j holds code 2j in its high nibble and code 2j+1 in its low nibble.
* dequantised weight = float32(c[code] * absmax), one rounding; the tensor-core operand
  is that value rounded to bf16 (round to nearest, ties to even).
"""
from __future__ import annotations

import numpy as np
from scipy.special import ndtri

BLOCK = 64
DELTA = 0.5 * ((1.0 - 1.0 / 32.0) + (1.0 - 1.0 / 30.0))


def codebook() -> np.ndarray:
    """The 16 NF4 values, ascending, float32 (see module docstring for the reading)."""
    pos = ndtri(np.linspace(DELTA, 0.5, 9, dtype=np.float64)[:-1])      # 8 values > 0
    neg = -ndtri(np.linspace(DELTA, 0.5, 8, dtype=np.float64)[:-1])     # 7 values < 0
    vals = np.sort(np.concatenate([neg, [0.0], pos]))
    vals = vals / vals.max()
    return vals.astype(np.float32)


def midpoints(cb: np.ndarray | None = None) -> np.ndarray:
    """m_k = float32((c_k + c_{k+1}) / 2), k = 0..14 (sum and halving in float64)."""
    c = (codebook() if cb is None else cb).astype(np.float64)
    return ((c[:-1] + c[1:]) * 0.5).astype(np.float32)


def quantize(x: np.ndarray):
    """Blockwise NF4 codes of a tensor.

    x: any-shape float32 array (the bf16 source widened to float32); it is flattened
    row-major.  Returns (codes uint8 [n_blocks*64], absmax float32 [n_blocks]).
    """
    flat = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    n = flat.size
    nb = (n + BLOCK - 1) // BLOCK
    pad = np.zeros(nb * BLOCK, np.float32)
    pad[:n] = flat
    blocks = pad.reshape(nb, BLOCK)
    absmax = np.abs(blocks).max(axis=1).astype(np.float32)
    m = midpoints()
    codes = np.full((nb, BLOCK), 7, np.uint8)
    nz = absmax > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (blocks[nz] / absmax[nz, None]).astype(np.float32)   # IEEE float32 divide
    # the code is the count of midpoints strictly below q, counted one midpoint at a time
    count = np.zeros(q.shape, np.uint8)
    below = np.empty(q.shape, bool)
    for mk in m:
        np.greater(q, mk, out=below)
        count += below.view(np.uint8)
    codes[nz] = count
    codes = codes.reshape(-1)
    codes[n:] = 7
    return codes, absmax


def pack(codes: np.ndarray) -> np.ndarray:
    """Two codes per byte, even-index code in the high nibble."""
    c = np.asarray(codes, np.uint8).reshape(-1)
    if c.size % 2:
        c = np.concatenate([c, np.array([7], np.uint8)])
    return ((c[0::2] << 4) | c[1::2]).astype(np.uint8)


def unpack(packed: np.ndarray, n: int) -> np.ndarray:
    p = np.asarray(packed, np.uint8).reshape(-1)
    c = np.empty(p.size * 2, np.uint8)
    c[0::2] = p >> 4
    c[1::2] = p & 0xF
    return c[:n]


def dequantize(codes: np.ndarray, absmax: np.ndarray, n: int) -> np.ndarray:
    """float32(c[code] * absmax) for the first n elements (flat order)."""
    cb = codebook()
    c = np.asarray(codes, np.uint8).reshape(-1)[:n]
    a = np.repeat(np.asarray(absmax, np.float32), BLOCK)[:n]
    return (cb[c] * a).astype(np.float32)


def quantize_tensor(w_bf16_bits: np.ndarray):
    """bf16 source tensor [out, in] -> (packed uint8 [numel/2], absmax float32)."""
    x = bf16_to_f32(w_bf16_bits)
    codes, absmax = quantize(x)
    return pack(codes[: x.size + (x.size % 2)]), absmax


def dequantize_tensor(packed: np.ndarray, absmax: np.ndarray, shape) -> np.ndarray:
    n = int(np.prod(shape))
    return dequantize(unpack(packed, n), absmax, n).reshape(shape)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even) and return them as float32.
    NaN is kept quiet; infinities pass through."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    out = (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32)
    nan = np.isnan(x)
    if nan.any():
        out = out.copy()
        out[nan] = np.float32(np.nan)
    return out
