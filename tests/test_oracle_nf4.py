"""Pins of the oracle's NF4 code against things other than itself: the normal CDF
(scipy.special.ndtr, the forward function, where the oracle uses the inverse), brute
force nearest-value search, hand-worked packing, torch's bf16 cast, and the store sizes
printed on the pages."""
import os

import numpy as np
from scipy.special import ndtr

from oracle import nf4, sizes
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_codebook_anchors_and_order():
    c = nf4.codebook()
    assert c.dtype == np.float32 and c.shape == (16,)
    assert c[0] == -1.0 and c[7] == 0.0 and c[15] == 1.0
    assert np.all(np.diff(c) > 0)
    assert (c < 0).sum() == 7 and (c > 0).sum() == 8


def test_codebook_is_normal_quantiles_at_even_probabilities():
    # Map the values back through the forward CDF: the positive ones must sit at 8 evenly
    # spaced probabilities from delta down towards 1/2, the negative ones at 7.
    c = nf4.codebook().astype(np.float64)
    # zmax is the quantile at delta; recover it from ndtr(zmax) == delta by bisection
    lo, hi = 0.0, 10.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if ndtr(mid) < nf4.DELTA:
            lo = mid
        else:
            hi = mid
    zmax = 0.5 * (lo + hi)
    pos = ndtr(c[8:][::-1] * zmax)             # descending probabilities
    neg = ndtr(-c[:7] * zmax)                  # c0 first: -c0 * zmax is the largest
    step_p = (nf4.DELTA - 0.5) / 8
    step_n = (nf4.DELTA - 0.5) / 7
    np.testing.assert_allclose(pos, nf4.DELTA - step_p * np.arange(8), atol=2e-7)
    np.testing.assert_allclose(neg, nf4.DELTA - step_n * np.arange(7), atol=2e-7)


def _nearest_code(q):
    """Brute force: index of the nearest codebook value, ties to the lower index."""
    c = nf4.codebook().astype(np.float64)
    d = np.abs(q.astype(np.float64)[..., None] - c)
    return d.argmin(axis=-1)


def test_codes_are_nearest_value_brute_force():
    rng = np.random.default_rng(1)
    x = synth.bf16_bits_to_f32(synth.to_bf16_bits(rng.standard_normal(64 * 400).astype(np.float32)))
    codes, absmax = nf4.quantize(x)
    q = (x.reshape(-1, 64) / absmax[:, None]).astype(np.float32).reshape(-1)
    want = _nearest_code(q)
    m = nf4.midpoints().astype(np.float64)
    # exact-midpoint rounding of the float32 midpoints may flip a value lying within
    # one float32 ulp of a midpoint; everywhere else the codes must be the nearest value
    near_mid = np.min(np.abs(q.astype(np.float64)[:, None] - m), axis=1) <= np.spacing(np.float32(1.0))
    assert np.array_equal(codes[~near_mid], want[~near_mid].astype(np.uint8))
    assert near_mid.mean() < 0.01


def test_half_step_bound():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(64 * 500) * 0.02).astype(np.float32)
    codes, absmax = nf4.quantize(x)
    w = nf4.dequantize(codes, absmax, x.size)
    c = nf4.codebook().astype(np.float64)
    gaps = np.diff(c)
    a = np.repeat(absmax, 64).astype(np.float64)
    q = x.astype(np.float64) / a
    k = np.clip(np.searchsorted(c, q) - 1, 0, 14)     # interval [c_k, c_k+1] holding q
    bound = a * gaps[k] / 2 + np.spacing(np.abs(w).astype(np.float32)).astype(np.float64) + 1e-30
    assert np.all(np.abs(x - w.astype(np.float64)) <= bound)


def test_codebook_values_round_trip_exactly():
    c = nf4.codebook()
    for a in (np.float32(0.037), np.float32(1.0), np.float32(3.5e-3)):
        x = (c[np.arange(64) % 16] * a).astype(np.float32)   # contains +-a, so absmax = a
        codes, absmax = nf4.quantize(x)
        assert absmax[0] == a
        assert np.array_equal(codes, (np.arange(64) % 16).astype(np.uint8))
        assert np.array_equal(nf4.dequantize(codes, absmax, 64), x)


def test_zero_block_and_tie_to_lower():
    codes, absmax = nf4.quantize(np.zeros(128, np.float32))
    assert np.all(codes == 7) and np.all(absmax == 0)
    assert np.all(nf4.dequantize(codes, absmax, 128) == 0)
    m = nf4.midpoints()
    for k in range(15):
        x = np.zeros(64, np.float32)
        x[0] = 1.0            # absmax 1, so x / absmax is exact
        x[1] = m[k]
        codes, _ = nf4.quantize(x)
        assert codes[1] == k, (k, codes[1])


def test_blocks_straddle_rows_and_partial_tail_is_padded():
    K = 96                                    # 1.5 blocks per row
    w = np.full((2, K), 1e-3, np.float32)
    w[0, 90] = 5.0                            # row 0's tail shares block 1 with row 1's head
    codes, absmax = nf4.quantize(w)
    assert absmax.shape == (3,)
    assert absmax[1] == np.float32(5.0)
    flat = nf4.dequantize(codes, absmax, w.size).reshape(2, K)
    assert np.all(flat[1, :32] == 0)          # 1e-3 / 5 rounds to the zero code
    assert np.all(flat[1, 32:] != 0)          # block 2 has absmax 1e-3
    # partial final block: 100 elements -> 2 blocks, tail codes are the zero code
    x = np.linspace(-1, 1, 100).astype(np.float32)
    codes, absmax = nf4.quantize(x)
    assert codes.size == 128 and np.all(codes[100:] == 7)
    assert absmax[1] == np.max(np.abs(x[64:]))


def test_pack_golden():
    lines = [l for l in open(os.path.join(GOLD, "nf4_pack.txt")) if not l.startswith("#")]
    codes = np.array(lines[0].split(":")[1].split(), np.uint8)
    want = np.array([int(b, 16) for b in lines[1].split(":")[1].split()], np.uint8)
    assert np.array_equal(nf4.pack(codes), want)
    assert np.array_equal(nf4.unpack(want, codes.size), codes)


def test_bf16_round_matches_torch_cast():
    import torch
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10.0,
                        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -1 - 2 ** -8, 0.0, -0.0,
                                  3.0e38, 1e-40, np.inf, -np.inf], np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = nf4.bf16_round(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert nf4.bf16_round(np.array([1 + 2 ** -8], np.float32))[0] == 1.0          # tie to even
    assert nf4.bf16_round(np.array([1 + 3 * 2 ** -8], np.float32))[0] == 1 + 2 ** -6


def _golden_sizes():
    out = {}
    for l in open(os.path.join(GOLD, "store_sizes.txt")):
        if l.startswith("#") or not l.strip():
            continue
        key, val, tol = l.split()[:3]
        out[key] = (float(val), float(tol))
    return out


def test_store_sizes_match_pages():
    g = _golden_sizes()
    # the bf16 3B store the pages print is exactly our bf16 byte count
    v, tol = g["qwen3b_bf16_store"]
    assert abs(sizes.store_payload_bytes(synth.QWEN3B_BF16) - v) <= tol * v
    # the pages' NF4 stores use one byte of scale per 64 weights; with that scale size our
    # weight counts reproduce their figures, which pins every projection shape
    for key, cfg in (("qwen3b_nf4_store_bnb", synth.QWEN3B_BF16), ("llama8b_nf4_store_bnb", synth.LLAMA8B)):
        v, tol = g[key]
        nw = sum(sizes.proj_numel(cfg).values()) * cfg.n_layers
        assert abs(nw * (0.5 + 1 / 64) - v) <= tol * v, key


def test_about_fourfold_and_large_layer_boundary():
    # "About Soup": NF4 shrinks the store about fourfold; "Read this first": 8B sits
    # below the ~165 MiB per-layer boundary, 32B above it
    cfg8 = synth.LLAMA8B
    nf = sizes.shard_payload_bytes(cfg8)
    bf = sizes.shard_payload_bytes(cfg8.with_(base_fmt="bf16"))
    assert 3.4 < bf / nf < 4.0
    assert nf < 165 * 2 ** 20 < sizes.shard_payload_bytes(synth.QWEN32B)
