"""Pins of the oracle's layer maths against closed forms, invariants, brute force and
finite differences (float64), so a dropped term, a wrong sign or index, or a transposed
operand anywhere in the forward or the hand-derived backward fails one of them."""
import math

import numpy as np
import pytest

from oracle import model, nf4
import synth

TINY = synth.TINY


def _tiny_weights(dtype, cfg=TINY):
    src = [synth.layer_source(cfg, i) for i in range(cfg.n_layers)]
    return model.weights_from_source(cfg, src, synth.embedding(cfg), synth.lm_head(cfg),
                                     synth.final_norm(cfg), dtype)


def test_b_zero_reproduces_base_exactly():
    cfg = TINY
    W = _tiny_weights(np.float32)
    tok = synth.tokens(cfg)
    lora0 = synth.lora_params(cfg, b_zero=True)
    a = model.forward(cfg, W, tok, lora0, keep_cache=False)
    b = model.forward(cfg, W, tok, None, keep_cache=False)
    for x, y in zip(a["hs"], b["hs"]):
        assert np.array_equal(x, y)
    assert np.array_equal(a["logits"], b["logits"]) and a["loss"] == b["loss"]


def test_attention_single_position_returns_v_of_mapped_head():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((2, 1, 4, 8))
    k = rng.standard_normal((2, 1, 2, 8))
    v = rng.standard_normal((2, 1, 2, 8))
    o, _ = model.attention(q, k, v)
    # heads 0,1 read kv head 0; heads 2,3 read kv head 1
    for h, g in ((0, 0), (1, 0), (2, 1), (3, 1)):
        assert np.array_equal(o[:, 0, h], v[:, 0, g])


def test_attention_zero_queries_is_causal_running_mean():
    rng = np.random.default_rng(1)
    S = 7
    q = np.zeros((1, S, 2, 4))
    k = rng.standard_normal((1, S, 1, 4))
    v = rng.standard_normal((1, S, 1, 4))
    o, _ = model.attention(q, k, v)
    want = np.cumsum(v[0, :, 0], axis=0) / np.arange(1, S + 1)[:, None]
    np.testing.assert_allclose(o[0, :, 0], want, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o[0, :, 1], want, rtol=1e-12, atol=1e-12)


def test_attention_brute_force_scalar_loops():
    rng = np.random.default_rng(2)
    B, S, nh, nkv, d = 1, 5, 4, 2, 3
    q = rng.standard_normal((B, S, nh, d))
    k = rng.standard_normal((B, S, nkv, d))
    v = rng.standard_normal((B, S, nkv, d))
    o, _ = model.attention(q, k, v)
    for h in range(nh):
        g = h // (nh // nkv)
        for i in range(S):
            sc = [sum(q[0, i, h, t] * k[0, j, g, t] for t in range(d)) / math.sqrt(d) for j in range(i + 1)]
            mx = max(sc)
            e = [math.exp(x - mx) for x in sc]
            z = sum(e)
            for t in range(d):
                want = sum(e[j] / z * v[0, j, g, t] for j in range(i + 1))
                assert abs(o[0, i, h, t] - want) < 1e-12


def test_rope_identity_at_zero_norm_preserving_and_relative():
    d, S = 16, 12
    cos, sin = model.rope_tables(S, d, 10000.0, np.float64)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((1, S, 1, d))
    y = model.rope(x, cos, sin)
    assert np.allclose(y[0, 0], x[0, 0])
    half = d // 2
    np.testing.assert_allclose(x[..., :half] ** 2 + x[..., half:] ** 2,
                               y[..., :half] ** 2 + y[..., half:] ** 2, rtol=1e-12)
    # <rope(q, m), rope(k, n)> depends only on m - n
    qv = rng.standard_normal(d)
    kv = rng.standard_normal(d)
    Q = model.rope(np.broadcast_to(qv, (1, S, 1, d)).copy(), cos, sin)[0, :, 0]
    K = model.rope(np.broadcast_to(kv, (1, S, 1, d)).copy(), cos, sin)[0, :, 0]
    for delta in (0, 1, 3):
        vals = [Q[m] @ K[m - delta] for m in range(delta, S)]
        np.testing.assert_allclose(vals, vals[0], rtol=1e-10, atol=1e-12)
    # backward is the transpose: <rope(x), g> == <x, rope_backward(g)>
    g = rng.standard_normal(y.shape)
    assert abs(np.sum(y * g) - np.sum(x * model.rope_backward(g, cos, sin))) < 1e-10


def test_rmsnorm_unit_rms():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5, 64)) * 3.0
    y, _ = model.rmsnorm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-12)


def test_uniform_logits_give_ln_vocab():
    V = 37
    logits = np.zeros((2, 9, V))
    tok = np.random.default_rng(5).integers(0, V, (2, 9))
    loss, _ = model.loss_of(logits, tok)
    assert abs(loss - math.log(V)) < 1e-12


def test_loss_brute_force():
    rng = np.random.default_rng(6)
    B, S, V = 2, 4, 6
    logits = rng.standard_normal((B, S, V))
    tok = rng.integers(0, V, (B, S))
    total, n = 0.0, 0
    for b in range(B):
        for t in range(S - 1):
            z = logits[b, t]
            total += -math.log(math.exp(z[tok[b, t + 1]]) / sum(math.exp(x) for x in z))
            n += 1
    assert abs(model.loss_of(logits, tok)[0] - total / n) < 1e-12


def test_layer_with_zero_output_projections_is_identity():
    cfg = TINY
    W = _tiny_weights(np.float64).layers[0]
    W = dict(W)
    W["o"] = np.zeros_like(W["o"])
    W["down"] = np.zeros_like(W["down"])
    rng = np.random.default_rng(7)
    h = rng.standard_normal((1, 8, cfg.hidden))
    cos, sin = model.rope_tables(8, cfg.head_dim, cfg.rope_theta, np.float64)
    out, _ = model.layer_forward(h, W, None, cfg, cos, sin)
    assert np.array_equal(out, h)


def test_lora_linear_matches_merged_weight():
    # y = x W^T + s (x A^T) B^T must equal x (W + s B A)^T
    rng = np.random.default_rng(8)
    x, W = rng.standard_normal((5, 12)), rng.standard_normal((7, 12))
    A, Bm = rng.standard_normal((3, 12)), rng.standard_normal((7, 3))
    y, _ = model.lora_linear(x, W, A, Bm, 2.0)
    np.testing.assert_allclose(y, x @ (W + 2.0 * Bm @ A).T, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", [0])
def test_finite_difference_gradients_float64(seed):
    """Central differences of the float64 loss on ~200 LoRA entries across both layers
    and all seven projections against the hand-derived backward."""
    cfg = TINY
    W = _tiny_weights(np.float64)
    tok = synth.tokens(cfg)
    lora = [[(a.astype(np.float64), b.astype(np.float64)) for a, b in layer]
            for layer in synth.lora_params(cfg)]
    fwd = model.forward(cfg, W, tok, lora, dtype=np.float64)
    grads, _ = model.backward(cfg, W, tok, lora, fwd, dtype=np.float64)
    rng = np.random.default_rng(seed)
    picks = []
    for li in range(cfg.n_layers):
        for pi in range(7):
            for which in (0, 1):
                shape = lora[li][pi][which].shape
                for _ in range(7):
                    picks.append((li, pi, which, tuple(int(rng.integers(0, s)) for s in shape)))
    fd, an = [], []
    for li, pi, which, idx in picks:
        t = lora[li][pi][which]
        h = 1e-3 * float(np.sqrt(np.mean(t * t)))
        old = t[idx]
        t[idx] = old + h
        lp = model.forward(cfg, W, tok, lora, dtype=np.float64, keep_cache=False)["loss"]
        t[idx] = old - h
        lm = model.forward(cfg, W, tok, lora, dtype=np.float64, keep_cache=False)["loss"]
        t[idx] = old
        fd.append((lp - lm) / (2 * h))
        an.append(grads[li][pi][which][idx])
    fd, an = np.array(fd), np.array(an)
    assert len(fd) >= 190
    err = np.abs(fd - an)
    # absolute floor: the rounding error of a central difference, ~loss * 2^-52 / h, is
    # ~1e-9 for the B entries (h = 1e-3 * rms(B) ~ 1e-6, loss ~ 7)
    assert np.all(err <= 1e-5 * np.abs(an) + 1e-9), (err.max(), np.abs(an).max())
    assert np.linalg.norm(fd - an) / np.linalg.norm(an) < 1e-6


def test_silu_hand_values():
    # silu(x) = x * sigmoid(x): values worked by hand from e^-1 = 0.36787944117144233
    np.testing.assert_allclose(model.silu(np.array([0.0, 1.0, -1.0])),
                               [0.0, 1.0 / 1.36787944117144233, -1.0 / (1.0 + math.e)], rtol=1e-15)
    assert abs(model.silu(np.array([40.0]))[0] - 40.0) < 1e-12


def test_rope_pairs_and_frequencies_hand_worked():
    # head_dim 4, theta 1e4: pair (0, 2) turns by pos * 1, pair (1, 3) by pos * 1e4^(-1/2)
    cos, sin = model.rope_tables(4, 4, 10000.0, np.float64)
    pos = 3
    for i, want in ((0, [math.cos(3), 0, math.sin(3), 0]),
                    (1, [0, math.cos(0.03), 0, math.sin(0.03)]),
                    (2, [-math.sin(3), 0, math.cos(3), 0]),
                    (3, [0, -math.sin(0.03), 0, math.cos(0.03)])):
        x = np.zeros((1, 4, 1, 4))
        x[0, pos, 0, i] = 1.0
        np.testing.assert_allclose(model.rope(x, cos, sin)[0, pos, 0], want, atol=1e-15)


def test_rmsnorm_hand_worked():
    # x = (3, 4): mean square 12.5; eps inside the root: 1 / sqrt(13)
    y, r = model.rmsnorm(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]), 0.5)
    np.testing.assert_allclose(y, [[3 / math.sqrt(13), 8 / math.sqrt(13)]], rtol=1e-15)
    np.testing.assert_allclose(r, [[1 / math.sqrt(13)]], rtol=1e-15)


def test_identity_like_layer_reduces_to_closed_form():
    """q = k = 0 makes every causal score equal, so attention is the running mean of v; with
    v taking the first head_dim features, o = I, gate = 2 I, up = I and down = I the layer is
        h' = h + [mean_{s<=t} n1[s, :4], same],   h'' = h' + silu(2 n2) * n2
    with n1, n2 the RMS-normalised h, h'.  Checks which projection feeds which, the causal
    mask, both residuals and the gate/up order."""
    cfg = TINY.with_(hidden=8, inter=8, n_heads=2, n_kv_heads=1, head_dim=4, rms_eps=1e-5)
    H, S = 8, 5
    W = {"q": np.zeros((8, 8)), "k": np.zeros((4, 8)), "v": np.eye(4, 8), "o": np.eye(8),
         "gate": 2 * np.eye(8), "up": np.eye(8), "down": np.eye(8),
         "ln1": np.ones(8), "ln2": np.ones(8)}
    rng = np.random.default_rng(11)
    h = rng.standard_normal((1, S, H))
    cos, sin = model.rope_tables(S, 4, cfg.rope_theta, np.float64)
    out, _ = model.layer_forward(h, W, None, cfg, cos, sin)

    def norm(x):
        return x / np.sqrt((x * x).mean(-1, keepdims=True) + cfg.rms_eps)
    n1 = norm(h[0])
    run_mean = np.cumsum(n1[:, :4], axis=0) / np.arange(1, S + 1)[:, None]
    h1 = h[0] + np.concatenate([run_mean, run_mean], axis=1)
    n2 = norm(h1)
    want = h1 + (2 * n2) / (1 + np.exp(-2 * n2)) * n2
    np.testing.assert_allclose(out[0], want, rtol=1e-12, atol=1e-12)


def test_weights_from_source_maps_each_tensor():
    """Every projection lands under its own name with its [out, in] shape: the NF4 base stays
    within each 64-block's half-step of its own bf16 source (a swapped pair of equal-shape
    projections breaks that), and a bf16 base is the source itself."""
    cb = nf4.codebook().astype(np.float64)
    half_gap = float(np.max(np.diff(cb))) / 2
    for cfg in (TINY, TINY.with_(base_fmt="bf16")):
        W = _tiny_weights(np.float64, cfg)
        for i in range(cfg.n_layers):
            src = synth.layer_source(cfg, i)
            for p in model.PROJ:
                ref = nf4.bf16_to_f32(src[p]).astype(np.float64)
                got = W.layers[i][p]
                assert got.shape == cfg.proj_shape(p), (p, got.shape)
                if cfg.base_fmt == "bf16":
                    assert np.array_equal(got, ref), p
                else:
                    blocks = np.abs(ref.reshape(-1, 64)).max(axis=1, keepdims=True)
                    err = np.abs(got.reshape(-1, 64) - ref.reshape(-1, 64))
                    assert np.all(err <= blocks * half_gap * (1 + 1e-6)), (i, p)
            for n in ("ln1", "ln2"):
                assert np.array_equal(W.layers[i][n], nf4.bf16_to_f32(src[n]))
        assert np.array_equal(W.embed, nf4.bf16_to_f32(synth.embedding(cfg)))
        assert np.array_equal(W.lm_head, nf4.bf16_to_f32(synth.lm_head(cfg)))


def test_logits_of_identity_head_is_the_normalised_state():
    rng = np.random.default_rng(12)
    hL = rng.standard_normal((3, 4))
    w_f = np.array([1.0, 2.0, 0.5, 1.0])
    z, _ = model.logits_of(hL, w_f, 3.0 * np.eye(4), 1e-6)
    want = 3.0 * hL / np.sqrt((hL * hL).mean(-1, keepdims=True) + 1e-6) * w_f
    np.testing.assert_allclose(z, want, rtol=1e-13)
