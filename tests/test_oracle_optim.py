"""Pins of the oracle's AdamW and gradient accumulation against closed forms, an independent
library implementation (torch.optim.AdamW on the CPU), Adam's scale invariance, the
batch/accumulation identity of a mean loss and a first-order prediction of the loss change,
so a missing bias correction, a misplaced epsilon, swapped betas, a decay applied to the
wrong tensor or an unscaled accumulated gradient each fail one of them."""
import numpy as np
import pytest
import torch

from oracle import model, optim
import synth

TINY = synth.TINY


def _tiny_weights(dtype, cfg=TINY):
    src = [synth.layer_source(cfg, i) for i in range(cfg.n_layers)]
    return model.weights_from_source(cfg, src, synth.embedding(cfg), synth.lm_head(cfg),
                                     synth.final_norm(cfg), dtype)


@pytest.mark.parametrize("c", [3e-8, -1e-8, 2.5e-3, -4.0])
def test_constant_gradient_moves_by_lr_times_c_over_abs_c_plus_eps(c):
    # with a constant gradient c both bias-corrected moments are exact: m_hat = c and
    # v_hat = c^2, so every step moves p by -lr * c / (|c| + eps).  At |c| ~ eps this
    # separates eps outside the square root from eps inside it.
    lr, eps = 1e-3, 1e-8
    p0 = np.array([0.7, -0.2, 0.0])
    p, m, v = p0.copy(), np.zeros(3), np.zeros(3)
    for t in range(1, 6):
        p, m, v = optim.adamw_step(p, np.full(3, c), m, v, t, lr, eps=eps)
        want = p0 - t * lr * c / (abs(c) + eps)
        np.testing.assert_allclose(p, want, rtol=0, atol=1e-15 + 1e-12 * t * lr)


def test_two_steps_hand_worked():
    # t=2: m_hat = (b1 g1 + g2) / (1 + b1), v_hat = (b2 g1^2 + g2^2) / (1 + b2)
    b1, b2, lr, eps = 0.8, 0.95, 0.01, 1e-6
    g1, g2 = np.array([0.3, -2.0]), np.array([-0.1, 0.5])
    p0 = np.array([1.0, -1.0])
    p, m, v = optim.adamw_step(p0, g1, 0 * p0, 0 * p0, 1, lr, b1, b2, eps)
    p, m, v = optim.adamw_step(p, g2, m, v, 2, lr, b1, b2, eps)
    mh = (b1 * g1 + g2) / (1 + b1)
    vh = (b2 * g1 ** 2 + g2 ** 2) / (1 + b2)
    want = p0 - lr * g1 / (np.abs(g1) + eps) - lr * mh / (np.sqrt(vh) + eps)
    np.testing.assert_allclose(p, want, rtol=1e-14, atol=0)
    np.testing.assert_allclose(m, b1 * (1 - b1) * g1 + (1 - b1) * g2, rtol=1e-14)
    np.testing.assert_allclose(v, b2 * (1 - b2) * g1 ** 2 + (1 - b2) * g2 ** 2, rtol=1e-14)


def test_zero_gradient_is_pure_decoupled_decay():
    lr, wd = 0.05, 0.1
    p0 = np.array([2.0, -3.0, 0.5])
    p, m, v = p0.copy(), np.zeros(3), np.zeros(3)
    for t in range(1, 8):
        p, m, v = optim.adamw_step(p, np.zeros(3), m, v, t, lr, weight_decay=wd)
    np.testing.assert_allclose(p, p0 * (1 - lr * wd) ** 7, rtol=1e-14)
    assert not m.any() and not v.any()


def test_matches_torch_adamw_float64():
    rng = np.random.default_rng(3)
    shape = (5, 7)
    p0 = rng.standard_normal(shape)
    hp = dict(lr=3e-3, betas=(0.85, 0.99), eps=1e-7, weight_decay=0.02)
    t_p = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([t_p], foreach=False, **hp)
    p, m, v = p0.copy(), np.zeros(shape), np.zeros(shape)
    for t in range(1, 7):
        g = rng.standard_normal(shape) * 10.0 ** rng.integers(-6, 1)
        t_p.grad = torch.from_numpy(g.copy())
        opt.step()
        p, m, v = optim.adamw_step(p, g, m, v, t, hp["lr"], *hp["betas"], hp["eps"],
                                   hp["weight_decay"])
    st = opt.state[t_p]
    np.testing.assert_allclose(p, t_p.detach().numpy(), rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-13, atol=1e-300)


def test_scale_invariance_and_grad_scale():
    # Adam is invariant to scaling the gradient together with eps; grad_scale undoes a
    # scale applied to the gradient before the moments.
    rng = np.random.default_rng(4)
    p0, k = rng.standard_normal(9), 1024.0
    gs = [rng.standard_normal(9) for _ in range(4)]
    a = (p0.copy(), np.zeros(9), np.zeros(9))
    b = (p0.copy(), np.zeros(9), np.zeros(9))
    c = (p0.copy(), np.zeros(9), np.zeros(9))
    for t, g in enumerate(gs, start=1):
        a = optim.adamw_step(*a[:1], g, *a[1:], t, 0.01, eps=1e-6)
        b = optim.adamw_step(*b[:1], k * g, *b[1:], t, 0.01, eps=k * 1e-6)
        c = optim.adamw_step(*c[:1], k * g, *c[1:], t, 0.01, eps=1e-6, grad_scale=1.0 / k)
    np.testing.assert_allclose(b[0], a[0], rtol=1e-13)
    np.testing.assert_allclose(c[0], a[0], rtol=1e-13)
    np.testing.assert_allclose(c[1], a[1], rtol=1e-13)


def test_accumulated_micro_batches_equal_the_batched_gradient():
    # the loss is a mean over positions, so for two equal-length sequences the gradient of
    # the batch of both is half the sum of the two micro-batch gradients
    cfg = TINY.with_(seq=16)
    W = _tiny_weights(np.float64, cfg)
    lora = [[(a.astype(np.float64), b.astype(np.float64)) for a, b in layer]
            for layer in synth.lora_params(cfg)]
    rng = np.random.default_rng(5)
    tok = rng.integers(0, cfg.vocab, size=(2, cfg.seq)).astype(np.int32)

    def grads(t):
        f = model.forward(cfg, W, t, lora, dtype=np.float64)
        return model.backward(cfg, W, t, lora, f, dtype=np.float64)[0]

    both = grads(tok)
    g0, g1 = grads(tok[:1]), grads(tok[1:])
    for li in range(cfg.n_layers):
        for pi in range(7):
            for w in (0, 1):
                acc = optim.accumulate([g0[li][pi][w], g1[li][pi][w]])
                np.testing.assert_allclose(0.5 * acc, both[li][pi][w], rtol=1e-9,
                                           atol=1e-12 * np.abs(both[li][pi][w]).max())


def test_first_step_changes_the_loss_as_first_order_predicts():
    # the first AdamW step moves every entry by -lr g / (|g| + eps) (t = 1, no decay), so the
    # loss changes by -lr sum g^2 / (|g| + eps) to first order; lr = 0 leaves it unchanged
    cfg = TINY.with_(seq=16)
    W = _tiny_weights(np.float64, cfg)
    lora = synth.lora_params(cfg)
    tok = synth.tokens(cfg)[:, :16]
    f = model.forward(cfg, W, tok, [[(a.astype(np.float64), b.astype(np.float64)) for a, b in l]
                                    for l in lora], dtype=np.float64)
    g, _ = model.backward(cfg, W, tok, [[(a.astype(np.float64), b.astype(np.float64))
                                         for a, b in l] for l in lora], f, dtype=np.float64)
    eps, lr = 1e-8, 1e-6
    pred = -lr * sum(float(np.sum(x * x / (np.abs(x) + eps)))
                     for layer in g for pair in layer for x in pair)
    losses, _ = optim.train(cfg, W, [[tok], [tok]], lora, lr=lr, eps=eps, dtype=np.float64)
    assert pred < 0
    assert abs((losses[1] - losses[0]) / pred - 1.0) < 1e-2, (losses, pred)
    same, _ = optim.train(cfg, W, [[tok], [tok]], lora, lr=0.0, dtype=np.float64)
    assert same[0] == same[1] == losses[0]


def test_train_with_accumulation_takes_one_step_per_group():
    # two micro-batches of one sequence each, accumulated and scaled by 1/2, reach the same
    # parameters as one batch of both (the batched gradient identity above), float64
    cfg = TINY.with_(seq=16)
    W = _tiny_weights(np.float64, cfg)
    lora = synth.lora_params(cfg)
    rng = np.random.default_rng(6)
    tok = rng.integers(0, cfg.vocab, size=(2, cfg.seq)).astype(np.int32)
    _, acc = optim.train(cfg, W, [[tok[:1], tok[1:]]], lora, lr=1e-3, weight_decay=0.01,
                         dtype=np.float64)
    _, bat = optim.train(cfg, W, [[tok]], lora, lr=1e-3, weight_decay=0.01, dtype=np.float64)
    for la, lb in zip(acc, bat):
        for pa, pb in zip(la, lb):
            for x, y in zip(pa, pb):
                np.testing.assert_allclose(x, y, rtol=1e-7, atol=1e-12)
