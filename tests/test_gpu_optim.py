"""GPU parity of training over several steps: the AdamW kernel, gradient accumulation over
micro-batches and a multi-step run of the tiny stack, all through the C ABI.

Bars:
* AdamW against the float64 oracle fed the same float32 inputs (and the float32-rounded
  hyper-parameters): per element within a few float32 rounding steps of the terms involved
  (bounds derived below);
* accumulation: old + g in one float addition, so two accumulated micro-batches equal the
  float32 sum of the two separately computed gradients bit for bit;
* several optimizer steps streamed vs resident: every loss, adapter and moment bit for bit
  ("Layer streaming: fine-tune a model that does not fit in your card", "Bit-exact is two
  claims, not one");
* each step against the oracle, recomputed from the GPU's own adapters at that step (AdamW
  turns near-zero gradients into +-lr steps, so two runs that differ by rounding drift apart;
  checking step by step keeps the bars those of one step): loss within 1e-3 relative,
  accumulated gradients relative L2 <= 2e-2 and cosine >= 0.999, the update within float32
  rounding of the oracle's AdamW applied to the GPU's gradient.
"""
import numpy as np
import pytest

import synth
from oracle import model, optim

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

U = 2.0 ** -24  # float32 unit roundoff


def _f32(x):
    return float(np.float32(x))


def _adamw_tols(p0, g, m0, v0, t, lr, b1, b2, eps, wd, gs):
    """Per-element bounds for the float32 kernel against the float64 oracle.
    m, v: the scaled gradient, two products and the sum, plus g^2 for v — at most 4 (m) and 6
    (v) roundings of the terms' magnitudes (m's terms can cancel, so the bound is on the terms,
    not on m).  p: the update u = m_hat / D with D = sqrt(v_hat) + eps takes m's absolute
    error divided by D (doubled for the roundings of 1/(1 - b1^t) and the quotient), and a
    relative error from D (half of v's, the square root, the host-rounded 1/sqrt(1 - b2^t),
    the product and the sum) and from the quotient and lr/(1 - b1^t) — bounded by 32
    roundings of lr |u|; p's own two terms by 4 roundings."""
    gg = np.float64(gs) * g
    tm = 4 * U * (np.abs(b1 * m0) + np.abs((1 - b1) * gg))
    tv = 6 * U * (np.abs(b2 * v0) + np.abs((1 - b2) * gg * gg))
    p1, m1, v1 = optim.adamw_step(p0, g, m0, v0, t, lr, b1, b2, eps, wd, gs)
    bc1, bc2 = 1 - b1 ** t, 1 - b2 ** t
    D = np.sqrt(v1 / bc2) + eps
    u = (m1 / bc1) / D
    tp = 4 * U * (np.abs(p0) + np.abs(lr * wd * p0)) + 2 * lr * (tm / bc1) / D + 32 * U * lr * np.abs(u)
    return (p1, m1, v1), (tp, tm, tv)


@pytest.mark.parametrize("n,offset", [(1, 0), (3, 0), (4099, 0), (4099, 1), ((1 << 20) + 3, 0),
                                      (1 << 20, 1)])
@pytest.mark.parametrize("t,wd,gs", [(1, 0.0, 1.0), (7, 0.01, 0.5)])
def test_adamw_kernel_matches_oracle(n, offset, t, wd, gs):
    from nf4_dequant_gemm_blockwise_b300 import api
    rng = np.random.default_rng(n + 31 * t)
    p0 = (rng.standard_normal(n) * 0.05).astype(np.float32)
    scale = 10.0 ** rng.integers(-7, 0, size=n)
    g = (rng.standard_normal(n) * scale).astype(np.float32)
    g[rng.random(n) < 0.01] = 0.0  # exact zeros
    if t == 1:
        m0 = np.zeros(n, np.float32)
        v0 = np.zeros(n, np.float32)
    else:
        m0 = (rng.standard_normal(n) * scale * 0.3).astype(np.float32)
        v0 = ((rng.standard_normal(n) * scale) ** 2).astype(np.float32)
    lr, b1, b2, eps = _f32(2e-4), _f32(0.9), _f32(0.999), _f32(1e-8)
    wd, gs = _f32(wd), _f32(gs)

    def dev(x):  # offset 1 float: the buffers are 4- but not 16-byte aligned (scalar path)
        buf = torch.zeros(n + offset, dtype=torch.float32, device="cuda")
        buf[offset:] = torch.from_numpy(x).cuda()
        return buf, buf[offset:]
    (_, P), (_, G), (_, M), (_, V) = dev(p0), dev(g), dev(m0), dev(v0)
    api.adamw_step(P, G, M, V, n, t, lr, b1, b2, eps, wd, gs)
    torch.cuda.synchronize()
    got = [x.cpu().numpy().astype(np.float64) for x in (P, M, V)]
    want, tol = _adamw_tols(p0.astype(np.float64), g.astype(np.float64), m0.astype(np.float64),
                            v0.astype(np.float64), t, lr, b1, b2, eps, wd, gs)
    for name, a, b, tl in zip("pmv", got, want, tol):
        err = np.abs(a - b)
        bad = np.flatnonzero(err > tl)
        assert bad.size == 0, (name, bad[:5], err[bad[:5]], tl[bad[:5]])
    assert np.array_equal(G.cpu().numpy(), g)  # the gradient is read only


def test_adamw_zero_length_enqueues_nothing():
    from nf4_dequant_gemm_blockwise_b300 import api
    x = torch.zeros(4, device="cuda")
    y, m, v = torch.zeros(4, device="cuda"), torch.zeros(4, device="cuda"), torch.zeros(4, device="cuda")
    before = api.kernel_launches()
    api.adamw_step(x, y, m, v, 0, 1, 1e-3)
    assert api.kernel_launches() == before


# ------------------------------------------------------------------------- the tiny stack
def _session(cfg, resident, store=None):
    from nf4_dequant_gemm_blockwise_b300.session import StreamedLoRA
    return StreamedLoRA(cfg, lambda i: synth.layer_source(cfg, i), synth.embedding(cfg),
                        synth.lm_head(cfg), synth.final_norm(cfg), synth.lora_params(cfg),
                        cfg.batch, cfg.seq, n_slots=2, resident=resident, store=store)


def _tok(cfg, seed):
    return torch.from_numpy(synth.tokens(cfg, seed=seed)).cuda()


def _rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _cos(a, b):
    a, b = np.asarray(a, np.float64).ravel(), np.asarray(b, np.float64).ravel()
    return float(a @ b / max(np.linalg.norm(a) * np.linalg.norm(b), 1e-300))


@pytest.fixture(scope="module")
def tiny_pair():
    cfg = synth.TINY
    s = _session(cfg, resident=False)
    r = _session(cfg, resident=True, store=s.store)
    W = model.weights_from_source(cfg, [synth.layer_source(cfg, i) for i in range(cfg.n_layers)],
                                  synth.embedding(cfg), synth.lm_head(cfg), synth.final_norm(cfg))
    yield cfg, s, r, W
    r.close()
    s.close()


def test_accumulate_adds_in_one_float_addition(tiny_pair):
    cfg, s, _, _ = tiny_pair
    t1, t2 = _tok(cfg, 21), _tok(cfg, 22)
    s.fwd(t1)
    s.bwd()
    s.sync()
    g1 = s.grad_flat.cpu().numpy()
    s.fwd(t2)
    s.bwd()
    s.sync()
    g2 = s.grad_flat.cpu().numpy()
    s.fwd(t1)
    s.bwd()
    s.fwd(t2)
    s.bwd(accumulate=True)
    s.sync()
    acc = s.grad_flat.cpu().numpy()
    assert np.abs(g1).max() > 0 and np.abs(g2).max() > 0
    assert np.array_equal(acc.view(np.uint32), (g1 + g2).view(np.uint32))


def _train(sess, cfg, steps, lr, wd, record=False):
    """Run the optimizer steps; with record, snapshot what the oracle needs at each step."""
    k = max(len(m) for m in steps)
    losses = torch.zeros(len(steps) * k, dtype=torch.float32, device="cuda")
    trace = []
    for t, micro in enumerate(steps):
        if not record:
            sess.train_step(micro, losses[t * k:], lr, weight_decay=wd)
            continue
        sess.sync()
        snap = {"adapters": sess.adapters(), "p": sess.params.cpu().numpy(),
                "m": sess.exp_avg.cpu().numpy(), "v": sess.exp_avg_sq.cpu().numpy()}
        sess.compute.wait_stream(torch.cuda.current_stream())
        for i, tok in enumerate(micro):
            B, S = tok.shape
            sess.stream.fwd(tok, B, S, sess.lora_A, sess.lora_B, losses[t * k + i:t * k + i + 1])
            sess.bwd(accumulate=i > 0)
        sess.sync()
        snap["g"] = sess.grad_flat.cpu().numpy()
        snap["grads"] = sess.grads()
        sess.optimizer_step(lr, weight_decay=wd, grad_scale=1.0 / len(micro))
        trace.append(snap)
    sess.sync()
    out = {"loss": losses.cpu().numpy(), "p": sess.params.cpu().numpy(),
           "m": sess.exp_avg.cpu().numpy(), "v": sess.exp_avg_sq.cpu().numpy()}
    return out, trace


def _bits(x):
    return np.asarray(x, np.float32).view(np.uint32)


def test_several_steps_streamed_equal_resident_and_track_the_oracle(tiny_pair):
    cfg, s, r, W = tiny_pair
    steps = [[_tok(cfg, 100 + 2 * t), _tok(cfg, 101 + 2 * t)] for t in range(3)]
    lr, wd = 1e-3, 0.01
    init = _flat_lora(cfg, s.n_params)
    _reset(s, init)
    _reset(r, init)
    a, _ = _train(s, cfg, steps, lr, wd)
    b, _ = _train(r, cfg, steps, lr, wd)
    for key in ("loss", "p", "m", "v"):
        assert np.array_equal(_bits(a[key]), _bits(b[key])), key
    moved = np.abs(a["p"] - init)
    assert moved.max() > 0.5 * lr and np.count_nonzero(moved) > 0.9 * np.count_nonzero(init)

    # the same run, step by step, against the oracle from the GPU's own state
    _reset(s, init)
    c, trace = _train(s, cfg, steps, lr, wd, record=True)
    for key in ("loss", "p", "m", "v"):  # recording changes nothing on the device
        assert np.array_equal(_bits(a[key]), _bits(c[key])), key
    b1, b2, eps = _f32(0.9), _f32(0.999), _f32(1e-8)
    for t, (snap, micro) in enumerate(zip(trace, steps), start=1):
        lora = snap["adapters"]
        per = []
        for i, tok in enumerate(micro):
            tk = tok.cpu().numpy()
            fwd = model.forward(cfg, W, tk, lora)
            got = float(c["loss"][(t - 1) * 2 + i])
            assert abs(got - fwd["loss"]) <= 1e-3 * fwd["loss"], (t, i, got, fwd["loss"])
            per.append(model.backward(cfg, W, tk, lora, fwd)[0])
        for li in range(cfg.n_layers):
            for p in range(7):
                for w in range(2):
                    want = optim.accumulate([g[li][p][w] for g in per])
                    got = snap["grads"][li][p][w]
                    assert _rel_l2(got, want) <= 2e-2, (t, li, p, w, _rel_l2(got, want))
                    assert _cos(got, want) >= 0.999, (t, li, p, w)
        nxt = trace[t] if t < len(trace) else c
        want, tol = _adamw_tols(snap["p"].astype(np.float64), snap["g"].astype(np.float64),
                                snap["m"].astype(np.float64), snap["v"].astype(np.float64), t,
                                _f32(lr), b1, b2, eps, _f32(wd), _f32(0.5))
        for name, w, tl in zip("pmv", want, tol):
            err = np.abs(nxt[name].astype(np.float64) - w)
            assert np.all(err <= tl), (t, name, float(err.max()))


def _reset(sess, init):
    """Fresh adapters and optimizer state, ordered before the session's next kernels."""
    sess.params.copy_(torch.from_numpy(init).cuda())
    sess.exp_avg.zero_()
    sess.exp_avg_sq.zero_()
    sess.opt_step = 0
    torch.cuda.synchronize()


def _flat_lora(cfg, n):
    """The session's flat adapter layout filled from the seeded adapters."""
    flat = [t for layer in synth.lora_params(cfg) for pair in layer for t in pair]
    host = np.zeros(n, np.float32)
    o = 0
    for t in flat:
        host[o:o + t.size] = t.ravel()
        o += -(-t.size // 64) * 64
    return host


def test_training_step_peak_memory_within_the_plan(tiny_pair):
    """"About Soup": peak device memory is bounded by one layer's working set plus the resident
    parts; soup_peak_bytes makes that bound exact for a training run (adapters, gradients and
    AdamW moments included).  Measured: torch's peak over building a session and one training
    step, less what the caller adds (token ids, loss buffers; 512-byte allocation rounding)."""
    from nf4_dequant_gemm_blockwise_b300 import api
    cfg = synth.TINY
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    tok = _tok(cfg, 5)
    losses = torch.zeros(1, dtype=torch.float32, device="cuda")
    sess = _session(cfg, resident=False)
    sess.train_step([tok], losses, 1e-3)
    sess.sync()
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated() - base
    sess.close()
    predicted, ws = api.peak_bytes(cfg, cfg.batch, cfg.seq, n_slots=2)
    n_tensors = 12  # device tensors the session and this test allocate
    assert peak <= predicted + 512 * n_tensors, (peak, predicted)
    assert peak >= predicted - ws  # the resident parts alone are allocated
