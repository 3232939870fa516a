"""GPU parity of the whole streamed LoRA step (forward + backward through the C ABI).

Bars ("Layer streaming: fine-tune a model that does not fit in your card", "Bit-exact is
two claims, not one"; "Read this first"):
* streamed vs resident on the GPU: logits, loss, every layer output, dL/dh at every layer
  boundary and every LoRA gradient bit for bit — forward and backward separately;
* GPU vs the float32 oracle: logits and layer outputs relative L2 <= 1e-2, logits max
  abs error <= 5e-2, LoRA gradients relative L2 <= 2e-2 and cosine >= 0.999 per tensor;
* a deliberately stale slot (the pages' control) must break the gradients.
The tiny stack is compared end to end with the oracle; the 8B-, 32B- and 3B-shaped stacks
(full sizes) layer by layer: the oracle recomputes sampled layers from the GPU's own layer
inputs and upstream gradients.
"""
import numpy as np
import pytest

import synth
from oracle import model, nf4

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL_FWD_REL = 1e-2
TOL_LOGIT_ABS = 5e-2
TOL_GRAD_REL = 2e-2
TOL_GRAD_COS = 0.999


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def cosine(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / max(np.linalg.norm(a) * np.linalg.norm(b), 1e-300))


def _session(cfg, resident, store=None, n_slots=2, lora=None, keep_activations=False):
    from nf4_dequant_gemm_blockwise_b300.session import StreamedLoRA
    return StreamedLoRA(cfg, lambda i: synth.layer_source(cfg, i), synth.embedding(cfg),
                        synth.lm_head(cfg), synth.final_norm(cfg),
                        lora if lora is not None else synth.lora_params(cfg),
                        cfg.batch, cfg.seq, n_slots=n_slots, resident=resident, store=store,
                        keep_activations=keep_activations)


def _run(sess, cfg, want_logits=True):
    M = cfg.batch * cfg.seq
    tok = torch.from_numpy(synth.tokens(cfg)).cuda()
    logits = torch.empty((M, cfg.vocab), dtype=torch.float32, device="cuda") if want_logits else None
    lay = torch.empty((cfg.n_layers + 1, M, cfg.hidden), dtype=torch.float32, device="cuda")
    dh = torch.empty_like(lay)
    sess.step(tok, logits=logits, layer_out=lay, dh_out=dh)
    sess.sync()
    out = {"loss": float(sess.loss.item()), "layers": lay.cpu().numpy(), "dh": dh.cpu().numpy(),
           "grads": sess.grads()}
    if want_logits:
        out["logits"] = logits.cpu().numpy()
    return out


def _assert_bit_equal(a, b):
    assert a["loss"] == b["loss"]
    assert np.array_equal(a["layers"].view(np.uint32), b["layers"].view(np.uint32))
    if "logits" in a and "logits" in b:
        assert np.array_equal(a["logits"].view(np.uint32), b["logits"].view(np.uint32))
    assert np.array_equal(a["dh"].view(np.uint32), b["dh"].view(np.uint32))
    n_exact = 0
    for la, lb in zip(a["grads"], b["grads"]):
        for (ga, gb), (ha, hb) in zip(la, lb):
            assert np.array_equal(ga.view(np.uint32), ha.view(np.uint32))
            assert np.array_equal(gb.view(np.uint32), hb.view(np.uint32))
            n_exact += 2
    return n_exact


# ----------------------------------------------------------------------------- tiny stack
@pytest.fixture(scope="module")
def tiny():
    cfg = synth.TINY
    s = _session(cfg, resident=False)
    r = _session(cfg, resident=True, store=s.store)
    out = {"cfg": cfg, "stream": _run(s, cfg), "resident": _run(r, cfg), "s": s, "r": r}
    # the oracle, end to end, float32
    W = model.weights_from_source(cfg, [synth.layer_source(cfg, i) for i in range(cfg.n_layers)],
                                  synth.embedding(cfg), synth.lm_head(cfg), synth.final_norm(cfg))
    tok = synth.tokens(cfg)
    lora = synth.lora_params(cfg)
    fwd = model.forward(cfg, W, tok, lora)
    grads, dhs = model.backward(cfg, W, tok, lora, fwd)
    out["oracle"] = {"fwd": fwd, "grads": grads, "dhs": dhs}
    yield out
    r.close()
    s.close()


def test_tiny_streamed_equals_resident_bitwise(tiny):
    n = _assert_bit_equal(tiny["stream"], tiny["resident"])
    assert n == 2 * 7 * tiny["cfg"].n_layers


def test_tiny_forward_matches_oracle(tiny):
    cfg, g, o = tiny["cfg"], tiny["stream"], tiny["oracle"]["fwd"]
    M = cfg.batch * cfg.seq
    for i in range(cfg.n_layers + 1):
        assert rel_l2(g["layers"][i], o["hs"][i].reshape(M, -1)) <= TOL_FWD_REL, i
    lo = o["logits"].reshape(M, -1)
    assert rel_l2(g["logits"], lo) <= TOL_FWD_REL
    assert np.abs(g["logits"] - lo).max() <= TOL_LOGIT_ABS
    assert abs(g["loss"] - o["loss"]) <= 1e-3 * o["loss"]


def test_tiny_backward_matches_oracle(tiny):
    cfg, g, o = tiny["cfg"], tiny["stream"], tiny["oracle"]
    for li in range(cfg.n_layers):
        for p in range(7):
            for w in range(2):
                got, want = g["grads"][li][p][w], o["grads"][li][p][w]
                assert rel_l2(got, want) <= TOL_GRAD_REL, (li, p, w, rel_l2(got, want))
                assert cosine(got, want) >= TOL_GRAD_COS, (li, p, w)
    M = cfg.batch * cfg.seq
    for i in range(cfg.n_layers + 1):
        assert rel_l2(g["dh"][i], o["dhs"][i].reshape(M, -1)) <= TOL_GRAD_REL, i


def test_tiny_repeat_step_is_deterministic(tiny):
    again = _run(tiny["s"], tiny["cfg"])
    _assert_bit_equal(tiny["stream"], again)


def test_tiny_stale_slot_control_is_caught(tiny):
    """The pages' repair was gated against a control that reproduced the defect; here a
    host switch makes the backward read a neighbouring layer's slot."""
    from nf4_dequant_gemm_blockwise_b300 import api
    s = tiny["s"]
    s.stream.debug(api.DBG_STALE_SLOT, 1)
    try:
        bad = _run(s, tiny["cfg"])
    finally:
        s.stream.debug(api.DBG_STALE_SLOT, 0)
    assert np.array_equal(bad["layers"], tiny["resident"]["layers"])      # forward still exact
    differs = sum(not np.array_equal(a[w], b[w]) for la, lb in zip(bad["grads"], tiny["resident"]["grads"])
                  for a, b in zip(la, lb) for w in range(2))
    assert differs > 0
    clean = _run(s, tiny["cfg"])
    _assert_bit_equal(clean, tiny["resident"])


def test_tiny_adapters_off_forward_is_the_base(tiny):
    """The reference forward of preference losses: the streamed base with the adapters
    switched off.  Streamed == resident bitwise; against the oracle with no LoRA at the forward
    bars; no backward may follow it; the next step with adapters is unaffected."""
    from nf4_dequant_gemm_blockwise_b300 import api
    cfg = tiny["cfg"]
    M = cfg.batch * cfg.seq
    tok = torch.from_numpy(synth.tokens(cfg)).cuda()
    outs = []
    for sess in (tiny["s"], tiny["r"]):
        logits = torch.empty((M, cfg.vocab), dtype=torch.float32, device="cuda")
        lay = torch.empty((cfg.n_layers + 1, M, cfg.hidden), dtype=torch.float32, device="cuda")
        loss = torch.zeros(1, dtype=torch.float32, device="cuda")
        sess.reference_fwd(tok, loss, logits=logits, layer_out=lay)
        sess.sync()
        outs.append((float(loss.item()), logits.cpu().numpy(), lay.cpu().numpy()))
        with pytest.raises(api.SoupError) as e:
            sess.bwd()
        assert e.value.code == api.ESTATE
    (ls, zs, hs), (lr_, zr, hr) = outs
    assert ls == lr_
    assert np.array_equal(zs.view(np.uint32), zr.view(np.uint32))
    assert np.array_equal(hs.view(np.uint32), hr.view(np.uint32))
    W = model.weights_from_source(cfg, [synth.layer_source(cfg, i) for i in range(cfg.n_layers)],
                                  synth.embedding(cfg), synth.lm_head(cfg), synth.final_norm(cfg))
    o = model.forward(cfg, W, synth.tokens(cfg), None, keep_cache=False)
    for i in range(cfg.n_layers + 1):
        assert rel_l2(hs[i], o["hs"][i].reshape(M, -1)) <= TOL_FWD_REL, i
    lo = o["logits"].reshape(M, -1)
    assert rel_l2(zs, lo) <= TOL_FWD_REL
    assert np.abs(zs - lo).max() <= TOL_LOGIT_ABS
    assert abs(ls - o["loss"]) <= 1e-3 * o["loss"]
    assert not np.array_equal(zs, tiny["stream"]["logits"])  # the adapters do change the output
    _assert_bit_equal(tiny["stream"], _run(tiny["s"], cfg))


def test_tiny_pageable_store_stays_exact(tiny):
    """The fallback when page-locking fails ("Layer streaming: fine-tune a model that does not
    fit in your card", "Measured numbers": pageable copies lose the overlap): the same shard
    bytes in a pageable arena stream to the same results, bit for bit."""
    from nf4_dequant_gemm_blockwise_b300 import api
    cfg = tiny["cfg"]
    paged = api.Store(cfg, force_pageable=True)
    for i in range(cfg.n_layers):
        paged.put_shard(i, tiny["s"].store.shard_bytes(i))
    assert paged.info()[2] is False
    s = _session(cfg, resident=False, store=paged)
    try:
        out = _run(s, cfg)
    finally:
        s.close()
        paged.free()
    _assert_bit_equal(tiny["resident"], out)


@pytest.mark.parametrize("resident", [False, True])
def test_tiny_kept_activations_equal_recompute_bitwise(tiny, resident):
    """"How it works": with stream_recompute off the backward uses the forward's activations
    of every layer instead of re-running each layer; the same kernels produced them from the
    same inputs, so every output and gradient is bitwise that of the recomputing stream."""
    s = _session(tiny["cfg"], resident=resident, store=tiny["s"].store, keep_activations=True)
    try:
        k1 = _run(s, tiny["cfg"])
        k2 = _run(s, tiny["cfg"])  # a second step over the kept buffers
    finally:
        s.close()
    _assert_bit_equal(tiny["stream"], k1)
    _assert_bit_equal(tiny["stream"], k2)


@pytest.mark.parametrize("batch,seq", [(1, 16), (2, 4)])
def test_small_token_count_step(batch, seq):
    """B*S <= 16 tokens: every base projection (the fused q/k/v with three LoRA segments, the
    residual-adding o and down projections, the dX GEMMs) takes the small-M path.  Same bars:
    bit-exact streamed vs resident, and the oracle tolerances."""
    cfg = synth.TINY.with_(batch=batch, seq=seq)
    s = _session(cfg, resident=False)
    r = _session(cfg, resident=True, store=s.store)
    try:
        gs, gr = _run(s, cfg), _run(r, cfg)
    finally:
        r.close()
        s.close()
    _assert_bit_equal(gs, gr)
    W = model.weights_from_source(cfg, [synth.layer_source(cfg, i) for i in range(cfg.n_layers)],
                                  synth.embedding(cfg), synth.lm_head(cfg), synth.final_norm(cfg))
    tok = synth.tokens(cfg)
    lora = synth.lora_params(cfg)
    fwd = model.forward(cfg, W, tok, lora)
    grads, dhs = model.backward(cfg, W, tok, lora, fwd)
    M = batch * seq
    for i in range(cfg.n_layers + 1):
        assert rel_l2(gs["layers"][i], fwd["hs"][i].reshape(M, -1)) <= TOL_FWD_REL, i
    lo = fwd["logits"].reshape(M, -1)
    assert rel_l2(gs["logits"], lo) <= TOL_FWD_REL
    assert np.abs(gs["logits"] - lo).max() <= TOL_LOGIT_ABS
    for li in range(cfg.n_layers):
        for p in range(7):
            for w in range(2):
                got, want = gs["grads"][li][p][w], grads[li][p][w]
                assert rel_l2(got, want) <= TOL_GRAD_REL, (li, p, w, rel_l2(got, want))
                assert cosine(got, want) >= TOL_GRAD_COS, (li, p, w)
    for i in range(cfg.n_layers + 1):
        assert rel_l2(gs["dh"][i], dhs[i].reshape(M, -1)) <= TOL_GRAD_REL, i


def test_tiny_b_zero_gives_exact_zero_dA():
    cfg = synth.TINY
    s = _session(cfg, resident=False, lora=synth.lora_params(cfg, b_zero=True))
    try:
        out = _run(s, cfg, want_logits=False)
    finally:
        s.close()
    for layer in out["grads"]:
        for dA, dB in layer:
            assert not dA.any()            # du = s dY B = 0 exactly
            assert np.abs(dB).max() > 0


def test_errors_are_reported():
    from nf4_dequant_gemm_blockwise_b300 import api
    cfg = synth.TINY
    s = _session(cfg, resident=False)
    try:
        with pytest.raises(api.SoupError) as e:
            s.bwd()
        assert e.value.code == api.ESTATE
        tok = torch.zeros((cfg.batch, cfg.seq * 2), dtype=torch.int32, device="cuda")
        with pytest.raises(api.SoupError) as e:
            s.fwd(tok)
        assert e.value.code == api.EINVAL
        small = torch.empty(1024, dtype=torch.uint8, device="cuda")
        with pytest.raises(api.SoupError) as e:
            api.Stream(s.store, 1, 64, small, s.embed, s.lm_head, s.final, s.compute, s.copy)
        assert e.value.code == api.ENOMEM
    finally:
        s.close()


# ----------------------------------------------------------------------------- full sizes
def _oracle_layer_check(cfg, g, li, M):
    """Recompute layer li in float32 from the GPU's own input h_li and upstream gradient."""
    src = synth.layer_source(cfg, li)
    W = model.weights_from_source(cfg, [src], synth.embedding(cfg.with_(vocab=2)),
                                  synth.embedding(cfg.with_(vocab=2)), synth.final_norm(cfg)).layers[0]
    lora = model.lora_dict(synth.lora_params(cfg.with_(n_layers=li + 1))[li], np.float32)
    cos, sin = model.rope_tables(cfg.seq, cfg.head_dim, cfg.rope_theta, np.float32)
    h_in = g["layers"][li].reshape(cfg.batch, cfg.seq, cfg.hidden)
    out, cache = model.layer_forward(h_in, W, lora, cfg, cos, sin)
    assert rel_l2(g["layers"][li + 1], out.reshape(M, -1)) <= TOL_FWD_REL, li
    dh_out = g["dh"][li + 1].reshape(cfg.batch, cfg.seq, cfg.hidden)
    dh_in, grads = model.layer_backward(dh_out, cache, W, lora, cfg, cos, sin)
    assert rel_l2(g["dh"][li], dh_in.reshape(M, -1)) <= TOL_GRAD_REL, li
    for p, name in enumerate(model.PROJ):
        for w in range(2):
            got, want = g["grads"][li][p][w], grads[name][w]
            assert rel_l2(got, want) <= TOL_GRAD_REL, (li, name, w, rel_l2(got, want))
            assert cosine(got, want) >= TOL_GRAD_COS, (li, name, w)


def _full_size(cfg, check_layers, logit_rows=64):
    M = cfg.batch * cfg.seq
    from nf4_dequant_gemm_blockwise_b300 import api
    from nf4_dequant_gemm_blockwise_b300.session import StreamedLoRA
    store = api.Store(cfg, allow_pageable=True)
    srcs = synth.layer_sources
    for i0 in range(0, cfg.n_layers, 8):
        for i, src in zip(range(i0, min(cfg.n_layers, i0 + 8)), srcs(cfg, range(i0, min(cfg.n_layers, i0 + 8)))):
            store.put_layer(i, [src[t] for t in synth.LAYER_TENSORS])
    lora = synth.lora_params(cfg)
    mk = lambda res: StreamedLoRA(cfg, None, synth.embedding(cfg), synth.lm_head(cfg), synth.final_norm(cfg),
                                  lora, cfg.batch, cfg.seq, n_slots=2, resident=res, store=store)
    s = mk(False)
    g = _run(s, cfg)
    s.close()
    torch.cuda.empty_cache()
    r = mk(True)
    gr = _run(r, cfg)
    r.close()
    n = _assert_bit_equal(g, gr)
    assert n == 14 * cfg.n_layers
    del gr
    for li in check_layers:
        _oracle_layer_check(cfg, g, li, M)
    # logits on sampled rows, loss from the full logits
    rows = np.linspace(0, M - 1, logit_rows).astype(int)
    w_lm = nf4.bf16_to_f32(synth.lm_head(cfg))
    lo, _ = model.logits_of(g["layers"][-1][rows], nf4.bf16_to_f32(synth.final_norm(cfg)), w_lm, cfg.rms_eps)
    assert rel_l2(g["logits"][rows], lo) <= TOL_FWD_REL
    assert np.abs(g["logits"][rows] - lo).max() <= TOL_LOGIT_ABS
    loss, _ = model.loss_of(g["logits"].reshape(cfg.batch, cfg.seq, -1), synth.tokens(cfg))
    assert abs(g["loss"] - loss) <= 1e-4 * loss
    store.free()


def test_llama8b_b1_full_size():
    cfg = synth.LLAMA8B
    _full_size(cfg, [0, 1, 15, 30, 31])


def test_qwen32b_large_layers_full_size():
    cfg = synth.QWEN32B
    _full_size(cfg, [0, 31, 63])


def test_qwen3b_bf16_full_size():
    cfg = synth.QWEN3B_BF16
    _full_size(cfg, [0, 35])
