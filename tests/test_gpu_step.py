"""GPU parity of the whole streamed LoRA step (forward + backward through the C ABI).

Bars ("Layer streaming: fine-tune a model that does not fit in your card", "Bit-exact is
two claims, not one"; "Read this first"):
* streamed vs resident on the GPU: logits, loss, every layer output, dL/dh at every layer
  boundary and every LoRA gradient bit for bit — forward and backward separately;
* GPU vs the float32 oracle: logits and layer outputs relative L2 <= 1e-2, logits max
  abs error <= 5e-2, LoRA gradients relative L2 <= 2e-2 and cosine >= 0.999 per tensor;
* a deliberately stale slot (the pages' control) must break the gradients.
The tiny stack is compared end to end with the oracle; the 8B-, 32B- and 3B-shaped stacks
(full sizes) layer by layer: the oracle recomputes every layer from the GPU's own layer inputs
and upstream gradients (tests/layer_oracle.py runs the layers on the host cores in parallel).
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


def _session(cfg, resident, store=None, n_slots=2, lora=None, keep_activations=False,
             stream_head=False):
    from nf4_dequant_gemm_blockwise_b300.session import StreamedLoRA
    return StreamedLoRA(cfg, lambda i: synth.layer_source(cfg, i), synth.embedding(cfg),
                        synth.lm_head(cfg), synth.final_norm(cfg),
                        lora if lora is not None else synth.lora_params(cfg),
                        cfg.batch, cfg.seq, n_slots=n_slots, resident=resident, store=store,
                        keep_activations=keep_activations, stream_head=stream_head)


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
def _assert_layer_figures(figs):
    """The oracle bars on every checked layer: output and dL/dh within the forward / gradient
    relative L2, every LoRA gradient within relative L2 2e-2 and cosine 0.999."""
    n = 0
    for per_layer in figs:
        for f in per_layer:
            assert f["out_rel"] <= TOL_FWD_REL, f
            assert f["dh_rel"] <= TOL_GRAD_REL, f
            for name, w, rel, cos in f["grads"]:
                assert rel <= TOL_GRAD_REL, (f["layer"], f["batch"], name, w, rel)
                assert cos >= TOL_GRAD_COS, (f["layer"], f["batch"], name, w, cos)
                n += 1
    return n


def _cases(cfg, runs, li):
    """The GPU's figures of layer li in each run, as the oracle's layer check takes them."""
    out = []
    for c, g in runs:
        B, S, H = c.batch, c.seq, c.hidden
        out.append({"h_in": g["layers"][li].reshape(B, S, H), "h_out": g["layers"][li + 1],
                    "dh_out": g["dh"][li + 1].reshape(B, S, H), "dh_in": g["dh"][li],
                    "grads": g["grads"][li]})
    return out


def _start_oracle(cfg, runs, layers=None, checks=None):
    """Queue the oracle's check of `layers` (default: every layer) of each run on host worker
    processes; the GPU work goes on meanwhile.  Returns the pool (pass it back to add more)."""
    import layer_oracle
    checks = checks or layer_oracle.LayerChecks(cfg.n_layers)
    checks.submit(cfg, range(cfg.n_layers) if layers is None else layers,
                  lambda li: _cases(cfg, runs, li))
    return checks


def _finish_oracle(checks, expected):
    """Wait for the queued checks and apply the bars; `expected` gradient tensors in all."""
    res = checks.results()
    n = _assert_layer_figures([res[li] for li in sorted(res)])
    assert n == expected


def _build_store(cfg):
    from nf4_dequant_gemm_blockwise_b300 import api
    store = api.Store(cfg, allow_pageable=True)
    for i0 in range(0, cfg.n_layers, 8):
        idx = list(range(i0, min(cfg.n_layers, i0 + 8)))
        for i, src in zip(idx, synth.layer_sources(cfg, idx)):
            store.put_layer(i, [src[t] for t in synth.LAYER_TENSORS])
    return store


def _full_run(cfg, store, lora, resident=False, n_slots=2, keep_activations=False, stream_head=False):
    from nf4_dequant_gemm_blockwise_b300.session import StreamedLoRA
    s = StreamedLoRA(cfg, None, synth.embedding(cfg), synth.lm_head(cfg), synth.final_norm(cfg), lora,
                     cfg.batch, cfg.seq, n_slots=n_slots, resident=resident, store=store,
                     keep_activations=keep_activations, stream_head=stream_head)
    try:
        return _run(s, cfg)
    finally:
        s.close()
        torch.cuda.empty_cache()


def _head_checks(cfg, g, logit_rows=64):
    """Logits on sampled rows against the oracle's head, the loss from the full logits."""
    M = cfg.batch * cfg.seq
    rows = np.linspace(0, M - 1, logit_rows).astype(int)
    w_lm = nf4.bf16_to_f32(synth.lm_head(cfg))
    lo, _ = model.logits_of(g["layers"][-1][rows], nf4.bf16_to_f32(synth.final_norm(cfg)), w_lm, cfg.rms_eps)
    assert rel_l2(g["logits"][rows], lo) <= TOL_FWD_REL
    assert np.abs(g["logits"][rows] - lo).max() <= TOL_LOGIT_ABS
    loss, _ = model.loss_of(g["logits"].reshape(cfg.batch, cfg.seq, -1), synth.tokens(cfg))
    assert abs(g["loss"] - loss) <= 1e-4 * loss


def _full_size(cfg):
    """Streamed == resident bit for bit on everything, and every layer against the oracle (on
    the host cores while the GPU runs the resident comparison)."""
    store = _build_store(cfg)
    lora = synth.lora_params(cfg)
    try:
        g = _full_run(cfg, store, lora)
        checks = _start_oracle(cfg, [(cfg, g)])
        n = _assert_bit_equal(g, _full_run(cfg, store, lora, resident=True))
        assert n == 14 * cfg.n_layers
        _head_checks(cfg, g)
        _finish_oracle(checks, 14 * cfg.n_layers)
    finally:
        store.free()


# layers of the 8B stack at B=4 checked against the oracle (every layer is checked at B=1)
B4_ORACLE_LAYERS = (0, 1, 8, 15, 23, 30, 31)


def test_llama8b_full_size():
    """The 8B-shaped stack at both of its batch sizes (B=1 and B=4, S=512): streamed == resident
    bit for bit with two slots, with eight slots and with the streamed head (B=1), and with kept
    activations (B=4, the backward re-runs no layer); every layer at B=1 and a spread of
    layers at B=4 against the oracle."""
    cfg1 = synth.LLAMA8B
    cfg4 = synth.LLAMA8B.with_(batch=4)
    store = _build_store(cfg1)
    lora = synth.lora_params(cfg1)
    try:
        g1 = _full_run(cfg1, store, lora)
        checks = _start_oracle(cfg1, [(cfg1, g1)])
        assert _assert_bit_equal(g1, _full_run(cfg1, store, lora, resident=True)) == 14 * cfg1.n_layers
        _assert_bit_equal(g1, _full_run(cfg1, store, lora, n_slots=8))
        _assert_bit_equal(g1, _full_run(cfg1, store, lora, stream_head=True))
        _head_checks(cfg1, g1)
        g4 = _full_run(cfg4, store, lora)
        _start_oracle(cfg4, [(cfg4, g4)], layers=B4_ORACLE_LAYERS, checks=checks)
        assert _assert_bit_equal(g4, _full_run(cfg4, store, lora, resident=True)) == 14 * cfg4.n_layers
        _assert_bit_equal(g4, _full_run(cfg4, store, lora, keep_activations=True))
        _head_checks(cfg4, g4)
        _finish_oracle(checks, 14 * (cfg1.n_layers + len(B4_ORACLE_LAYERS)))
    finally:
        store.free()


def test_qwen32b_large_layers_full_size():
    """64 layers of 261.6 MiB each (every layer above the pages' ~165 MiB threshold)."""
    _full_size(synth.QWEN32B)


def test_qwen3b_bf16_full_size():
    _full_size(synth.QWEN3B_BF16)


@pytest.mark.parametrize("keep", [False, True])
def test_tiny_eight_slots_equal_resident_bitwise(tiny, keep):
    """stream_buffers' upper bound: eight device slots (more slots than the stack has layers
    here, so the slot choice keeps every layer after its first copy), recomputing and with
    kept activations, two steps in a row."""
    s = _session(tiny["cfg"], resident=False, store=tiny["s"].store, n_slots=8, keep_activations=keep)
    try:
        a, b = _run(s, tiny["cfg"]), _run(s, tiny["cfg"])
    finally:
        s.close()
    _assert_bit_equal(tiny["resident"], a)
    _assert_bit_equal(tiny["resident"], b)


@pytest.mark.parametrize("tied", [False, True])
def test_tiny_stream_head_equals_resident_tables_bitwise(tiny, tied):
    """"Measured numbers": the embedding and the head move into the store and reuse one device
    buffer.  The gather reads the rows from the page-locked store and the head GEMMs read the
    buffer: every output and gradient is bitwise that of resident tables, two steps in a row,
    untied and tied (the embedding is the head), and the device total drops by the tables."""
    from nf4_dequant_gemm_blockwise_b300 import api
    cfg = tiny["cfg"].with_(tied=tied)
    if tied:
        ref = _session(cfg, resident=True)
        want = _run(ref, cfg)
        store = ref.store
    else:
        ref, want, store = None, tiny["resident"], tiny["s"].store
    s = _session(cfg, resident=False, store=store, stream_head=True)
    try:
        a, b = _run(s, cfg), _run(s, cfg)
    finally:
        s.close()
        if ref is not None:
            ref.close()
    _assert_bit_equal(want, a)
    _assert_bit_equal(want, b)
    # untied: two resident tables give way to one buffer; tied: the one table moves into it
    sh, base = api.peak_bytes(cfg, cfg.batch, cfg.seq, stream_head=True)[0], api.peak_bytes(cfg, cfg.batch, cfg.seq)[0]
    assert (sh <= base + 1024) if tied else (sh < base)
