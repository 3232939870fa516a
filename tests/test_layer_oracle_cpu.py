"""The host-parallel layer check the full-size GPU tests use (tests/layer_oracle.py), run on
the CPU against the oracle's own end-to-end step: fed the oracle's layer inputs, upstream
gradients and results, every figure must come out at zero (same arithmetic), and a planted
error in one layer's output or one gradient must show up in that layer's figures only."""
import numpy as np

import layer_oracle
import synth
from oracle import model


def _oracle_run(cfg):
    W = model.weights_from_source(cfg, [synth.layer_source(cfg, i) for i in range(cfg.n_layers)],
                                  synth.embedding(cfg), synth.lm_head(cfg), synth.final_norm(cfg))
    tok = synth.tokens(cfg)
    lora = synth.lora_params(cfg)
    fwd = model.forward(cfg, W, tok, lora)
    grads, dhs = model.backward(cfg, W, tok, lora, fwd)
    M = cfg.batch * cfg.seq
    return {"layers": np.stack([h.reshape(M, -1) for h in fwd["hs"]]),
            "dh": np.stack([d.reshape(M, -1) for d in dhs]), "grads": grads}


def _cases(cfg, g, li):
    B, S, H = cfg.batch, cfg.seq, cfg.hidden
    return [{"h_in": g["layers"][li].reshape(B, S, H), "h_out": g["layers"][li + 1],
             "dh_out": g["dh"][li + 1].reshape(B, S, H), "dh_in": g["dh"][li], "grads": g["grads"][li]}]


def test_layer_checks_reproduce_the_oracle_and_catch_a_planted_error():
    cfg = synth.TINY
    g = _oracle_run(cfg)
    figs = layer_oracle.check_layers(cfg, range(cfg.n_layers), lambda li: _cases(cfg, g, li))
    for per_layer in figs:
        (f,) = per_layer
        assert f["out_rel"] < 1e-6 and f["dh_rel"] < 1e-6
        assert all(rel < 1e-6 and cos > 1 - 1e-9 for _, _, rel, cos in f["grads"])
    bad = dict(g)
    bad["layers"] = g["layers"].copy()
    bad["layers"][2] *= 1.05                                  # layer 1's output is off by 5%
    bad["grads"] = [list(x) for x in g["grads"]]
    dA, dB = bad["grads"][0][4]
    bad["grads"][0][4] = (dA, -dB)                            # layer 0, gate: dB sign flipped
    figs = layer_oracle.check_layers(cfg, range(cfg.n_layers), lambda li: _cases(cfg, bad, li))
    f0, f1 = figs[0][0], figs[1][0]
    assert f1["out_rel"] > 0.04 and f0["out_rel"] < 1e-6
    gate_b = [x for x in f0["grads"] if x[0] == "gate" and x[1] == "B"][0]
    assert gate_b[3] < -0.99
    assert all(cos > 1 - 1e-9 for name, w, rel, cos in f1["grads"])
