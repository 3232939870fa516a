"""The oracle's layer-by-layer check of a full-size streamed step, spread over host processes.

For each decoder layer the oracle quantises the layer's own bf16 source (oracle.nf4), runs the
layer forward and its hand-derived backward in float32 (oracle.model) from the GPU's layer
input and upstream gradient, and measures the GPU's layer output, dL/dh and the 14 LoRA
gradients against it.  The checks are independent per layer, so they run in worker processes
started with `spawn` (a fork after the first CUDA call would hang); each worker limits its BLAS
threads so that the workers share the host's cores.  The parent asserts on the returned
figures.  Test infrastructure only.
"""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np


def _rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _cosine(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / max(np.linalg.norm(a) * np.linalg.norm(b), 1e-300))


def _init_worker(root, blas_threads):
    import sys
    if root not in sys.path:
        sys.path.insert(0, root)
    try:
        from threadpoolctl import threadpool_limits
        globals()["_limits"] = threadpool_limits(blas_threads)
    except ImportError:
        pass


def check_layer(cfg, li, cases):
    """Oracle figures for layer li.  cases: list of dicts, one per run of the layer (batch
    sizes may differ), with the GPU's h_in [B,S,H], h_out, dh_out, dh_in (float32) and grads
    (7 pairs (dA, dB)).  Returns one dict of figures per case."""
    import synth
    from oracle import model

    src = synth.layer_source(cfg, li)
    W = model.weights_from_source(cfg, [src], synth.embedding(cfg.with_(vocab=2)),
                                  synth.embedding(cfg.with_(vocab=2)), synth.final_norm(cfg)).layers[0]
    del src
    lora = model.lora_dict(synth.lora_params(cfg.with_(n_layers=li + 1))[li], np.float32)
    out = []
    for c in cases:
        B, S = c["h_in"].shape[:2]
        cos, sin = model.rope_tables(S, cfg.head_dim, cfg.rope_theta, np.float32)
        h_out, cache = model.layer_forward(c["h_in"], W, lora, cfg, cos, sin)
        dh_in, grads = model.layer_backward(c["dh_out"], cache, W, lora, cfg, cos, sin)
        del cache
        fig = {"layer": li, "batch": B, "out_rel": _rel_l2(c["h_out"], h_out.reshape(c["h_out"].shape)),
               "dh_rel": _rel_l2(c["dh_in"], dh_in.reshape(c["dh_in"].shape)), "grads": []}
        for p, name in enumerate(model.PROJ):
            for w in range(2):
                got, want = c["grads"][p][w], grads[name][w]
                fig["grads"].append((name, "AB"[w], _rel_l2(got, want), _cosine(got, want)))
        out.append(fig)
    return out


def _workers(n_layers, gb_per_worker):
    cores = os.cpu_count() or 1
    try:
        import psutil
        avail_gb = psutil.virtual_memory().available / 2 ** 30
    except ImportError:
        avail_gb = 64.0
    return max(1, min(cores, n_layers, int(avail_gb // gb_per_worker)))


class LayerChecks:
    """A pool of worker processes checking layers while the caller goes on (with the GPU).
    submit(cfg, layers, cases_of) queues layer checks (cases_of(li) builds that layer's cases
    from the GPU results, called here, in the parent); results() waits for all of them and
    returns {layer: figures} in submission order per layer."""

    def __init__(self, n_layers, gb_per_worker=8.0):
        self.n = _workers(n_layers, gb_per_worker)
        threads = max(1, (os.cpu_count() or 1) // self.n)
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        self.ex = cf.ProcessPoolExecutor(max_workers=self.n, mp_context=mp.get_context("spawn"),
                                         initializer=_init_worker, initargs=(root, threads))
        self.futures = []

    def submit(self, cfg, layers, cases_of):
        for li in layers:
            self.futures.append((li, self.ex.submit(check_layer, cfg, li, cases_of(li))))

    def results(self):
        out = {}
        try:
            for li, f in self.futures:
                out.setdefault(li, []).extend(f.result())
        finally:
            self.ex.shutdown()
        return out


def check_layers(cfg, layers, cases_of, gb_per_worker=8.0):
    """Run check_layer for every layer in `layers` and wait: the figures in layer order."""
    layers = list(layers)
    lc = LayerChecks(len(layers), gb_per_worker)
    lc.submit(cfg, layers, cases_of)
    res = lc.results()
    return [res[li] for li in layers]
