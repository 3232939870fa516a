#!/usr/bin/env python
"""Streamed NF4 LoRA training step on the Llama-3.1-8B-shaped stack (B=1, S=512, r=16, two
device slots), seeded synthetic weights and tokens.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  `value` = tokens/s of whole training steps (forward,
backward, AdamW on the adapters) timed with CUDA events on the compute stream, inputs
already on the device; `e2e` = the same
through host buffers (token ids copied in from pinned memory and the loss read back every
step).  The weights are streamed from the pinned host store by the step itself in both.
`roofline` covers the NF4-dequant tensor-core GEMMs (all base-weight projections of the
step, forward, recompute and dX), timed live with CUDA events around each launch during
the timed steps.  `cpu_baseline` times the CPU oracle on one decoder layer plus the output
head, scaled to the whole stack.  With N > 1 (torchrun) every rank runs an independent
replica ("replicas only": the step has no exchange).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "streamed LoRA train tok/s (8B-shape NF4); dequant-GEMM % roofline; H2D GB/s"
UNIT = "tokens/s"
LR = 2e-4  # AdamW learning rate of the timed steps (a usual LoRA rate; the pages give none)


def _train_step(sess, tok):
    """One training step: streamed forward + backward, then AdamW on every adapter."""
    sess.step(tok)
    sess.optimizer_step(LR)


# DRAM traffic of the NF4 GEMM launches of a step, from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum, a one-pass metric set, averaged over 388 consecutive NF4 GEMM launches
# of the 8B step at B = 1, S = 512).  Valid only for the GEMM source it was taken on: reported
# while the hash of these files matches, null otherwise.
GEMM_TRAFFIC = {"sha256": "34eec8b91d99ce5d3cc37ed7a5d2ae4156a2f98656264a277574afb8cdffe2f7",
                "bytes_per_launch": 39.44e6, "algorithmic_bytes_per_launch": 55.43e6}
GEMM_SOURCES = ("nf4_dequant_gemm_blockwise_b300/csrc/gemm.cu", "nf4_dequant_gemm_blockwise_b300/csrc/gemm.h",
                "nf4_dequant_gemm_blockwise_b300/csrc/common.cuh")


def gemm_source_sha256():
    import hashlib
    h = hashlib.sha256()
    for rel in GEMM_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def gemm_traffic():
    """Measured bytes per GEMM launch if the capture matches the current kernel source."""
    if not GEMM_TRAFFIC or GEMM_TRAFFIC.get("sha256") != gemm_source_sha256():
        return None
    return GEMM_TRAFFIC["bytes_per_launch"]


def max_over_ranks(dist, values, device="cpu"):
    """Entry-wise maximum over ranks (the slowest replica sets the job's step time)."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def job_tokens_per_s(world, tokens_per_rank, ms_per_step):
    """Whole-job throughput: every rank steps its own replica over tokens_per_rank tokens, and
    the job advances at the pace of the slowest rank (ms_per_step = max over ranks)."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--batch", type=int, default=1)
    p.add_argument("--seq", type=int, default=None)
    p.add_argument("--slots", type=int, default=2)
    p.add_argument("--config", default="llama8b", choices=["llama8b", "qwen3b", "qwen32b"],
                   help="stack shape: the 8B NF4 stack (default, the headline workload), the 3B stack "
                        "with a bf16 base (S=512), or the 32B NF4 stack of large layers (S=1024)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--pageable", action="store_true",
                   help="stream from a pageable (not page-locked) copy of the store, to measure "
                        "what the pageable fallback costs")
    p.add_argument("--no-overlap", action="store_true", help="skip the resident comparison run")
    p.add_argument("--no-variants", action="store_true",
                   help="skip the extra batch-4 / eight-slot measurements")
    p.add_argument("--micro", action="store_true",
                   help="single-projection microbench instead of the step: one JSON line per (shape, M)")
    p.add_argument("--micro-shape", default="14336x4096,4096x14336", help="NxK list")
    p.add_argument("--micro-m", default="1,16,128,512,2048,8192")
    p.add_argument("--micro-iters", type=int, default=10)
    p.add_argument("--micro-attn", default=None, metavar="BxSxHxKVxD,...",
                   help="attention microbench instead of the step: forward and backward of causal GQA "
                        "attention at each shape, e.g. 1x512x32x8x128 (the 8B layer at B=1, S=512)")
    return p.parse_args()


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sus": d["bf16_tflops_sustained"],
                "src": "measured"}
    return {"hbm": 6400.0, "bf16": 1800.0, "bf16_sus": 1400.0, "src": "fallback"}


def _stack(args):
    """The stack the step runs on: --config picks the shape; --batch / --seq override the
    8B stack's (the 3B and 32B stacks keep their own sequence length unless --seq is given)."""
    import synth
    base = {"llama8b": synth.LLAMA8B, "qwen3b": synth.QWEN3B_BF16, "qwen32b": synth.QWEN32B}[args.config]
    seq = args.seq if (args.seq is not None) else base.seq
    return base.with_(batch=args.batch, seq=seq)


def _workload(cfg, slots):
    return {"workload": f"{cfg.name}: streamed LoRA training step (fwd+bwd+AdamW), {cfg.n_layers} layers, hidden "
                        f"{cfg.hidden}, inter {cfg.inter}, {cfg.n_heads}/{cfg.n_kv_heads} heads, vocab "
                        f"{cfg.vocab}, {cfg.base_fmt.upper()} base{', tied head' if cfg.tied else ''}, "
                        f"r={cfg.lora_r}, {slots} device slots, AdamW lr {LR}",
            "global_batch": cfg.batch, "seq_len": cfg.seq, "tokens_per_step": cfg.batch * cfg.seq,
            "parallelism": "replicas", "l2": "inputs larger than L2 (whole store re-streamed each step)"}


# ------------------------------------------------------------------------------ clocks
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------ oracle baseline
def run_oracle_timed(cfg):
    """Estimated oracle step time: L x (layer fwd + layer bwd + AdamW on the layer's adapters)
    + head fwd + head bwd."""
    import numpy as np

    import synth
    from oracle import model, nf4, optim

    src = synth.layer_source(cfg, 0)
    W = model.weights_from_source(cfg, [src], synth.embedding(cfg.with_(vocab=2)),
                                  synth.embedding(cfg.with_(vocab=2)), synth.final_norm(cfg)).layers[0]
    lora = model.lora_dict(synth.lora_params(cfg.with_(n_layers=1))[0], np.float32)
    w_lm = nf4.bf16_to_f32(synth.lm_head(cfg))
    w_f = nf4.bf16_to_f32(synth.final_norm(cfg))
    tok = synth.tokens(cfg)
    h = nf4.bf16_to_f32(synth.embedding(cfg))[tok.astype(np.int64)]
    cos, sin = model.rope_tables(cfg.seq, cfg.head_dim, cfg.rope_theta, np.float32)
    M = cfg.batch * cfg.seq

    def one(parts=False):
        ta = time.perf_counter()
        out, cache = model.layer_forward(h, W, lora, cfg, cos, sin)
        tb = time.perf_counter()
        logits, (xn, r) = model.logits_of(out.reshape(M, -1), w_f, w_lm, cfg.rms_eps)
        model.loss_of(logits.reshape(cfg.batch, cfg.seq, -1), tok)
        dz = model.loss_backward(logits.reshape(cfg.batch, cfg.seq, -1), tok).reshape(M, -1)
        dh = model.rmsnorm_backward(dz @ w_lm, out.reshape(M, -1), w_f, r).reshape(out.shape)
        tc = time.perf_counter()
        _, grads = model.layer_backward(dh, cache, W, lora, cfg, cos, sin)
        for p in model.PROJ:
            for t, g in zip(lora[p], grads[p]):
                optim.adamw_step(t, g, np.zeros_like(g), np.zeros_like(g), 1, LR)
        td = time.perf_counter()
        layer = (tb - ta) + (td - tc)
        head = tc - tb
        if parts:
            return cfg.n_layers * layer + head, td - ta, layer, head
        return cfg.n_layers * layer + head, td - ta

    return one


def oracle_tiny_step_s():
    """Wall time of the oracle's whole tiny-stack step (2 layers, S=64: forward, loss, backward,
    AdamW on every adapter), best of 3."""
    import numpy as np

    import synth
    from oracle import model, optim

    cfg = synth.TINY
    W = model.weights_from_source(cfg, [synth.layer_source(cfg, i) for i in range(cfg.n_layers)],
                                  synth.embedding(cfg), synth.lm_head(cfg), synth.final_norm(cfg))
    tok = synth.tokens(cfg)
    lora = synth.lora_params(cfg)
    best = float("inf")
    for _ in range(3):
        t0 = time.perf_counter()
        fwd = model.forward(cfg, W, tok, lora)
        grads, _ = model.backward(cfg, W, tok, lora, fwd)
        for layer_g, layer_p in zip(grads, lora):
            for (dA, dB), (A, B) in zip(layer_g, layer_p):
                optim.adamw_step(A, dA, np.zeros_like(dA), np.zeros_like(dA), 1, LR)
                optim.adamw_step(B, dB, np.zeros_like(dB), np.zeros_like(dB), 1, LR)
        best = min(best, time.perf_counter() - t0)
    return best


def _threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


# ------------------------------------------------------------------------------ reference arm
def run_reference(args, rank):
    import synth
    cfg = _stack(args)
    if rank != 0:
        return
    one = run_oracle_timed(cfg)
    for _ in range(args.warmup):
        one()
    est, wall, parts = [], [], []
    for _ in range(args.steps):
        e, w, layer_s, head_s = one(parts=True)
        est.append(e)
        wall.append(w)
        parts.append((layer_s, head_s))
    step_s = statistics.mean(est)
    value = cfg.batch * cfg.seq / step_s
    layer_ms = statistics.mean(p[0] for p in parts) * 1e3
    head_ms = statistics.mean(p[1] for p in parts) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": _workload(cfg, args.slots),
            "estimated": True,
            "estimate": {"per_layer_ms": layer_ms, "layers": cfg.n_layers, "head_ms": head_ms,
                         "formula": f"ms_per_step = {cfg.n_layers} x per_layer_ms + head_ms",
                         "wall_ms_per_timed_sample": statistics.mean(wall) * 1e3},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": _threads(), "kind": "oracle",
                             "sample": "each step: one decoder layer forward+backward+AdamW and the output "
                                       "head forward+backward of the same workload, on the CPU "
                                       f"oracle; step time estimated as {cfg.n_layers} x layer + head "
                                       "(the whole stack is not run)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ microbench
def run_micro(args):
    """Single-projection NF4 dequant-GEMM + LoRA: forward (half operands), dX (bf16) and the
    LoRA gradients, each launch timed alone with CUDA events after an L2 flush."""
    import numpy as np
    import torch

    import synth
    from nf4_dequant_gemm_blockwise_b300 import api

    peaks = _peaks()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    r, s = synth.MICRO_R, 2.0
    for shp in args.micro_shape.split(","):
        N, K = (int(v) for v in shp.lower().split("x"))
        codes, absmax = api.nf4_quantize_host(synth.micro_weight(N, K))
        codes_d, absmax_d = torch.from_numpy(codes).cuda(), torch.from_numpy(absmax).cuda()
        A, B = synth.micro_lora(N, K, r)
        A_d, B_d = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        for M in (int(v) for v in args.micro_m.split(",")):
            x32 = synth.bf16_bits_to_f32(synth.activations_bf16(M, K, key=1))
            x = torch.from_numpy(x32.astype(np.float16).view(np.int16)).cuda()
            dy = torch.from_numpy(synth.activations_bf16(M, N, key=2).view(np.int16)).cuda()
            y = torch.empty((M, N), dtype=torch.int16, device="cuda")
            dx = torch.empty((M, K), dtype=torch.float32, device="cuda")
            dA = torch.empty((r, K), dtype=torch.float32, device="cuda")
            dB = torch.empty((N, r), dtype=torch.float32, device="cuda")
            scratch = torch.empty(api.proj_scratch_bytes(M, N, K, r), dtype=torch.uint8, device="cuda")
            st = torch.cuda.current_stream()
            calls = {
                "fwd": lambda: api.proj_fwd(x, M, N, K, codes_d, absmax_d, None, A_d, B_d, r, s, y, scratch, st),
                "dx": lambda: api.proj_dx(dy, M, N, K, codes_d, absmax_d, None, A_d, B_d, r, s, dx, scratch, st),
                "grad": lambda: api.proj_lora_grad(x, dy, M, N, K, A_d, B_d, r, s, dA, dB, scratch, st),
                # the dequant GEMM kernel alone (no adapter: r = 0)
                "fwd_gemm": lambda: api.proj_fwd(x, M, N, K, codes_d, absmax_d, None, None, None, 0, s, y, scratch, st),
                "dx_gemm": lambda: api.proj_dx(dy, M, N, K, codes_d, absmax_d, None, None, None, 0, s, dx, scratch, st),
            }
            out = {"micro": True, "shape": [N, K], "M": M, "r": r}
            wbytes = N * K * 0.5 + N * K / 64 * 4
            for name, fn in calls.items():
                for _ in range(2):
                    fn()
                ts = []
                for _ in range(args.micro_iters):
                    flush.fill_(1)
                    # keep the stream busy while the host enqueues the call, so the timed
                    # region holds device work only (no host launch latency)
                    torch.cuda._sleep(1_000_000)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(st)
                    fn()
                    e1.record(st)
                    e1.synchronize()
                    ts.append(e0.elapsed_time(e1) * 1e-3)
                t = statistics.median(ts)
                rr = 0 if name.endswith("_gemm") else r
                fwd_like = name.startswith("fwd")
                if name == "grad":
                    flops = 4.0 * M * r * (N + K)
                    byts = 2.0 * M * (N + K) + 4.0 * r * (N + K) * 2
                elif fwd_like:
                    flops = 2.0 * M * N * K + 2.0 * M * rr * (N + K)
                    byts = wbytes + 2.0 * M * K + 2.0 * M * N + 2.0 * rr * (N + K)
                else:
                    flops = 2.0 * M * N * K + 2.0 * M * rr * (N + K)
                    byts = wbytes + 2.0 * M * N + 4.0 * M * K + 2.0 * rr * (N + K)
                t_hbm = byts / (peaks["hbm"] * 1e9)
                t_tc = flops / (peaks["bf16"] * 1e12)
                bound = "hbm" if t_hbm >= t_tc else "tensor"
                out[name] = {"us": t * 1e6, "tflops": flops / t / 1e12, "gbs": byts / t / 1e9,
                             "bound": bound, "frac": max(t_hbm, t_tc) / t}
            out["peak_source"] = f"{peaks['src']}: hbm {peaks['hbm']} GB/s, bf16 burst {peaks['bf16']} TFLOP/s"
            if not args.no_cpu_baseline:
                out["cpu_baseline"] = run_micro_oracle(N, K, M, r, s, codes, absmax, A, B)
            print(json.dumps(out), flush=True)


def run_micro_attn(args):
    """Causal GQA attention alone (soup_attn_fwd / soup_attn_bwd), each call timed with CUDA
    events after an L2 flush; flops count the causal half of every S x S x d product (2 in the
    forward; 5 in the backward: score recompute, dP, dV, dQ, dK), as in the step's roofline."""
    import torch

    from nf4_dequant_gemm_blockwise_b300 import api

    peaks = _peaks()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()
    g = torch.Generator(device="cuda").manual_seed(0)
    for shp in args.micro_attn.split(","):
        B, S, nh, nkv, d = (int(v) for v in shp.lower().split("x"))
        M, ld = B * S, (nh + 2 * nkv) * d
        qkv = torch.randn((M, ld), generator=g, device="cuda").half().view(torch.int16)
        o = torch.empty((M, nh * d), dtype=torch.int16, device="cuda")
        lse = torch.empty((B, nh, S), dtype=torch.float32, device="cuda")
        do = (torch.randn((M, nh * d), generator=g, device="cuda") * 0.05).bfloat16().view(torch.int16)
        dqkv = torch.empty((M, ld), dtype=torch.float32, device="cuda")
        scratch = torch.empty(api.attn_bwd_scratch_bytes(B, S, nh, nkv, d), dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        calls = {
            "fwd": (2, lambda: api.attn_fwd(qkv, B, S, nh, nkv, d, o, lse, err, st)),
            "bwd": (5, lambda: api.attn_bwd(qkv, o, do, lse, B, S, nh, nkv, d, scratch, dqkv, err, st)),
        }
        out = {"micro_attn": True, "B": B, "S": S, "n_heads": nh, "n_kv_heads": nkv, "head_dim": d,
               "path": "tcgen05" if d in (64, 128) and nh % nkv == 0 and nh // nkv <= 8 else "mma.sync"}
        for name, (mats, fn) in calls.items():
            for _ in range(3):
                fn()
            ts = []
            for _ in range(args.micro_iters):
                flush.fill_(1)
                torch.cuda._sleep(1_000_000)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                fn()
                e1.record(st)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e-3)
            t = statistics.median(ts)
            flops = float(mats) * B * nh * S * (S + 1) * d
            out[name] = {"us": t * 1e6, "tflops": flops / t / 1e12, "frac": flops / t / 1e12 / peaks["bf16"]}
        torch.cuda.synchronize()
        out["errors"] = int(err.item())
        out["peak_source"] = f"{peaks['src']}: bf16 burst {peaks['bf16']} TFLOP/s"
        print(json.dumps(out), flush=True)


def run_micro_oracle(N, K, M, r, s, codes, absmax, A, B, cap_rows=512):
    """The CPU oracle on one microbench projection: forward (dequantise + x W^T + LoRA) and
    backward (dequantise + dX + dA/dB), float32 NumPy.  Above cap_rows rows the products of a
    cap_rows-row slice are timed and scaled by M / cap_rows (they are linear in M); the
    dequantisation is timed once and counted in both."""
    import numpy as np

    import synth
    from oracle import model, nf4

    rows = min(M, cap_rows)
    x = synth.bf16_bits_to_f32(synth.activations_bf16(M, K, key=1))[:rows]
    x = x.astype(np.float16).astype(np.float32)
    dy = synth.bf16_bits_to_f32(synth.activations_bf16(M, N, key=2))[:rows]
    t0 = time.perf_counter()
    W = nf4.dequantize_tensor(codes, absmax, (N, K))
    t1 = time.perf_counter()
    _, u = model.lora_linear(x, W, A, B, s)
    t2 = time.perf_counter()
    model.lora_linear_backward(dy, x, u, W, A, B, s)
    t3 = time.perf_counter()
    scale = M / rows
    deq = t1 - t0  # once per call, like the kernels' dequantisation
    return {"fwd_us": (deq + (t2 - t1) * scale) * 1e6, "bwd_us": (deq + (t3 - t2) * scale) * 1e6,
            "cores": _threads(), "kind": "oracle",
            "sample": f"products on {rows} of {M} rows, scaled by {scale:g}; one dequantisation "
                      f"per call"}


# ------------------------------------------------------------------------------ our arm
def h2d_peak_gbs(torch):
    n = 1 << 30
    h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    h.fill_(1)
    d = torch.empty(n, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    best = 0.0
    for _ in range(10):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            a.record(s)
            d.copy_(h, non_blocking=True)
            b.record(s)
        b.synchronize()
        best = max(best, n / (a.elapsed_time(b) * 1e-3) / 1e9)
    del h, d
    return best


def run_ours(args, rank, world, local_rank, dist):
    import numpy as np
    import torch

    import synth
    from nf4_dequant_gemm_blockwise_b300 import api
    from nf4_dequant_gemm_blockwise_b300.session import StreamedLoRA

    torch.cuda.set_device(local_rank)
    cfg = _stack(args)
    B, S = cfg.batch, cfg.seq
    peaks = _peaks()
    h2d_peak = h2d_peak_gbs(torch)

    t_build = time.perf_counter()
    store = api.Store(cfg, allow_pageable=True)
    for i0 in range(0, cfg.n_layers, 8):
        idx = list(range(i0, min(cfg.n_layers, i0 + 8)))
        for i, src in zip(idx, synth.layer_sources(cfg, idx)):
            store.put_layer(i, [src[t] for t in synth.LAYER_TENSORS])
    if args.pageable:
        paged = api.Store(cfg, force_pageable=True)
        for i in range(cfg.n_layers):
            paged.put_shard(i, store.shard_bytes(i))
        store.free()
        store = paged
    t_build = time.perf_counter() - t_build
    _, store_bytes, pinned = store.info()

    torch.cuda.reset_peak_memory_stats()
    lora = synth.lora_params(cfg)
    sess = StreamedLoRA(cfg, None, synth.embedding(cfg), synth.lm_head(cfg), synth.final_norm(cfg),
                        lora, B, S, n_slots=args.slots, store=store)
    tok_host = torch.from_numpy(synth.tokens(cfg)).pin_memory()
    tok_dev = tok_host.cuda()
    loss_host = torch.zeros(1, dtype=torch.float32).pin_memory()

    for _ in range(args.warmup):
        _train_step(sess, tok_dev)
    sess.sync()
    torch.cuda.synchronize()

    # ---- timed region: device-resident inputs
    clocks = Clocks(local_rank)
    clocks.start()
    time.sleep(0.3)
    sess.stream.debug(api.DBG_PROFILE, 1)
    sess.stream.stats(reset=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    l0 = api.kernel_launches()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(sess.compute)
    for _ in range(args.steps):
        _train_step(sess, tok_dev)
    e1.record(sess.compute)
    sess.sync()
    torch.cuda.synchronize()
    launches = api.kernel_launches() - l0
    ms_total = e0.elapsed_time(e1)
    clk = clocks.stop()
    st = sess.stream.stats(reset=True)
    sess.stream.debug(api.DBG_PROFILE, 0)
    if dist is not None:
        dist.barrier()
    peak_alloc = torch.cuda.max_memory_allocated()

    # ---- the AdamW launch alone (all adapters, one launch; 1.2 GB of state > L2)
    o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    o0.record(sess.compute)
    for _ in range(5):
        sess.optimizer_step(LR)
    o1.record(sess.compute)
    sess.sync()
    torch.cuda.synchronize()
    opt_ms = o0.elapsed_time(o1) / 5
    opt_gbs = 28 * sess.n_params / (opt_ms * 1e-3) / 1e9  # p, g, m, v read; p, m, v written

    # ---- end to end through the public API, timed by the host clock: every step copies its
    # token ids in from pinned host memory and reads its loss back into pinned host memory (the
    # loop a trainer runs), and the clock stops after the final synchronise, so host-side stalls
    # (enqueue, copies, the loss read) count
    for _ in range(2):
        _train_step(sess, tok_dev)
    sess.sync()
    torch.cuda.synchronize()
    sess.stream.stats(reset=True)  # count the timed end-to-end steps' copies only
    losses_host = torch.zeros(args.steps, dtype=torch.float32).pin_memory()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    for k in range(args.steps):
        with torch.cuda.stream(sess.compute):
            tok_dev.copy_(tok_host, non_blocking=True)
        sess.fwd(tok_dev)
        sess.bwd()
        sess.optimizer_step(LR)
        with torch.cuda.stream(sess.compute):
            losses_host[k:k + 1].copy_(sess.loss, non_blocking=True)
    sess.sync()
    torch.cuda.synchronize()
    ms_e2e = (time.perf_counter() - h0) * 1e3
    st_e2e = sess.stream.stats(reset=True)
    loss_val = float(losses_host[-1].item())

    # ---- resident run of the same kernels: the compute-only step time (for the overlap)
    ms_res = None
    if not args.no_overlap:
        sess_r = StreamedLoRA(cfg, None, synth.embedding(cfg), synth.lm_head(cfg), synth.final_norm(cfg),
                              lora, B, S, resident=True, store=store)
        for _ in range(args.warmup):
            _train_step(sess_r, tok_dev)
        sess_r.sync()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(sess_r.compute)
        for _ in range(args.steps):
            _train_step(sess_r, tok_dev)
        g1.record(sess_r.compute)
        sess_r.sync()
        torch.cuda.synchronize()
        ms_res = g0.elapsed_time(g1) / args.steps
        sess_r.close()
        del sess_r  # its device buffers (the whole store, resident) go before anything else is measured
        torch.cuda.empty_cache()

    # ---- every kernel family of the step, event-timed per launch group over a few extra steps
    # (not the timed run: the events themselves cost a little)
    prof_steps = 3
    sess.stream.debug(api.DBG_PROFILE, 2)
    sess.stream.kernel_stats(reset=True)
    for _ in range(prof_steps):
        _train_step(sess, tok_dev)
    sess.sync()
    fams = sess.stream.kernel_stats(reset=True)
    sess.stream.debug(api.DBG_PROFILE, 0)
    kernels = []
    for f in fams:
        if f["ms"] <= 0:
            continue
        if f["tensor_bound"]:
            ach, peak, unit = f["flops"] / (f["ms"] * 1e-3) / 1e12, peaks["bf16_sus"], "TFLOP/s"
        else:
            ach, peak, unit = f["bytes"] / (f["ms"] * 1e-3) / 1e9, peaks["hbm"], "GB/s"
        kernels.append({"family": f["name"], "bound": "tensor" if f["tensor_bound"] else "hbm",
                        "launch_groups_per_step": f["launches"] / prof_steps,
                        "ms_per_step": f["ms"] / prof_steps, "flops_per_step": f["flops"] / prof_steps,
                        "bytes_per_step": f["bytes"] / prof_steps, "achieved": ach, "unit": unit,
                        "peak": peak, "frac": ach / peak})

    # ---- max over ranks
    ms_step, ms_e2e_step = max_over_ranks(dist, [ms_total / args.steps, ms_e2e / args.steps], "cuda")
    tokens = B * S
    value = job_tokens_per_s(world, tokens, ms_step)
    e2e_value = job_tokens_per_s(world, tokens, ms_e2e_step)

    # roofline of the NF4 dequant GEMMs (tensor-bound at this token count)
    gemm_tflops = st["gemm_flops"] / (st["gemm_ms"] * 1e-3) / 1e12 if st["gemm_ms"] else None
    peak_tc = peaks["bf16_sus"]
    copy_s = st["copy_ms"] * 1e-3
    h2d_gbs = st["copy_bytes"] / copy_s / 1e9 if copy_s else None
    t_copy = st["copy_ms"] / args.steps
    overlap = None
    if ms_res is not None:
        exposed = ms_step - max(t_copy, ms_res)
        overlap = {"t_step_ms": ms_step, "t_copy_ms": t_copy, "t_compute_resident_ms": ms_res,
                   "hidden_fraction": 1.0 - max(exposed, 0.0) / min(t_copy, ms_res) if min(t_copy, ms_res) > 0 else None}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 fwd / bf16 bwd operands, f32 accumulate", "data": "synthetic",
        "config": dict(_workload(cfg, args.slots), **({"store": "pageable"} if args.pageable else {})),
        "e2e": {"value": e2e_value, "unit": UNIT, "clock": "host (perf_counter), final synchronise included",
                "h2d_bytes_per_step": tok_host.numel() * 4 + st_e2e["copy_bytes"] / args.steps,
                "d2h_bytes_per_step": 4},
        "gpu_launches": launches,
        "roofline": {"kernel": "nf4_dequant_gemm (tcgen05; all base-weight projections, fwd + recompute + dX)",
                     "bound": "tensor", "achieved": gemm_tflops, "peak": peak_tc, "unit": "TFLOP/s",
                     "frac": gemm_tflops / peak_tc if gemm_tflops else None, "traffic": gemm_traffic(),
                     "peak_source": f"{peaks['src']} bf16 sustained", "launches": st["gemm_launches"],
                     "avg_launch_us": st["gemm_ms"] * 1e3 / max(st["gemm_launches"], 1),
                     "share_of_step": st["gemm_ms"] / ms_total if ms_total else None},
        "h2d": {"achieved_gbs": h2d_gbs, "pinned_peak_gbs": h2d_peak,
                "frac": h2d_gbs / h2d_peak if h2d_gbs else None, "bytes_per_step": st["copy_bytes"] / args.steps,
                "copies_per_step": st["copies"] / args.steps, "store_bytes": store_bytes, "pinned": pinned},
        "overlap": overlap,
        "kernels": {"method": f"CUDA events around every launch group on the compute stream over {prof_steps} "
                              "extra steps (profiling mode 2, outside the timed run); algorithmic flops or "
                              f"bytes per family; peaks: {peaks['src']} bf16 sustained / HBM copy",
                    "families": kernels},
        "optimizer": {"kernel": "adamw (float32 state, one launch over all adapters)",
                      "params": sess.n_params, "ms": opt_ms, "bound": "hbm", "achieved_gbs": opt_gbs,
                      "frac": opt_gbs / peaks["hbm"], "bytes_per_param": 28},
        "peak_vram_bytes": peak_alloc,
        "peak_vram_predicted_bytes": api.peak_bytes(cfg, B, S, n_slots=args.slots)[0],
        "store_build_s": t_build,
        "loss": loss_val,
        "clocks": clk,
    }
    sess.close()
    del sess
    torch.cuda.empty_cache()
    # ---- extra configurations of the same store: batch 4 (the pages' other 8B batch), eight
    # device slots (stream_buffers' upper bound) and kept activations (stream_recompute: off);
    # same timing method, fewer steps
    if not args.no_variants and args.config == "llama8b":
        variants = []
        for vb, vslots, keep, shead in ((4, args.slots, False, False), (1, 8, False, False),
                                        (4, 8, False, False), (1, args.slots, True, False),
                                        (4, args.slots, True, False), (1, args.slots, False, True)):
            vcfg = cfg.with_(batch=vb)
            torch.cuda.synchronize()
            torch.cuda.reset_peak_memory_stats()
            v_base = torch.cuda.memory_allocated()  # anything still held outside this variant
            vs = StreamedLoRA(vcfg, None, synth.embedding(cfg), synth.lm_head(cfg), synth.final_norm(cfg),
                              lora, vb, S, n_slots=vslots, store=store, keep_activations=keep,
                              stream_head=shead)
            vtok = torch.from_numpy(synth.tokens(vcfg)).cuda()
            for _ in range(args.warmup):
                _train_step(vs, vtok)
            vs.sync()
            torch.cuda.synchronize()
            vs.stream.stats(reset=True)          # count the timed steps' copies only
            nsteps = max(3, args.steps // 2)
            v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            v0.record(vs.compute)
            for _ in range(nsteps):
                _train_step(vs, vtok)
            v1.record(vs.compute)
            vs.sync()
            torch.cuda.synchronize()
            vms = v0.elapsed_time(v1) / nsteps
            vst = vs.stream.stats(reset=True)
            v_peak = torch.cuda.max_memory_allocated() - v_base
            variants.append({"batch": vb, "slots": vslots, "keep_activations": keep, "stream_head": shead,
                             "tokens_per_step": vb * S,
                             "value": world * vb * S / (vms * 1e-3), "ms_per_step": vms,
                             "copies_per_step": vst["copies"] / nsteps, "steps": nsteps,
                             "peak_vram_bytes": v_peak,
                             "peak_vram_predicted_bytes": api.peak_bytes(vcfg, vb, S, n_slots=vslots,
                                                                         keep_activations=keep,
                                                                         stream_head=shead)[0]})
            vs.close()
            del vs  # free its device buffers before the next variant's peak is measured
            torch.cuda.empty_cache()
        line["variants"] = variants
    if rank == 0 and not args.no_cpu_baseline:
        one = run_oracle_timed(cfg)
        est = [one()[0] for _ in range(2)]
        step_s = min(est)
        line["cpu_baseline"] = {"value": tokens / step_s, "unit": UNIT, "cores": _threads(), "kind": "oracle",
                                "sample": f"one decoder layer fwd+bwd+AdamW and the output head fwd+bwd of this "
                                          f"workload on the CPU oracle (float32 NumPy), step time = "
                                          f"{cfg.n_layers} x layer + head; best of 2",
                                "tiny_step_s": oracle_tiny_step_s()}
    store.free()
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = _args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as td
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local_rank)
        td.init_process_group(backend)
        dist = td
    if args.impl == "reference":
        run_reference(args, rank)
    elif args.micro_attn:
        if rank == 0:
            run_micro_attn(args)
    elif args.micro:
        if rank == 0:
            run_micro(args)
    else:
        run_ours(args, rank, world, local_rank, dist)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
