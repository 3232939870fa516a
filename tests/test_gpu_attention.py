"""The attention kernels on their own, through soup_attn_fwd / soup_attn_bwd, against the oracle.

"Layer streaming: fine-tune a model that does not fit in your card", "How it works": the layer
is the model family's own, so its attention is plain causal grouped-query attention.  The
oracle (oracle.model.attention / attention_backward, float64 here) takes the very half-precision
q, k, v and bf16 dO the kernels read.

Bars, from the operand formats: the forward rounds P and the output to IEEE half (relative
2^-11 each), so the output is held to relative L2 <= 2e-3; the backward forms every product
with a gradient from bf16 operands (relative 2^-9 each: v, k, q, P and dS), so dv is held to
relative L2 <= 1e-2.  dq and dk come from dS = P (dP - rowsum(dP P)), a difference of two terms
each rounded on its own, so their error scales with the terms, not with the difference (at
S = 1 the difference is exactly zero): ||err|| <= 1e-2 (||want|| + ||gross||), where gross is
the same product with (P dP) in place of dS.  The log-sum-exp is float throughout: absolute
error <= 1e-3 in base-2 units.  The backward is deterministic: two runs are bitwise equal.

Shapes cover one position, ragged tails shorter than one 64-row tile, several 128-row tiles,
clusters of 1, 2, 4, 5 and 8 query heads per key/value head, both head dims, S = 512 and 1024,
and a 16-to-1 grouping that the warp-level path takes.
"""
import numpy as np
import pytest

import synth
from oracle import model

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CASES = [  # B, S, n_heads, n_kv_heads, head_dim
    (1, 1, 4, 2, 64),
    (2, 63, 4, 2, 64),
    (1, 200, 8, 2, 128),
    (2, 130, 8, 1, 64),
    (1, 300, 10, 2, 128),
    (1, 512, 8, 2, 128),
    (2, 512, 4, 4, 128),
    (1, 1024, 4, 1, 128),
    (1, 1024, 4, 2, 64),
    (1, 96, 16, 1, 64),
]


def _inputs(B, S, nh, nkv, d, seed):
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((B, S, nh, d)) * 1.5).astype(np.float16)
    k = rng.standard_normal((B, S, nkv, d)).astype(np.float16)
    v = rng.standard_normal((B, S, nkv, d)).astype(np.float16)
    do = synth.bf16_bits_to_f32(synth.to_bf16_bits(
        (rng.standard_normal((B, S, nh, d)) * 0.05).astype(np.float32)))
    return q, k, v, do


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _cos(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / max(np.linalg.norm(a) * np.linalg.norm(b), 1e-300))


def _lse2(q, k):
    """Base-2 log-sum-exp of each row's visible scaled scores [B, nh, S] (float64)."""
    B, S, nh, d = q.shape
    nkv = k.shape[2]
    out = np.zeros((B, nh, S))
    mask = np.triu(np.ones((S, S), bool), 1)
    for b in range(B):
        for h in range(nh):
            g = model.kv_head_of(h, nh, nkv)
            s = np.where(mask, -np.inf, (q[b, :, h] @ k[b, :, g].T) / np.sqrt(d))
            m = s.max(axis=-1, keepdims=True)
            out[b, h] = (np.log(np.exp(s - m).sum(axis=-1)) + m[:, 0]) / np.log(2.0)
    return out


def _gross(do, q, k, v, p):
    """||(P o dP) K|| / sqrt(d) and ||(P o dP)^T Q|| / sqrt(d) summed over heads: the size of the
    uncentred terms of dq and dk (float64)."""
    B, S, nh, d = q.shape
    nkv = k.shape[2]
    gq = np.zeros_like(q)
    gk = np.zeros_like(k)
    for b in range(B):
        for h in range(nh):
            g = model.kv_head_of(h, nh, nkv)
            t = p[b, h] * (do[b, :, h] @ v[b, :, g].T)
            gq[b, :, h] = t @ k[b, :, g] / np.sqrt(d)
            gk[b, :, g] += t.T @ q[b, :, h] / np.sqrt(d)
    return np.linalg.norm(gq), np.linalg.norm(gk)


def _run(case, seed=0):
    from nf4_dequant_gemm_blockwise_b300 import api
    B, S, nh, nkv, d = case
    q, k, v, do = _inputs(B, S, nh, nkv, d, seed)
    M = B * S
    ld = (nh + 2 * nkv) * d
    qkv = np.concatenate([q.reshape(M, nh * d), k.reshape(M, nkv * d), v.reshape(M, nkv * d)], axis=1)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    qkv_d = dev(qkv.view(np.int16))
    o_d = torch.empty((M, nh * d), dtype=torch.int16, device="cuda")
    lse_d = torch.empty((B, nh, S), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.attn_fwd(qkv_d, B, S, nh, nkv, d, o_d, lse_d, err)
    do_d = dev(synth.to_bf16_bits(do.reshape(M, nh * d)).view(np.int16))
    scratch = torch.zeros(api.attn_bwd_scratch_bytes(B, S, nh, nkv, d), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        dqkv = torch.full((M, ld), float("nan"), dtype=torch.float32, device="cuda")
        api.attn_bwd(qkv_d, o_d, do_d, lse_d, B, S, nh, nkv, d, scratch, dqkv, err)
        outs.append(dqkv)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o = o_d.cpu().numpy().view(np.float16).astype(np.float64).reshape(B, S, nh, d)
    return (q, k, v, do), o, lse_d.cpu().numpy(), outs[0].cpu().numpy(), outs[1].cpu().numpy()


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d_S%d_h%d_kv%d_d%d" % c)
def test_attention_matches_oracle(case):
    B, S, nh, nkv, d = case
    (q, k, v, do), o, lse, dqkv, dqkv2 = _run(case)
    q64, k64, v64, do64 = (x.astype(np.float64) for x in (q, k, v, do))
    o_ref, p = model.attention(q64, k64, v64)
    assert _rel(o, o_ref) <= 2e-3
    assert np.max(np.abs(lse - _lse2(q64, k64))) <= 1e-3
    dq, dk, dv = model.attention_backward(do64, q64, k64, v64, p)
    M = B * S
    got_q = dqkv[:, :nh * d].reshape(B, S, nh, d)
    got_k = dqkv[:, nh * d:(nh + nkv) * d].reshape(B, S, nkv, d)
    got_v = dqkv[:, (nh + nkv) * d:].reshape(B, S, nkv, d)
    gq, gk = _gross(do64, q64, k64, v64, p)
    for name, got, want, gross in (("dq", got_q, dq, gq), ("dk", got_k, dk, gk), ("dv", got_v, dv, 0.0)):
        assert np.all(np.isfinite(got)), name
        err = float(np.linalg.norm(np.asarray(got, np.float64) - want))
        assert err <= 1e-2 * (np.linalg.norm(want) + gross), (name, err, np.linalg.norm(want), gross)
    for name, got, want in (("dq", got_q, dq), ("dk", got_k, dk), ("dv", got_v, dv)):
        if S >= 64:  # well away from the cancellation of the smallest cases
            assert _rel(got, want) <= 1e-2, (name, _rel(got, want))
            assert _cos(got, want) >= 0.9999, (name, _cos(got, want))
    assert np.array_equal(dqkv.view(np.uint32), dqkv2.view(np.uint32))
    assert dqkv.shape == (M, (nh + 2 * nkv) * d)


def test_attention_empty_is_a_no_op():
    from nf4_dequant_gemm_blockwise_b300 import api
    z = torch.zeros(16, dtype=torch.int16, device="cuda")
    f = torch.zeros(16, dtype=torch.float32, device="cuda")
    api.attn_fwd(z, 0, 64, 4, 2, 64, z, f)
    api.attn_fwd(z, 2, 0, 4, 2, 64, z, f)
    s = torch.zeros(256, dtype=torch.uint8, device="cuda")
    api.attn_bwd(z, z, z, f, 0, 64, 4, 2, 64, s, f)
    torch.cuda.synchronize()


def test_attention_rejects_bad_shapes():
    from nf4_dequant_gemm_blockwise_b300 import api
    z = torch.zeros(16, dtype=torch.int16, device="cuda")
    f = torch.zeros(16, dtype=torch.float32, device="cuda")
    for args in ((1, 8, 4, 3, 64), (1, 8, 4, 2, 96), (-1, 8, 4, 2, 64)):
        with pytest.raises(api.SoupError) as e:
            api.attn_fwd(z, *args, z, f)
        assert e.value.code == api.EINVAL
