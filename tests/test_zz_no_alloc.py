"""soup_proj_fwd_noalloc — the single-projection forward for callers that cannot allocate
device memory (a host application that owns the device-memory budget, or a caller that cannot
afford cudaMalloc's synchronisation) — checked through the C ABI against soup_proj_fwd, the
entry point that takes caller-provided scratch, on two calls in a row, and against the oracle.
After every call soup_proj_noalloc_status must report that no kernel raised its error flag.

This file is collected last on purpose, so a run that stops at the first failure has already
run every other test.  It passes alone in a fresh process and after the other tests (the
static scratch keeps the previous call's contents; the entry point clears what must start at
zero, and the shared error flag is cleared by each status read)."""
import numpy as np
import pytest

import synth
from oracle import nf4

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _f16(t):
    return t.cpu().numpy().view(np.uint16).view(np.float16).astype(np.float64)


def _rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


# (M, N, K, r, weight format).  M <= 16 takes the small-M path, whose per-CTA partial strips
# live in the static array (the largest share of it at N=14336); r = 0 is the plain dequant
# GEMM; "bf16" streams un-quantised weights.
CASES = [
    (130, 4096, 14336, 16, "nf4"), (512, 14336, 4096, 16, "nf4"), (64, 1376, 256, 16, "nf4"),
    (1, 14336, 4096, 16, "nf4"), (16, 14336, 4096, 16, "nf4"),
    (1, 4096, 14336, 16, "nf4"), (16, 4096, 14336, 16, "nf4"),
    (16, 14336, 4096, 0, "nf4"), (512, 4096, 4096, 0, "nf4"),
    (192, 512, 1024, 16, "bf16"), (16, 512, 1024, 16, "bf16"),
]


@pytest.mark.parametrize("M,N,K,r,fmt", CASES)
def test_noalloc_matches_scratch_entry_point_twice(M, N, K, r, fmt):
    from nf4_dequant_gemm_blockwise_b300 import api
    s = 2.0
    w = synth.normal_bf16(0, "layer", (8000 + N, K), (N, K), 0.02)
    x32 = nf4.bf16_to_f32(synth.activations_bf16(M, K, key=9))
    x = _dev(x32.astype(np.float16).view(np.uint16))
    A, B = synth.micro_lora(N, K, max(r, 1))
    A_d, B_d = (_dev(A), _dev(B)) if r else (None, None)
    if fmt == "nf4":
        packed, absmax = nf4.quantize_tensor(w)
        wargs = (_dev(packed), _dev(absmax), None)
        w_used = nf4.dequantize_tensor(packed, absmax, (N, K)).astype(np.float64)
    else:
        wargs = (None, None, _dev(w))
        w_used = nf4.bf16_to_f32(w).astype(np.float64)
    ref = torch.empty((M, N), dtype=torch.int16, device="cuda")
    scratch = torch.zeros(api.proj_scratch_bytes(M, N, K, r), dtype=torch.uint8, device="cuda")
    api.proj_fwd(x, M, N, K, *wargs, A_d, B_d, r, s, ref, scratch)
    api.proj_status(scratch, M, N, K)
    want = _f16(ref)
    # the oracle: float64 products of the unrounded operands (x is exactly half here)
    xh = x32.astype(np.float16).astype(np.float64)
    oracle = xh @ w_used.T
    if r:
        oracle = oracle + s * (xh @ A.T.astype(np.float64)) @ B.T.astype(np.float64)
    for _ in range(2):
        y = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
        api.proj_fwd_noalloc(x, M, N, K, *wargs, A_d, B_d, r, s, y)
        api.proj_noalloc_status()          # no kernel gave up a wait or overflowed
        got = _f16(y)
        # same operands; only the float summation order may differ (no split-K here), so the
        # results agree to the half-precision output rounding
        tol = 2.0 ** -10 * np.abs(want) + 2e-3 * np.sqrt(np.mean(want ** 2))
        assert np.all(np.abs(got - want) <= tol)
        assert _rel_l2(got, oracle) <= 2e-3, _rel_l2(got, oracle)


def test_noalloc_rejects_oversized_calls():
    from nf4_dequant_gemm_blockwise_b300 import api
    M, N, K = 65536, 14336, 4096      # working memory far beyond the static scratch
    x = torch.zeros((1,), dtype=torch.int16, device="cuda")
    y = torch.zeros((1,), dtype=torch.int16, device="cuda")
    codes = torch.zeros((1,), dtype=torch.uint8, device="cuda")
    absmax = torch.zeros((1,), dtype=torch.float32, device="cuda")
    A = torch.zeros((1,), dtype=torch.float32, device="cuda")
    with pytest.raises(api.SoupError) as e:
        api.proj_fwd_noalloc(x, M, N, K, codes, absmax, None, A, A, 16, 2.0, y)
    assert e.value.code == api.EINVAL
    assert "static scratch" in str(e.value)
    api.proj_noalloc_status()
