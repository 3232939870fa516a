"""GPU parity of the single-projection kernels against the oracle (all calls go through the
C ABI).  The forward runs on IEEE-half operands (as in the step) or bf16 ones; dX on bf16.
Operands are the oracle's: NF4 codes and absmax from oracle.nf4, dequantised values from
oracle.nf4.dequantize.  Two references are used:

* the exact-operand reference: the same 16-bit operands the kernel is defined on (x and the
  dequantised W rounded to the GEMM's 16-bit format) multiplied in float64 — the
  tensor-core result must match it to float32-accumulation accuracy plus the final output
  rounding;
* the oracle's float32 layer maths (unrounded W) — relative L2 <= 1e-2, the step's bar.

Token counts up to 16 take the small-M path, whose operands differ: the 16-bit operand is the
codebook value itself and the block scale is applied in float (forward: to each 64-wide
block's partial dot product; dX: to the gradient before its bf16 rounding), with the LoRA
term in float.  Its exact-operand reference models exactly those operands.
"""
import numpy as np
import pytest

import synth
from oracle import nf4

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from nf4_dequant_gemm_blockwise_b300 import api as a
    return a


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def _weights(N, K, seed=0):
    w_bits = synth.micro_weight(N, K, seed) if (N, K) in synth.MICRO_SHAPES else \
        synth.normal_bf16(seed, "layer", (7000 + N, K), (N, K), 0.02)
    packed, absmax = nf4.quantize_tensor(w_bits)
    wdq = nf4.dequantize_tensor(packed, absmax, (N, K))          # float32, the oracle's W
    return w_bits, packed, absmax, wdq


def _h16(x):
    """float32 -> IEEE half values (round to nearest even), returned as float32."""
    return np.asarray(x, np.float32).astype(np.float16).astype(np.float32)


def _tf32(x):
    """float32 -> TF32 (10 explicit mantissa bits; nearest, ties away from zero), as float64."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = ((b + 0x1000) & 0xFFFFE000).astype(np.uint32)
    return b.view(np.float32).astype(np.float64)


def _rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def test_dequant_bit_exact(api):
    N, K = 300, 688                                   # blocks straddle rows
    _, packed, absmax, wdq = _weights(N, K)
    n = N * K
    f = torch.empty(n, dtype=torch.float32, device="cuda")
    b = torch.empty(n, dtype=torch.int16, device="cuda")
    api.nf4_dequant(_dev(packed), _dev(absmax), n, f, b)
    torch.cuda.synchronize()
    assert np.array_equal(f.cpu().numpy().view(np.uint32), wdq.reshape(-1).view(np.uint32))
    want_b = synth.to_bf16_bits(wdq.reshape(-1))
    assert np.array_equal(b.cpu().numpy().view(np.uint16), want_b)


SHAPES = [  # (M, N, K): tiles, ragged M / N, the fallback (K % 256 != 0), microbench shapes;
    # (130, 4096, 14336) takes split-K; (2100, 14336, 4096) forward and (2100, 4096, 14336) dX
    # take two 128-row m-tiles per CTA with a ragged last m-tile.  M <= 16 takes the small-M
    # path: (9, 32, 1024) has more CTAs than strips, so every strip is summed from partials;
    # (3, 48, 4096), (5, 4096, 14336) and (16, 14336, 4096) cut strips at CTA boundaries.
    (128, 256, 256), (200, 512, 512), (64, 1376, 256), (64, 256, 688), (1, 256, 256),
    (130, 4096, 14336), (128, 14336, 4096), (16, 14336, 4096), (2100, 14336, 4096),
    (2100, 4096, 14336), (9, 32, 1024), (3, 48, 4096), (5, 4096, 14336), (1, 14336, 4096),
    # two m-tiles per CTA with split-K (and a ragged second m-tile pair at M=300)
    (512, 4096, 4096), (300, 4096, 14336),
]


def _small_m(M, N, K):
    """Whether the library takes the small-M path for this NF4 projection."""
    return 1 <= M <= 16 and N % 16 == 0 and K % 64 == 0


def _codes(packed, N, K):
    return nf4.unpack(packed, N * K).reshape(N, K // 64, 64)


def _small_fwd_exact(xh, packed, absmax, N, K):
    """y = sum over blocks b of absmax[n, b] * (x_b . half(c[code_b])), in float64."""
    codes = _codes(packed, N, K)
    table = nf4.codebook().astype(np.float16).astype(np.float64)
    a = absmax.reshape(N, K // 64).astype(np.float64)
    y = np.zeros((xh.shape[0], N))
    for b in range(K // 64):
        y += (xh[:, 64 * b:64 * b + 64] @ table[codes[:, b, :]].T) * a[:, b]
    return y


def _small_dx_exact(dy32, packed, absmax, N, K):
    """dx[:, block b] = bf16(dY * absmax[:, b]) . bf16(c[code_b]), in float64."""
    codes = _codes(packed, N, K)
    table = nf4.bf16_round(nf4.codebook()).astype(np.float64)
    dx = np.empty((dy32.shape[0], K))
    for b in range(K // 64):
        dya = nf4.bf16_round((dy32 * absmax.reshape(N, K // 64)[:, b][None, :]).astype(np.float32))
        dx[:, 64 * b:64 * b + 64] = dya.astype(np.float64) @ table[codes[:, b, :]]
    return dx


def _rows(M):
    """Rows checked against the float64 references (all of them up to 512)."""
    return np.arange(M) if M <= 512 else np.unique(np.linspace(0, M - 1, 300).astype(int))


def _lora(N, K, r=16):
    return synth.micro_lora(N, K, r)


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("f16", [True, False])
def test_proj_fwd(api, M, N, K, f16):
    r, s = 16, 2.0
    w_bits, packed, absmax, wdq = _weights(N, K)
    x32 = nf4.bf16_to_f32(synth.activations_bf16(M, K, key=1))
    if f16:
        x_in = x32.astype(np.float16).view(np.uint16)
        rnd = _h16
    else:
        x_in = synth.to_bf16_bits(x32)
        rnd = nf4.bf16_round
    A, B = _lora(N, K, r)
    y = torch.empty((M, N), dtype=torch.int16, device="cuda")
    scratch = torch.zeros(api.proj_scratch_bytes(M, N, K, r), dtype=torch.uint8, device="cuda")
    api.proj_fwd(_dev(x_in), M, N, K, _dev(packed), _dev(absmax), None, _dev(A), _dev(B), r, s, y,
                 scratch, x_f16=f16)
    api.proj_status(scratch, M, N, K)
    torch.cuda.synchronize()
    rows = _rows(M)
    yb = y.cpu().numpy().view(np.uint16)[rows]
    got = yb.view(np.float16).astype(np.float32) if f16 else synth.bf16_bits_to_f32(yb)
    x32 = x32[rows]
    xf = rnd(x32).astype(np.float64)
    wb = rnd(wdq).astype(np.float64)
    lora = s * (xf @ A.T.astype(np.float64)) @ B.T.astype(np.float64)
    ulp = 2.0 ** -10 if f16 else 2.0 ** -8
    if f16 and _small_m(M, N, K):
        exact = _small_fwd_exact(xf, packed, absmax, N, K) + lora
        tol = ulp * np.abs(exact) + 1e-4 * np.sqrt(np.mean(exact ** 2))
    else:
        exact = xf @ wb.T + lora
        tol = ulp * np.abs(exact) + 2e-3 * np.sqrt(np.mean(exact ** 2))
    bad = np.abs(got - exact) > tol
    assert not bad.any(), (bad.sum(), np.abs(got - exact).max())
    oracle = x32.astype(np.float64) @ wdq.T.astype(np.float64) + lora   # unrounded operands
    assert _rel_l2(got, oracle) <= (2e-3 if f16 else 1e-2)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_proj_dx(api, M, N, K):
    r, s = 16, 2.0
    w_bits, packed, absmax, wdq = _weights(N, K)
    dy_bits = synth.activations_bf16(M, N, key=2)
    A, B = _lora(N, K, r)
    dx = torch.empty((M, K), dtype=torch.float32, device="cuda")
    scratch = torch.zeros(api.proj_scratch_bytes(M, N, K, r), dtype=torch.uint8, device="cuda")
    api.proj_dx(_dev(dy_bits), M, N, K, _dev(packed), _dev(absmax), None, _dev(A), _dev(B), r, s, dx, scratch)
    api.proj_status(scratch, M, N, K)      # no kernel gave up a bounded wait
    torch.cuda.synchronize()
    rows = _rows(M)
    got = dx.cpu().numpy().astype(np.float64)[rows]
    dyf = nf4.bf16_to_f32(dy_bits).astype(np.float64)[rows]
    wb = nf4.bf16_round(wdq).astype(np.float64)
    du = s * (dyf @ B.astype(np.float64))
    if _small_m(M, N, K):
        # float LoRA term on this path
        exact = _small_dx_exact(dyf.astype(np.float32), packed, absmax, N, K) + du @ A.astype(np.float64)
        tol = 1e-4 * np.abs(exact) + 1e-4 * np.sqrt(np.mean(exact ** 2))
    else:
        exact = dyf @ wb + nf4.bf16_round(du.astype(np.float32)).astype(np.float64) @ \
            nf4.bf16_round(A).astype(np.float64)
        tol = 1e-4 * np.abs(exact) + 1e-3 * np.sqrt(np.mean(exact ** 2))
    bad = np.abs(got - exact) > tol
    assert not bad.any(), (bad.sum(), np.abs(got - exact).max())
    oracle = dyf @ wdq.astype(np.float64) + du @ A.astype(np.float64)
    assert _rel_l2(got, oracle) <= 1e-2


@pytest.mark.parametrize("rep", range(6))
def test_proj_dx_two_mtile_repeat(api, rep):
    """dX with two 128-row m-tiles per CTA, a ragged last m-tile and the LoRA extension,
    repeated: the result must be identical every time (fixed summation order)."""
    M, N, K, r, s = 2100, 4096, 14336, 16, 2.0
    _, packed, absmax, _ = _weights(N, K)
    dy = _dev(synth.activations_bf16(M, N, key=2))
    A, B = _lora(N, K, r)
    args = (_dev(packed), _dev(absmax), None, _dev(A), _dev(B), r, s)
    scratch = torch.zeros(api.proj_scratch_bytes(M, N, K, r), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        dx = torch.full((M, K), float("nan"), dtype=torch.float32, device="cuda")
        api.proj_dx(dy, M, N, K, *args, dx, scratch)
        api.proj_status(scratch, M, N, K)
        outs.append(dx.cpu().numpy())
    assert np.isfinite(outs[0]).all()
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


@pytest.mark.parametrize("M,N,K", [(64, 256, 256), (513, 1376, 256), (512, 4096, 14336)])
@pytest.mark.parametrize("f16", [True, False])
def test_proj_lora_grad(api, M, N, K, f16):
    r, s = 16, 2.0
    x32 = nf4.bf16_to_f32(synth.activations_bf16(M, K, key=3))
    x_in = x32.astype(np.float16).view(np.uint16) if f16 else synth.to_bf16_bits(x32)
    dy_bits = synth.activations_bf16(M, N, key=4)
    A, B = _lora(N, K, r)
    dA = torch.empty((r, K), dtype=torch.float32, device="cuda")
    dB = torch.empty((N, r), dtype=torch.float32, device="cuda")
    scratch = torch.empty(api.proj_scratch_bytes(M, N, K, r), dtype=torch.uint8, device="cuda")
    api.proj_lora_grad(_dev(x_in), _dev(dy_bits), M, N, K, _dev(A), _dev(B), r, s, dA, dB, scratch,
                       x_f16=f16)
    torch.cuda.synchronize()
    # exact-operand reference: the 16-bit x and dY are exact in TF32; the float operands A, B,
    # u = x A^T and du = s dY B are rounded to TF32 where the kernels stage them
    xf = (_h16(x32) if f16 else x32).astype(np.float64)
    dyf = nf4.bf16_to_f32(dy_bits).astype(np.float64)
    u = xf @ _tf32(A).T
    du = s * (dyf @ _tf32(B))
    want_dB = s * dyf.T @ _tf32(u)
    want_dA = _tf32(du).T @ xf
    # 2e-4: u and du are float intermediates whose last bits depend on the tensor core's
    # accumulation order, so an element near a TF32 rounding boundary may round the other way
    # than in this model (one TF32 step, 2^-11, on that element)
    assert _rel_l2(dB.cpu().numpy(), want_dB) < 2e-4
    assert _rel_l2(dA.cpu().numpy(), want_dA) < 2e-4
    # and the unrounded product, to the step's gradient bar
    assert _rel_l2(dB.cpu().numpy(), s * dyf.T @ (xf @ A.T.astype(np.float64))) < 2e-3
    assert _rel_l2(dA.cpu().numpy(), s * (dyf @ B.astype(np.float64)).T @ xf) < 2e-3


@pytest.mark.parametrize("f16", [True, False])
def test_bf16_weight_path(api, f16):
    """bf16 base weights (the un-quantised streamed base) through the same kernels; with half
    activations the weight tile is converted to half in shared memory."""
    M, N, K, r, s = 192, 512, 1024, 16, 2.0
    w_bits = synth.normal_bf16(0, "layer", (9000, 1), (N, K), 0.02)
    x32 = nf4.bf16_to_f32(synth.activations_bf16(M, K, key=5))
    x_in = x32.astype(np.float16).view(np.uint16) if f16 else synth.to_bf16_bits(x32)
    dy_bits = synth.activations_bf16(M, N, key=6)
    A, B = _lora(N, K, r)
    scratch = torch.empty(api.proj_scratch_bytes(M, N, K, r), dtype=torch.uint8, device="cuda")
    y = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dx = torch.empty((M, K), dtype=torch.float32, device="cuda")
    wd = _dev(w_bits)
    api.proj_fwd(_dev(x_in), M, N, K, None, None, wd, _dev(A), _dev(B), r, s, y, scratch, x_f16=f16)
    api.proj_dx(_dev(dy_bits), M, N, K, None, None, wd, _dev(A), _dev(B), r, s, dx, scratch)
    torch.cuda.synchronize()
    w = nf4.bf16_to_f32(w_bits).astype(np.float64)
    xf = x32.astype(np.float64)
    dyf = nf4.bf16_to_f32(dy_bits).astype(np.float64)
    want_y = xf @ w.T + s * (xf @ A.T) @ B.T
    want_dx = dyf @ w + s * (dyf @ B) @ A
    yb = y.cpu().numpy().view(np.uint16)
    got_y = yb.view(np.float16).astype(np.float32) if f16 else synth.bf16_bits_to_f32(yb)
    assert _rel_l2(got_y, want_y) < (2e-3 if f16 else 5e-3)
    assert _rel_l2(dx.cpu().numpy(), want_dx) < 5e-3
