"""Failure detection on the GPU, in the forms that fault, trap or hang nothing.

"Layer streaming: fine-tune a model that does not fit in your card", "Troubleshooting": a read
that wedges is given up after a bounded wait and reported; a failure must surface as an error,
never as wrong numbers.  Here:
* soup_sync with a zero budget while a step is still running returns SOUP_ETIMEDOUT, and the
  step, waited for properly afterwards, is bitwise unchanged;
* a host-side delay before every shard copy changes timing only: the streamed run still equals
  the resident run bit for bit;
* a kernel whose bounded wait on a barrier that nothing signals gives up raises the error flag:
  soup_sync returns SOUP_ETIMEDOUT once, and the next step on the same handle is clean;
* a forward operand beyond the IEEE-half range raises SOUP_ERANGE from soup_sync (the step) and
  from soup_proj_status / soup_proj_noalloc_status (one projection), and the flag is cleared
  by that read.
"""
import numpy as np
import pytest

import synth
from oracle import nf4

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _session(cfg, resident=False, store=None, source=None):
    from nf4_dequant_gemm_blockwise_b300.session import StreamedLoRA
    src = source or (lambda i: synth.layer_source(cfg, i))
    return StreamedLoRA(cfg, src, synth.embedding(cfg), synth.lm_head(cfg), synth.final_norm(cfg),
                        synth.lora_params(cfg), cfg.batch, cfg.seq, resident=resident, store=store)


def _outputs(sess, cfg):
    M = cfg.batch * cfg.seq
    lay = torch.empty((cfg.n_layers + 1, M, cfg.hidden), dtype=torch.float32, device="cuda")
    return lay


def _fetch(sess, lay):
    return float(sess.loss.item()), lay.cpu().numpy(), sess.grads()


def _equal(a, b):
    assert a[0] == b[0]
    assert np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32))
    for la, lb in zip(a[2], b[2]):
        for (ga, gb), (ha, hb) in zip(la, lb):
            assert np.array_equal(ga.view(np.uint32), ha.view(np.uint32))
            assert np.array_equal(gb.view(np.uint32), hb.view(np.uint32))


@pytest.fixture(scope="module")
def pair():
    cfg = synth.TINY
    s = _session(cfg)
    r = _session(cfg, resident=True, store=s.store)
    tok = torch.from_numpy(synth.tokens(cfg)).cuda()
    lay = _outputs(r, cfg)
    r.step(tok, layer_out=lay)
    r.sync()
    ref = _fetch(r, lay)
    yield cfg, s, tok, ref
    r.close()
    s.close()


def test_sync_with_zero_budget_times_out_then_completes(pair):
    from nf4_dequant_gemm_blockwise_b300 import api
    cfg, s, tok, ref = pair
    lay = _outputs(s, cfg)
    with torch.cuda.stream(s.compute):
        torch.cuda._sleep(200_000_000)          # ~0.1 s of device time ahead of the step
    s.step(tok, layer_out=lay)
    with pytest.raises(api.SoupError) as e:
        s.stream.sync(0)
    assert e.value.code == api.ETIMEDOUT
    s.sync()                                    # the real wait succeeds
    _equal(_fetch(s, lay), ref)


def test_copy_delay_changes_timing_only(pair):
    from nf4_dequant_gemm_blockwise_b300 import api
    cfg, s, tok, ref = pair
    s.stream.debug(api.DBG_COPY_DELAY_US, 3000)
    try:
        lay = _outputs(s, cfg)
        s.step(tok, layer_out=lay)
        s.sync()
        got = _fetch(s, lay)
    finally:
        s.stream.debug(api.DBG_COPY_DELAY_US, 0)
    _equal(got, ref)


def test_bounded_wait_gives_up_and_is_reported_once(pair):
    from nf4_dequant_gemm_blockwise_b300 import api
    cfg, s, tok, ref = pair
    s.stream.debug(api.DBG_WAIT_PROBE, 2000)     # a wait that nothing ends, given ~2 ms
    with pytest.raises(api.SoupError) as e:
        s.sync()
    assert e.value.code == api.ETIMEDOUT
    assert "bounded wait" in str(e.value)
    lay = _outputs(s, cfg)                       # the handle stays usable
    s.step(tok, layer_out=lay)
    s.sync()
    _equal(_fetch(s, lay), ref)


def test_half_range_overflow_in_the_step_is_reported():
    """Layer 1's input-norm weight set to 60000: its normalised input leaves the half range."""
    from nf4_dequant_gemm_blockwise_b300 import api
    cfg = synth.TINY

    def source(i):
        src = synth.layer_source(cfg, i)
        if i == 1:
            src["ln1"] = synth.to_bf16_bits(np.full(cfg.hidden, 60000.0, np.float32))
        return src

    s = _session(cfg, source=source)
    try:
        tok = torch.from_numpy(synth.tokens(cfg)).cuda()
        s.fwd(tok)
        with pytest.raises(api.SoupError) as e:
            s.sync()
        assert e.value.code == api.ERANGE
    finally:
        s.close()


def test_half_range_overflow_in_a_projection_is_reported():
    """y = x W^T with x = 1000 and W = 100 over K = 256: 2.56e7, far beyond the half range."""
    from nf4_dequant_gemm_blockwise_b300 import api
    M, N, K, r = 128, 256, 256, 0
    x = torch.from_numpy(np.full((M, K), 1000.0, np.float16).view(np.int16)).cuda()
    w = torch.from_numpy(synth.to_bf16_bits(np.full((N, K), 100.0, np.float32)).view(np.int16)).cuda()
    y = torch.empty((M, N), dtype=torch.int16, device="cuda")
    scratch = torch.zeros(api.proj_scratch_bytes(M, N, K, r), dtype=torch.uint8, device="cuda")
    api.proj_fwd(x, M, N, K, None, None, w, None, None, r, 2.0, y, scratch)
    with pytest.raises(api.SoupError) as e:
        api.proj_status(scratch, M, N, K)
    assert e.value.code == api.ERANGE
    api.proj_status(scratch, M, N, K)           # cleared by the read
    # the same through the entry point that allocates nothing, and its own status call
    api.proj_fwd_noalloc(x, M, N, K, None, None, w, None, None, r, 2.0, y)
    with pytest.raises(api.SoupError) as e:
        api.proj_noalloc_status()
    assert e.value.code == api.ERANGE
    api.proj_noalloc_status()
    # in range: a clean status
    x1 = torch.from_numpy(np.full((M, K), 0.01, np.float16).view(np.int16)).cuda()
    api.proj_fwd_noalloc(x1, M, N, K, None, None, w, None, None, r, 2.0, y)
    api.proj_noalloc_status()
    got = y.cpu().numpy().view(np.float16).astype(np.float64)
    want = np.float64(np.float16(0.01)) * 100.0 * K
    assert np.allclose(got, want, rtol=2e-3)
