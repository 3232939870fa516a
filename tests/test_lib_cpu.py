"""CPU checks of the C-ABI library: it loads without a GPU, exports every entry point the
header declares, and its host-side logic (codebook, packer, shard layout, memory plan) agrees
with the oracle.  No device work is launched here."""
import os
import re

import numpy as np
import pytest

import synth
from oracle import nf4, sizes

api = pytest.importorskip("nf4_dequant_gemm_blockwise_b300.api")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "soup.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(soup_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol():
    import ctypes
    lib = ctypes.CDLL(api.LIB_PATH)
    declared = _declared()
    assert len(declared) >= 20
    for name in declared:
        assert hasattr(lib, name), name


def test_codebook_matches_oracle_bitwise():
    assert np.array_equal(api.nf4_codebook().view(np.uint32), nf4.codebook().view(np.uint32))


@pytest.mark.parametrize("n", [64 * 1000, 64 * 37 + 13, 688 * 256, 1])
def test_host_packer_bit_exact(n):
    rng = np.random.default_rng(n)
    x = (rng.standard_normal(n) * 0.02).astype(np.float32)
    x[rng.integers(0, n, size=max(1, n // 500))] = 0.0
    if n > 200:
        x[64:128] = 0.0                                # an all-zero block
    bits = synth.to_bf16_bits(x)
    codes, absmax = api.nf4_quantize_host(bits, n_threads=4)
    oc, oa = nf4.quantize(nf4.bf16_to_f32(bits))
    assert np.array_equal(absmax.view(np.uint32), oa.view(np.uint32))
    assert np.array_equal(codes, nf4.pack(oc[: n + (n % 2)]))


def test_host_packer_ties_go_low():
    m = nf4.midpoints()
    x = np.zeros(64, np.float32)
    x[0] = 1.0
    x[1:16] = m
    codes, _ = api.nf4_quantize_host(synth.to_bf16_bits(x))
    # midpoints are not all bf16-representable: compare with the oracle on the same bf16 input
    oc, _ = nf4.quantize(nf4.bf16_to_f32(synth.to_bf16_bits(x)))
    assert np.array_equal(codes, nf4.pack(oc))


@pytest.mark.parametrize("cfg", [synth.TINY, synth.LLAMA8B, synth.QWEN32B, synth.QWEN3B_BF16])
def test_shard_layout_matches_payload(cfg):
    lay = api.shard_layout_of(cfg)
    assert lay.payload == sizes.shard_payload_bytes(cfg)
    assert lay.stride % 4096 == 0 and lay.payload <= lay.stride < lay.payload + 16 * 1024
    for g in range(4):
        assert lay.w_off[g] % 1024 == 0 and lay.a_off[g] % 1024 == 0
    assert lay.ln1_off % 1024 == 0 and lay.ln2_off % 1024 == 0


def test_store_shard_bytes_match_oracle_packing():
    cfg = synth.TINY
    st = api.Store(cfg, allow_pageable=True)            # no GPU here: pageable fallback
    src = [synth.layer_source(cfg, i) for i in range(cfg.n_layers)]
    for i, s in enumerate(src):
        st.put_layer(i, [s[t] for t in synth.LAYER_TENSORS])
    lay = api.shard_layout_of(cfg)
    groups = [("q", "k", "v"), ("o",), ("gate", "up"), ("down",)]
    for i in range(cfg.n_layers):
        sh = st.shard_bytes(i)
        for g, names in enumerate(groups):
            packed = np.concatenate([nf4.quantize_tensor(src[i][p])[0] for p in names])
            absm = np.concatenate([nf4.quantize_tensor(src[i][p])[1] for p in names])
            assert np.array_equal(sh[lay.w_off[g]: lay.w_off[g] + lay.w_bytes[g]], packed)
            got_a = sh[lay.a_off[g]: lay.a_off[g] + lay.a_bytes[g]].view(np.float32)
            assert np.array_equal(got_a.view(np.uint32), absm.view(np.uint32))
        assert np.array_equal(sh[lay.ln1_off: lay.ln1_off + 2 * cfg.hidden].view(np.uint16), src[i]["ln1"])
    st.free()


def test_memory_plan_bounds_streaming_by_slots():
    cfg = synth.LLAMA8B
    lay = api.shard_layout_of(cfg)
    ws2 = api.workspace_bytes(cfg, 1, 512, n_slots=2)
    ws8 = api.workspace_bytes(cfg, 1, 512, n_slots=8)
    wsr = api.workspace_bytes(cfg, 1, 512, resident=True)
    # weights on the device: n_slots shards when streamed, every shard when resident
    assert ws8 - ws2 == 6 * lay.stride
    assert wsr - ws2 == (cfg.n_layers - 2) * lay.stride
    tot, ws = api.peak_bytes(cfg, 1, 512, n_slots=2)
    assert ws == ws2
    assert tot - ws == sizes.resident_bytes(cfg)
    # streaming keeps the device copy of the base to two shards (< 1/10 of the store here)
    assert 2 * lay.stride < sizes.store_payload_bytes(cfg) / 10


def test_invalid_config_is_rejected():
    bad = synth.TINY.with_(head_dim=96)
    with pytest.raises(api.SoupError) as e:
        api.shard_layout_of(bad)
    assert e.value.code == api.EINVAL
    with pytest.raises(api.SoupError):
        api.workspace_bytes(synth.TINY, 1, 64, n_slots=9)


def test_adamw_and_accumulate_arguments_are_checked_before_any_launch():
    # every case below fails validation on the host, so no CUDA call is made
    def rc(*args, **kw):
        with pytest.raises(api.SoupError) as e:
            api.adamw_step(*args, **kw)
        return e.value.code
    n = 1024
    a, b, c, d = 1 << 20, 2 << 20, 3 << 20, 4 << 20  # disjoint fake device addresses
    assert rc(a, b, c, d, n, 0, 1e-3) == api.EINVAL                 # step numbers start at 1
    assert rc(a, b, c, d, n, 1, 1e-3, beta1=1.0) == api.EINVAL      # beta outside [0, 1)
    assert rc(a, b, c, d, n, 1, 1e-3, beta2=-0.5) == api.EINVAL
    assert rc(a, b, c, d, -1, 1, 1e-3) == api.EINVAL                # negative size
    assert rc(a, None, c, d, n, 1, 1e-3) == api.EINVAL              # NULL buffer
    assert rc(a, a + 4 * n - 4, c, d, n, 1, 1e-3) == api.EINVAL     # param and grad overlap
    assert rc(a, b, c, c + 8, n, 1, 1e-3) == api.EINVAL             # m and v overlap
    assert "overlap" in api.last_error()
    arr = (api.C.c_void_p * 1)()
    assert api.lib.soup_step_bwd_ex(None, arr, arr, None, api.BWD_ACCUMULATE) == api.EINVAL


def test_keep_activations_plan_adds_one_activation_set_per_layer():
    # the activation set of one layer: mid residual (float), x1, x2 (16-bit), qkv, attention
    # output, LSE (float per head), gate/up (reserved as float), SwiGLU output, and the LoRA
    # down-projections of the four groups (float + 16-bit, 64 wide), each 1024-byte aligned
    cfg = synth.LLAMA8B
    B, S = 1, 512
    M, H, I = B * S, cfg.hidden, cfg.inter
    qd, kvd = cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    al = lambda n: -(-n // 1024) * 1024
    one = (al(4 * M * H) + 2 * al(2 * M * H) + al(2 * M * (qd + 2 * kvd)) + al(2 * M * qd)
           + al(4 * M * cfg.n_heads) + al(4 * M * I) + al(2 * M * I)
           + 4 * (al(4 * M * 64) + al(2 * M * 64)))
    base = api.workspace_bytes(cfg, B, S, n_slots=2)
    keep = api.workspace_bytes(cfg, B, S, n_slots=2, keep_activations=True)
    assert keep - base == (cfg.n_layers - 1) * one
    both = api.workspace_bytes(cfg, B, S, resident=True, keep_activations=True)
    assert both - api.workspace_bytes(cfg, B, S, resident=True) == (cfg.n_layers - 1) * one
    tot, ws = api.peak_bytes(cfg, B, S, n_slots=2, keep_activations=True)
    assert ws == keep and tot - ws == sizes.resident_bytes(cfg)
    out = api.C.c_uint64()
    assert api.lib.soup_workspace_bytes(api.C.byref(api.make_cfg(cfg)), B, S, 2, 8,
                                        api.C.byref(out)) == api.EINVAL


@pytest.mark.parametrize("cfg", [synth.LLAMA8B, synth.QWEN3B_BF16])
def test_stream_head_plan_trades_the_tables_for_one_vocabulary_buffer(cfg):
    # "Measured numbers": the embedding and the untied head move into the store and reuse one
    # device buffer.  The workspace grows by one [vocab, hidden] bf16 table (1024-byte aligned)
    # and the resident tables (two untied, one tied) leave the run's device total.
    B, S = 1, 512
    table = 2 * cfg.vocab * cfg.hidden
    base = api.workspace_bytes(cfg, B, S, n_slots=2)
    sh = api.workspace_bytes(cfg, B, S, n_slots=2, stream_head=True)
    assert sh - base == -(-table // 1024) * 1024
    tot, ws = api.peak_bytes(cfg, B, S, n_slots=2, stream_head=True)
    assert ws == sh
    assert tot - ws == sizes.resident_bytes(cfg) - table * (1 if cfg.tied else 2)
    tot0, _ = api.peak_bytes(cfg, B, S, n_slots=2)
    assert tot0 - tot == table * (1 if cfg.tied else 2) - (-(-table // 1024) * 1024)


def test_put_head_checks_its_arguments():
    cfg = synth.TINY
    st = api.Store(cfg)
    e = synth.embedding(cfg)
    with pytest.raises(api.SoupError) as ex:
        st.put_head(e, None)                      # untied: the head is required
    assert ex.value.code == api.EINVAL
    tied = api.Store(cfg.with_(tied=True))
    with pytest.raises(api.SoupError) as ex:
        tied.put_head(e, e)                       # tied: no separate head
    assert ex.value.code == api.EINVAL
    st.free()
    tied.free()


def test_forced_pageable_store_and_raw_shard_copy():
    # a store filled shard by shard from another store's bytes is byte-identical, and a store
    # created with page-locking skipped reports itself pageable without a warning
    cfg = synth.TINY
    a = api.Store(cfg)
    for i in range(cfg.n_layers):
        src = synth.layer_source(cfg, i)
        a.put_layer(i, [src[t] for t in synth.LAYER_TENSORS])
    b = api.Store(cfg, force_pageable=True)
    assert not b.pageable_warning and b.info()[2] is False
    for i in range(cfg.n_layers):
        b.put_shard(i, a.shard_bytes(i))
    for i in range(cfg.n_layers):
        assert np.array_equal(a.shard_bytes(i), b.shard_bytes(i))
    with pytest.raises(api.SoupError):
        b.put_shard(0, a.shard_bytes(0)[:-16])
    with pytest.raises(api.SoupError):
        b.put_shard(cfg.n_layers, a.shard_bytes(0))
    a.free()
    b.free()


def test_c_abi_from_plain_c(tmp_path):
    """The library used from C99 through include/soup.h alone (gcc, no Python in between):
    the codebook and the host quantiser agree bit for bit with the oracle, the layout and
    memory plan with the binding's, and argument errors come back as SOUP_EINVAL."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = os.path.join(root, "nf4_dequant_gemm_blockwise_b300")
    exe = str(tmp_path / "abi_smoke")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(root, "include"),
                    os.path.join(root, "tests", "c", "abi_smoke.c"), "-L", pkg, "-lsoup",
                    f"-Wl,-rpath,{pkg}", "-o", exe], check=True)
    # the header is also valid C++ (the library's own translation units include it too)
    subprocess.run(["g++", "-std=c++17", "-fsyntax-only", "-x", "c++",
                    os.path.join(root, "include", "soup.h")], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    kv = {ln.split(" ", 1)[0]: ln.split(" ", 1)[1] for ln in out.strip().splitlines()}
    cb = np.array([int(h, 16) for h in kv["codebook"].split()], np.uint32)
    assert np.array_equal(cb, nf4.codebook().astype(np.float32).view(np.uint32))
    # the program's input: k / 17 in float32 for k = (37 i mod 101) - 50, rounded to bf16
    k = (np.arange(130) * 37 % 101 - 50).astype(np.float32)
    bits = (k / np.float32(17)).view(np.uint32)
    bits = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)
    packed, absmax = nf4.quantize_tensor(bits)
    assert np.array_equal(np.array([int(h, 16) for h in kv["codes"].split()], np.uint8), packed)
    assert np.array_equal(np.array([int(h, 16) for h in kv["absmax"].split()], np.uint32),
                          absmax.astype(np.float32).view(np.uint32))
    cfg = synth.TINY
    assert int(kv["stride"]) == api.shard_layout_of(cfg).stride
    ws0, ws2 = (int(v) for v in kv["workspace"].split())
    assert ws0 == api.workspace_bytes(cfg, 1, 64) and ws2 == api.workspace_bytes(cfg, 1, 64, keep_activations=True)
    assert int(kv["peak"]) == api.peak_bytes(cfg, 1, 64)[0]
    assert int(kv["bad_mode"]) == api.EINVAL and int(kv["short_shard"]) == api.EINVAL
    nbytes, pinned, first = kv["store"].split()
    assert int(nbytes) == cfg.n_layers * api.shard_layout_of(cfg).stride and pinned == "0" and first == "5a"
    assert int(kv["adamw_step0"]) == api.EINVAL and "step numbers start at 1" in kv["last_error"]


@pytest.mark.parametrize("n_threads", [1, 3, 16])
def test_host_packer_special_values_and_threads(n_threads):
    # bf16 subnormals, negative zeros, an all-negative block, a block whose absmax is a
    # subnormal, and a ragged tail: same bits as the oracle at any thread count
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(64 * 9 + 5) * 0.02).astype(np.float32)
    x[0:64] = -np.abs(x[0:64])                              # all negative
    x[64:128] = rng.standard_normal(64).astype(np.float32) * np.float32(1e-39)  # subnormals
    x[128:192:3] = np.float32(-0.0)                          # negative zeros
    x[192] = np.float32(3e-39)
    bits = synth.to_bf16_bits(x)
    codes, absmax = api.nf4_quantize_host(bits, n_threads=n_threads)
    oc, oa = nf4.quantize(nf4.bf16_to_f32(bits))
    assert np.array_equal(absmax.view(np.uint32), oa.view(np.uint32))
    assert np.array_equal(codes, nf4.pack(oc[: x.size + (x.size % 2)]))


def test_attention_entry_points_check_their_arguments_first():
    """soup_attn_fwd / soup_attn_bwd reject bad shapes (kv heads not dividing the query heads,
    head dims other than 64 / 128, negative sizes) and NULL buffers with SOUP_EINVAL before any
    device work; an empty batch or sequence is a no-op that touches nothing."""
    z = 16  # any non-NULL address: nothing is dereferenced on these paths
    for B, S, nh, nkv, d in ((1, 8, 4, 3, 64), (1, 8, 4, 2, 96), (-1, 8, 4, 2, 64), (1, -2, 4, 2, 64),
                             (1, 8, 0, 1, 64), (1, 8, 4, 0, 64)):
        with pytest.raises(api.SoupError) as e:
            api.attn_fwd(z, B, S, nh, nkv, d, z, z)
        assert e.value.code == api.EINVAL
        assert api.attn_bwd_scratch_bytes(B, S, nh, nkv, d) == 0
    api.attn_fwd(z, 0, 64, 4, 2, 64, z, z)
    api.attn_fwd(z, 2, 0, 4, 2, 64, z, z)
    with pytest.raises(api.SoupError) as e:
        api.attn_fwd(None, 1, 8, 4, 2, 64, z, z)
    assert e.value.code == api.EINVAL
    lib = api.lib
    rc = lib.soup_attn_bwd(z, z, z, z, 1, 8, 4, 2, 64, z, 0, z, None, 0)  # scratch too small
    assert rc == api.EINVAL
    rc = lib.soup_attn_bwd(z, z, z, z, 1, 8, 4, 2, 64, 17, 1 << 30, z, None, 0)  # misaligned scratch
    assert rc == api.EINVAL


@pytest.mark.parametrize("nh,nkv,d", [(32, 8, 128), (4, 2, 64), (40, 8, 128), (16, 1, 64)])
def test_attention_backward_scratch_covers_its_buffers(nh, nkv, d):
    """The backward's scratch holds the row sums D [B, nh, S] (float) and a bf16 copy of the
    fused q|k|v rows [B*S, (nh + 2 nkv) d] (or, on the warp-level path, per-head dK/dV partials);
    it grows with B and S and never falls below the first two."""
    prev = 0
    for B, S in ((1, 1), (1, 63), (1, 512), (2, 512), (4, 1024)):
        n = api.attn_bwd_scratch_bytes(B, S, nh, nkv, d)
        assert n >= 4 * B * nh * S + 2 * B * S * (nh + 2 * nkv) * d
        assert n >= prev
        prev = n
