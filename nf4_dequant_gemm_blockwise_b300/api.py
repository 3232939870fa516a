"""ctypes binding of the C ABI in include/soup.h, with the same names.

PyTorch supplies device memory and streams; tensors are passed as raw pointers.  Every call
checks the status code and raises :class:`SoupError` with the library's message.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsoup.so")

OK, EINVAL, ENOMEM, ECUDA, ESTATE, ETIMEDOUT, EPAGEABLE, ERANGE = 0, -1, -2, -3, -4, -5, -6, -7
FMT_BF16, FMT_NF4 = 0, 1
DBG_PROFILE, DBG_STALE_SLOT, DBG_COPY_DELAY_US, DBG_WAIT_PROBE = 1, 2, 3, 4
PROJ = ("q", "k", "v", "o", "gate", "up", "down")


class SoupError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"soup error {code}: {msg}")
        self.code = code


class soup_cfg(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("hidden", C.c_int32), ("inter", C.c_int32),
                ("n_heads", C.c_int32), ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("vocab", C.c_int32), ("tied", C.c_int32), ("rope_theta", C.c_float),
                ("rms_eps", C.c_float), ("base_fmt", C.c_int32), ("lora_r", C.c_int32),
                ("lora_alpha", C.c_float)]


class soup_shard_layout(C.Structure):
    _fields_ = [("stride", C.c_uint64), ("payload", C.c_uint64),
                ("w_off", C.c_uint64 * 4), ("w_bytes", C.c_uint64 * 4),
                ("a_off", C.c_uint64 * 4), ("a_bytes", C.c_uint64 * 4),
                ("ln1_off", C.c_uint64), ("ln2_off", C.c_uint64),
                ("n_out", C.c_int32 * 4), ("n_in", C.c_int32 * 4)]


class soup_stats(C.Structure):
    _fields_ = [("steps_fwd", C.c_uint64), ("steps_bwd", C.c_uint64), ("copies", C.c_uint64),
                ("copy_bytes", C.c_uint64), ("copy_ms", C.c_double),
                ("gemm_launches", C.c_uint64), ("gemm_ms", C.c_double),
                ("gemm_flops", C.c_double), ("gemm_bytes", C.c_double)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}


class soup_kernel_stat(C.Structure):
    _fields_ = [("name", C.c_char * 32), ("tensor_bound", C.c_int32), ("launches", C.c_uint64),
                ("ms", C.c_double), ("flops", C.c_double), ("bytes", C.c_double)]


class soup_adamw(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float),
                ("eps", C.c_float), ("weight_decay", C.c_float), ("grad_scale", C.c_float)]


BWD_ACCUMULATE = 1
STORE_PAGEABLE = 2
MODE_RESIDENT, MODE_KEEP_ACTIVATIONS, MODE_STREAM_HEAD = 1, 2, 4


def _mode(resident, keep_activations, stream_head=False) -> int:
    return ((MODE_RESIDENT if resident else 0) | (MODE_KEEP_ACTIVATIONS if keep_activations else 0)
            | (MODE_STREAM_HEAD if stream_head else 0))


def _load() -> C.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run python -m nf4_dequant_gemm_blockwise_b300.build")
    lib = C.CDLL(LIB_PATH)
    P, U64, I32, F32, VP = C.c_void_p, C.c_uint64, C.c_int, C.c_float, C.c_void_p
    sig = {
        "soup_last_error": (C.c_char_p, []),
        "soup_version": (C.c_char_p, []),
        "soup_kernel_launches": (C.c_uint64, []),

        "soup_nf4_codebook": (I32, [P]),
        "soup_shard_layout_of": (I32, [C.POINTER(soup_cfg), C.POINTER(soup_shard_layout)]),
        "soup_nf4_quantize_host": (I32, [P, C.c_int64, P, P, I32]),
        "soup_store_create": (I32, [C.POINTER(soup_cfg), I32, C.POINTER(VP)]),
        "soup_store_put_layer": (I32, [VP, I32, C.POINTER(P), I32]),
        "soup_store_put_shard": (I32, [VP, I32, P, U64]),
        "soup_store_put_head": (I32, [VP, P, P]),
        "soup_store_build": (I32, [C.POINTER(soup_cfg), C.POINTER(P), I32, C.POINTER(VP)]),
        "soup_store_info": (I32, [VP, C.POINTER(P), C.POINTER(U64), C.POINTER(I32)]),
        "soup_store_free": (None, [VP]),
        "soup_workspace_bytes": (I32, [C.POINTER(soup_cfg), I32, I32, I32, I32, C.POINTER(U64)]),
        "soup_peak_bytes": (U64, [C.POINTER(soup_cfg), I32, I32, I32, I32, C.POINTER(U64)]),
        "soup_stream_init": (I32, [VP, C.POINTER(soup_cfg), I32, I32, P, U64, P, P, P, C.c_size_t,
                                   C.c_size_t, I32, I32, C.POINTER(VP)]),
        "soup_step_fwd": (I32, [VP, P, I32, I32, C.POINTER(P), C.POINTER(P), P, P, P]),
        "soup_step_bwd": (I32, [VP, C.POINTER(P), C.POINTER(P), P]),
        "soup_step_bwd_ex": (I32, [VP, C.POINTER(P), C.POINTER(P), P, I32]),
        "soup_adamw_step": (I32, [P, P, P, P, C.c_int64, C.POINTER(soup_adamw), C.c_int64,
                                  C.c_size_t]),
        "soup_sync": (I32, [VP, I32]),
        "soup_stream_stats": (I32, [VP, C.POINTER(soup_stats), I32]),
        "soup_stream_kernel_stats": (I32, [VP, C.POINTER(soup_kernel_stat), I32, C.POINTER(I32), I32]),
        "soup_stream_debug": (I32, [VP, I32, I32]),
        "soup_stream_free": (None, [VP]),
        "soup_proj_scratch_bytes": (I32, [I32, I32, I32, I32, C.POINTER(U64)]),
        "soup_proj_fwd": (I32, [P, I32, I32, I32, P, P, P, P, P, I32, F32, I32, P, P, U64, C.c_size_t]),
        "soup_proj_dx": (I32, [P, I32, I32, I32, P, P, P, P, P, I32, F32, P, P, U64, C.c_size_t]),
        "soup_proj_lora_grad": (I32, [P, P, I32, I32, I32, P, P, I32, F32, I32, P, P, P, U64, C.c_size_t]),
        "soup_nf4_dequant": (I32, [P, P, C.c_int64, P, P, C.c_size_t]),
        "soup_proj_fwd_noalloc": (I32, [P, I32, I32, I32, P, P, P, P, P, I32, F32, I32, P, C.c_size_t]),
        "soup_proj_status": (I32, [P, I32, I32, I32, C.c_size_t]),
        "soup_proj_noalloc_status": (I32, [C.c_size_t]),
        "soup_attn_fwd": (I32, [P, I32, I32, I32, I32, I32, P, P, P, C.c_size_t]),
        "soup_attn_bwd_scratch_bytes": (U64, [I32, I32, I32, I32, I32]),
        "soup_attn_bwd": (I32, [P, P, P, P, I32, I32, I32, I32, I32, P, U64, P, P, C.c_size_t]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()

# every entry point include/soup.h declares (the CPU tests check the exports against it)
EXPORTS = tuple(sorted(n for n in dir(lib) if n.startswith("soup_")))


def _check(rc: int, allow=()) -> int:
    if rc != OK and rc not in allow:
        raise SoupError(rc, lib.soup_last_error().decode())
    return rc


def last_error() -> str:
    return lib.soup_last_error().decode()


def version() -> str:
    return lib.soup_version().decode()


def kernel_launches() -> int:
    return int(lib.soup_kernel_launches())



def _ptr(x) -> int | None:
    """Device or host address of a torch tensor / numpy array / int (None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


def make_cfg(cfg) -> soup_cfg:
    """soup_cfg from any object with the stack's fields (n_layers, hidden, ..., base_fmt
    'nf4'|'bf16', lora_r, lora_alpha)."""
    fmt = cfg.base_fmt
    if isinstance(fmt, str):
        fmt = FMT_NF4 if fmt == "nf4" else FMT_BF16
    return soup_cfg(cfg.n_layers, cfg.hidden, cfg.inter, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim,
                    cfg.vocab, int(bool(cfg.tied)), float(cfg.rope_theta), float(cfg.rms_eps), fmt,
                    cfg.lora_r, float(cfg.lora_alpha))


def nf4_codebook() -> np.ndarray:
    out = np.zeros(16, np.float32)
    _check(lib.soup_nf4_codebook(out.ctypes.data))
    return out


def shard_layout_of(cfg) -> soup_shard_layout:
    c = make_cfg(cfg)
    out = soup_shard_layout()
    _check(lib.soup_shard_layout_of(C.byref(c), C.byref(out)))
    return out


def nf4_quantize_host(src_bf16_bits: np.ndarray, n_threads: int = 0):
    """Host packer: bf16 bit patterns -> (packed codes uint8, absmax float32)."""
    src = np.ascontiguousarray(src_bf16_bits, np.uint16).reshape(-1)
    n = src.size
    codes = np.empty((n + 1) // 2, np.uint8)
    absmax = np.empty((n + 63) // 64, np.float32)
    _check(lib.soup_nf4_quantize_host(src.ctypes.data, n, codes.ctypes.data, absmax.ctypes.data,
                                      n_threads))
    return codes, absmax


def workspace_bytes(cfg, max_batch, max_seq, n_slots=2, resident=False, keep_activations=False,
                    stream_head=False) -> int:
    c = make_cfg(cfg)
    out = C.c_uint64()
    _check(lib.soup_workspace_bytes(C.byref(c), max_batch, max_seq, n_slots,
                                    _mode(resident, keep_activations, stream_head), C.byref(out)))
    return out.value


def peak_bytes(cfg, batch, seq, n_slots=2, resident=False, keep_activations=False, stream_head=False):
    """(total device bytes of a run, workspace part)."""
    c = make_cfg(cfg)
    ws = C.c_uint64()
    tot = lib.soup_peak_bytes(C.byref(c), batch, seq, n_slots,
                              _mode(resident, keep_activations, stream_head), C.byref(ws))
    if tot == 0:
        raise SoupError(EINVAL, last_error())
    return tot, ws.value


class Store:
    """One page-locked host arena holding every layer's shard (soup_store_*)."""

    def __init__(self, cfg, allow_pageable: bool = True, force_pageable: bool = False):
        """force_pageable: skip page-locking (to measure the pageable fallback)."""
        self.cfg = make_cfg(cfg)
        h = C.c_void_p()
        rc = lib.soup_store_create(C.byref(self.cfg), STORE_PAGEABLE if force_pageable else int(allow_pageable),
                                   C.byref(h))
        self.pageable_warning = rc == EPAGEABLE
        _check(rc, allow=(EPAGEABLE,))
        self.handle = h

    def put_layer(self, layer: int, tensors, n_threads: int = 0):
        """tensors: nine bf16-bit arrays q,k,v,o,gate,up,down ([out,in]) and ln1, ln2."""
        arrs = [np.ascontiguousarray(t, np.uint16) for t in tensors]
        ptrs = (C.c_void_p * 9)(*[a.ctypes.data for a in arrs])
        _check(lib.soup_store_put_layer(self.handle, layer, ptrs, n_threads))

    def put_shard(self, layer: int, shard: np.ndarray):
        """Fill a shard from its bytes (e.g. another store's ``shard_bytes``)."""
        b = np.ascontiguousarray(shard, np.uint8)
        _check(lib.soup_store_put_shard(self.handle, layer, b.ctypes.data, b.nbytes))

    def put_head(self, embed: np.ndarray, lm_head: np.ndarray | None):
        """The embedding and the untied output head (None when tied), bf16 bits [vocab,
        hidden], for streams with stream_head=True."""
        e = np.ascontiguousarray(embed, np.uint16)
        h = None if lm_head is None else np.ascontiguousarray(lm_head, np.uint16)
        _check(lib.soup_store_put_head(self.handle, e.ctypes.data, None if h is None else h.ctypes.data))

    def info(self):
        base, nb, pinned = C.c_void_p(), C.c_uint64(), C.c_int()
        _check(lib.soup_store_info(self.handle, C.byref(base), C.byref(nb), C.byref(pinned)))
        return base.value, nb.value, bool(pinned.value)

    def shard_bytes(self, layer: int) -> np.ndarray:
        """A numpy view of one shard in the arena (host memory)."""
        base, _, _ = self.info()
        lay = shard_layout_of_cfg(self.cfg)
        buf = (C.c_uint8 * lay.stride).from_address(base + layer * lay.stride)
        return np.frombuffer(buf, np.uint8)

    def free(self):
        if self.handle:
            lib.soup_store_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def shard_layout_of_cfg(c: soup_cfg) -> soup_shard_layout:
    out = soup_shard_layout()
    _check(lib.soup_shard_layout_of(C.byref(c), C.byref(out)))
    return out


class Stream:
    """A stream handle: a store bound to a device workspace and two CUDA streams."""

    def __init__(self, store: Store, max_batch, max_seq, workspace, embed, lm_head, final_norm,
                 compute_stream, copy_stream, n_slots=2, resident=False, keep_activations=False,
                 stream_head=False):
        self.store = store
        self.cfg = store.cfg
        ws_need = C.c_uint64()
        mode = _mode(resident, keep_activations, stream_head)
        _check(lib.soup_workspace_bytes(C.byref(self.cfg), max_batch, max_seq, n_slots, mode,
                                        C.byref(ws_need)))
        self.keep = (workspace, embed, lm_head, final_norm)
        h = C.c_void_p()
        _check(lib.soup_stream_init(store.handle, C.byref(self.cfg), max_batch, max_seq, _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _ptr(embed),
                                    _ptr(lm_head), _ptr(final_norm), compute_stream.cuda_stream,
                                    copy_stream.cuda_stream, n_slots, mode, C.byref(h)))
        self.handle = h

    def fwd(self, tokens, B, S, lora_A, lora_B, loss, logits=None, layer_out=None):
        """lora_A = lora_B = None: adapters switched off (the base alone)."""
        if lora_A is None and lora_B is None:
            a = b = None
        else:
            n = len(lora_A)
            a = (C.c_void_p * n)(*[_ptr(t) for t in lora_A])
            b = (C.c_void_p * n)(*[_ptr(t) for t in lora_B])
        self._lora = (a, b, lora_A, lora_B)
        _check(lib.soup_step_fwd(self.handle, _ptr(tokens), B, S, a, b, _ptr(loss), _ptr(logits),
                                 _ptr(layer_out)))

    def bwd(self, dA, dB, dh_out=None, accumulate=False):
        n = len(dA)
        a = (C.c_void_p * n)(*[_ptr(t) for t in dA])
        b = (C.c_void_p * n)(*[_ptr(t) for t in dB])
        if accumulate:
            _check(lib.soup_step_bwd_ex(self.handle, a, b, _ptr(dh_out), BWD_ACCUMULATE))
        else:
            _check(lib.soup_step_bwd(self.handle, a, b, _ptr(dh_out)))

    def sync(self, timeout_ms: int = 60000):
        _check(lib.soup_sync(self.handle, timeout_ms))

    def stats(self, reset: bool = False) -> dict:
        s = soup_stats()
        _check(lib.soup_stream_stats(self.handle, C.byref(s), int(reset)))
        return s.as_dict()

    def kernel_stats(self, reset: bool = False) -> list:
        """Per kernel family (profiling mode 2): name, tensor_bound, launches, ms, flops, bytes."""
        n = C.c_int()
        _check(lib.soup_stream_kernel_stats(self.handle, None, 0, C.byref(n), 0))
        arr = (soup_kernel_stat * max(n.value, 1))()
        _check(lib.soup_stream_kernel_stats(self.handle, arr, n.value, C.byref(n), int(reset)))
        return [{"name": a.name.decode(), "tensor_bound": bool(a.tensor_bound), "launches": a.launches,
                 "ms": a.ms, "flops": a.flops, "bytes": a.bytes} for a in arr[:n.value]]

    def debug(self, what: int, value: int):
        _check(lib.soup_stream_debug(self.handle, what, value))

    def free(self):
        if getattr(self, "handle", None):
            lib.soup_stream_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def proj_scratch_bytes(M, N, K, r) -> int:
    out = C.c_uint64()
    _check(lib.soup_proj_scratch_bytes(M, N, K, r, C.byref(out)))
    return out.value


def proj_fwd(x, M, N, K, codes, absmax, w_bf16, A, B, r, s, y, scratch, stream=0, x_f16=True):
    _check(lib.soup_proj_fwd(_ptr(x), M, N, K, _ptr(codes), _ptr(absmax), _ptr(w_bf16), _ptr(A),
                             _ptr(B), r, s, int(x_f16), _ptr(y), _ptr(scratch),
                             scratch.numel() * scratch.element_size(), _stream(stream)))


def proj_fwd_noalloc(x, M, N, K, codes, absmax, w_bf16, A, B, r, s, y, stream=0, x_f16=True):
    """soup_proj_fwd with the library's static device scratch (no allocation by anyone)."""
    _check(lib.soup_proj_fwd_noalloc(_ptr(x), M, N, K, _ptr(codes), _ptr(absmax), _ptr(w_bf16),
                                     _ptr(A), _ptr(B), r, s, int(x_f16), _ptr(y), _stream(stream)))


def proj_noalloc_status(stream=0):
    """Wait for `stream` and raise if a proj_fwd_noalloc call since the last check reported a
    kernel error (bounded wait given up, half-precision overflow); clears the shared flag."""
    _check(lib.soup_proj_noalloc_status(_stream(stream)))


def attn_fwd(qkv, B, S, n_heads, n_kv_heads, head_dim, o, lse, err=None, stream=0):
    """Causal GQA attention of one layer (soup_attn_fwd): qkv half [B*S, (nh + 2 nkv) d] ->
    o half [B*S, nh d], lse float [B, nh, S]; err: optional device int32 for error bits."""
    _check(lib.soup_attn_fwd(_ptr(qkv), B, S, n_heads, n_kv_heads, head_dim, _ptr(o), _ptr(lse),
                             _ptr(err), _stream(stream)))


def attn_bwd_scratch_bytes(B, S, n_heads, n_kv_heads, head_dim) -> int:
    return int(lib.soup_attn_bwd_scratch_bytes(B, S, n_heads, n_kv_heads, head_dim))


def attn_bwd(qkv, o, dO, lse, B, S, n_heads, n_kv_heads, head_dim, scratch, dqkv, err=None, stream=0):
    """Backward of attn_fwd (soup_attn_bwd): dO bf16 [B*S, nh d] -> dqkv float in qkv's layout."""
    _check(lib.soup_attn_bwd(_ptr(qkv), _ptr(o), _ptr(dO), _ptr(lse), B, S, n_heads, n_kv_heads,
                             head_dim, _ptr(scratch), scratch.numel() * scratch.element_size(),
                             _ptr(dqkv), _ptr(err), _stream(stream)))


def proj_dx(dy, M, N, K, codes, absmax, w_bf16, A, B, r, s, dx, scratch, stream=0):
    _check(lib.soup_proj_dx(_ptr(dy), M, N, K, _ptr(codes), _ptr(absmax), _ptr(w_bf16), _ptr(A),
                            _ptr(B), r, s, _ptr(dx), _ptr(scratch),
                            scratch.numel() * scratch.element_size(), _stream(stream)))


def proj_status(scratch, M, N, K, stream=0):
    """Raise SoupError(ETIMEDOUT) if a kernel of the projections that used `scratch` gave up a
    bounded wait; clears the flag.  Waits for the stream."""
    _check(lib.soup_proj_status(_ptr(scratch), M, N, K, _stream(stream)))


def proj_lora_grad(x, dy, M, N, K, A, B, r, s, dA, dB, scratch, stream=0, x_f16=True):
    _check(lib.soup_proj_lora_grad(_ptr(x), _ptr(dy), M, N, K, _ptr(A), _ptr(B), r, s, int(x_f16), _ptr(dA),
                                   _ptr(dB), _ptr(scratch), scratch.numel() * scratch.element_size(),
                                   _stream(stream)))


def nf4_dequant(codes, absmax, n, out_f32=None, out_bf16=None, stream=0):
    _check(lib.soup_nf4_dequant(_ptr(codes), _ptr(absmax), n, _ptr(out_f32), _ptr(out_bf16),
                                _stream(stream)))


def adamw_step(param, grad, m, v, n, step, lr, beta1=0.9, beta2=0.999, eps=1e-8,
               weight_decay=0.0, grad_scale=1.0, stream=0):
    """One in-place AdamW step over n floats of device buffers (soup_adamw_step)."""
    hp = soup_adamw(lr, beta1, beta2, eps, weight_decay, grad_scale)
    _check(lib.soup_adamw_step(_ptr(param), _ptr(grad), _ptr(m), _ptr(v), n, C.byref(hp), step,
                               _stream(stream)))


def _stream(s) -> int:
    if s is None or isinstance(s, int):
        return s or 0
    return s.cuda_stream
