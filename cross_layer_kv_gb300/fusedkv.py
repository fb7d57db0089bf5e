"""Thin ctypes binding of libfusedkv.so (include/fusedkv.h).

Argument marshalling only: every function keeps the C name, takes torch
tensors (device memory owned by the caller) or plain ints, checks shapes and
dtypes against the context, and forwards raw pointers.  All arithmetic runs in
the library's CUDA kernels; if the library is missing this module raises.
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Sequence

import torch

from . import build as _build

FKV_OK = 0
FKV_ERR_INVALID_ARG = 1
FKV_ERR_UNSUPPORTED = 2
FKV_ERR_CUDA = 3
FKV_ERR_TIMEOUT = 4
FKV_ERR_WORKSPACE = 5
FKV_ERR_DEVICE_ARG = 6

FKV_VANILLA, FKV_LITE, FKV_FUSED, FKV_SCALED = 0, 1, 2, 3
MODES = {"vanilla": FKV_VANILLA, "lite": FKV_LITE, "fused": FKV_FUSED, "scaled": FKV_SCALED}
FKV_BF16, FKV_F32 = 0, 1

# Kernel launches per call: decode = 1 (split + in-kernel merge); append = 1.
DECODE_LAUNCHES_PER_CALL = 1
APPEND_LAUNCHES_PER_CALL = 1

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "fusedkv.h")


class FkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (what, status_string(status), status))


class fkv_config(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int),
        ("batch", ctypes.c_int),
        ("max_seq", ctypes.c_int),
        ("num_q_heads", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("store_upper", ctypes.c_int),
        ("softmax_scale", ctypes.c_float),
        ("decode_ctas", ctypes.c_int),
    ]


_LIB: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_SIGS = {
    "fkv_create": (ctypes.c_int, [ctypes.POINTER(fkv_config), ctypes.POINTER(_P)]),
    "fkv_destroy": (None, [_P]),
    "fkv_bind_layer_cache": (ctypes.c_int, [_P, ctypes.c_int, _P, _P]),
    "fkv_q4_row_bytes": (ctypes.c_size_t, [ctypes.c_int]),
    "fkv_bind_layer_cache_q4": (ctypes.c_int, [_P, ctypes.c_int, _P, _P]),
    "fkv_set_fusion_weights": (ctypes.c_int, [_P, ctypes.c_int, _P, _P, _P, _P]),
    "fkv_set_sources": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int]),
    "fkv_set_window": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int]),
    "fkv_set_ring_rows": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int]),
    "fkv_append_kv": (ctypes.c_int, [_P, ctypes.c_int, _P, _P, _P, ctypes.c_int, _P]),
    "fkv_decode_workspace_bytes": (ctypes.c_size_t, [_P]),
    "fkv_decode_attn": (ctypes.c_int, [_P, _P, ctypes.c_int, ctypes.c_int, _P, _P, _P,
                                       ctypes.c_size_t, _P]),
    "fkv_decode_attn_noalloc": (ctypes.c_int, [_P, _P, ctypes.c_int, ctypes.c_int, _P, _P, _P]),
    "fkv_prefill_attn": (ctypes.c_int, [_P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P]),
    "fkv_prefill_attn_chunk": (ctypes.c_int, [_P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, _P, _P]),
    "fkv_get_device_status": (ctypes.c_int, [_P, _P]),
    "fkv_set_wait_limit": (ctypes.c_int, [_P, ctypes.c_ulonglong]),
    "fkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}


def header_symbols(path: str = HEADER) -> Sequence[str]:
    """Function names declared in include/fusedkv.h."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fkv_\w+)\s*\(", text)))


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the in-tree libfusedkv.so."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB
    if not os.path.exists(path) or not _build.up_to_date():
        if not build_if_missing:
            raise FileNotFoundError("libfusedkv.so is not built: run cross_layer_kv_gb300.build")
        _build.build()
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def status_string(status: int) -> str:
    return load().fkv_status_string(status).decode()


def _check(status: int, what: str):
    if status != FKV_OK:
        raise FkvError(status, what)


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    raise TypeError("expected a tensor, an int pointer or None, got %r" % type(x))


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


class Context:
    """An fkv_ctx plus references to the caller buffers bound to it (kept
    alive for as long as the context can read them)."""

    def __init__(self, num_layers: int, batch: int, max_seq: int, num_q_heads: int,
                 num_kv_heads: int, head_dim: int, dtype: str = "bf16", store_upper: bool = False,
                 softmax_scale: float = 0.0, decode_ctas: int = 0):
        self.cfg = fkv_config(num_layers, batch, max_seq, num_q_heads, num_kv_heads, head_dim,
                              FKV_F32 if dtype in ("f32", "fp32", torch.float32) else FKV_BF16,
                              1 if store_upper else 0, softmax_scale, decode_ctas)
        self.torch_dtype = torch.float32 if self.cfg.dtype == FKV_F32 else torch.bfloat16
        self._lib = load()
        h = ctypes.c_void_p()
        _check(self._lib.fkv_create(ctypes.byref(self.cfg), ctypes.byref(h)), "fkv_create")
        self.handle = h
        self._keep = {}
        self._ring = {}   # layer -> ring rows (layers with full-length caches absent)

    # -- lifetime --------------------------------------------------------
    def close(self):
        if getattr(self, "handle", None):
            self._lib.fkv_destroy(self.handle)
            self.handle = None
            self._keep.clear()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- shape checks (marshalling only) ---------------------------------
    def _rows(self, layer: int) -> int:
        """Cache rows per (batch row, KV head) of a layer: S_max, or its ring's rows."""
        return self._ring.get(layer) or self.cfg.max_seq

    def _cache_shape(self, layer: int):
        c = self.cfg
        return (c.batch, c.num_kv_heads, self._rows(layer), c.head_dim)

    def _need(self, t: torch.Tensor, shape, dtype, name):
        if not isinstance(t, torch.Tensor):
            return
        if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_contiguous():
            raise ValueError("%s: expected contiguous %s %s, got %s %s" %
                             (name, dtype, tuple(shape), t.dtype, tuple(t.shape)))

    # -- the C calls -----------------------------------------------------
    def fkv_bind_layer_cache(self, layer: int, k, v):
        self._need(k, self._cache_shape(layer), self.torch_dtype, "k cache")
        self._need(v, self._cache_shape(layer), self.torch_dtype, "v cache")
        _check(self._lib.fkv_bind_layer_cache(self.handle, layer, _ptr(k), _ptr(v)),
               "fkv_bind_layer_cache")
        self._keep[("kv", layer)] = (k, v)

    def fkv_q4_row_bytes(self) -> int:
        return int(self._lib.fkv_q4_row_bytes(self.cfg.head_dim))

    def q4_cache(self, device="cuda", rows: Optional[int] = None) -> torch.Tensor:
        """A zeroed uint8 [B, H_kv, rows (default S_max), fkv_q4_row_bytes(D)] buffer."""
        c = self.cfg
        return torch.zeros((c.batch, c.num_kv_heads, rows or c.max_seq, self.fkv_q4_row_bytes()),
                           dtype=torch.uint8, device=device)

    def fkv_bind_layer_cache_q4(self, layer: int, k_rec, v_rec):
        c = self.cfg
        shape = (c.batch, c.num_kv_heads, self._rows(layer), self.fkv_q4_row_bytes())
        self._need(k_rec, shape, torch.uint8, "k records")
        self._need(v_rec, shape, torch.uint8, "v records")
        _check(self._lib.fkv_bind_layer_cache_q4(self.handle, layer, _ptr(k_rec), _ptr(v_rec)),
               "fkv_bind_layer_cache_q4")
        self._keep[("kv", layer)] = (k_rec, v_rec)

    def fkv_set_fusion_weights(self, layer: int, a_first, a_second, b_first, b_second):
        shape = (self.cfg.num_kv_heads, self.cfg.head_dim)
        for n, t in zip(("a_first", "a_second", "b_first", "b_second"),
                        (a_first, a_second, b_first, b_second)):
            self._need(t, shape, torch.float32, n)
        _check(self._lib.fkv_set_fusion_weights(self.handle, layer, _ptr(a_first), _ptr(a_second),
                                                _ptr(b_first), _ptr(b_second)),
               "fkv_set_fusion_weights")
        self._keep[("w", layer)] = (a_first, a_second, b_first, b_second)

    def fkv_set_sources(self, layer: int, mode, k_first: int, k_second: int = 0, v_first: int = 0,
                        v_second: int = 0):
        m = MODES[mode] if isinstance(mode, str) else int(mode)
        _check(self._lib.fkv_set_sources(self.handle, layer, m, k_first, k_second, v_first,
                                         v_second), "fkv_set_sources")

    def fkv_set_window(self, layer: int, window: int):
        _check(self._lib.fkv_set_window(self.handle, layer, window), "fkv_set_window")

    def fkv_set_ring_rows(self, layer: int, rows: int):
        """Make a layer's caches rings of `rows` rows (0: full length).  Bind
        the layer's caches after this call: the bind checks their row count."""
        _check(self._lib.fkv_set_ring_rows(self.handle, layer, rows), "fkv_set_ring_rows")
        if rows in (0, self.cfg.max_seq):
            self._ring.pop(layer, None)
        else:
            self._ring[layer] = rows

    def fkv_append_kv(self, layer: int, k_new, v_new, pos, T: Optional[int] = None, stream=None):
        c = self.cfg
        if T is None:
            T = k_new.shape[2]
        shape = (c.batch, c.num_kv_heads, T, c.head_dim)
        self._need(k_new, shape, self.torch_dtype, "k_new")
        self._need(v_new, shape, self.torch_dtype, "v_new")
        self._need(pos, (c.batch,), torch.int32, "pos")
        _check(self._lib.fkv_append_kv(self.handle, layer, _ptr(k_new), _ptr(v_new), _ptr(pos), T,
                                       _stream(stream)), "fkv_append_kv")

    def fkv_decode_workspace_bytes(self) -> int:
        return int(self._lib.fkv_decode_workspace_bytes(self.handle))

    def workspace(self, device="cuda") -> torch.Tensor:
        """A caller-owned workspace buffer of the required size."""
        n = (self.fkv_decode_workspace_bytes() + 15) // 16 * 16
        return torch.empty(n, dtype=torch.uint8, device=device)

    def fkv_decode_attn(self, q, layer: int, mode, seq_lens, out, workspace, stream=None):
        c = self.cfg
        shape = (c.batch, c.num_q_heads, c.head_dim)
        self._need(q, shape, self.torch_dtype, "q")
        self._need(out, shape, self.torch_dtype, "out")
        self._need(seq_lens, (c.batch,), torch.int32, "seq_lens")
        m = MODES[mode] if isinstance(mode, str) else int(mode)
        nbytes = workspace.numel() * workspace.element_size() if isinstance(workspace, torch.Tensor) \
            else int(getattr(workspace, "nbytes", 0))
        _check(self._lib.fkv_decode_attn(self.handle, _ptr(q), layer, m, _ptr(seq_lens), _ptr(out),
                                         _ptr(workspace), nbytes, _stream(stream)),
               "fkv_decode_attn")
        return out

    def fkv_decode_attn_noalloc(self, q, layer: int, mode, seq_lens, out, stream=None):
        """fkv_decode_attn for callers that cannot allocate: the partials live
        in the library's own 4 MiB of static device memory."""
        c = self.cfg
        shape = (c.batch, c.num_q_heads, c.head_dim)
        self._need(q, shape, self.torch_dtype, "q")
        self._need(out, shape, self.torch_dtype, "out")
        self._need(seq_lens, (c.batch,), torch.int32, "seq_lens")
        m = MODES[mode] if isinstance(mode, str) else int(mode)
        _check(self._lib.fkv_decode_attn_noalloc(self.handle, _ptr(q), layer, m, _ptr(seq_lens),
                                                 _ptr(out), _stream(stream)),
               "fkv_decode_attn_noalloc")
        return out

    def fkv_prefill_attn(self, q, layer: int, mode, S: int, out, stream=None):
        c = self.cfg
        shape = (c.batch, c.num_q_heads, S, c.head_dim)
        self._need(q, shape, self.torch_dtype, "q")
        self._need(out, shape, self.torch_dtype, "out")
        m = MODES[mode] if isinstance(mode, str) else int(mode)
        _check(self._lib.fkv_prefill_attn(self.handle, _ptr(q), layer, m, S, _ptr(out),
                                          _stream(stream)), "fkv_prefill_attn")
        return out

    def fkv_prefill_attn_chunk(self, q, layer: int, mode, q_start: int, C: int, out, stream=None):
        c = self.cfg
        shape = (c.batch, c.num_q_heads, C, c.head_dim)
        self._need(q, shape, self.torch_dtype, "q")
        self._need(out, shape, self.torch_dtype, "out")
        m = MODES[mode] if isinstance(mode, str) else int(mode)
        _check(self._lib.fkv_prefill_attn_chunk(self.handle, _ptr(q), layer, m, q_start, C, _ptr(out),
                                                _stream(stream)), "fkv_prefill_attn_chunk")
        return out

    def fkv_get_device_status(self, stream=None) -> int:
        """The device status code (FKV_OK, FKV_ERR_DEVICE_ARG, FKV_ERR_TIMEOUT);
        synchronises the stream and clears the word."""
        return int(self._lib.fkv_get_device_status(self.handle, _stream(stream)))

    def fkv_set_wait_limit(self, limit_ns: int):
        """Failure-path tests only: the limit of every bounded device wait of
        this context's later kernels (1 s by default; 0 makes every wait
        report a timeout at once).  Synchronous."""
        _check(self._lib.fkv_set_wait_limit(self.handle, int(limit_ns)), "fkv_set_wait_limit")
