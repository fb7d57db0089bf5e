"""CPU checks of the C-ABI boundary: the library builds, loads, exports every
function include/fusedkv.h declares, and rejects bad arguments on the host
before any CUDA call."""

import ctypes

import pytest
import torch

import cross_layer_kv_gb300 as fkv
from cross_layer_kv_gb300 import fusedkv as B


def test_library_exports_every_header_symbol():
    lib = fkv.load()
    names = fkv.header_symbols()
    assert set(names) >= {"fkv_create", "fkv_destroy", "fkv_bind_layer_cache",
                          "fkv_set_fusion_weights", "fkv_append_kv", "fkv_decode_workspace_bytes",
                          "fkv_decode_attn", "fkv_prefill_attn", "fkv_get_device_status",
                          "fkv_status_string"}
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(B._SIGS), "binding and header disagree"


def test_status_strings():
    seen = set()
    for s in range(7):
        txt = fkv.status_string(s)
        assert txt and txt != "unknown status"
        seen.add(txt)
    assert len(seen) == 7
    assert fkv.status_string(99) == "unknown status"


def _cfg(**kw):
    base = dict(num_layers=4, batch=1, max_seq=256, num_q_heads=4, num_kv_heads=2, head_dim=64,
                dtype=B.FKV_F32, store_upper=0, softmax_scale=0.0, decode_ctas=0)
    base.update(kw)
    return B.fkv_config(**base)


def _create(cfg):
    lib = fkv.load()
    h = ctypes.c_void_p(1234)
    s = lib.fkv_create(ctypes.byref(cfg), ctypes.byref(h))
    return s, h


@pytest.mark.parametrize("kw,status", [
    (dict(num_layers=3), B.FKV_ERR_INVALID_ARG),
    (dict(num_layers=0), B.FKV_ERR_INVALID_ARG),
    (dict(batch=0), B.FKV_ERR_INVALID_ARG),
    (dict(max_seq=0), B.FKV_ERR_INVALID_ARG),
    (dict(num_q_heads=3), B.FKV_ERR_INVALID_ARG),
    (dict(dtype=7), B.FKV_ERR_INVALID_ARG),
    (dict(softmax_scale=-1.0), B.FKV_ERR_INVALID_ARG),
    (dict(softmax_scale=float("nan")), B.FKV_ERR_INVALID_ARG),
    (dict(decode_ctas=-1), B.FKV_ERR_INVALID_ARG),
    (dict(batch=1025), B.FKV_ERR_INVALID_ARG),
    (dict(batch=1024, num_kv_heads=64, max_seq=1 << 15), B.FKV_ERR_INVALID_ARG),
    (dict(head_dim=72), B.FKV_ERR_UNSUPPORTED),
    (dict(num_q_heads=16, num_kv_heads=2), B.FKV_ERR_UNSUPPORTED),
])
def test_create_rejects_bad_configs_before_cuda(kw, status):
    s, h = _create(_cfg(**kw))
    assert s == status
    assert h.value is None


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_create_without_gpu_reports_cuda_error():
    s, h = _create(_cfg())
    assert s == B.FKV_ERR_CUDA
    assert h.value is None


def test_null_context_is_rejected_everywhere():
    lib = fkv.load()
    assert lib.fkv_bind_layer_cache(None, 1, 16, 16) == B.FKV_ERR_INVALID_ARG
    assert lib.fkv_set_fusion_weights(None, 3, 16, 16, 16, 16) == B.FKV_ERR_INVALID_ARG
    assert lib.fkv_append_kv(None, 1, 16, 16, 16, 1, None) == B.FKV_ERR_INVALID_ARG
    assert lib.fkv_decode_attn(None, 16, 3, 2, 16, 16, 16, 1 << 20, None) == B.FKV_ERR_INVALID_ARG
    assert lib.fkv_prefill_attn(None, 16, 3, 2, 8, 16, None) == B.FKV_ERR_INVALID_ARG
    assert lib.fkv_get_device_status(None, None) == B.FKV_ERR_INVALID_ARG
    assert lib.fkv_decode_workspace_bytes(None) == 0
    lib.fkv_destroy(None)


def test_create_null_out_pointer():
    lib = fkv.load()
    cfg = _cfg()
    assert lib.fkv_create(ctypes.byref(cfg), None) == B.FKV_ERR_INVALID_ARG
    assert lib.fkv_create(None, ctypes.byref(ctypes.c_void_p())) == B.FKV_ERR_INVALID_ARG
