"""GPU check of fkv_append_kv: a pure copy, compared bit for bit with the
oracle's append."""

import numpy as np
import pytest
import torch

import oracle as O
from cross_layer_kv_gb300 import fusedkv as B
from cross_layer_kv_gb300 import synth
from parity import f64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("bf16", 80), ("f32", 96), ("bf16", 128)])
@pytest.mark.parametrize("T", [1, 5])
def test_append_matches_oracle(dtype, D, T):
    Bt, H, S = 3, 2, 40
    ctx = B.Context(4, Bt, S, 4, H, D, dtype)
    tdt = ctx.torch_dtype
    g = torch.Generator(device="cuda").manual_seed(1)
    k = torch.randn(Bt, H, S, D, generator=g, device="cuda").to(tdt)
    v = torch.randn(Bt, H, S, D, generator=g, device="cuda").to(tdt)
    kn = torch.randn(Bt, H, T, D, generator=g, device="cuda").to(tdt)
    vn = torch.randn(Bt, H, T, D, generator=g, device="cuda").to(tdt)
    pos = torch.tensor([0, 17, S - T], dtype=torch.int32, device="cuda")
    k0, v0 = f64(k), f64(v)
    ctx.fkv_bind_layer_cache(2, k, v)
    ctx.fkv_append_kv(2, kn, vn, pos)
    assert ctx.fkv_get_device_status() == B.FKV_OK
    np.testing.assert_array_equal(f64(k), O.append_kv(k0, f64(kn), pos.tolist()))
    np.testing.assert_array_equal(f64(v), O.append_kv(v0, f64(vn), pos.tolist()))
    ctx.close()


def test_append_out_of_range_skipped_and_flagged():
    Bt, H, S, D = 2, 1, 16, 64
    ctx = B.Context(2, Bt, S, 1, H, D, "bf16")
    k = torch.zeros(Bt, H, S, D, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    kn = torch.ones(Bt, H, 2, D, dtype=torch.bfloat16, device="cuda")
    pos = torch.tensor([15, 3], dtype=torch.int32, device="cuda")  # 15 + 2 > 16
    ctx.fkv_bind_layer_cache(1, k, v)
    ctx.fkv_append_kv(1, kn, kn, pos)
    assert ctx.fkv_get_device_status() == B.FKV_ERR_DEVICE_ARG
    assert torch.all(k[0] == 0)
    assert torch.all(k[1, :, 3:5] == 1) and torch.all(k[1, :, 5:] == 0)
    ctx.close()


def test_append_to_upper_layer_needs_store_upper():
    ctx = B.Context(4, 1, 8, 2, 1, 64, "bf16")
    k = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.FkvError) as e:
        ctx.fkv_bind_layer_cache(3, k, k)
    assert e.value.status == B.FKV_ERR_UNSUPPORTED
    ctx.close()
