"""fkv_decode_attn_noalloc: decode attention for callers that cannot allocate
device memory (a process whose memory is fully held by its own pool, or a
plugin interface that hands over only one operation's operands).  It must give
the workspace entry point's answer, call after call, from the library's own
static scratch array.

Kept in a file of its own that pytest collects last."""

import pytest
import torch

from cross_layer_kv_gb300 import fusedkv as B
from cross_layer_kv_gb300 import synth
from parity import DecodeSetup, assert_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("w,dtype", [(synth.M332, "bf16"), (synth.TINY, "f32")],
                         ids=["332M-bf16", "tiny-f32"])
def test_noalloc_matches_workspace_entry_point_twice(w, dtype):
    layer = w.num_layers
    s = DecodeSetup(w, layer, ["fused", "lite"], seed=21)
    ref_fused = s.run("fused").clone()
    ref_lite = s.run("lite").clone()
    out = torch.empty_like(s.q)
    # two calls in a row, different modes, so a stale array would show
    for mode, ref in (("fused", ref_fused), ("lite", ref_lite), ("fused", ref_fused)):
        out.fill_(float("nan"))
        s.ctx.fkv_decode_attn_noalloc(s.q, layer, mode, s.lens, out)
        assert_close(f64(out), f64(ref), dtype, "noalloc %s" % mode)
    assert s.ctx.fkv_get_device_status() == B.FKV_OK
    s.close()


def test_noalloc_rejects_workspace_above_limit():
    # 1024 x 64 KV heads need far more than 4 MiB of partials
    ctx = B.Context(4, 1024, 8, 128, 64, 128, "bf16")
    assert ctx.fkv_decode_workspace_bytes() > (4 << 20)
    q = torch.zeros(1024, 128, 128, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(1024, dtype=torch.int32, device="cuda")
    k = torch.zeros(1024, 64, 8, 128, dtype=torch.bfloat16, device="cuda")
    ctx.fkv_bind_layer_cache(1, k, k)
    with pytest.raises(B.FkvError) as e:
        ctx.fkv_decode_attn_noalloc(q, 1, "vanilla", lens, q.clone())
    assert e.value.status == B.FKV_ERR_WORKSPACE
    ctx.close()
