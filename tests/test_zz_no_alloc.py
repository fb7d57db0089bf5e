"""fkv_decode_attn_noalloc: decode attention for callers that cannot allocate
device memory (a process whose memory is fully held by its own pool, or a
plugin interface that hands over only one operation's operands).  It runs the
same kernel as fkv_decode_attn on the same split, so its output must equal the
workspace entry point's bit for bit, call after call, from the library's own
static scratch array; and it must match the float64 oracle.

Kept in a file of its own that pytest collects last."""

import numpy as np
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


def _pairs(w):
    # one query head of every (batch row, KV head) unit
    return sorted({(b, kh * w.group + (b + kh) % w.group)
                   for b in range(w.batch) for kh in range(w.kv_heads)})


@pytest.mark.parametrize("w,dtype", [(synth.M332, "bf16"), (synth.TINY, "f32")],
                         ids=["332M-bf16", "tiny-f32"])
def test_noalloc_matches_workspace_entry_point_twice(w, dtype):
    layer = w.num_layers
    s = DecodeSetup(w, layer, ["fused", "lite"], seed=21)
    ref_fused = s.run("fused").clone()
    ref_lite = s.run("lite").clone()
    pairs = _pairs(w)
    oracle = {m: s.oracle(m, pairs) for m in ("fused", "lite")}
    out = torch.empty_like(s.q)
    # calls in a row, different modes, so a stale array would show
    for mode, ref in (("fused", ref_fused), ("lite", ref_lite), ("fused", ref_fused)):
        out.fill_(float("nan"))
        s.ctx.fkv_decode_attn_noalloc(s.q, layer, mode, s.lens, out)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), "noalloc %s differs from the workspace call" % mode
        got = f64(out)
        sel = np.stack([got[b, h] for b, h in pairs])
        assert_close(sel, oracle[mode], dtype, "noalloc %s vs oracle" % mode)
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


def test_noalloc_graph_replays_with_another_context_between():
    """A noalloc call captured in a CUDA graph, replayed with new queries,
    while a second context with another batch and head count (so another
    layout of partials and arrival counts in the shared array) makes eager
    noalloc calls between the replays.  One replay is forced to time out; the
    next replay is right without any clearing by the caller, since every
    call clears its own arrival counts."""
    # large enough that every warp streams several tiles (copies in flight
    # when its first wait reports the timeout)
    w = synth.Workload("noalloc-graph", 4, 8, 8192, 16, 8, 64, "bf16")
    s = DecodeSetup(w, 4, ["fused"], seed=40,
                    lens=[8192, 4000, 33, 8191, 1, 6000, 8192, 5000])
    pairs = _pairs(w)
    w2 = synth.Workload("noalloc-other", 4, 5, 900, 8, 4, 80, "bf16")
    s2 = DecodeSetup(w2, 3, ["lite"], seed=41, lens=[900, 1, 450, 899, 77])
    ref2 = s2.oracle("lite")
    out2 = torch.empty_like(s2.q)
    s.ctx.fkv_decode_attn_noalloc(s.q, 4, "fused", s.lens, s.out)   # first call: set-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        s.ctx.fkv_decode_attn_noalloc(s.q, 4, "fused", s.lens, s.out)
    for i in range(4):
        s.q.copy_(synth.make_query(w, 4, 200 + i, "cuda"))
        s.out.fill_(float("nan"))
        timed_out = i == 2
        if timed_out:
            s.ctx.fkv_set_wait_limit(0)
        g.replay()
        torch.cuda.synchronize()
        if timed_out:
            assert s.ctx.fkv_get_device_status() == B.FKV_ERR_TIMEOUT
            s.ctx.fkv_set_wait_limit(10 ** 9)
        else:
            got = f64(s.out)
            assert_close(np.stack([got[b, h] for b, h in pairs]), s.oracle("fused", pairs),
                         "bf16", "replay %d" % i)
            assert s.ctx.fkv_get_device_status() == B.FKV_OK
        out2.fill_(float("nan"))
        s2.ctx.fkv_decode_attn_noalloc(s2.q, 3, "lite", s2.lens, out2)
        torch.cuda.synchronize()
        assert_close(f64(out2), ref2, "bf16", "second context after replay %d" % i)
        assert s2.ctx.fkv_get_device_status() == B.FKV_OK
    del g
    s.close()
    s2.close()
