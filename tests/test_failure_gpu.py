"""The failure path of the bounded device waits, forced without any fault.

Every kernel spins on its mbarriers with a wall-clock limit; a wait that runs
out records FKV_ERR_TIMEOUT in the context's device status, lets the copies
and tensor-core products it has in flight finish, frees its tensor memory and
returns.  fkv_set_wait_limit(0) (a test-only call) makes every wait report a
timeout at once, so these tests drive that path on kernels that do no
out-of-bounds access.  Then, with the limit
restored, the next call must be right: the context stays usable.  For a
decode call replayed from a CUDA graph, the header's advice is followed
(zero the workspace after a replay that timed out)."""

import numpy as np
import pytest
import torch

import oracle as O
from cross_layer_kv_gb300 import fusedkv as B
from cross_layer_kv_gb300 import synth
from parity import DecodeSetup, assert_close, f64

pytestmark = pytest.mark.gpu

DEFAULT_LIMIT_NS = 10 ** 9


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    yield
    torch.cuda.synchronize()


# Every warp of the split streams several tiles here (8 x 8 units of up to
# 8192 rows over one CTA per SM), so a timed-out warp has copies in flight.
W_DEC = synth.Workload("timeout-decode", 4, 8, 8192, 16, 8, 64, "bf16")
LENS = [8192, 4000, 33, 8191, 1, 6000, 8192, 5000]


def _pairs(w):
    return sorted({(b, kh * w.group + (b + kh) % w.group)
                   for b in range(w.batch) for kh in range(w.kv_heads)})


def _check(s, mode, what):
    got = f64(s.out)
    pairs = _pairs(s.w)
    assert_close(np.stack([got[b, h] for b, h in pairs]), s.oracle(mode, pairs), "bf16", what)


def test_set_wait_limit_rejects_above_default():
    s = DecodeSetup(synth.TINY, 3, ["fused"], seed=1)
    with pytest.raises(B.FkvError) as e:
        s.ctx.fkv_set_wait_limit(DEFAULT_LIMIT_NS + 1)
    assert e.value.status == B.FKV_ERR_INVALID_ARG
    s.close()


@pytest.mark.parametrize("mode", ["fused", "lite"])
def test_decode_timeout_then_recovers(mode):
    s = DecodeSetup(W_DEC, 4, [mode], seed=50, lens=LENS)
    s.ctx.fkv_set_wait_limit(0)
    s.run(mode)
    assert s.ctx.fkv_get_device_status() == B.FKV_ERR_TIMEOUT
    assert s.ctx.fkv_get_device_status() == B.FKV_OK   # read and cleared
    s.ctx.fkv_set_wait_limit(DEFAULT_LIMIT_NS)
    # arrival counts left by the stopped call carry its own tag: no clearing needed
    s.out.fill_(float("nan"))
    s.run(mode)
    assert s.ctx.fkv_get_device_status() == B.FKV_OK
    _check(s, mode, "after a timed-out call, %s" % mode)
    s.close()


def test_decode_graph_replay_after_timeout_with_zeroed_workspace():
    mode = "fused"
    s = DecodeSetup(W_DEC, 4, [mode], seed=51, lens=LENS)
    s.run(mode)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        s.ctx.fkv_decode_attn(s.q, s.layer, mode, s.lens, s.out, s.ws)
    s.out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert s.ctx.fkv_get_device_status() == B.FKV_OK
    _check(s, mode, "first replay")
    # a replay that times out (the limit lives in device memory, so the
    # captured launch reads the new value)
    s.ctx.fkv_set_wait_limit(0)
    g.replay()
    torch.cuda.synchronize()
    assert s.ctx.fkv_get_device_status() == B.FKV_ERR_TIMEOUT
    s.ctx.fkv_set_wait_limit(DEFAULT_LIMIT_NS)
    # as the header says: zero the workspace before the next replay
    s.ws.zero_()
    for i in range(2):
        s.q.copy_(synth.make_query(W_DEC, 4, 300 + i, "cuda"))
        s.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert s.ctx.fkv_get_device_status() == B.FKV_OK
        _check(s, mode, "replay %d after the timed-out one" % i)
    del g
    s.close()


def test_decode_q4_timeout_then_recovers():
    w = W_DEC
    ctx = B.Context(w.num_layers, w.batch, w.seq, w.q_heads, w.kv_heads, w.head_dim, "bf16")
    recs = {}   # layer -> host records, quantised by the oracle
    keep = []
    for l in (1, 2):
        k, v = synth.make_cache(w, l, 52, "cuda")
        recs[l] = tuple(O.q4_pack(*O.q4_quantize(x.to("cpu", torch.float32).numpy()))
                        for x in (k, v))
        kr, vr = (torch.from_numpy(r).to("cuda") for r in recs[l])
        ctx.fkv_bind_layer_cache_q4(l, kr, vr)
        keep.append((kr, vr))
    wts = synth.make_weights(w, 4, 52, "cuda")
    ctx.fkv_set_fusion_weights(4, *wts)
    q = synth.make_query(w, 4, 52, "cuda")
    lens = torch.tensor(LENS, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    ws = ctx.workspace("cuda")
    torch.cuda.synchronize()
    ctx.fkv_set_wait_limit(0)
    ctx.fkv_decode_attn(q, 4, "fused", lens, out, ws)
    assert ctx.fkv_get_device_status() == B.FKV_ERR_TIMEOUT
    ctx.fkv_set_wait_limit(DEFAULT_LIMIT_NS)
    out.fill_(float("nan"))
    ctx.fkv_decode_attn(q, 4, "fused", lens, out, ws)
    assert ctx.fkv_get_device_status() == B.FKV_OK
    # against the oracle over the dequantised records, sampled units
    D = w.head_dim
    got = f64(out)
    pairs = _pairs(w)
    ref, sel = [], []
    for b, h in pairs:
        kh = h // w.group
        n = LENS[b]
        kc = {l: O.q4_dequantize_records(recs[l][0][b:b + 1, kh:kh + 1, :n], D) for l in (1, 2)}
        vc = {l: O.q4_dequantize_records(recs[l][1][b:b + 1, kh:kh + 1, :n], D) for l in (1, 2)}
        ws4 = {4: tuple(f64(x[kh:kh + 1]) for x in wts)}
        ref.append(O.decode_attn(f64(q[b:b + 1, h:h + 1]), 4, w.num_layers, "fused", kc, vc, [n],
                                 weights=ws4)[0, 0])
        sel.append(got[b, h])
    assert_close(np.stack(sel), np.stack(ref), "bf16", "4-bit after a timed-out call")
    ctx.close()


class _Prefill:
    def __init__(self, D, mode, S=1024, B_=2, seed=60):
        self.w = synth.Workload("timeout-prefill", 4, B_, S, 4, 2, D, "bf16")
        w = self.w
        self.mode, self.S = mode, S
        need = [4] if mode == "vanilla" else [1, 2]
        self.ctx = B.Context(4, B_, S, 4, 2, D, "bf16", store_upper=(mode == "vanilla"))
        self.caches = {l: synth.make_cache(w, l, seed, "cuda") for l in need}
        for l, (k, v) in self.caches.items():
            self.ctx.fkv_bind_layer_cache(l, k, v)
        self.wts = synth.make_weights(w, 4, seed, "cuda")
        self.ctx.fkv_set_fusion_weights(4, *self.wts)
        g = torch.Generator(device="cuda").manual_seed(seed)
        self.q = torch.randn(B_, 4, S, D, generator=g, device="cuda").to(torch.bfloat16)
        self.out = torch.empty_like(self.q)

    def run(self):
        self.ctx.fkv_prefill_attn(self.q, 4, self.mode, self.S, self.out)

    def check(self, what):
        rows = [0, 1, 127, 128, 500, 1023]
        got = f64(self.out)
        ws = {4: tuple(f64(x) for x in self.wts)}
        for b, h in ((0, 0), (1, 3)):
            kh = h // 2
            kc = {l: f64(k[b:b + 1, kh:kh + 1]) for l, (k, v) in self.caches.items()}
            vc = {l: f64(v[b:b + 1, kh:kh + 1]) for l, (k, v) in self.caches.items()}
            wsb = {4: tuple(x[kh:kh + 1] for x in ws[4])}
            ref = O.prefill_attn(f64(self.q[b:b + 1, h:h + 1]), 4, 4, self.mode, kc, vc,
                                 weights=wsb, rows=rows)[0, 0]
            assert_close(got[b, h, rows], ref, "bf16", "%s b=%d h=%d" % (what, b, h))


@pytest.mark.parametrize("D,mode", [(64, "vanilla"), (96, "fused"), (128, "fused")],
                         ids=["one-source-128-key", "fused-112-key", "fused-D128-64-key"])
def test_prefill_timeout_then_recovers(D, mode):
    p = _Prefill(D, mode)
    p.ctx.fkv_set_wait_limit(0)
    p.run()
    assert p.ctx.fkv_get_device_status() == B.FKV_ERR_TIMEOUT
    p.ctx.fkv_set_wait_limit(DEFAULT_LIMIT_NS)
    p.out.fill_(float("nan"))
    p.run()
    assert p.ctx.fkv_get_device_status() == B.FKV_OK
    p.check("prefill %s D=%d after a timed-out call" % (mode, D))
    p.ctx.close()
