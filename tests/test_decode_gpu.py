"""GPU parity of fkv_decode_attn against the float64 oracle, through the C ABI.

Small cases compare every output element; the full-size workloads (the
launch configuration the benchmark times) compare sampled (batch, head) rows
that the oracle computes one at a time."""

import dataclasses

import numpy as np
import pytest
import torch

from cross_layer_kv_gb300 import synth
from cross_layer_kv_gb300 import fusedkv as B
from parity import DecodeSetup, assert_close, f64

pytestmark = pytest.mark.gpu

MODES = ("vanilla", "lite", "fused")
ALL_MODES = MODES + ("scaled",)


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("layer", [1, 2, 3, 4])
def test_tiny_fp32_all_layers(mode, layer):
    """L=4, B=1, S=256, 4 Q / 2 KV heads, D=64, fp32, seed 0: max-abs 1e-5."""
    s = DecodeSetup(synth.TINY, layer, [mode])
    got = f64(s.run(mode))
    assert s.ctx.fkv_get_device_status() == B.FKV_OK
    assert_close(got, s.oracle(mode), "f32", "tiny %s layer %d" % (mode, layer))
    s.close()


def _small(D, G, dtype="bf16", S=700, Bt=3, L=6):
    return synth.Workload("small", L, Bt, S, 2 * G, 2, D, dtype)


@pytest.mark.parametrize("D", [64, 80, 96, 128])
@pytest.mark.parametrize("G", [1, 2, 4])
@pytest.mark.parametrize("mode", MODES)
def test_small_bf16_ragged(D, G, mode):
    w = _small(D, G)
    lens = [700, 1, 333]
    s = DecodeSetup(w, 5, [mode], seed=3, lens=lens)
    got = f64(s.run(mode))
    assert s.ctx.fkv_get_device_status() == B.FKV_OK
    assert_close(got, s.oracle(mode), "bf16", "D=%d G=%d %s" % (D, G, mode))
    s.close()


@pytest.mark.parametrize("D", [80, 128])
@pytest.mark.parametrize("mode", ["lite", "fused"])
def test_small_fp32(D, mode):
    w = _small(D, 2, dtype="f32", S=513, Bt=2)
    s = DecodeSetup(w, 6, [mode], seed=4, lens=[513, 77])
    assert_close(f64(s.run(mode)), s.oracle(mode), "f32", "fp32 D=%d %s" % (D, mode))
    s.close()


@pytest.mark.parametrize("ctas", [1, 2, 5, 37])
def test_split_count_invariance(ctas):
    """Any split grid gives the oracle's answer (fused, ragged)."""
    w = _small(64, 2, S=2048, Bt=5)
    lens = [2048, 1500, 9, 1024, 1]
    s = DecodeSetup(w, 4, ["fused"], seed=5, lens=lens, decode_ctas=ctas)
    assert_close(f64(s.run("fused")), s.oracle("fused"), "bf16", "ctas=%d" % ctas)
    s.close()


@pytest.mark.parametrize("ctas", [1, 3, 7])
@pytest.mark.parametrize("mode", ["vanilla", "fused"])
def test_many_short_units_per_cta(ctas, mode):
    """Each CTA's range holds many short (b, kh) units, with empty sequences
    between them: most warps draw no tile of most units and write weight-0
    records, and units span CTA boundaries."""
    w = _small(64, 2, S=300, Bt=16)
    lens = [1, 0, 57, 300, 3, 0, 0, 120, 48, 49, 2, 0, 211, 96, 5, 17]
    s = DecodeSetup(w, 4, [mode], seed=8, lens=lens, decode_ctas=ctas)
    got = f64(s.run(mode))
    # a length of 0 is flagged (and gives a zero row); the others are exact
    assert s.ctx.fkv_get_device_status() == B.FKV_ERR_DEVICE_ARG
    pairs = [(b, hq) for b in range(len(lens)) if lens[b] > 0 for hq in range(w.q_heads)]
    want = s.oracle(mode, pairs)
    assert_close(np.stack([got[b, hq] for b, hq in pairs]), want, "bf16",
                 "ctas=%d %s" % (ctas, mode))
    assert np.all(got[[b for b in range(len(lens)) if lens[b] == 0]] == 0)
    s.close()


@pytest.mark.parametrize("mode", ["vanilla", "fused"])
def test_cuda_graph_replay(mode):
    """A decode call captured in a CUDA graph is right on every replay, with
    new queries each time.  A replay repeats the captured call's epoch, so the
    unit arrival words must not carry a finished count from one replay into
    the next."""
    w = _small(64, 2, S=1500, Bt=3)
    s = DecodeSetup(w, 4, [mode], seed=31, lens=[1500, 700, 33])
    s.run(mode)  # an eager call first
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        s.ctx.fkv_decode_attn(s.q, s.layer, mode, s.lens, s.out, s.ws)
    for i in range(3):
        s.q.copy_(synth.make_query(w, s.layer, 100 + i, "cuda"))
        s.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_close(f64(s.out), s.oracle(mode), "bf16", "replay %d %s" % (i, mode))
    assert s.ctx.fkv_get_device_status() == B.FKV_OK
    del g
    s.close()


def test_cuda_graph_decode_step_matches_eager():
    """A whole decode step captured once in a CUDA graph and replayed gives,
    bit for bit, what eager calls give on the same new rows and queries.
    The step appends into the storage layers, then makes the storage-layer
    calls and the fused upper-layer calls."""
    w = _small(64, 2, S=600, Bt=2, L=4)  # storage layers 1-2, upper layers 3-4
    L, n = w.num_layers, w.n
    ctx = B.Context(L, w.batch, w.seq, w.q_heads, w.kv_heads, w.head_dim, w.dtype)
    caches = [synth.make_cache(w, l, 0, "cuda") for l in range(1, n + 1)]
    for l, (k, v) in enumerate(caches, start=1):
        ctx.fkv_bind_layer_cache(l, k, v)
    for l in range(n + 1, L + 1):
        ctx.fkv_set_fusion_weights(l, *synth.make_weights(w, l, 0, "cuda"))
    lens = torch.tensor([600, 311], dtype=torch.int32, device="cuda")
    pos = lens - 1
    dt = ctx.torch_dtype
    q = torch.empty(L, w.batch, w.q_heads, w.head_dim, dtype=dt, device="cuda")
    kn = torch.empty(n, w.batch, w.kv_heads, 1, w.head_dim, dtype=dt, device="cuda")
    vn = torch.empty_like(kn)
    out = torch.empty_like(q)
    ws = ctx.workspace("cuda")

    def step():
        for l in range(1, n + 1):
            ctx.fkv_append_kv(l, kn[l - 1], vn[l - 1], pos, 1)
        for l in range(1, L + 1):
            ctx.fkv_decode_attn(q[l - 1], l, "fused" if l > n else "vanilla", lens, out[l - 1], ws)

    def fill(seed):
        g = torch.Generator(device="cuda").manual_seed(seed)
        for x in (q, kn, vn):
            x.copy_(torch.randn(x.shape, generator=g, device="cuda").to(dt))

    fill(1)
    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=torch.cuda.Stream()):
        step()
    for seed in (2, 3, 4):
        fill(seed)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        got = out.clone()
        out.fill_(float("nan"))
        step()
        torch.cuda.synchronize()
        assert not torch.isnan(got).any()
        assert torch.equal(got, out), "replay with inputs %d" % seed
    assert ctx.fkv_get_device_status() == B.FKV_OK
    del graph
    ctx.close()


def test_more_warps_than_rows():
    """A grid with more warps than cache rows (empty warp ranges)."""
    w = _small(64, 2, S=16, Bt=2)
    s = DecodeSetup(w, 4, ["fused", "lite"], seed=6, lens=[3, 5], decode_ctas=64)
    for m in ("fused", "lite"):
        assert_close(f64(s.run(m)), s.oracle(m), "bf16", m)
    s.close()


def test_lite_equals_fused_with_zero_one_weights():
    """Lite (K^n, V^1) and fused with (a1, an, b1, bn) = (0, 1, 1, 0) agree."""
    w = _small(96, 2, S=1000, Bt=2)
    s = DecodeSetup(w, 4, ["lite", "fused"], seed=7, lens=[1000, 640])
    z = torch.zeros_like(s.weights[0])
    o = torch.ones_like(s.weights[0])
    s.ctx.fkv_set_fusion_weights(4, z, o, o, z)
    lite = f64(s.run("lite")).copy()
    fused = f64(s.run("fused"))
    assert np.max(np.abs(lite - fused)) <= 1e-2
    assert_close(fused, s.oracle("lite"), "bf16", "fused(0,1,1,0) vs lite oracle")
    s.close()


def test_untied_and_negative_weights():
    """Weights of any sign, untied across RoPE pairs, are used as given."""
    w = _small(64, 2, S=300, Bt=2)
    s = DecodeSetup(w, 6, ["fused"], seed=8, lens=[300, 299], tie_keys=False, weight_std=1.5)
    s.weights[2].neg_()
    assert_close(f64(s.run("fused")), s.oracle("fused"), "bf16", "untied")
    s.close()


def test_out_of_range_lengths_flagged():
    """Length 0 gives a zero row, a length above S_max is clamped; both set
    FKV_ERR_DEVICE_ARG in the device status, the other rows stay correct."""
    w = _small(64, 2, S=256, Bt=3)
    s = DecodeSetup(w, 5, ["fused"], seed=9, lens=[0, 9999, 100])
    got = f64(s.run("fused"))
    assert s.ctx.fkv_get_device_status() == B.FKV_ERR_DEVICE_ARG
    assert s.ctx.fkv_get_device_status() == B.FKV_OK  # cleared
    assert np.all(got[0] == 0)
    s.lens = torch.tensor([1, 256, 100], dtype=torch.int32, device="cuda")
    ref = s.oracle("fused")
    assert_close(got[1:], ref[1:], "bf16", "clamped")
    s.close()


def test_host_validation_launches_nothing():
    w = _small(64, 2, S=64, Bt=1)
    s = DecodeSetup(w, 4, ["fused"], seed=10, lens=[64])
    with pytest.raises(B.FkvError) as e:
        s.ctx.fkv_decode_attn(s.q, 4, "fused", s.lens, s.out, s.ws[:16])
    assert e.value.status == B.FKV_ERR_WORKSPACE
    with pytest.raises(B.FkvError) as e:
        s.ctx.fkv_decode_attn(s.q, 4, "vanilla", s.lens, s.out, s.ws)   # no own cache
    assert e.value.status == B.FKV_ERR_UNSUPPORTED
    with pytest.raises(B.FkvError) as e:
        s.ctx.fkv_decode_attn(s.q, 7, "fused", s.lens, s.out, s.ws)
    assert e.value.status == B.FKV_ERR_INVALID_ARG
    with pytest.raises(B.FkvError) as e:
        s.ctx.fkv_decode_attn(s.q.data_ptr() + 2, 4, "fused", s.lens, s.out, s.ws)
    assert e.value.status == B.FKV_ERR_INVALID_ARG
    s.close()


# ---------------------------------------------------------------------------
# full-size workloads, sampled rows
# ---------------------------------------------------------------------------

def _every_unit(w):
    return [(b, kh) for b in range(w.batch) for kh in range(w.kv_heads)]


@pytest.mark.parametrize("w", [synth.M332, synth.B1_5, synth.B4], ids=lambda w: w.name)
@pytest.mark.parametrize("mode", ALL_MODES)
def test_full_size_every_unit(w, mode):
    """The benchmark's workloads in its launch configuration: every query
    head of every (batch row, KV head) unit against the oracle, so that every
    CTA position, stream-K boundary and merge of the timed launch is checked."""
    layer = w.num_layers  # the top reconstruction layer
    s = DecodeSetup(w, layer, [mode], seed=0)
    got = f64(s.run(mode))
    assert s.ctx.fkv_get_device_status() == B.FKV_OK
    G = w.group
    units = _every_unit(w)
    ref = s.oracle_units(mode, units)
    sel = np.stack([got[b, kh * G:(kh + 1) * G] for b, kh in units])
    assert_close(sel, ref, "bf16", "%s %s" % (w.name, mode))
    s.close()
    torch.cuda.empty_cache()


def test_full_size_storage_layer():
    w = synth.M332
    s = DecodeSetup(w, 1, ["fused"], seed=0)
    got = f64(s.run("fused"))
    G = w.group
    units = _every_unit(w)
    assert_close(np.stack([got[b, kh * G:(kh + 1) * G] for b, kh in units]),
                 s.oracle_units("fused", units), "bf16", "storage layer 1")
    s.close()


def test_workspace_garbage_and_reuse():
    """The workspace needs no clearing: random bytes in it, or counts left by
    earlier calls of other shapes, do not change the result."""
    w = _small(80, 2, S=900, Bt=4)
    s = DecodeSetup(w, 5, ["fused", "lite"], seed=13, lens=[900, 17, 450, 1])
    g = torch.Generator(device="cuda").manual_seed(5)
    s.ws.copy_(torch.randint(0, 256, s.ws.shape, generator=g, device="cuda", dtype=torch.uint8))
    ref_f, ref_l = s.oracle("fused"), s.oracle("lite")
    for _ in range(3):
        assert_close(f64(s.run("fused")), ref_f, "bf16", "fused, dirty workspace")
        assert_close(f64(s.run("lite")), ref_l, "bf16", "lite, dirty workspace")
    assert s.ctx.fkv_get_device_status() == B.FKV_OK
    s.close()



# ---------------------------------------------------------------------------
# source-layer choice and single-source channel scaling (FusedKV slides,
# Table 17 and Fig.8)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("D", [64, 80, 128])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_scaled_mode_default_sources(D, dtype):
    w = _small(D, 2, dtype=dtype, S=600, Bt=3)
    s = DecodeSetup(w, 6, ["scaled"], seed=14, lens=[600, 300, 5])
    assert_close(f64(s.run("scaled")), s.oracle("scaled"), dtype, "scaled D=%d" % D)
    s.close()


@pytest.mark.parametrize("mode,src", [
    ("lite", (2, 0, 3, 0)),       # middle-layer K, V source 3
    ("lite", (1, 0, 3, 0)),       # reversed sharing K^1, V^n (n = 3)
    ("scaled", (2, 0, 1, 0)),
    ("fused", (2, 3, 3, 1)),
    ("fused", (3, 3, 1, 1)),      # both weights on one layer
])
def test_custom_sources(mode, src):
    w = _small(64, 2, S=512, Bt=2)   # 6 layers, storage 1..3
    s = DecodeSetup(w, 5, [mode], seed=15, lens=[512, 100], sources={mode: src})
    assert_close(f64(s.run(mode)), s.oracle(mode), "bf16", "%s %s" % (mode, src))
    s.close()


def test_set_sources_rejects_non_storage_layers():
    w = _small(64, 2, S=64, Bt=1)
    s = DecodeSetup(w, 5, ["lite"], seed=16, lens=[64])
    for args in (("lite", 4, 0, 1, 0), ("fused", 1, 5, 1, 1), ("vanilla", 1, 1, 1, 1),
                 ("lite", 0, 0, 1, 0)):
        with pytest.raises(B.FkvError) as e:
            s.ctx.fkv_set_sources(5, *args)
        assert e.value.status == B.FKV_ERR_INVALID_ARG
    with pytest.raises(B.FkvError):
        s.ctx.fkv_set_sources(2, "lite", 1, 0, 1, 0)   # a storage layer has no sources
    s.close()



# ---------------------------------------------------------------------------
# sliding-window layers (hybrid SWA, FusedKV slides "MoE and hybrid SWA")
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("window", [1, 37, 300, 2000])
@pytest.mark.parametrize("mode", ALL_MODES)
@pytest.mark.parametrize("D", [64, 80])
def test_window_decode(window, mode, D):
    w = _small(D, 2, S=700, Bt=3)
    s = DecodeSetup(w, 5, [mode], seed=17, lens=[700, 1, 333], window=window)
    assert_close(f64(s.run(mode)), s.oracle(mode), "bf16", "W=%d %s D=%d" % (window, mode, D))
    assert s.ctx.fkv_get_device_status() == B.FKV_OK
    s.close()


@pytest.mark.parametrize("mode", MODES)
def test_window_decode_full_size_332M(mode):
    """332M workload with the pages' window of 512 (every unit)."""
    w = synth.M332
    s = DecodeSetup(w, w.num_layers, [mode], seed=0, window=512)
    got = f64(s.run(mode))
    G = w.group
    units = _every_unit(w)
    assert_close(np.stack([got[b, kh * G:(kh + 1) * G] for b, kh in units]),
                 s.oracle_units(mode, units), "bf16", "332M W=512 %s" % mode)
    s.close()
    torch.cuda.empty_cache()


def test_set_window_rejects():
    w = _small(64, 2, S=64, Bt=1)
    s = DecodeSetup(w, 5, ["lite"], seed=18, lens=[64])
    for layer, win in ((0, 4), (7, 4), (5, -1)):
        with pytest.raises(B.FkvError):
            s.ctx.fkv_set_window(layer, win)
    s.close()
