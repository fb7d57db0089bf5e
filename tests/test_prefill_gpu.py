"""GPU parity of fkv_prefill_attn (causal, tcgen05 tensor cores) against the
float64 oracle, through the C ABI.  bf16 bars: max-abs 2e-2, rel-L2 5e-3."""

import numpy as np
import pytest
import torch

import oracle as O
from cross_layer_kv_gb300 import fusedkv as B
from cross_layer_kv_gb300 import synth
from parity import assert_close, f64

pytestmark = pytest.mark.gpu

MODES = ("vanilla", "lite", "fused")


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    yield
    torch.cuda.synchronize()


class PrefillSetup:
    def __init__(self, w, layer, mode, S, seed=0, tie_keys=True, sources=None, window=0):
        self.w, self.layer, self.mode, self.S = w, layer, mode, S
        self.sources = sources
        self.window = window
        n = w.n
        need = [layer] if (layer <= n or mode == "vanilla") else sorted({1, n})
        if sources:
            need = sorted(set(need) | set(range(1, n + 1)))
        self.ctx = B.Context(w.num_layers, w.batch, w.seq, w.q_heads, w.kv_heads, w.head_dim,
                             "bf16", store_upper=any(l > n for l in need))
        self.caches = {}
        for l in need:
            k, v = synth.make_cache(w, l, seed, "cuda")
            self.caches[l] = (k, v)
            self.ctx.fkv_bind_layer_cache(l, k, v)
        self.weights = None
        if layer > n:
            self.weights = synth.make_weights(w, layer, seed, "cuda", tie_keys=tie_keys)
            self.ctx.fkv_set_fusion_weights(layer, *self.weights)
        if sources:
            self.ctx.fkv_set_sources(layer, mode, *sources)
        if window:
            self.ctx.fkv_set_window(layer, window)
        g = torch.Generator(device="cuda").manual_seed(seed + 99)
        self.q = torch.randn(w.batch, w.q_heads, S, w.head_dim, generator=g,
                             device="cuda").to(torch.bfloat16)
        self.out = torch.full_like(self.q, float("nan"))

    def run(self):
        self.ctx.fkv_prefill_attn(self.q, self.layer, self.mode, self.S, self.out)
        return self.out

    def source_kwargs(self):
        src = self.sources
        if not src:
            return {}
        if self.mode == "fused":
            return {"k_sources": (src[0], src[1]), "v_sources": (src[2], src[3])}
        return {"k_sources": (src[0],), "v_sources": (src[2],)}

    def oracle(self, bh=None, rows=None):
        w = self.w
        G = w.group
        sk = self.source_kwargs()
        sk["window"] = self.window
        ws = ({self.layer: tuple(f64(x) for x in self.weights)} if self.weights else None)
        if bh is None:
            kc = {l: f64(k) for l, (k, v) in self.caches.items()}
            vc = {l: f64(v) for l, (k, v) in self.caches.items()}
            return O.prefill_attn(f64(self.q), self.layer, w.num_layers, self.mode, kc, vc,
                                  weights=ws, rows=rows, **sk)
        b, h = bh
        kh = h // G
        kc = {l: f64(k[b:b + 1, kh:kh + 1, :self.S]) for l, (k, v) in self.caches.items()}
        vc = {l: f64(v[b:b + 1, kh:kh + 1, :self.S]) for l, (k, v) in self.caches.items()}
        if ws:
            ws = {self.layer: tuple(x[kh:kh + 1] for x in ws[self.layer])}
        return O.prefill_attn(f64(self.q[b:b + 1, h:h + 1]), self.layer, w.num_layers, self.mode,
                              kc, vc, weights=ws, rows=rows, **sk)[0, 0]

    def close(self):
        self.ctx.close()


def _w(D, G, S_max, Bt=2, L=4):
    return synth.Workload("p", L, Bt, S_max, 2 * G, 2, D, "bf16")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("D", [64, 80, 96, 128])
def test_prefill_small(mode, D):
    w = _w(D, 2, 320)
    s = PrefillSetup(w, 4, mode, 300, seed=1)
    got = f64(s.run())
    assert s.ctx.fkv_get_device_status() == B.FKV_OK
    assert_close(got, s.oracle(), "bf16", "prefill D=%d %s" % (D, mode))
    s.close()


@pytest.mark.parametrize("S", [1, 2, 63, 64, 65, 128, 129, 256])
def test_prefill_lengths_fused(S):
    w = _w(96, 2, 256)
    s = PrefillSetup(w, 3, "fused", S, seed=2)
    assert_close(f64(s.run()), s.oracle(), "bf16", "S=%d" % S)
    s.close()


@pytest.mark.parametrize("G", [1, 2])
@pytest.mark.parametrize("S", [1, 2, 127, 128, 129, 255, 256, 257, 384, 513])
def test_prefill_lengths_single_source(S, G):
    """One-source layers run 128-key tiles with two 128-row groups per CTA
    (two heads, or two row tiles of one head when G = 1): every length from
    one row to several tiles with a ragged tail, both pairings."""
    w = _w(64, G, 520)
    s = PrefillSetup(w, 2, "vanilla", S, seed=20 + G)
    assert_close(f64(s.run()), s.oracle(), "bf16", "S=%d G=%d" % (S, G))
    assert s.ctx.fkv_get_device_status() == B.FKV_OK
    s.close()


@pytest.mark.parametrize("mode", ["vanilla", "lite"])
def test_prefill_group_one_window_chunks(mode):
    """G = 1 with a sliding window and chunks starting off the tile grid: the
    second row tile of a CTA starts 128 positions later than the first, so
    its leading key tiles can lie wholly before its window."""
    w = _w(128, 1, 700)
    s = PrefillSetup(w, 4, mode, 700, seed=23, window=100)
    assert_close(f64(s.run()), s.oracle(), "bf16", "G=1 W=100 %s" % mode)
    for a, c in ((0, 257), (257, 300), (557, 143)):
        qc = s.q[:, :, a:a + c].contiguous()
        oc = torch.empty_like(qc)
        s.ctx.fkv_prefill_attn_chunk(qc, 4, mode, a, c, oc)
        assert_close(f64(oc), _chunk_oracle(s, qc, a), "bf16", "G=1 chunk %d+%d" % (a, c))
    s.close()


@pytest.mark.parametrize("mode", ["lite", "fused"])
def test_prefill_group_one(mode):
    w = _w(64, 1, 200)
    s = PrefillSetup(w, 3, mode, 200, seed=3)
    assert_close(f64(s.run()), s.oracle(), "bf16", "G=1 %s" % mode)
    s.close()


@pytest.mark.parametrize("G", [1, 2])
def test_prefill_fused_head_dim_128(G):
    """Fused layers with D = 128 run the 64-key kernel (the 112-key fused
    kernel keeps Q in tensor memory, which does not fit at D = 128): both
    pairings, several tiles and a ragged tail."""
    w = _w(128, G, 330)
    s = PrefillSetup(w, 4, "fused", 321, seed=30 + G)
    assert_close(f64(s.run()), s.oracle(), "bf16", "fused D=128 G=%d" % G)
    assert s.ctx.fkv_get_device_status() == B.FKV_OK
    s.close()


@pytest.mark.parametrize("D", [64, 80, 96])
def test_prefill_fused_group_one_window_chunks(D):
    """The 112-key fused kernel with one head per KV head (two row tiles per
    CTA), a sliding window and chunks that start off the tile grid."""
    w = _w(D, 1, 600)
    s = PrefillSetup(w, 4, "fused", 600, seed=40 + D, window=150)
    assert_close(f64(s.run()), s.oracle(), "bf16", "fused G=1 W=150 D=%d" % D)
    for a, c in ((0, 113), (113, 300), (413, 187)):
        qc = s.q[:, :, a:a + c].contiguous()
        oc = torch.empty_like(qc)
        s.ctx.fkv_prefill_attn_chunk(qc, 4, "fused", a, c, oc)
        assert_close(f64(oc), _chunk_oracle(s, qc, a), "bf16", "fused G=1 chunk %d+%d" % (a, c))
    s.close()


def test_prefill_storage_layer_and_untied():
    w = _w(128, 2, 190)
    s = PrefillSetup(w, 1, "fused", 190, seed=4)
    assert_close(f64(s.run()), s.oracle(), "bf16", "storage layer")
    s.close()
    s = PrefillSetup(w, 3, "fused", 190, seed=5, tie_keys=False)
    assert_close(f64(s.run()), s.oracle(), "bf16", "untied")
    s.close()


def test_prefill_rejects():
    w = _w(64, 2, 64)
    s = PrefillSetup(w, 3, "fused", 64)
    with pytest.raises(B.FkvError) as e:   # S > S_max, checked by the library
        s.ctx.fkv_prefill_attn(s.q.data_ptr(), 3, "fused", 65, s.out.data_ptr())
    assert e.value.status == B.FKV_ERR_INVALID_ARG
    with pytest.raises(B.FkvError) as e:
        s.ctx.fkv_prefill_attn(s.q, 3, "vanilla", 64, s.out)
    assert e.value.status == B.FKV_ERR_UNSUPPORTED
    s.close()
    ctx = B.Context(4, 1, 64, 2, 1, 64, "f32")
    q = torch.zeros(1, 2, 8, 64, device="cuda")
    with pytest.raises(B.FkvError) as e:
        ctx.fkv_prefill_attn(q, 1, "vanilla", 8, q.clone())
    assert e.value.status in (B.FKV_ERR_UNSUPPORTED, B.FKV_ERR_INVALID_ARG)
    ctx.close()


# Full-size checks: eight (batch row, query head) pairs that cover every batch
# row, both heads of a KV head and both ends of the head range; in each, the
# first and last row of every 128-row query tile.
_FULL_PAIRS = [(0, 0), (0, 1), (1, 6), (1, 7), (2, 9), (2, 14), (3, 3), (3, 15)]
_TILE_EDGES = sorted({r for t in range(8192 // 128) for r in (128 * t, 128 * t + 127)})


@pytest.mark.parametrize("mode", MODES)
def test_prefill_full_size_sampled(mode):
    """650M-shaped workload (B=4, S=8192, 16/8 heads, D=96): the first and
    last row of every query tile of eight (b, h) pairs."""
    w = synth.M650_PREFILL
    s = PrefillSetup(w, w.num_layers, mode, w.seq, seed=0)
    got = f64(s.run())
    assert s.ctx.fkv_get_device_status() == B.FKV_OK
    for b, h in _FULL_PAIRS:
        ref = s.oracle((b, h), rows=_TILE_EDGES)
        assert_close(got[b, h, _TILE_EDGES], ref, "bf16", "650M %s b=%d h=%d" % (mode, b, h))
    s.close()
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# chunked prefill over an existing cache
# ---------------------------------------------------------------------------

def _chunk_oracle(s, q, q_start, bh=None, rows=None):
    w = s.w
    ws = ({s.layer: tuple(f64(x) for x in s.weights)} if s.weights else None)
    n = q_start + q.shape[2]
    if bh is None:
        kc = {l: f64(k[:, :, :n]) for l, (k, v) in s.caches.items()}
        vc = {l: f64(v[:, :, :n]) for l, (k, v) in s.caches.items()}
        return O.chunk_prefill_attn(f64(q), q_start, s.layer, w.num_layers, s.mode, kc, vc,
                                    weights=ws, window=s.window)
    b, h = bh
    kh = h // w.group
    kc = {l: f64(k[b:b + 1, kh:kh + 1, :n]) for l, (k, v) in s.caches.items()}
    vc = {l: f64(v[b:b + 1, kh:kh + 1, :n]) for l, (k, v) in s.caches.items()}
    if ws:
        ws = {s.layer: tuple(x[kh:kh + 1] for x in ws[s.layer])}
    qq = q[b:b + 1, h:h + 1]
    if rows is not None:
        # rows of the chunk, each a one-row chunk at its own position
        return np.stack([O.chunk_prefill_attn(f64(qq[:, :, r:r + 1]), q_start + r, s.layer,
                                              w.num_layers, s.mode, kc, vc, weights=ws,
                                              window=s.window)[0, 0, 0]
                         for r in rows])
    return O.chunk_prefill_attn(f64(qq), q_start, s.layer, w.num_layers, s.mode, kc, vc,
                                weights=ws, window=s.window)[0, 0]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("D", [64, 96])
def test_prefill_chunks_reassemble_full(mode, D):
    w = _w(D, 2, 320)
    S = 300
    s = PrefillSetup(w, 4, mode, S, seed=6)
    full = f64(s.run()).copy()
    parts = []
    for a, c in ((0, 100), (100, 1), (101, 77), (178, 122)):
        qc = s.q[:, :, a:a + c].contiguous()
        oc = torch.empty_like(qc)
        s.ctx.fkv_prefill_attn_chunk(qc, 4, mode, a, c, oc)
        parts.append(f64(oc))
        assert_close(parts[-1], _chunk_oracle(s, qc, a), "bf16", "chunk %d+%d %s" % (a, c, mode))
    got = np.concatenate(parts, axis=2)
    assert_close(got, s.oracle(), "bf16", "reassembled %s" % mode)
    assert np.max(np.abs(got - full)) <= 2e-2
    s.close()


def test_last_prompt_position_is_a_decode_call():
    """The first generated token needs only the last prompt position in the
    upper layers: one decode call of length S gives prefill's last row."""
    w = _w(96, 2, 256)
    S = 201
    s = PrefillSetup(w, 4, "fused", S, seed=8)
    full = f64(s.run())
    q_last = s.q[:, :, S - 1].contiguous()
    out = torch.empty_like(q_last)
    lens = torch.full((w.batch,), S, dtype=torch.int32, device="cuda")
    ws = s.ctx.workspace()
    s.ctx.fkv_decode_attn(q_last, 4, "fused", lens, out, ws)
    assert_close(f64(out), full[:, :, S - 1], "bf16", "decode vs prefill last row")
    s.close()


def test_prefill_chunk_rejects():
    w = _w(64, 2, 128)
    s = PrefillSetup(w, 3, "fused", 64)
    for q_start, c in ((-1, 8), (120, 9), (0, 0)):
        with pytest.raises(B.FkvError) as e:
            s.ctx.fkv_prefill_attn_chunk(s.q.data_ptr(), 3, "fused", q_start, c, s.out.data_ptr())
        assert e.value.status == B.FKV_ERR_INVALID_ARG
    s.close()


@pytest.mark.parametrize("mode", ["fused", "lite"])
def test_prefill_chunk_full_size_sampled(mode):
    """650M workload: the second half of an 8192-token prompt as one chunk
    (q_start = 4096, C = 4096) over the cached first half."""
    w = synth.M650_PREFILL
    s = PrefillSetup(w, w.num_layers, mode, 4096, seed=0)
    q_start = 4096
    s.ctx.fkv_prefill_attn_chunk(s.q, w.num_layers, mode, q_start, 4096, s.out)
    got = f64(s.out)
    rows = [r for r in _TILE_EDGES if r < 4096]
    for b, h in _FULL_PAIRS:
        ref = _chunk_oracle(s, s.q, q_start, bh=(b, h), rows=rows)
        assert_close(got[b, h, rows], ref, "bf16", "650M chunk %s b=%d h=%d" % (mode, b, h))
    s.close()
    torch.cuda.empty_cache()



@pytest.mark.parametrize("mode,src,D", [
    ("scaled", None, 64), ("scaled", None, 96), ("scaled", (2, 0, 1, 0), 80),
    ("lite", (1, 0, 3, 0), 64), ("fused", (2, 3, 3, 1), 96),
])
def test_prefill_sources_and_scaled(mode, src, D):
    w = synth.Workload("p6", 6, 2, 260, 4, 2, D, "bf16")   # storage layers 1..3
    s = PrefillSetup(w, 5, mode, 250, seed=9, sources=src)
    assert_close(f64(s.run()), s.oracle(), "bf16", "prefill %s %s D=%d" % (mode, src, D))
    s.close()



@pytest.mark.parametrize("window", [1, 16, 64, 100, 300])
@pytest.mark.parametrize("mode", ["vanilla", "fused", "scaled"])
def test_prefill_window(window, mode):
    w = _w(96, 2, 320)
    s = PrefillSetup(w, 4, mode, 300, seed=10, window=window)
    assert_close(f64(s.run()), s.oracle(), "bf16", "prefill W=%d %s" % (window, mode))
    s.close()


def test_prefill_window_chunk():
    w = _w(64, 2, 400)
    s = PrefillSetup(w, 4, "fused", 400, seed=11, window=77)
    for a, c in ((0, 130), (130, 200), (330, 70)):
        qc = s.q[:, :, a:a + c].contiguous()
        oc = torch.empty_like(qc)
        s.ctx.fkv_prefill_attn_chunk(qc, 4, "fused", a, c, oc)
        assert_close(f64(oc), _chunk_oracle(s, qc, a), "bf16", "window chunk %d+%d" % (a, c))
    s.close()
