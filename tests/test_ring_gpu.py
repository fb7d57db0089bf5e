"""Ring caches for sliding-window layers (fkv_set_ring_rows), on the GPU
through the C ABI, against the float64 oracle.

A window layer attends only to its last W positions ([Slides] "MoE and hybrid
SWA"), so its caches need only R >= W rows: position t of a sequence at row
t % R.  The oracle works on ordinary full-length caches; the GPU gets the
same positions laid out in rings, so every check is the windowed attention
of the oracle over the full caches."""

import numpy as np
import pytest
import torch

import oracle as O
from cross_layer_kv_gb300 import fusedkv as B
from cross_layer_kv_gb300 import synth
from parity import assert_close, f64

pytestmark = pytest.mark.gpu

ALL_MODES = ("vanilla", "lite", "fused", "scaled")


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    yield
    torch.cuda.synchronize()


def ring_of(full: torch.Tensor, lens, R: int) -> torch.Tensor:
    """[B, H, S, ...] caches by position -> [B, H, R, ...] rings holding each
    sequence's last R positions (position t at row t % R; other rows zero)."""
    shape = list(full.shape)
    shape[2] = R
    ring = torch.zeros(shape, dtype=full.dtype, device=full.device)
    for b, L in enumerate(lens):
        t = torch.arange(max(0, L - R), L, device=full.device)
        ring[b][:, t % R] = full[b][:, t]
    return ring


class RingSetup:
    """A decode call of `layer` whose source caches (and the layer's own) are
    rings of R rows, with the layer's window W."""

    def __init__(self, w, layer, mode, R, W, lens, seed=0, dtype=None):
        self.w, self.layer, self.mode, self.W = w, layer, mode, W
        n = w.n
        need = [layer] if (layer <= n or mode == "vanilla") else sorted({1, n})
        self.ctx = B.Context(w.num_layers, w.batch, w.seq, w.q_heads, w.kv_heads, w.head_dim,
                             w.dtype, store_upper=any(l > n for l in need))
        self.lens = [int(x) for x in lens]
        self.full = {}
        self.keep = []
        for l in need:
            k, v = synth.make_cache(w, l, seed, "cuda")
            self.full[l] = (k, v)
            self.ctx.fkv_set_ring_rows(l, R)
            kr, vr = ring_of(k, self.lens, R), ring_of(v, self.lens, R)
            self.keep.append((kr, vr))
            self.ctx.fkv_bind_layer_cache(l, kr, vr)
        self.weights = None
        if layer > n:
            self.weights = synth.make_weights(w, layer, seed, "cuda")
            self.ctx.fkv_set_fusion_weights(layer, *self.weights)
        self.ctx.fkv_set_window(layer, W)
        self.q = synth.make_query(w, layer, seed, "cuda")
        self.lens_t = torch.tensor(self.lens, dtype=torch.int32, device="cuda")
        self.out = torch.empty_like(self.q)
        self.ws = self.ctx.workspace()

    def run(self):
        self.ctx.fkv_decode_attn(self.q, self.layer, self.mode, self.lens_t, self.out, self.ws)
        return self.out

    def oracle_units(self, units):
        w, G = self.w, self.w.group
        out = []
        for b, kh in units:
            L = self.lens[b]
            kc = {l: f64(k[b:b + 1, kh:kh + 1, :L]) for l, (k, v) in self.full.items()}
            vc = {l: f64(v[b:b + 1, kh:kh + 1, :L]) for l, (k, v) in self.full.items()}
            ws = ({self.layer: tuple(f64(x[kh:kh + 1]) for x in self.weights)}
                  if self.weights else None)
            o = O.decode_attn(f64(self.q[b:b + 1, kh * G:(kh + 1) * G]), self.layer, w.num_layers,
                              self.mode, kc, vc, [L], weights=ws, window=self.W)
            out.append(o[0])
        return np.stack(out)

    def check(self, what):
        got = f64(self.run())
        assert self.ctx.fkv_get_device_status() == B.FKV_OK
        G = self.w.group
        units = [(b, kh) for b in range(self.w.batch) for kh in range(self.w.kv_heads)]
        ref = self.oracle_units(units)
        sel = np.stack([got[b, kh * G:(kh + 1) * G] for b, kh in units])
        assert_close(sel, ref, self.w.dtype, what)

    def close(self):
        self.ctx.close()


def _w(D, G=2, S=1500, Bt=4, L=6, dtype="bf16"):
    return synth.Workload("ring", L, Bt, S, 2 * G, 2, D, dtype)


# lengths: shorter than the ring, a multiple of it, and wrapped at various rows
LENS = [1500, 1200, 299, 1033]


@pytest.mark.parametrize("mode", ALL_MODES)
@pytest.mark.parametrize("D", [64, 80, 128])
def test_ring_decode_matches_windowed_oracle(mode, D):
    s = RingSetup(_w(D), 5, mode, R=300, W=300, lens=LENS, seed=1)
    s.check("ring R=300 W=300 %s D=%d" % (mode, D))
    s.close()


@pytest.mark.parametrize("R,W", [(512, 100), (257, 257), (64, 1)])
@pytest.mark.parametrize("mode", ["fused", "lite"])
def test_ring_larger_than_window(R, W, mode):
    s = RingSetup(_w(96), 6, mode, R=R, W=W, lens=[1500, 511, 513, 64], seed=2)
    s.check("ring R=%d W=%d %s" % (R, W, mode))
    s.close()


@pytest.mark.parametrize("G", [1, 4])
def test_ring_group_sizes_and_storage_layer(G):
    w = _w(64, G=G)
    for layer, mode in ((2, "vanilla"), (5, "fused")):
        s = RingSetup(w, layer, mode, R=200, W=150, lens=LENS, seed=3)
        s.check("ring G=%d layer %d" % (G, layer))
        s.close()


def test_ring_fp32():
    s = RingSetup(_w(64, dtype="f32", S=700), 5, "fused", R=128, W=128, lens=[700, 127, 128, 385],
                  seed=4)
    s.check("ring fp32")
    s.close()


def test_ring_full_size_332M_window_512():
    """The 332M workload with window-512 layers whose caches are 512-row
    rings (1/16 of the full-length bytes): every unit."""
    w = synth.M332
    lens = [w.seq - (37 * b) % 700 for b in range(w.batch)]   # different wrap points
    for mode in ("fused", "lite"):
        s = RingSetup(w, w.num_layers, mode, R=512, W=512, lens=lens, seed=0)
        s.check("332M ring 512 %s" % mode)
        s.close()
        torch.cuda.empty_cache()


def test_ring_append_wraps():
    """fkv_append_kv writes position p + i at row (p + i) % R, across the end."""
    w = _w(64, S=400, Bt=3)
    R, T = 100, 7
    ctx = B.Context(w.num_layers, w.batch, w.seq, w.q_heads, w.kv_heads, w.head_dim, "bf16")
    ctx.fkv_set_ring_rows(1, R)
    k = torch.zeros(w.batch, w.kv_heads, R, w.head_dim, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    ctx.fkv_bind_layer_cache(1, k, v)
    g = torch.Generator(device="cuda").manual_seed(7)
    kn = torch.randn(w.batch, w.kv_heads, T, w.head_dim, generator=g, device="cuda").to(torch.bfloat16)
    vn = torch.randn(w.batch, w.kv_heads, T, w.head_dim, generator=g, device="cuda").to(torch.bfloat16)
    pos = [96, 0, 393]   # wraps at row 100; starts at row 0; positions 393..399 -> rows 93..99
    ctx.fkv_append_kv(1, kn, vn, torch.tensor(pos, dtype=torch.int32, device="cuda"))
    assert ctx.fkv_get_device_status() == B.FKV_OK
    ek, ev = torch.zeros_like(k), torch.zeros_like(v)
    for b, p in enumerate(pos):
        for i in range(T):
            ek[b, :, (p + i) % R] = kn[b, :, i]
            ev[b, :, (p + i) % R] = vn[b, :, i]
    assert torch.equal(k, ek) and torch.equal(v, ev)
    with pytest.raises(B.FkvError) as e:   # more new rows than the ring holds
        big = torch.zeros(w.batch, w.kv_heads, R + 1, w.head_dim, dtype=torch.bfloat16, device="cuda")
        ctx.fkv_append_kv(1, big, big, torch.zeros(w.batch, dtype=torch.int32, device="cuda"))
    assert e.value.status == B.FKV_ERR_INVALID_ARG
    ctx.close()


def test_ring_q4_decode():
    """4-bit ring caches (records quantised by the oracle on the CPU)."""
    w = _w(64, S=900, Bt=3)
    R, W = 256, 200
    lens = [900, 255, 600]
    n, layer = w.n, 5
    ctx = B.Context(w.num_layers, w.batch, w.seq, w.q_heads, w.kv_heads, w.head_dim, "bf16")
    D = w.head_dim
    deq = {}
    keep = []
    for l in (1, n):
        k, v = synth.make_cache(w, l, 9, "cuda")
        ctx.fkv_set_ring_rows(l, R)
        recs = []
        for x in (k, v):
            rec = torch.from_numpy(O.q4_pack(*O.q4_quantize(x.to("cpu", torch.float32).numpy())))
            recs.append(rec)
        deq[l] = tuple(O.q4_dequantize_records(r.numpy(), D) for r in recs)
        kr, vr = (ring_of(r.to("cuda"), lens, R) for r in recs)
        keep.append((kr, vr))
        ctx.fkv_bind_layer_cache_q4(l, kr, vr)
    wts = synth.make_weights(w, layer, 9, "cuda")
    ctx.fkv_set_fusion_weights(layer, *wts)
    ctx.fkv_set_window(layer, W)
    q = synth.make_query(w, layer, 9, "cuda")
    out = torch.empty_like(q)
    ctx.fkv_decode_attn(q, layer, "fused", torch.tensor(lens, dtype=torch.int32, device="cuda"),
                        out, ctx.workspace())
    assert ctx.fkv_get_device_status() == B.FKV_OK
    kc = {l: d[0] for l, d in deq.items()}
    vc = {l: d[1] for l, d in deq.items()}
    ref = O.decode_attn(f64(q), layer, w.num_layers, "fused", kc, vc, lens,
                        weights={layer: tuple(f64(x) for x in wts)}, window=W)
    assert_close(f64(out), ref, "bf16", "q4 ring")
    ctx.close()


def test_ring_prefill_before_wrap_and_rejections():
    """Prefill over ring caches while the prompt's positions have not wrapped;
    rings the kernels cannot tile past that, and inconsistent set-ups, are
    refused."""
    w = _w(96, S=600, Bt=2)
    R, S = 320, 300
    n, layer = w.n, 5
    ctx = B.Context(w.num_layers, w.batch, w.seq, w.q_heads, w.kv_heads, w.head_dim, "bf16")
    full = {}
    for l in (1, n):
        k, v = synth.make_cache(w, l, 11, "cuda")
        full[l] = (k, v)
        ctx.fkv_set_ring_rows(l, R)
        ctx.fkv_bind_layer_cache(l, k[:, :, :R].contiguous(), v[:, :, :R].contiguous())
    wts = synth.make_weights(w, layer, 11, "cuda")
    ctx.fkv_set_fusion_weights(layer, *wts)
    ctx.fkv_set_window(layer, 100)
    g = torch.Generator(device="cuda").manual_seed(12)
    q = torch.randn(w.batch, w.q_heads, S, w.head_dim, generator=g, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(q)
    ctx.fkv_prefill_attn(q, layer, "fused", S, out)
    assert ctx.fkv_get_device_status() == B.FKV_OK
    kc = {l: f64(k[:, :, :S]) for l, (k, v) in full.items()}
    vc = {l: f64(v[:, :, :S]) for l, (k, v) in full.items()}
    ref = O.prefill_attn(f64(q), layer, w.num_layers, "fused", kc, vc,
                         weights={layer: tuple(f64(x) for x in wts)}, window=100)
    assert_close(f64(out), ref, "bf16", "prefill over a ring before it wraps")
    # past the ring's rows, a ring that is not a whole number of key tiles
    # (320 rows against the fused kernel's 112-key tiles) is refused
    qc = q[:, :, :40].contiguous()
    with pytest.raises(B.FkvError) as e:
        ctx.fkv_prefill_attn_chunk(qc, layer, "fused", R - 20, 40, torch.empty_like(qc))
    assert e.value.status == B.FKV_ERR_UNSUPPORTED
    lens = torch.full((w.batch,), 500, dtype=torch.int32, device="cuda")
    qd = torch.zeros(w.batch, w.q_heads, w.head_dim, dtype=torch.bfloat16, device="cuda")
    ws = ctx.workspace()
    # a window wider than the ring, and no window at all, are refused
    for win in (R + 1, 0):
        ctx.fkv_set_window(layer, win)
        with pytest.raises(B.FkvError) as e:
            ctx.fkv_decode_attn(qd, layer, "fused", lens, qd.clone(), ws)
        assert e.value.status == B.FKV_ERR_INVALID_ARG
    # sources with different ring sizes are refused
    ctx.fkv_set_window(layer, 100)
    ctx.fkv_set_ring_rows(n, 0)
    k, v = full[n]
    ctx.fkv_bind_layer_cache(n, k, v)
    with pytest.raises(B.FkvError) as e:
        ctx.fkv_decode_attn(qd, layer, "fused", lens, qd.clone(), ws)
    assert e.value.status == B.FKV_ERR_UNSUPPORTED
    for bad in (-1, w.seq + 1):
        with pytest.raises(B.FkvError) as e:
            ctx.fkv_set_ring_rows(1, bad)
        assert e.value.status == B.FKV_ERR_INVALID_ARG
    ctx.close()


# (mode, D, G): the one-source kernel (128-key tiles), the fused kernel for
# D <= 96 (112-key tiles; G = 1 puts two row tiles of one head in a CTA) and
# the fused D = 128 kernel (64-key tiles)
_WRAP_CASES = [("lite", 64, 2), ("vanilla", 80, 1), ("fused", 96, 2), ("fused", 64, 1),
               ("fused", 128, 1), ("scaled", 128, 2)]


@pytest.mark.parametrize("mode,D,G", _WRAP_CASES)
def test_ring_chunked_prefill_wraps(mode, D, G):
    """A prompt streamed in chunks through rings of 896 rows (a whole number
    of every kernel's key tiles): each chunk's K/V appended, then the chunk's
    causal windowed attention, against the oracle over full-length caches.
    The chunks cross the ring's end, start on and off the tile grid, and the
    longest one meets C + W - 1 = R exactly."""
    R, W = 896, 300
    chunks = [(0, 500), (500, 597), (1097, 333), (1430, 470), (1900, 401)]
    S_all = chunks[-1][0] + chunks[-1][1]
    w = _w(D, G=G, S=S_all, Bt=2)
    n, layer = w.n, 5
    need = [layer] if mode == "vanilla" else sorted({1, n})
    ctx = B.Context(w.num_layers, w.batch, w.seq, w.q_heads, w.kv_heads, w.head_dim, "bf16",
                    store_upper=(mode == "vanilla"))
    full, rings = {}, {}
    for l in need:
        k, v = synth.make_cache(w, l, 60 + D, "cuda")
        full[l] = (k, v)
        ctx.fkv_set_ring_rows(l, R)
        kr = torch.zeros(w.batch, w.kv_heads, R, D, dtype=torch.bfloat16, device="cuda")
        rings[l] = (kr, torch.zeros_like(kr))
        ctx.fkv_bind_layer_cache(l, *rings[l])
    wts = synth.make_weights(w, layer, 60 + D, "cuda")
    ctx.fkv_set_fusion_weights(layer, *wts)
    ctx.fkv_set_window(layer, W)
    g = torch.Generator(device="cuda").manual_seed(61 + D)
    q = torch.randn(w.batch, w.q_heads, S_all, D, generator=g, device="cuda").to(torch.bfloat16)
    ws = {layer: tuple(f64(x) for x in wts)}
    for q0, C in chunks:
        pos = torch.full((w.batch,), q0, dtype=torch.int32, device="cuda")
        for l in need:
            k, v = full[l]
            ctx.fkv_append_kv(l, k[:, :, q0:q0 + C].contiguous(), v[:, :, q0:q0 + C].contiguous(),
                              pos)
        qc = q[:, :, q0:q0 + C].contiguous()
        oc = torch.empty_like(qc)
        ctx.fkv_prefill_attn_chunk(qc, layer, mode, q0, C, oc)
        assert ctx.fkv_get_device_status() == B.FKV_OK
        kc = {l: f64(k[:, :, :q0 + C]) for l, (k, v) in full.items()}
        vc = {l: f64(v[:, :, :q0 + C]) for l, (k, v) in full.items()}
        ref = O.chunk_prefill_attn(f64(qc), q0, layer, w.num_layers, mode, kc, vc,
                                   weights=ws, window=W)
        assert_close(f64(oc), ref, "bf16", "%s D=%d G=%d chunk %d+%d" % (mode, D, G, q0, C))
    # once wrapped: a chunk too long for its window, and no window, are refused
    qc = q[:, :, :W].contiguous()
    ctx.fkv_set_window(layer, R - W + 2)
    with pytest.raises(B.FkvError) as e:
        ctx.fkv_prefill_attn_chunk(qc, layer, mode, S_all - W, W, torch.empty_like(qc))
    assert e.value.status == B.FKV_ERR_UNSUPPORTED
    ctx.fkv_set_window(layer, 0)
    with pytest.raises(B.FkvError) as e:
        ctx.fkv_prefill_attn_chunk(qc, layer, mode, S_all - W, W, torch.empty_like(qc))
    assert e.value.status == B.FKV_ERR_INVALID_ARG
    ctx.close()
