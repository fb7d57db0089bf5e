"""4-bit KV caches (FusedKV slides, "Four-bit KV quantization is the stronger
combination", Table 14) on the GPU, through the C ABI.

* fkv_append_kv on a 4-bit layer quantises exactly as the oracle does (bit
  for bit: codes, bf16 scale and minimum, padding);
* fkv_decode_attn over 4-bit sources -- caches quantised by the oracle on the
  CPU -- matches the oracle's attention over the dequantised caches."""

import numpy as np
import pytest
import torch

import oracle as O
from cross_layer_kv_gb300 import fusedkv as B
from cross_layer_kv_gb300 import synth
from parity import assert_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    yield
    torch.cuda.synchronize()


def _records(x_bf16: torch.Tensor) -> torch.Tensor:
    """Oracle quantisation of a bf16 tensor [..., D] -> uint8 records on the GPU."""
    x = x_bf16.detach().to("cpu", torch.float32).numpy()
    return torch.from_numpy(O.q4_pack(*O.q4_quantize(x))).to(x_bf16.device)


@pytest.mark.parametrize("D", [64, 80, 96, 128])
def test_append_q4_bit_exact(D):
    Bt, H, S, T = 3, 2, 24, 5
    ctx = B.Context(4, Bt, S, 4, H, D, "bf16")
    g = torch.Generator(device="cuda").manual_seed(D)
    kn = (torch.randn(Bt, H, T, D, generator=g, device="cuda") * 3).to(torch.bfloat16)
    vn = torch.randn(Bt, H, T, D, generator=g, device="cuda").to(torch.bfloat16)
    kn[0, 0, 0, :16] = 1.25            # a constant group
    kn[0, 0, 1, :16] = torch.arange(16, device="cuda").to(torch.bfloat16)  # on the grid
    kr, vr = ctx.q4_cache(), ctx.q4_cache()
    kr.fill_(0xAB)
    vr.fill_(0xCD)
    ctx.fkv_bind_layer_cache_q4(2, kr, vr)
    pos = torch.tensor([0, 11, S - T], dtype=torch.int32, device="cuda")
    ctx.fkv_append_kv(2, kn, vn, pos)
    assert ctx.fkv_get_device_status() == B.FKV_OK
    rk = kr.cpu().numpy()
    rv = vr.cpu().numpy()
    ek, ev = _records(kn).cpu().numpy(), _records(vn).cpu().numpy()
    for b in range(Bt):
        p = int(pos[b])
        np.testing.assert_array_equal(rk[b, :, p:p + T], ek[b])
        np.testing.assert_array_equal(rv[b, :, p:p + T], ev[b])
        # rows outside the append untouched
        other = np.ones(S, bool)
        other[p:p + T] = False
        assert np.all(rk[b][:, other] == 0xAB) and np.all(rv[b][:, other] == 0xCD)
    ctx.close()


class Q4Setup:
    """A decode call whose source layers are 4-bit (quantised by the oracle)."""

    def __init__(self, w, layer, mode, seed=0, lens=None, window=0, sources=None):
        self.w, self.layer, self.mode = w, layer, mode
        n = w.n
        need = [layer] if (layer <= n or mode == "vanilla") else sorted({1, n})
        if sources:
            need = sorted(set(need) | set(range(1, n + 1)))
        self.ctx = B.Context(w.num_layers, w.batch, w.seq, w.q_heads, w.kv_heads, w.head_dim,
                             "bf16", store_upper=any(l > n for l in need))
        self.deq = {}
        self.keep = []
        for l in need:
            k, v = synth.make_cache(w, l, seed, "cuda")
            kr, vr = _records(k), _records(v)
            self.keep.append((kr, vr))
            self.ctx.fkv_bind_layer_cache_q4(l, kr, vr)
            D = w.head_dim
            self.deq[l] = (O.q4_dequantize_records(kr.cpu().numpy(), D),
                           O.q4_dequantize_records(vr.cpu().numpy(), D))
            del k, v
        self.weights = None
        if layer > n:
            self.weights = synth.make_weights(w, layer, seed, "cuda")
            self.ctx.fkv_set_fusion_weights(layer, *self.weights)
        self.sources = sources
        if sources:
            self.ctx.fkv_set_sources(layer, mode, *sources)
        self.window = window
        if window:
            self.ctx.fkv_set_window(layer, window)
        self.q = synth.make_query(w, layer, seed, "cuda")
        self.lens = (synth.make_seq_lens(w, seed, "cuda") if lens is None else
                     torch.tensor(lens, dtype=torch.int32, device="cuda"))
        self.out = torch.empty_like(self.q)
        self.ws = self.ctx.workspace()

    def run(self):
        self.ctx.fkv_decode_attn(self.q, self.layer, self.mode, self.lens, self.out, self.ws)
        return self.out

    def oracle(self, pairs=None):
        kw = {"window": self.window}
        if self.sources:
            s = self.sources
            kw.update({"k_sources": (s[0], s[1]), "v_sources": (s[2], s[3])} if self.mode == "fused"
                      else {"k_sources": (s[0],), "v_sources": (s[2],)})
        ws = ({self.layer: tuple(f64(x) for x in self.weights)} if self.weights else None)
        kc = {l: k for l, (k, v) in self.deq.items()}
        vc = {l: v for l, (k, v) in self.deq.items()}
        lens = self.lens.cpu().tolist()
        if pairs is None:
            return O.decode_attn(f64(self.q), self.layer, self.w.num_layers, self.mode, kc, vc,
                                 lens, weights=ws, **kw)
        G = self.w.group
        out = []
        for b, h in pairs:
            kh = h // G
            n = lens[b]
            kcs = {l: x[b:b + 1, kh:kh + 1, :n] for l, x in kc.items()}
            vcs = {l: x[b:b + 1, kh:kh + 1, :n] for l, x in vc.items()}
            wss = ({self.layer: tuple(x[kh:kh + 1] for x in ws[self.layer])} if ws else None)
            out.append(O.decode_attn(f64(self.q[b:b + 1, h:h + 1]), self.layer, self.w.num_layers,
                                     self.mode, kcs, vcs, [n], weights=wss, **kw)[0, 0])
        return np.stack(out)

    def close(self):
        self.ctx.close()


def _small(D, G=2, S=600, Bt=3, L=6):
    return synth.Workload("q4", L, Bt, S, 2 * G, 2, D, "bf16")


@pytest.mark.parametrize("D", [64, 80, 96, 128])
@pytest.mark.parametrize("mode", ["vanilla", "lite", "fused", "scaled"])
def test_q4_decode(D, mode):
    s = Q4Setup(_small(D), 5, mode, seed=31, lens=[600, 1, 257])
    assert_close(f64(s.run()), s.oracle(), "bf16", "q4 D=%d %s" % (D, mode))
    assert s.ctx.fkv_get_device_status() == B.FKV_OK
    s.close()


@pytest.mark.parametrize("mode", ["lite", "fused"])
def test_q4_decode_group_one_window_sources(mode):
    w = _small(64, G=1, S=500, Bt=2)
    src = (2, 3, 3, 1) if mode == "fused" else (2, 0, 3, 0)
    s = Q4Setup(w, 5, mode, seed=32, lens=[500, 333], window=100, sources=src)
    assert_close(f64(s.run()), s.oracle(), "bf16", "q4 G=1 window %s" % mode)
    s.close()


@pytest.mark.parametrize("mode", ["lite", "fused"])
def test_q4_decode_full_size_332M(mode):
    w = synth.M332
    s = Q4Setup(w, w.num_layers, mode, seed=0)
    got = f64(s.run())
    rng = np.random.default_rng(33)
    pairs = sorted(set(zip(rng.integers(0, 32, 5).tolist(), rng.integers(0, 16, 5).tolist())))
    assert_close(np.stack([got[b, h] for b, h in pairs]), s.oracle(pairs), "bf16",
                 "q4 332M %s" % mode)
    s.close()
    torch.cuda.empty_cache()


def test_q4_rejects_mixed_formats_and_prefill():
    w = _small(64, S=64, Bt=1)
    ctx = B.Context(w.num_layers, 1, 64, 4, 2, 64, "bf16")
    k = torch.zeros(1, 2, 64, 64, dtype=torch.bfloat16, device="cuda")
    kr = ctx.q4_cache()
    ctx.fkv_bind_layer_cache(1, k, k)          # bf16 layer 1
    ctx.fkv_bind_layer_cache_q4(3, kr, kr)     # 4-bit layer 3 (n = 3)
    wts = [torch.ones(2, 64, device="cuda") for _ in range(4)]
    ctx.fkv_set_fusion_weights(5, *wts)
    q = torch.zeros(1, 4, 64, dtype=torch.bfloat16, device="cuda")
    lens = torch.full((1,), 64, dtype=torch.int32, device="cuda")
    with pytest.raises(B.FkvError) as e:
        ctx.fkv_decode_attn(q, 5, "fused", lens, q.clone(), ctx.workspace())
    assert e.value.status == B.FKV_ERR_UNSUPPORTED
    qp = torch.zeros(1, 4, 8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.FkvError) as e:
        ctx.fkv_prefill_attn(qp, 3, "vanilla", 8, qp.clone())
    assert e.value.status == B.FKV_ERR_UNSUPPORTED
    ctx.close()
    cf = B.Context(4, 1, 8, 2, 1, 64, "f32")
    with pytest.raises(B.FkvError) as e:
        cf.fkv_bind_layer_cache_q4(1, torch.zeros(1, 1, 8, 48, dtype=torch.uint8, device="cuda"),
                                   torch.zeros(1, 1, 8, 48, dtype=torch.uint8, device="cuda"))
    assert e.value.status == B.FKV_ERR_UNSUPPORTED
    cf.close()


@pytest.mark.parametrize("mode", ["fused", "scaled"])
def test_q4_decode_full_size_4B(mode):
    """4B-shaped workload (B=4, S=131072, 32/16 heads, D=80) with 4-bit
    source caches quantised by the oracle on the CPU one batch row at a time;
    every (batch row, KV head) unit against the oracle over the dequantised
    records."""
    w = synth.B4
    D, G, n = w.head_dim, w.group, w.n
    layer = w.num_layers
    ctx = B.Context(w.num_layers, w.batch, w.seq, w.q_heads, w.kv_heads, D, "bf16")
    host = {}   # layer -> (k records, v records) as host uint8 arrays
    keep = []
    for l in sorted({1, n}):
        k, v = synth.make_cache(w, l, 0, "cuda")
        recs = []
        for x in (k, v):
            rec_h = np.empty((w.batch, w.kv_heads, w.seq, O.q4_row_bytes(D)), dtype=np.uint8)
            for b in range(w.batch):
                xb = x[b].to("cpu", torch.float32).numpy()
                rec_h[b] = O.q4_pack(*O.q4_quantize(xb))
            recs.append(rec_h)
        del k, v
        torch.cuda.empty_cache()
        kr, vr = (torch.from_numpy(r).to("cuda") for r in recs)
        ctx.fkv_bind_layer_cache_q4(l, kr, vr)
        keep.append((kr, vr))
        host[l] = tuple(recs)
    wts = synth.make_weights(w, layer, 0, "cuda")
    ctx.fkv_set_fusion_weights(layer, *wts)
    q = synth.make_query(w, layer, 0, "cuda")
    lens = synth.make_seq_lens(w, 0, "cuda")
    out = torch.empty_like(q)
    ctx.fkv_decode_attn(q, layer, mode, lens, out, ctx.workspace())
    assert ctx.fkv_get_device_status() == B.FKV_OK
    got = f64(out)
    L = lens.cpu().tolist()
    qh = f64(q)
    wn = tuple(f64(x) for x in wts)
    ref, sel = [], []
    for b in range(w.batch):
        for kh in range(w.kv_heads):
            nb = L[b]
            kc = {l: O.q4_dequantize_records(r[0][b:b + 1, kh:kh + 1, :nb], D) for l, r in host.items()}
            vc = {l: O.q4_dequantize_records(r[1][b:b + 1, kh:kh + 1, :nb], D) for l, r in host.items()}
            ws = {layer: tuple(x[kh:kh + 1] for x in wn)}
            ref.append(O.decode_attn(qh[b:b + 1, kh * G:(kh + 1) * G], layer, w.num_layers, mode,
                                     kc, vc, [nb], weights=ws)[0])
            sel.append(got[b, kh * G:(kh + 1) * G])
    assert_close(np.stack(sel), np.stack(ref), "bf16", "q4 4B %s" % mode)
    ctx.close()
    keep.clear()
    torch.cuda.empty_cache()
