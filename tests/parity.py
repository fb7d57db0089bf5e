"""Shared test helpers: tolerances, comparisons, and building a library
context from a seeded synthetic workload.  Test infrastructure only."""

from __future__ import annotations

import numpy as np
import torch

# Parity bars: bf16 I/O max-abs 2e-2 and relative L2 5e-3; fp32 max-abs 1e-5.
BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3
F32_MAX_ABS = 1e-5


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def errors(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite output"
    max_abs = float(np.max(np.abs(got - ref))) if got.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got - ref))
    return max_abs, rel


def assert_close(got, ref, dtype: str, what: str = ""):
    max_abs, rel = errors(got, ref)
    if dtype == "f32":
        assert max_abs <= F32_MAX_ABS, "%s: max-abs %.3g > %.1g" % (what, max_abs, F32_MAX_ABS)
    else:
        assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_L2, \
            "%s: max-abs %.3g (bar %.1g), rel-L2 %.3g (bar %.1g)" % (
                what, max_abs, BF16_MAX_ABS, rel, BF16_REL_L2)
    return max_abs, rel


# ---------------------------------------------------------------------------
# GPU set-up from a synthetic workload (only the layers a call reads)
# ---------------------------------------------------------------------------

def layers_read(w, layer, mode):
    n = w.n
    if layer <= n or mode == "vanilla":
        return [layer]
    return sorted({1, n})   # lite, scaled and fused default sources


class DecodeSetup:
    """Caches, weights, query and lengths of one decode call on the GPU, bound
    to a library context."""

    def __init__(self, w, layer, modes, seed=0, device="cuda", lens=None, decode_ctas=0,
                 weight_std=0.3, tie_keys=True, sources=None, window=0):
        """``sources``: {mode: (k_first, k_second, v_first, v_second)} to
        reconstruct from other storage layers (all storage layers are bound)."""
        import cross_layer_kv_gb300 as fkv
        from cross_layer_kv_gb300 import synth
        self.w = w
        self.layer = layer
        self.sources = dict(sources or {})
        need = sorted({l for m in modes for l in layers_read(w, layer, m)})
        if self.sources:
            need = sorted(set(need) | set(range(1, w.n + 1)))
        store_upper = any(l > w.n for l in need)
        self.ctx = fkv.Context(w.num_layers, w.batch, w.seq, w.q_heads, w.kv_heads, w.head_dim,
                               w.dtype, store_upper=store_upper, decode_ctas=decode_ctas)
        self.caches = {}
        for l in need:
            k, v = synth.make_cache(w, l, seed, device)
            self.caches[l] = (k, v)
            self.ctx.fkv_bind_layer_cache(l, k, v)
        self.weights = None
        if layer > w.n:
            self.weights = synth.make_weights(w, layer, seed, device, tie_keys=tie_keys,
                                              std=weight_std)
            self.ctx.fkv_set_fusion_weights(layer, *self.weights)
        for m, src in self.sources.items():
            self.ctx.fkv_set_sources(layer, m, *src)
        self.window = window
        if window:
            self.ctx.fkv_set_window(layer, window)
        self.q = synth.make_query(w, layer, seed, device)
        if lens is None:
            self.lens = synth.make_seq_lens(w, seed, device)
        else:
            self.lens = torch.as_tensor(lens, dtype=torch.int32, device=device)
        self.ws = self.ctx.workspace(device)
        self.out = torch.empty_like(self.q)

    def run(self, mode):
        self.ctx.fkv_decode_attn(self.q, self.layer, mode, self.lens, self.out, self.ws)
        return self.out

    def source_kwargs(self, mode):
        src = self.sources.get(mode)
        if not src:
            return {}
        if mode == "fused":
            return {"k_sources": (src[0], src[1]), "v_sources": (src[2], src[3])}
        return {"k_sources": (src[0],), "v_sources": (src[2],)}

    def oracle(self, mode, pairs=None):
        """float64 oracle output, all (b, hq) or the listed pairs."""
        import oracle as O
        w = self.w
        lens = self.lens.cpu().tolist()
        G = w.group
        sk = self.source_kwargs(mode)
        sk["window"] = self.window
        if pairs is None:
            kc = {l: f64(k) for l, (k, v) in self.caches.items()}
            vc = {l: f64(v) for l, (k, v) in self.caches.items()}
            ws = {self.layer: tuple(f64(x) for x in self.weights)} if self.weights else None
            return O.decode_attn(f64(self.q), self.layer, w.num_layers, mode, kc, vc, lens,
                                 weights=ws, **sk)
        out = []
        for b, hq in pairs:
            kh = hq // G
            n = lens[b]
            kc = {l: f64(k[b:b + 1, kh:kh + 1, :n]) for l, (k, v) in self.caches.items()}
            vc = {l: f64(v[b:b + 1, kh:kh + 1, :n]) for l, (k, v) in self.caches.items()}
            ws = ({self.layer: tuple(f64(x[kh:kh + 1]) for x in self.weights)}
                  if self.weights else None)
            o = O.decode_attn(f64(self.q[b:b + 1, hq:hq + 1]), self.layer, w.num_layers, mode,
                              kc, vc, [n], weights=ws, **sk)
            out.append(o[0, 0])
        return np.stack(out)

    def oracle_units(self, mode, units):
        """float64 oracle outputs ``[len(units), G, D]``: all G query heads of
        each listed (b, kv_head) unit, one oracle call per unit."""
        import oracle as O
        w = self.w
        lens = self.lens.cpu().tolist()
        G = w.group
        sk = self.source_kwargs(mode)
        sk["window"] = self.window
        out = []
        for b, kh in units:
            n = lens[b]
            kc = {l: f64(k[b:b + 1, kh:kh + 1, :n]) for l, (k, v) in self.caches.items()}
            vc = {l: f64(v[b:b + 1, kh:kh + 1, :n]) for l, (k, v) in self.caches.items()}
            ws = ({self.layer: tuple(f64(x[kh:kh + 1]) for x in self.weights)}
                  if self.weights else None)
            o = O.decode_attn(f64(self.q[b:b + 1, kh * G:(kh + 1) * G]), self.layer, w.num_layers,
                              mode, kc, vc, [n], weights=ws, **sk)
            out.append(o[0])
        return np.stack(out)

    def close(self):
        self.ctx.close()
        self.caches.clear()
