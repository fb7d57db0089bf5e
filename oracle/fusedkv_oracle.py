"""Plain float64 CPU oracle for FusedKV upper-layer attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (no kernels, headers, tables or helpers); the two
meet only through the seeded input arrays that the tests hand to both.

Everything here is written for a reader to check against the pages by eye:
NumPy float64, whole tensors materialised, no blocking, no fusion, no
reordering beyond what the definitions state.

Sources cited below (titles of the pages, then the section / equation / table):

* [Slides] "FusedKV: Reconstructing KV Caches with Cross-Layer Fusion" --
  reading presentation of Lin et al., arXiv:2512.03870v3.
* [Notes] "FusedKV: 通过跨层融合重构 KV 缓存" -- reading notes on the same
  paper (sections 2.1-2.5 follow the paper's Sec.2).

Readings of points the pages leave open:

* layers are 1-based, L = 2n, storage layers 1..n, reconstruction layers
  n+1..L ([Notes] §2.1, Eq.(1));
* the fusion weights of a target layer are one vector over the full K/V
  projection width, stored as ``[H_kv, D]`` (the pages use a simplified
  single-matrix notation, [Slides] Eqs.(4)-(5); [Notes] §2.1 says real code adds
  batch and head axes);
* the RoPE rotation pair is (j, j + D/2) ("rotate-half" storage);
* softmax scale 1/sqrt(D), no bias, no soft-capping;
* GQA: query head h reads KV head floor(h / G), G = H_q / H_kv;
* decode attends over positions [0, seq_len) with the new token already
  appended ([Notes] §2.3: storage caches are updated first);
* causal prefill from position 0, inclusive diagonal.

Parity status of every function is stated in its docstring; all are pinned by
``tests/test_oracle.py`` except where a docstring says "parity unpinned".
"""

from __future__ import annotations

import math
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

VANILLA = "vanilla"
LITE = "lite"
FUSED = "fused"
SCALED = "scaled"   # single-source channel scaling, [Slides] Fig.8 ablation
MODES = (VANILLA, LITE, FUSED, SCALED)


# ---------------------------------------------------------------------------
# Layer partition and source map  ([Notes] §2.1 Eq.(1); [Slides] "Lite
# separates the key source from the value source", Eq.(6))
# ---------------------------------------------------------------------------

def num_storage_layers(num_layers: int) -> int:
    """n = L / 2 for an even layer count L ([Notes] §2.1: L = 2n)."""
    if num_layers < 2 or num_layers % 2:
        raise ValueError("L must be even and >= 2")
    return num_layers // 2


def is_storage_layer(layer: int, num_layers: int) -> bool:
    """Storage layers are {1..n}; reconstruction layers are {n+1..L}."""
    if not 1 <= layer <= num_layers:
        raise ValueError("layer out of range (1-based)")
    return layer <= num_storage_layers(num_layers)


def kv_sources(layer: int, num_layers: int, mode: str,
               k_sources: Optional[Tuple[int, int]] = None,
               v_sources: Optional[Tuple[int, int]] = None) -> dict:
    """Which stored caches a layer's K and V come from.

    Returns ``{"k": [src...], "v": [src...], "weighted": bool}``.

    * storage layer (any mode), or vanilla: its own cache;
    * lite ([Slides] Eq.(6)): K^i = K^n, V^i = V^1;
    * fused ([Slides] Eqs.(4)-(5)): K^i from {K^1, K^n}, V^i from {V^1, V^n};
    * scaled ([Slides] Fig.8, "learnable channel weights" on the Lite
      sources): K^i = a (.) K^n, V^i = b (.) V^1.

    ``k_sources`` / ``v_sources`` override the source layers (the source-layer
    ablation of [Slides] "Source-layer choice", Table 17, and the reversed
    sharing K^1, V^n of Fig.8); lite and scaled use the first entry of each.
    """
    n = num_storage_layers(num_layers)
    if mode not in MODES:
        raise ValueError(mode)
    if is_storage_layer(layer, num_layers) or mode == VANILLA:
        return {"k": [layer], "v": [layer], "weighted": False}
    ks = tuple(k_sources) if k_sources is not None else None
    vs = tuple(v_sources) if v_sources is not None else None
    if mode in (LITE, SCALED):
        k = ks[0] if ks else n
        v = vs[0] if vs else 1
        return {"k": [k], "v": [v], "weighted": mode == SCALED}
    return {"k": list(ks) if ks else [1, n], "v": list(vs) if vs else [1, n],
            "weighted": True}


# ---------------------------------------------------------------------------
# Reconstruction  ([Slides] Eqs.(4)-(6); [Notes] §2.3)
# ---------------------------------------------------------------------------

def reconstruct_kv(layer: int, num_layers: int, mode: str,
                   k_caches: Dict[int, np.ndarray], v_caches: Dict[int, np.ndarray],
                   weights: Optional[Dict[int, Sequence[np.ndarray]]] = None,
                   k_sources=None, v_sources=None) -> Tuple[np.ndarray, np.ndarray]:
    """Materialise K^i, V^i in float64.

    Caches are ``[B, H_kv, S, D]`` (any float dtype; cast to float64).
    ``weights[layer] = (a_first, a_second, b_first, b_second)``, each
    ``[H_kv, D]``: the per-target-layer channel weights of Eqs.(4)-(5),
    broadcast over batch and tokens.  No sign or normalisation constraint
    ([Slides] "FusedKV learns two-source, channel-wise fusion").
    """
    src = kv_sources(layer, num_layers, mode, k_sources, v_sources)
    if not src["weighted"]:
        return (np.asarray(k_caches[src["k"][0]], dtype=np.float64),
                np.asarray(v_caches[src["v"][0]], dtype=np.float64))
    a1, an, b1, bn = (np.asarray(w, dtype=np.float64) for w in weights[layer])
    if len(src["k"]) == 1:
        # scaled: one source each, weighted by the first key / value weights
        k = np.asarray(k_caches[src["k"][0]], dtype=np.float64)
        v = np.asarray(v_caches[src["v"][0]], dtype=np.float64)
        return a1[None, :, None, :] * k, b1[None, :, None, :] * v
    k1 = np.asarray(k_caches[src["k"][0]], dtype=np.float64)
    kn = np.asarray(k_caches[src["k"][1]], dtype=np.float64)
    v1 = np.asarray(v_caches[src["v"][0]], dtype=np.float64)
    vn = np.asarray(v_caches[src["v"][1]], dtype=np.float64)
    # weights [H_kv, D] -> [1, H_kv, 1, D]: one value per (head, channel),
    # the same for every batch row and token
    w = lambda x: x[None, :, None, :]
    k_i = w(a1) * k1 + w(an) * kn
    v_i = w(b1) * v1 + w(bn) * vn
    return k_i, v_i


# ---------------------------------------------------------------------------
# Softmax attention (the plain definition; vanilla attention of [Slides]
# Table 1 is standard attention, queries stay layer-specific)
# ---------------------------------------------------------------------------

def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """o = softmax(scale * k q) ^T v for one query vector.

    q ``[D]``, k ``[T, D]``, v ``[T, D]`` -> ``[D]``.  T >= 1.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = scale * (k @ q)
    p = np.exp(s - s.max())
    p = p / p.sum()
    return p @ v


def decode_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                     seq_lens: Sequence[int], scale: Optional[float] = None,
                     window: int = 0) -> np.ndarray:
    """One decode step of GQA softmax attention.

    q ``[B, H_q, D]``; k, v ``[B, H_kv, S, D]``; each sequence b attends over
    positions ``[0, seq_lens[b])``, or only the last ``window`` of them for a
    sliding-window layer (window > 0; the hybrid SWA layers of [Slides]
    "MoE and hybrid SWA").  Query head h reads KV head h // G.
    Returns float64 ``[B, H_q, D]``.
    """
    B, H_q, D = q.shape
    H_kv = k.shape[1]
    if H_q % H_kv:
        raise ValueError("H_q must be a multiple of H_kv")
    G = H_q // H_kv
    if scale is None:
        scale = default_scale(D)
    out = np.empty((B, H_q, D), dtype=np.float64)
    for b in range(B):
        n = int(seq_lens[b])
        if not 1 <= n <= k.shape[2]:
            raise ValueError("sequence length out of range")
        lo = max(0, n - window) if window > 0 else 0
        for h in range(H_q):
            kv = h // G
            out[b, h] = attend(q[b, h], k[b, kv, lo:n], v[b, kv, lo:n], scale)
    return out


def prefill_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                      scale: Optional[float] = None,
                      rows: Optional[Sequence[int]] = None, window: int = 0) -> np.ndarray:
    """Causal GQA attention over a prompt that starts at position 0.

    q ``[B, H_q, S, D]``; k, v ``[B, H_kv, >=S, D]``.  Query position m sees
    key positions t <= m (inclusive diagonal), and with window > 0 only
    t > m - window.  With ``rows`` given, only those query positions are
    computed and the result is ``[B, H_q, len(rows), D]``.
    """
    B, H_q, S, D = q.shape
    H_kv = k.shape[1]
    G = H_q // H_kv
    if scale is None:
        scale = default_scale(D)
    rows = list(range(S)) if rows is None else [int(r) for r in rows]
    out = np.empty((B, H_q, len(rows), D), dtype=np.float64)
    for b in range(B):
        for h in range(H_q):
            kv = h // G
            kk = np.asarray(k[b, kv], dtype=np.float64)
            vv = np.asarray(v[b, kv], dtype=np.float64)
            qq = np.asarray(q[b, h], dtype=np.float64)
            for i, m in enumerate(rows):
                lo = max(0, m + 1 - window) if window > 0 else 0
                out[b, h, i] = attend(qq[m], kk[lo:m + 1], vv[lo:m + 1], scale)
    return out


def decode_attn(q, layer, num_layers, mode, k_caches, v_caches, seq_lens,
                weights=None, scale=None, k_sources=None, v_sources=None, window=0):
    """A decode attention call of one layer: reconstruct, then attend."""
    k_i, v_i = reconstruct_kv(layer, num_layers, mode, k_caches, v_caches,
                              weights, k_sources, v_sources)
    return decode_attention(q, k_i, v_i, seq_lens, scale, window)


def prefill_attn(q, layer, num_layers, mode, k_caches, v_caches,
                 weights=None, scale=None, rows=None, k_sources=None, v_sources=None,
                 window=0):
    """A causal prefill attention call of one layer: reconstruct, then attend."""
    S = q.shape[2]
    k_i, v_i = reconstruct_kv(layer, num_layers, mode,
                              {l: c[:, :, :S] for l, c in k_caches.items()},
                              {l: c[:, :, :S] for l, c in v_caches.items()},
                              weights, k_sources, v_sources)
    return prefill_attention(q, k_i, v_i, scale, rows, window)


def chunk_prefill_attention(q: np.ndarray, q_start: int, k: np.ndarray, v: np.ndarray,
                            scale: Optional[float] = None, window: int = 0) -> np.ndarray:
    """Causal attention of a chunk of queries over an existing cache.

    q ``[B, H_q, C, D]`` holds the queries of positions q_start .. q_start+C-1;
    k, v ``[B, H_kv, >= q_start+C, D]``.  Query i sees key positions
    t <= q_start + i (the prompt rows before the chunk are already cached).
    With q_start = 0 this is ``prefill_attention``; with C = 1 it is one
    decode step over q_start + 1 cached rows.
    """
    B, H_q, C, D = q.shape
    H_kv = k.shape[1]
    G = H_q // H_kv
    if scale is None:
        scale = default_scale(D)
    out = np.empty((B, H_q, C, D), dtype=np.float64)
    for b in range(B):
        for h in range(H_q):
            kv = h // G
            for i in range(C):
                n = q_start + i + 1
                lo = max(0, n - window) if window > 0 else 0
                out[b, h, i] = attend(q[b, h, i], k[b, kv, lo:n], v[b, kv, lo:n], scale)
    return out


def chunk_prefill_attn(q, q_start, layer, num_layers, mode, k_caches, v_caches, weights=None,
                       scale=None, k_sources=None, v_sources=None, window=0):
    """A chunked causal prefill call of one layer: reconstruct rows
    [0, q_start + C), then attend."""
    n = q_start + q.shape[2]
    k_i, v_i = reconstruct_kv(layer, num_layers, mode,
                              {l: c[:, :, :n] for l, c in k_caches.items()},
                              {l: c[:, :, :n] for l, c in v_caches.items()},
                              weights, k_sources, v_sources)
    return chunk_prefill_attention(q, q_start, k_i, v_i, scale, window)


# ---------------------------------------------------------------------------
# Cache append ([Notes] §2.3: the storage caches take the new token's
# post-RoPE K/V before the upper layers attend)
# ---------------------------------------------------------------------------

def append_kv(cache: np.ndarray, new: np.ndarray, pos: Sequence[int]) -> np.ndarray:
    """cache[b, h, pos[b] + t, :] = new[b, h, t, :]; returns an updated copy."""
    out = np.array(cache, copy=True)
    T = new.shape[2]
    for b in range(cache.shape[0]):
        p = int(pos[b])
        if p < 0 or p + T > cache.shape[2]:
            raise ValueError("append out of range")
        out[b, :, p:p + T, :] = new[b]
    return out


# ---------------------------------------------------------------------------
# 4-bit KV cache ([Slides] "Four-bit KV quantization is the stronger
# combination", Table 14).  KIVI's grouping is not on the pages; this library
# quantises each token row of each head in groups of Q4_GROUP channels with
# an asymmetric uniform 4-bit code:
#     min = min(x_g), scale = bf16((max(x_g) - min) / 15)   (fp32 division),
#     code = clamp(rint((x - min) / scale), 0, 15)           (fp32, half to even),
#     x_hat = min + code * scale.
# A constant group (scale 0) stores code 0.  min and scale are stored as bf16
# (min is an input value, so exact); the codes use the stored scale.
# ---------------------------------------------------------------------------

Q4_GROUP = 16


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest bfloat16 (ties to even), returned as float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def q4_quantize(x: np.ndarray):
    """x ``[..., D]`` (bf16 values) -> codes uint8 ``[..., D]`` (0..15),
    scale and min float32 ``[..., D / Q4_GROUP]`` (bf16-representable)."""
    x = np.asarray(x, dtype=np.float32)
    D = x.shape[-1]
    g = x.reshape(x.shape[:-1] + (D // Q4_GROUP, Q4_GROUP))
    lo = g.min(axis=-1)
    hi = g.max(axis=-1)
    scale = bf16_round((hi - lo) / np.float32(15.0))
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint((g - lo[..., None]) / scale[..., None])
    q = np.where(scale[..., None] > 0, q, 0)
    codes = np.clip(q, 0, 15).astype(np.uint8).reshape(x.shape)
    return codes, scale.astype(np.float32), lo.astype(np.float32)


def q4_dequantize(codes: np.ndarray, scale: np.ndarray, lo: np.ndarray) -> np.ndarray:
    """x_hat = min + code * scale, float64 ``[..., D]``."""
    D = codes.shape[-1]
    c = np.asarray(codes, dtype=np.float64).reshape(codes.shape[:-1] + (D // Q4_GROUP, Q4_GROUP))
    xh = np.asarray(lo, np.float64)[..., None] + c * np.asarray(scale, np.float64)[..., None]
    return xh.reshape(codes.shape)


def q4_row_bytes(head_dim: int) -> int:
    """Bytes of one quantised row: codes (D/2), then (scale, min) bf16 pairs
    (D/4), padded to 16 bytes."""
    return (head_dim // 2 + head_dim // 4 + 15) // 16 * 16


def q4_pack(codes: np.ndarray, scale: np.ndarray, lo: np.ndarray) -> np.ndarray:
    """Rows ``[..., D]`` -> records ``[..., q4_row_bytes(D)]`` uint8: byte i of
    the codes holds channel 2i in its low and 2i+1 in its high nibble; then
    per group the bf16 bits of scale and of min (little-endian)."""
    D = codes.shape[-1]
    rb = q4_row_bytes(D)
    out = np.zeros(codes.shape[:-1] + (rb,), dtype=np.uint8)
    c = codes.astype(np.uint8)
    out[..., : D // 2] = c[..., 0::2] | (c[..., 1::2] << 4)
    sb = (np.ascontiguousarray(scale, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    mb = (np.ascontiguousarray(lo, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    pm = np.stack([sb, mb], axis=-1).reshape(codes.shape[:-1] + (D // Q4_GROUP * 2,))
    out[..., D // 2: D // 2 + D // 4] = pm.view(np.uint8).reshape(codes.shape[:-1] + (D // 4,))
    return out


def q4_unpack(rec: np.ndarray, head_dim: int):
    """Records -> (codes, scale, min), the inverse of ``q4_pack``."""
    D = head_dim
    rec = np.asarray(rec, dtype=np.uint8)
    b = rec[..., : D // 2]
    codes = np.empty(rec.shape[:-1] + (D,), dtype=np.uint8)
    codes[..., 0::2] = b & 0xF
    codes[..., 1::2] = b >> 4
    pm = np.ascontiguousarray(rec[..., D // 2: D // 2 + D // 4]).view(np.uint16)
    pm = pm.reshape(rec.shape[:-1] + (D // Q4_GROUP, 2)).astype(np.uint32) << 16
    f = pm.view(np.float32)
    return codes, f[..., 0].copy(), f[..., 1].copy()


def q4_dequantize_records(rec: np.ndarray, head_dim: int) -> np.ndarray:
    return q4_dequantize(*q4_unpack(rec, head_dim))


# ---------------------------------------------------------------------------
# RoPE and the pair-tying property ([Slides] "Post-RoPE fusion needs paired key
# weights", Eqs.(7)-(8); [Notes] §2.4)
# ---------------------------------------------------------------------------

def rope_angles(positions: np.ndarray, head_dim: int, base: float = 10000.0) -> np.ndarray:
    """theta[p, j] = pos_p * base^(-2j/D) for the D/2 rotation pairs."""
    half = head_dim // 2
    inv = base ** (-2.0 * np.arange(half, dtype=np.float64) / head_dim)
    return np.asarray(positions, dtype=np.float64)[..., None] * inv


def rope_rotate_half(x: np.ndarray, positions: np.ndarray, base: float = 10000.0) -> np.ndarray:
    """Rotate channel pairs (j, j + D/2) of ``x[..., T, D]`` by angle theta_j(pos).

    (x_j, x_{j+D/2}) -> (x_j cos - x_{j+D/2} sin, x_j sin + x_{j+D/2} cos).
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    th = rope_angles(positions, D, base)
    c, s = np.cos(th), np.sin(th)
    lo, hi = x[..., : D // 2], x[..., D // 2:]
    return np.concatenate([lo * c - hi * s, lo * s + hi * c], axis=-1)


def fused_key_scores(q: np.ndarray, q_pos: int, k_first: np.ndarray, k_second: np.ndarray,
                     k_pos: np.ndarray, a_first: np.ndarray, a_second: np.ndarray,
                     base: float = 10000.0) -> np.ndarray:
    """Unscaled scores  (R_m q) . (a_1 (.) R_t K^1_t + a_n (.) R_t K^n_t)  for each t.

    q ``[D]`` and keys ``[T, D]`` are pre-RoPE; RoPE is applied here at the
    given positions, then the keys are fused post-RoPE (the order the method
    uses: caches hold post-RoPE keys).
    """
    qr = rope_rotate_half(q[None, :], np.array([q_pos]), base)[0]
    k1 = rope_rotate_half(k_first, k_pos, base)
    kn = rope_rotate_half(k_second, k_pos, base)
    k = a_first[None, :] * k1 + a_second[None, :] * kn
    return k @ qr


def tied(a: np.ndarray) -> bool:
    """True when a[j] == a[j + D/2] for every rotation pair."""
    D = a.shape[-1]
    return bool(np.all(a[..., : D // 2] == a[..., D // 2:]))


# ---------------------------------------------------------------------------
# Cache capacity / I/O accounting ([Slides] "Capacity and bandwidth are
# different bottlenecks" and Table 1; [Notes] §2.5)
# ---------------------------------------------------------------------------

def stored_elements(mode: str, num_layers: int, seq: int, kv_heads: int, head_dim: int,
                    batch: int = 1) -> int:
    """Elements held in the KV cache (K and V, all layers that store)."""
    per_layer = 2 * batch * seq * kv_heads * head_dim
    if mode == VANILLA:
        return num_layers * per_layer
    return num_storage_layers(num_layers) * per_layer


def call_read_elements(layer: int, mode: str, num_layers: int, seq: int, kv_heads: int,
                       head_dim: int, batch: int = 1) -> int:
    # (scaled reads one K and one V source, like lite)
    """Cache elements one attention call of ``layer`` reads (K and V)."""
    src = kv_sources(layer, num_layers, mode)
    per_source = batch * seq * kv_heads * head_dim
    return per_source * (len(src["k"]) + len(src["v"]))


def step_read_elements(mode: str, num_layers: int, seq: int, kv_heads: int, head_dim: int,
                       batch: int = 1) -> int:
    """Cache elements one decode step reads over all L layers (attention only)."""
    return sum(call_read_elements(l, mode, num_layers, seq, kv_heads, head_dim, batch)
               for l in range(1, num_layers + 1))


# ---------------------------------------------------------------------------
# Brute force (pure-Python loops, tiny shapes only): Eqs.(4)-(6) element by
# element, then the softmax written out term by term.
# ---------------------------------------------------------------------------

def brute_force_decode(q, layer, num_layers, mode, k_caches, v_caches, seq_lens,
                       weights=None, scale=None):
    """Same result as ``decode_attn`` computed with explicit scalar loops."""
    B, H_q, D = q.shape
    H_kv = next(iter(k_caches.values())).shape[1]
    G = H_q // H_kv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    n = num_layers // 2
    out = [[[0.0] * D for _ in range(H_q)] for _ in range(B)]
    for b in range(B):
        T = int(seq_lens[b])
        for h in range(H_q):
            kv = h // G

            def key(t, d):
                if layer <= n or mode == VANILLA:
                    return float(k_caches[layer][b][kv][t][d])
                if mode == LITE:
                    return float(k_caches[n][b][kv][t][d])
                a1, an = weights[layer][0], weights[layer][1]
                return (float(a1[kv][d]) * float(k_caches[1][b][kv][t][d])
                        + float(an[kv][d]) * float(k_caches[n][b][kv][t][d]))

            def val(t, d):
                if layer <= n or mode == VANILLA:
                    return float(v_caches[layer][b][kv][t][d])
                if mode == LITE:
                    return float(v_caches[1][b][kv][t][d])
                b1, bn = weights[layer][2], weights[layer][3]
                return (float(b1[kv][d]) * float(v_caches[1][b][kv][t][d])
                        + float(bn[kv][d]) * float(v_caches[n][b][kv][t][d]))

            scores = []
            for t in range(T):
                acc = 0.0
                for d in range(D):
                    acc += float(q[b][h][d]) * key(t, d)
                scores.append(scale * acc)
            mx = max(scores)
            ex = [math.exp(s - mx) for s in scores]
            tot = sum(ex)
            for d in range(D):
                acc = 0.0
                for t in range(T):
                    acc += ex[t] * val(t, d)
                out[b][h][d] = acc / tot
    return np.array(out, dtype=np.float64)


def brute_force_prefill(q, k, v, scale=None):
    """Causal attention with scalar loops; q [B,H_q,S,D], k/v [B,H_kv,S,D]."""
    B, H_q, S, D = q.shape
    H_kv = k.shape[1]
    G = H_q // H_kv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, H_q, S, D), dtype=np.float64)
    for b in range(B):
        for h in range(H_q):
            kv = h // G
            for m in range(S):
                sc = []
                for t in range(m + 1):
                    sc.append(scale * sum(float(q[b, h, m, d]) * float(k[b, kv, t, d])
                                          for d in range(D)))
                mx = max(sc)
                ex = [math.exp(s - mx) for s in sc]
                tot = sum(ex)
                for d in range(D):
                    out[b, h, m, d] = sum(ex[t] * float(v[b, kv, t, d])
                                          for t in range(m + 1)) / tot
    return out
