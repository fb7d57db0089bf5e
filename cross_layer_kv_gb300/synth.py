"""Seeded synthetic workloads shaped like the FusedKV evaluation models.

This module only draws inputs.  It holds none of the attention or fusion
arithmetic: the CUDA library and the float64 oracle both receive the arrays it
makes and nothing else from it.

Recipe (the same for every workload, all draws from ``torch.Generator``
seeded per (workload seed, layer, tensor) so that one layer can be rebuilt on
its own):

* keys: pre-RoPE K ~ N(0, 1), then rotary embedding with base 10000,
  "rotate-half" pairing (channel j with j + D/2) at positions 0..S_max-1, and
  stored post-RoPE (the caches of the method hold post-RoPE keys);
* values ~ N(0, 1); queries ~ N(0, 1), taken as already rotated;
* fusion weights a, b ~ N(0.5, 0.3) per (target layer, KV head, channel), the
  key weights tied across each rotation pair (a[j] = a[j + D/2]);
* ragged lengths, where a workload has them, uniform integers in [S/2, S].

The rotary step here only synthesises realistic post-RoPE caches; the library
itself never applies RoPE.
"""

from __future__ import annotations

import dataclasses
import hashlib
from typing import Dict, Optional, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_layers: int
    batch: int
    seq: int
    q_heads: int
    kv_heads: int
    head_dim: int
    dtype: str  # "bf16" | "f32"
    ragged: bool = False
    kind: str = "decode"  # "decode" | "prefill"
    hidden: int = 0

    @property
    def n(self) -> int:
        return self.num_layers // 2

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4


# The five workloads: a tiny fp32 parity case and four shapes taken from the
# model table of the paper (332M / 650M / 1.5B / 4B), with GQA 2:1.
TINY = Workload("tiny-decode-f32", 4, 1, 256, 4, 2, 64, "f32")
M332 = Workload("332M-decode", 12, 32, 8192, 16, 8, 64, "bf16", hidden=1024)
B1_5 = Workload("1.5B-decode-ragged", 24, 16, 32768, 16, 8, 128, "bf16", ragged=True, hidden=2048)
M650_PREFILL = Workload("650M-prefill", 16, 4, 8192, 16, 8, 96, "bf16", kind="prefill", hidden=1536)
B4 = Workload("4B-decode-128k", 36, 4, 131072, 32, 16, 80, "bf16", hidden=2560)

WORKLOADS = {w.name: w for w in (TINY, M332, B1_5, M650_PREFILL, B4)}


def sub_seed(seed: int, *tags) -> int:
    """A stable 63-bit seed derived from the workload seed and string tags."""
    h = hashlib.sha256(("%d|" % seed + "|".join(str(t) for t in tags)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, seed: int, *tags) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(sub_seed(seed, *tags))
    return g


def _rotate_half_inplace(k: torch.Tensor, positions: torch.Tensor, base: float = 10000.0):
    """Apply rotary embedding (pairs j, j + D/2) to fp32 ``k[..., T, D]`` in place."""
    D = k.shape[-1]
    half = D // 2
    inv = base ** (-2.0 * torch.arange(half, device=k.device, dtype=torch.float64) / D)
    ang = positions.to(torch.float64)[:, None] * inv[None, :]
    c = torch.cos(ang).to(torch.float32)
    s = torch.sin(ang).to(torch.float32)
    lo = k[..., :half].clone()
    hi = k[..., half:]
    k[..., :half] = lo * c - hi * s
    k[..., half:] = lo * s + hi * c


def make_cache(w: Workload, layer: int, seed: int, device, seq: Optional[int] = None,
               batch: Optional[int] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Post-RoPE K and V caches ``[B, H_kv, S, D]`` of one layer."""
    S = seq or w.seq
    B = batch or w.batch
    shape = (B, w.kv_heads, S, w.head_dim)
    k = torch.empty(shape, dtype=w.torch_dtype, device=device)
    v = torch.empty(shape, dtype=w.torch_dtype, device=device)
    gk = _gen(device, seed, "k", layer)
    gv = _gen(device, seed, "v", layer)
    pos = torch.arange(S, device=device)
    # fill one batch row at a time so the fp32 temporary stays bounded
    for b in range(B):
        tmp = torch.randn((w.kv_heads, S, w.head_dim), generator=gk, device=device,
                          dtype=torch.float32)
        _rotate_half_inplace(tmp, pos)
        k[b].copy_(tmp)
        del tmp
        v[b].copy_(torch.randn((w.kv_heads, S, w.head_dim), generator=gv, device=device,
                               dtype=torch.float32))
    return k, v


def make_query(w: Workload, layer: int, seed: int, device, positions: int = 0) -> torch.Tensor:
    """q ~ N(0,1): ``[B, H_q, D]`` for decode, ``[B, H_q, S, D]`` for prefill."""
    g = _gen(device, seed, "q", layer)
    shape = ((w.batch, w.q_heads, positions, w.head_dim) if positions
             else (w.batch, w.q_heads, w.head_dim))
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(w.torch_dtype)


def make_weights(w: Workload, layer: int, seed: int, device, tie_keys: bool = True,
                 mean: float = 0.5, std: float = 0.3) -> Tuple[torch.Tensor, ...]:
    """(a_first, a_second, b_first, b_second), each fp32 ``[H_kv, D]``."""
    g = _gen(device, seed, "w", layer)
    D = w.head_dim
    out = []
    for i in range(4):
        x = torch.randn((w.kv_heads, D), generator=g, device=device, dtype=torch.float32)
        x = x * std + mean
        if tie_keys and i < 2:
            x[:, D // 2:] = x[:, : D // 2]
        out.append(x.contiguous())
    return tuple(out)


def make_seq_lens(w: Workload, seed: int, device) -> torch.Tensor:
    """int32 ``[B]``: S everywhere, or uniform in [S/2, S] for ragged workloads."""
    if not w.ragged:
        return torch.full((w.batch,), w.seq, dtype=torch.int32, device=device)
    g = _gen("cpu", seed, "lens")
    lens = torch.randint(w.seq // 2, w.seq + 1, (w.batch,), generator=g, dtype=torch.int64)
    return lens.to(torch.int32).to(device)


def make_model_inputs(w: Workload, seed: int, device, store_upper: bool = False,
                      layers=None) -> Dict[str, object]:
    """Caches of the storage layers (all layers if ``store_upper``), per-layer
    queries, fusion weights of the upper layers and the sequence lengths."""
    L, n = w.num_layers, w.n
    cache_layers = range(1, L + 1) if store_upper else range(1, n + 1)
    if layers is not None:
        cache_layers = [l for l in cache_layers if l in layers]
    caches = {l: make_cache(w, l, seed, device) for l in cache_layers}
    qpos = w.seq if w.kind == "prefill" else 0
    wanted = range(1, L + 1) if layers is None else layers
    queries = {l: make_query(w, l, seed, device, positions=qpos) for l in wanted}
    weights = {l: make_weights(w, l, seed, device) for l in wanted if l > n}
    lens = make_seq_lens(w, seed, device)
    return {"caches": caches, "q": queries, "weights": weights, "seq_lens": lens}
