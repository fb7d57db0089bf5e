"""Pins for the float64 oracle: facts fixed by the pages and by mathematics,
checked without the oracle checking itself.

Each test states what pins what:

* library routine: vanilla attention equals torch's scaled_dot_product_attention
  run in float64 on the CPU (GQA by explicit head repetition);
* special cases: one cached token returns that token's value row; a zero query
  returns the mean of the value rows;
* exact identities from the pages: Lite (K^n, V^1) is fused attention with
  weights (0, 1, 1, 0) ([Slides] Eq.(6) vs Eqs.(4)-(5)); fused attention with
  constant channel weights equals plain attention over the explicitly summed
  caches;
* closed form of [Slides] Eqs.(7)-(8): with pair-tied key weights, shifting every
  position by the same amount leaves the scores unchanged; untied weights break
  this, by an amount that vanishes as the pair weights are made equal;
* linearity of Eq.(5) in the value weights;
* brute-force scalar loops on tiny shapes;
* Table 1 and the notes' element counts (golden fixtures under tests/golden/).
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed=0):
    return np.random.default_rng(seed)


def _caches(rng, L, B, H_kv, S, D, layers=None):
    layers = layers or range(1, L + 1)
    k = {l: rng.standard_normal((B, H_kv, S, D)) for l in layers}
    v = {l: rng.standard_normal((B, H_kv, S, D)) for l in layers}
    return k, v


def _weights(rng, H_kv, D, tie=True):
    ws = []
    for i in range(4):
        x = rng.normal(0.5, 0.3, (H_kv, D))
        if tie and i < 2:
            x[:, D // 2:] = x[:, : D // 2]
        ws.append(x)
    return tuple(ws)


def _sdpa(q, k, v, causal=False, lens=None):
    """torch SDPA in float64; q [B,H_q,T,D], k/v [B,H_kv,S,D]."""
    G = q.shape[1] // k.shape[1]
    qt = torch.from_numpy(np.ascontiguousarray(q))
    kt = torch.from_numpy(np.ascontiguousarray(k)).repeat_interleave(G, dim=1)
    vt = torch.from_numpy(np.ascontiguousarray(v)).repeat_interleave(G, dim=1)
    if lens is None:
        return torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, is_causal=causal).numpy()
    outs = []
    for b, n in enumerate(lens):
        outs.append(torch.nn.functional.scaled_dot_product_attention(
            qt[b:b + 1], kt[b:b + 1, :, :n], vt[b:b + 1, :, :n]).numpy())
    return np.concatenate(outs, 0)


# --------------------------------------------------------------------------
# layer partition / sources ([Notes] §2.1, [Slides] Eq.(6) with its 16-layer
# example)
# --------------------------------------------------------------------------

def test_lite_sources_sixteen_layers_golden():
    g = _golden("lite_sources_16_layers.json")
    L = g["num_layers"]
    assert O.num_storage_layers(L) == len(g["storage_layers"])
    for l in range(1, L + 1):
        assert O.is_storage_layer(l, L) == (l in g["storage_layers"])
    for l in g["reconstruction_layers"]:
        src = O.kv_sources(l, L, O.LITE)
        assert src["k"] == [g["lite_key_source"]] and src["v"] == [g["lite_value_source"]]
        f = O.kv_sources(l, L, O.FUSED)
        assert f["k"] == g["fused_sources"] and f["v"] == g["fused_sources"]
    for l in g["storage_layers"]:
        for m in O.MODES:
            assert O.kv_sources(l, L, m) == {"k": [l], "v": [l], "weighted": False}


def test_partition_rejects_odd_and_out_of_range():
    with pytest.raises(ValueError):
        O.num_storage_layers(7)
    with pytest.raises(ValueError):
        O.is_storage_layer(0, 4)
    with pytest.raises(ValueError):
        O.is_storage_layer(5, 4)


# --------------------------------------------------------------------------
# softmax attention against a library routine and closed-form special cases
# --------------------------------------------------------------------------

@pytest.mark.parametrize("G", [1, 2, 4])
def test_decode_attention_matches_torch_sdpa(G):
    rng = _rng(1)
    B, H_kv, S, D = 3, 2, 37, 16
    q = rng.standard_normal((B, H_kv * G, D))
    k = rng.standard_normal((B, H_kv, S, D))
    v = rng.standard_normal((B, H_kv, S, D))
    lens = [37, 1, 20]
    got = O.decode_attention(q, k, v, lens)
    ref = _sdpa(q[:, :, None, :], k, v, lens=lens)[:, :, 0, :]
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_decode_attention_custom_scale_matches_sdpa():
    rng = _rng(2)
    q = rng.standard_normal((1, 2, 8))
    k = rng.standard_normal((1, 1, 9, 8))
    v = rng.standard_normal((1, 1, 9, 8))
    got = O.decode_attention(q, k, v, [9], scale=0.3)
    qt = torch.from_numpy(q[:, :, None, :])
    kt = torch.from_numpy(k).expand(1, 2, 9, 8)
    vt = torch.from_numpy(v).expand(1, 2, 9, 8)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=0.3)
    np.testing.assert_allclose(got, ref[:, :, 0].numpy(), atol=1e-12)


@pytest.mark.parametrize("G", [1, 2])
def test_prefill_attention_matches_torch_causal_sdpa(G):
    rng = _rng(3)
    B, H_kv, S, D = 2, 2, 23, 8
    q = rng.standard_normal((B, H_kv * G, S, D))
    k = rng.standard_normal((B, H_kv, S, D))
    v = rng.standard_normal((B, H_kv, S, D))
    got = O.prefill_attention(q, k, v)
    ref = _sdpa(q, k, v, causal=True)
    np.testing.assert_allclose(got, ref, atol=1e-12)
    rows = [0, 5, 22]
    got_rows = O.prefill_attention(q, k, v, rows=rows)
    np.testing.assert_allclose(got_rows, ref[:, :, rows], atol=1e-12)


def test_single_token_returns_value_row():
    rng = _rng(4)
    q = rng.standard_normal((2, 4, 8))
    k = rng.standard_normal((2, 2, 5, 8))
    v = rng.standard_normal((2, 2, 5, 8))
    out = O.decode_attention(q, k, v, [1, 1])
    for b in range(2):
        for h in range(4):
            np.testing.assert_array_equal(out[b, h], v[b, h // 2, 0])


def test_zero_query_returns_mean_value():
    rng = _rng(5)
    q = np.zeros((1, 2, 8))
    k = rng.standard_normal((1, 1, 11, 8))
    v = rng.standard_normal((1, 1, 11, 8))
    out = O.decode_attention(q, k, v, [7])
    np.testing.assert_allclose(out[0, 0], v[0, 0, :7].mean(0), atol=1e-14)
    np.testing.assert_allclose(out[0, 1], v[0, 0, :7].mean(0), atol=1e-14)


def test_prefill_first_row_is_first_value():
    rng = _rng(6)
    q = rng.standard_normal((1, 2, 4, 8))
    k = rng.standard_normal((1, 1, 4, 8))
    v = rng.standard_normal((1, 1, 4, 8))
    out = O.prefill_attention(q, k, v)
    np.testing.assert_array_equal(out[0, 0, 0], v[0, 0, 0])


def test_decode_rejects_empty_and_overlong():
    q = np.zeros((1, 1, 4))
    k = np.zeros((1, 1, 3, 4))
    with pytest.raises(ValueError):
        O.decode_attention(q, k, k, [0])
    with pytest.raises(ValueError):
        O.decode_attention(q, k, k, [4])


# --------------------------------------------------------------------------
# reconstruction ([Slides] Eqs.(4)-(6))
# --------------------------------------------------------------------------

def test_lite_equals_fused_with_zero_one_weights():
    rng = _rng(7)
    L, B, H_kv, S, D = 4, 2, 2, 19, 8
    kc, vc = _caches(rng, L, B, H_kv, S, D, layers=[1, 2])
    q = rng.standard_normal((B, 2 * H_kv, D))
    z, o = np.zeros((H_kv, D)), np.ones((H_kv, D))
    lens = [19, 6]
    for layer in (3, 4):
        lite = O.decode_attn(q, layer, L, O.LITE, kc, vc, lens)
        fused = O.decode_attn(q, layer, L, O.FUSED, kc, vc, lens, weights={layer: (z, o, o, z)})
        np.testing.assert_array_equal(lite, fused)


def test_fused_unit_weights_select_sources():
    """(a1, an, b1, bn) = (1, 0, 0, 1) is attention over (K^1, V^n): pins which
    weight goes with which source."""
    rng = _rng(8)
    L, B, H_kv, S, D = 6, 1, 2, 13, 8
    n = 3
    kc, vc = _caches(rng, L, B, H_kv, S, D, layers=[1, 2, 3])
    q = rng.standard_normal((B, 2 * H_kv, D))
    z, o = np.zeros((H_kv, D)), np.ones((H_kv, D))
    got = O.decode_attn(q, 5, L, O.FUSED, kc, vc, [13], weights={5: (o, z, z, o)})
    ref = _sdpa(q[:, :, None], kc[1], vc[n])[:, :, 0]
    np.testing.assert_allclose(got, ref, atol=1e-12)


def test_fused_constant_weights_match_sdpa_on_summed_caches():
    rng = _rng(9)
    L, B, H_kv, S, D = 4, 2, 2, 17, 8
    kc, vc = _caches(rng, L, B, H_kv, S, D, layers=[1, 2])
    q = rng.standard_normal((B, 4, D))
    c = (0.7, -1.3, 2.1, -0.4)
    ws = tuple(np.full((H_kv, D), x) for x in c)
    got = O.decode_attn(q, 3, L, O.FUSED, kc, vc, [17, 17], weights={3: ws})
    ref = _sdpa(q[:, :, None], c[0] * kc[1] + c[1] * kc[2], c[2] * vc[1] + c[3] * vc[2])[:, :, 0]
    np.testing.assert_allclose(got, ref, atol=1e-12)


def test_fused_per_head_channel_weights_match_sdpa():
    """Channel weights differ per (head, channel) and are broadcast over batch
    and tokens ([Slides] 'learned vectors broadcast over tokens')."""
    rng = _rng(10)
    L, B, H_kv, S, D = 4, 2, 2, 9, 6
    kc, vc = _caches(rng, L, B, H_kv, S, D, layers=[1, 2])
    q = rng.standard_normal((B, 4, D))
    ws = _weights(rng, H_kv, D, tie=False)
    got = O.decode_attn(q, 4, L, O.FUSED, kc, vc, [9, 9], weights={4: ws})
    k_i = np.empty_like(kc[1])
    v_i = np.empty_like(vc[1])
    for b in range(B):
        for h in range(H_kv):
            for t in range(S):
                k_i[b, h, t] = ws[0][h] * kc[1][b, h, t] + ws[1][h] * kc[2][b, h, t]
                v_i[b, h, t] = ws[2][h] * vc[1][b, h, t] + ws[3][h] * vc[2][b, h, t]
    np.testing.assert_allclose(got, _sdpa(q[:, :, None], k_i, v_i)[:, :, 0], atol=1e-12)


def test_value_weights_act_linearly():
    """For fixed scores, o(b1 V1 + bn Vn) = b1 o(V1) + bn o(Vn) (Eq.(5) is linear)."""
    rng = _rng(11)
    L, B, H_kv, S, D = 4, 1, 1, 15, 8
    kc, vc = _caches(rng, L, B, H_kv, S, D, layers=[1, 2])
    q = rng.standard_normal((B, 2, D))
    a1, an, b1, bn = _weights(rng, H_kv, D)
    z = np.zeros_like(b1)
    full = O.decode_attn(q, 3, L, O.FUSED, kc, vc, [15], weights={3: (a1, an, b1, bn)})
    only1 = O.decode_attn(q, 3, L, O.FUSED, kc, vc, [15], weights={3: (a1, an, np.ones_like(b1), z)})
    onlyn = O.decode_attn(q, 3, L, O.FUSED, kc, vc, [15], weights={3: (a1, an, z, np.ones_like(bn))})
    np.testing.assert_allclose(full, b1[0] * only1 + bn[0] * onlyn, atol=1e-12)


def test_negative_and_unnormalised_weights_accepted():
    rng = _rng(12)
    L = 4
    kc, vc = _caches(rng, L, 1, 1, 5, 4, layers=[1, 2])
    q = rng.standard_normal((1, 1, 4))
    ws = tuple(np.full((1, 4), x) for x in (-3.0, 5.0, -2.0, 7.5))
    out = O.decode_attn(q, 3, L, O.FUSED, kc, vc, [5], weights={3: ws})
    assert np.all(np.isfinite(out))


@pytest.mark.parametrize("mode", (O.VANILLA, O.LITE, O.FUSED))
@pytest.mark.parametrize("layer", [1, 2, 3, 4])
def test_brute_force_matches_vectorised_decode(mode, layer):
    rng = _rng(13)
    L, B, H_kv, S, D = 4, 2, 2, 7, 4
    kc, vc = _caches(rng, L, B, H_kv, S, D)
    q = rng.standard_normal((B, 4, D))
    ws = {l: _weights(rng, H_kv, D, tie=False) for l in (3, 4)}
    lens = [7, 3]
    a = O.decode_attn(q, layer, L, mode, kc, vc, lens, weights=ws)
    b = O.brute_force_decode(q, layer, L, mode, kc, vc, lens, weights=ws)
    np.testing.assert_allclose(a, b, atol=1e-12)


def test_brute_force_matches_vectorised_prefill():
    rng = _rng(14)
    q = rng.standard_normal((1, 4, 6, 4))
    k = rng.standard_normal((1, 2, 6, 4))
    v = rng.standard_normal((1, 2, 6, 4))
    np.testing.assert_allclose(O.prefill_attention(q, k, v), O.brute_force_prefill(q, k, v),
                               atol=1e-12)


def test_prefill_fused_uses_first_S_positions():
    rng = _rng(15)
    L, B, H_kv, Smax, S, D = 4, 1, 1, 12, 8, 4
    kc, vc = _caches(rng, L, B, H_kv, Smax, D, layers=[1, 2])
    q = rng.standard_normal((B, 2, S, D))
    ws = {3: _weights(rng, H_kv, D)}
    got = O.prefill_attn(q, 3, L, O.FUSED, kc, vc, weights=ws)
    a1, an, b1, bn = ws[3]
    k_i = a1[None, :, None] * kc[1][:, :, :S] + an[None, :, None] * kc[2][:, :, :S]
    v_i = b1[None, :, None] * vc[1][:, :, :S] + bn[None, :, None] * vc[2][:, :, :S]
    np.testing.assert_allclose(got, _sdpa(q, k_i, v_i, causal=True), atol=1e-12)


# --------------------------------------------------------------------------
# RoPE pair tying ([Slides] "Post-RoPE fusion needs paired key weights",
# Eqs.(7)-(8); [Notes] §2.4)
# --------------------------------------------------------------------------

def test_rope_is_a_rotation_with_relative_composition():
    rng = _rng(16)
    D = 16
    x = rng.standard_normal((5, D))
    y = rng.standard_normal((5, D))
    pos_x = np.array([0, 3, 10, 100, 7])
    pos_y = np.array([2, 3, 0, 50, 1000])
    rx, ry = O.rope_rotate_half(x, pos_x), O.rope_rotate_half(y, pos_y)
    # position 0 is the identity; norms are kept
    np.testing.assert_allclose(rx[0], x[0], atol=0)
    np.testing.assert_allclose(np.linalg.norm(rx, axis=1), np.linalg.norm(x, axis=1), atol=1e-12)
    # <R_m x, R_t y> = <x, R_{t-m} y>
    lhs = np.sum(rx * ry, axis=1)
    rhs = np.array([x[i] @ O.rope_rotate_half(y[i:i + 1], np.array([pos_y[i] - pos_x[i]]))[0]
                    for i in range(5)])
    np.testing.assert_allclose(lhs, rhs, atol=1e-10)
    # rotate-half pairs channel j with j + D/2: a rotation by pi/2 of pair 0
    e = np.zeros((1, D))
    e[0, 0] = 1.0
    th0 = O.rope_angles(np.array([1.0]), D)[0, 0]
    r = O.rope_rotate_half(e, np.array([1.0]))[0]
    assert r[0] == pytest.approx(math.cos(th0)) and r[D // 2] == pytest.approx(math.sin(th0))
    assert np.count_nonzero(np.abs(r) > 1e-15) == 2


def _scores_at_offset(q, k1, kn, a1, an, c):
    T = k1.shape[0]
    m = T - 1 + c
    return O.fused_key_scores(q, m, k1, kn, np.arange(T) + c, a1, an)


def test_tied_weights_make_scores_shift_invariant():
    rng = _rng(17)
    D, T = 32, 20
    q = rng.standard_normal(D)
    k1 = rng.standard_normal((T, D))
    kn = rng.standard_normal((T, D))
    a1, an, _, _ = (w[0] for w in _weights(rng, 1, D, tie=True))
    assert O.tied(a1) and O.tied(an)
    s0 = _scores_at_offset(q, k1, kn, a1, an, 0)
    for c in (1, 17, 4096):
        np.testing.assert_allclose(_scores_at_offset(q, k1, kn, a1, an, c), s0, atol=1e-10)


def test_untied_weights_break_shift_invariance_in_proportion():
    rng = _rng(18)
    D, T = 32, 20
    q = rng.standard_normal(D)
    k1 = rng.standard_normal((T, D))
    kn = rng.standard_normal((T, D))
    a1, an, _, _ = (w[0] for w in _weights(rng, 1, D, tie=True))
    delta = rng.standard_normal(D // 2)
    diffs = []
    for eps in (1.0, 0.1, 0.01):
        u = a1.copy()
        u[D // 2:] += eps * delta  # untie: w_j != w_{j+D/2}
        assert not O.tied(u)
        d = np.max(np.abs(_scores_at_offset(q, k1, kn, u, an, 37)
                          - _scores_at_offset(q, k1, kn, u, an, 0)))
        diffs.append(d)
    assert diffs[0] > 1e-3
    # the absolute-position term is proportional to (w_j - w_{j+D/2})
    assert diffs[1] == pytest.approx(diffs[0] * 0.1, rel=1e-6)
    assert diffs[2] == pytest.approx(diffs[0] * 0.01, rel=1e-6)


# --------------------------------------------------------------------------
# cache capacity / I/O ([Slides] Table 1; [Notes] §2.5 element counts)
# --------------------------------------------------------------------------

def test_table1_capacity_and_io_ratios():
    g = _golden("table1_capacity_io.json")
    L, S, H, D = 16, 1000, 4, 64
    LSHD = L * S * H * D
    for m in (O.VANILLA, O.LITE, O.FUSED):   # the three methods of Table 1
        assert O.stored_elements(m, L, S, H, D) / O.stored_elements(O.VANILLA, L, S, H, D) \
            == g["capacity"][m]
        assert O.step_read_elements(m, L, S, H, D) / O.step_read_elements(O.VANILLA, L, S, H, D) \
            == g["io"][m]
        assert O.step_read_elements(m, L, S, H, D) == g["elements_in_units_of_LSHD"][m + "_step"] * LSHD
    lower = sum(O.call_read_elements(l, O.FUSED, L, S, H, D) for l in range(1, L // 2 + 1))
    upper = sum(O.call_read_elements(l, O.FUSED, L, S, H, D) for l in range(L // 2 + 1, L + 1))
    assert lower == g["elements_in_units_of_LSHD"]["fused_lower_half"] * LSHD
    assert upper == g["elements_in_units_of_LSHD"]["fused_upper_half"] * LSHD
    # the plain element count of the pages: 2 L S H_kv D
    assert O.stored_elements(O.VANILLA, L, S, H, D) == 2 * LSHD


def test_gqa_composition_golden():
    g = _golden("composed_capacity.json")
    L, S, D, H_q = 8, 64, 16, 8
    mha = O.stored_elements(O.VANILLA, L, S, H_q, D)
    gqa = O.stored_elements(O.VANILLA, L, S, H_q // g["gqa_group"], D)
    fkv = O.stored_elements(O.FUSED, L, S, H_q // g["gqa_group"], D)
    assert gqa / mha == g["gqa_vs_mha"]
    assert fkv / mha == g["gqa_fusedkv_vs_mha"]
    # 4-bit payload on top of FusedKV, against fp16 vanilla with the same heads
    van = O.stored_elements(O.VANILLA, L, S, H_q // g["gqa_group"], D)
    assert (fkv * 4) / (van * 16) == g["fusedkv_4bit_vs_fp16_vanilla"]


# --------------------------------------------------------------------------
# append ([Notes] §2.3: new tokens enter the storage caches first)
# --------------------------------------------------------------------------

def test_append_writes_rows_at_offsets_only():
    rng = _rng(19)
    cache = rng.standard_normal((2, 2, 10, 4))
    new = rng.standard_normal((2, 2, 3, 4))
    out = O.append_kv(cache, new, [0, 7])
    np.testing.assert_array_equal(out[0, :, 0:3], new[0])
    np.testing.assert_array_equal(out[1, :, 7:10], new[1])
    np.testing.assert_array_equal(out[0, :, 3:], cache[0, :, 3:])
    np.testing.assert_array_equal(out[1, :, :7], cache[1, :, :7])
    with pytest.raises(ValueError):
        O.append_kv(cache, new, [8, 0])


# --------------------------------------------------------------------------
# chunked prefill over an existing cache (a prompt continued in chunks)
# --------------------------------------------------------------------------

def test_chunk_prefill_matches_sdpa_with_offset_mask():
    """Library pin: SDPA with an explicit boolean mask allowing key t for
    query i iff t <= q_start + i."""
    rng = _rng(20)
    B, H_kv, G, D, q_start, C = 2, 2, 2, 8, 11, 7
    n = q_start + C
    q = rng.standard_normal((B, H_kv * G, C, D))
    k = rng.standard_normal((B, H_kv, n + 3, D))
    v = rng.standard_normal((B, H_kv, n + 3, D))
    got = O.chunk_prefill_attention(q, q_start, k, v)
    mask = torch.tensor([[t <= q_start + i for t in range(n)] for i in range(C)])
    qt = torch.from_numpy(q)
    kt = torch.from_numpy(k[:, :, :n]).repeat_interleave(G, dim=1)
    vt = torch.from_numpy(v[:, :, :n]).repeat_interleave(G, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask).numpy()
    np.testing.assert_allclose(got, ref, atol=1e-12)


def test_chunks_reassemble_full_prefill_and_last_row_is_decode():
    rng = _rng(21)
    L, B, H_kv, S, D = 4, 1, 2, 30, 8
    kc, vc = _caches(rng, L, B, H_kv, S, D, layers=[1, 2])
    ws = {3: _weights(rng, H_kv, D)}
    q = rng.standard_normal((B, 4, S, D))
    full = O.prefill_attn(q, 3, L, O.FUSED, kc, vc, weights=ws)
    parts = [O.chunk_prefill_attn(q[:, :, a:b], a, 3, L, O.FUSED, kc, vc, weights=ws)
             for a, b in ((0, 9), (9, 10), (10, 30))]
    np.testing.assert_allclose(np.concatenate(parts, axis=2), full, atol=1e-12)
    last = O.decode_attn(q[:, :, S - 1], 3, L, O.FUSED, kc, vc, [S], weights=ws)
    np.testing.assert_allclose(full[:, :, S - 1], last, atol=1e-12)


# --------------------------------------------------------------------------
# source-layer choice ([Slides] Table 17, Fig.8): lite with other sources,
# reversed sharing, single-source channel scaling
# --------------------------------------------------------------------------

def test_lite_sources_override_selects_caches():
    rng = _rng(22)
    L, B, H_kv, S, D = 8, 1, 2, 12, 8
    kc, vc = _caches(rng, L, B, H_kv, S, D, layers=[1, 2, 3, 4])
    q = rng.standard_normal((B, 4, D))
    for ks, vs in (((3,), (1,)), ((1,), (4,)), ((2,), (2,))):
        got = O.decode_attn(q, 6, L, O.LITE, kc, vc, [S], k_sources=ks, v_sources=vs)
        ref = _sdpa(q[:, :, None], kc[ks[0]], vc[vs[0]])[:, :, 0]
        np.testing.assert_allclose(got, ref, atol=1e-12)
    # the default lite sources are K^n, V^1
    np.testing.assert_allclose(O.decode_attn(q, 6, L, O.LITE, kc, vc, [S]),
                               _sdpa(q[:, :, None], kc[4], vc[1])[:, :, 0], atol=1e-12)


def test_fused_sources_override():
    rng = _rng(23)
    L, B, H_kv, S, D = 8, 1, 1, 10, 4
    kc, vc = _caches(rng, L, B, H_kv, S, D, layers=[1, 2, 3, 4])
    q = rng.standard_normal((B, 2, D))
    c = (0.3, 1.7, -0.5, 2.0)
    ws = {7: tuple(np.full((H_kv, D), x) for x in c)}
    got = O.decode_attn(q, 7, L, O.FUSED, kc, vc, [S], weights=ws, k_sources=(2, 3),
                        v_sources=(4, 1))
    ref = _sdpa(q[:, :, None], c[0] * kc[2] + c[1] * kc[3], c[2] * vc[4] + c[3] * vc[1])[:, :, 0]
    np.testing.assert_allclose(got, ref, atol=1e-12)


def test_scaled_is_lite_with_unit_weights_and_fused_with_zero_second():
    rng = _rng(24)
    L, B, H_kv, S, D = 4, 2, 2, 15, 8
    kc, vc = _caches(rng, L, B, H_kv, S, D, layers=[1, 2])
    q = rng.standard_normal((B, 4, D))
    ones = tuple(np.ones((H_kv, D)) for _ in range(4))
    np.testing.assert_array_equal(
        O.decode_attn(q, 3, L, O.SCALED, kc, vc, [15, 6], weights={3: ones}),
        O.decode_attn(q, 3, L, O.LITE, kc, vc, [15, 6]))
    a1, an, b1, bn = _weights(rng, H_kv, D, tie=False)
    z = np.zeros_like(a1)
    got = O.decode_attn(q, 3, L, O.SCALED, kc, vc, [15, 6], weights={3: (a1, an, b1, bn)},
                        k_sources=(1,), v_sources=(2,))
    ref = O.decode_attn(q, 3, L, O.FUSED, kc, vc, [15, 6], weights={3: (a1, z, b1, z)},
                        k_sources=(1, 2), v_sources=(2, 1))
    np.testing.assert_allclose(got, ref, atol=1e-12)
    # and against SDPA on explicitly scaled caches
    ks = a1[None, :, None, :] * kc[1]
    vs = b1[None, :, None, :] * vc[2]
    np.testing.assert_allclose(got, _sdpa(q[:, :, None], ks, vs, lens=[15, 6])[:, :, 0], atol=1e-12)


# --------------------------------------------------------------------------
# sliding-window layers (hybrid SWA of [Slides] "MoE and hybrid SWA": window
# 512, three window layers per full-attention layer)
# --------------------------------------------------------------------------

def test_window_decode_matches_sdpa_on_last_rows_and_special_cases():
    rng = _rng(25)
    B, H_kv, S, D = 3, 2, 40, 8
    q = rng.standard_normal((B, 4, D))
    k = rng.standard_normal((B, H_kv, S, D))
    v = rng.standard_normal((B, H_kv, S, D))
    lens = [40, 7, 25]
    for W in (1, 5, 7, 64):
        got = O.decode_attention(q, k, v, lens, window=W)
        for b, n in enumerate(lens):
            lo = max(0, n - W)
            ref = _sdpa(q[b:b + 1, :, None], k[b:b + 1, :, lo:n], v[b:b + 1, :, lo:n])[0, :, 0]
            np.testing.assert_allclose(got[b], ref, atol=1e-12)
    # window 1: the newest value row; a window at least len: full attention
    w1 = O.decode_attention(q, k, v, lens, window=1)
    for b, n in enumerate(lens):
        np.testing.assert_array_equal(w1[b, 0], v[b, 0, n - 1])
    np.testing.assert_array_equal(O.decode_attention(q, k, v, lens, window=40),
                                  O.decode_attention(q, k, v, lens))


def test_window_prefill_matches_sdpa_band_mask():
    rng = _rng(26)
    B, H_kv, S, D, W = 1, 2, 30, 8, 6
    q = rng.standard_normal((B, 4, S, D))
    k = rng.standard_normal((B, H_kv, S, D))
    v = rng.standard_normal((B, H_kv, S, D))
    got = O.prefill_attention(q, k, v, window=W)
    mask = torch.tensor([[m - W < t <= m for t in range(S)] for m in range(S)])
    qt = torch.from_numpy(q)
    kt = torch.from_numpy(k).repeat_interleave(2, dim=1)
    vt = torch.from_numpy(v).repeat_interleave(2, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask).numpy()
    np.testing.assert_allclose(got, ref, atol=1e-12)
    # chunked, windowed: rows of the full windowed prefill
    part = O.chunk_prefill_attention(q[:, :, 11:20], 11, k, v, window=W)
    np.testing.assert_allclose(part, got[:, :, 11:20], atol=1e-12)


# --------------------------------------------------------------------------
# 4-bit KV cache ([Slides] Table 14); the grouping is this library's reading
# --------------------------------------------------------------------------

def test_bf16_round_matches_torch():
    rng = _rng(27)
    x = (rng.standard_normal(10000) * 10 ** rng.uniform(-5, 5, 10000)).astype(np.float32)
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0]   # exact ties
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(O.bf16_round(x), ref)


def test_q4_error_bound_codes_and_grid():
    rng = _rng(28)
    x = O.bf16_round(rng.standard_normal((7, 3, 64)).astype(np.float32))
    codes, scale, lo = O.q4_quantize(x)
    assert codes.dtype == np.uint8 and codes.max() <= 15
    xh = O.q4_dequantize(codes, scale, lo)
    # |x - x_hat| <= scale / 2 (+ the scale's own bf16 rounding over 15 steps)
    s = np.repeat(scale, O.Q4_GROUP, axis=-1).astype(np.float64)
    hi = np.repeat(x.reshape(7, 3, 4, 16).max(-1), 16, axis=-1)
    bound = 0.5 * s + np.abs(hi - (np.repeat(lo, 16, -1) + 15 * s)) + 1e-12
    assert np.all(np.abs(x - xh) <= bound)
    # values already on the grid round-trip exactly
    again = O.q4_quantize(O.bf16_round(xh.astype(np.float32)))
    np.testing.assert_array_equal(O.q4_dequantize(*again), O.q4_dequantize(codes, scale, lo))
    # a constant group stores code 0 and dequantises exactly
    cst = np.full((1, 16), 1.5, np.float32)
    c2, s2, l2 = O.q4_quantize(cst)
    assert np.all(c2 == 0) and s2[0, 0] == 0 and np.all(O.q4_dequantize(c2, s2, l2) == 1.5)


def test_q4_pack_roundtrip_and_layout():
    rng = _rng(29)
    for D in (64, 80, 96, 128):
        x = O.bf16_round(rng.standard_normal((2, 5, D)).astype(np.float32))
        codes, scale, lo = O.q4_quantize(x)
        rec = O.q4_pack(codes, scale, lo)
        assert rec.shape[-1] == O.q4_row_bytes(D) and rec.shape[-1] % 16 == 0
        c2, s2, l2 = O.q4_unpack(rec, D)
        np.testing.assert_array_equal(c2, codes)
        np.testing.assert_array_equal(s2, scale)
        np.testing.assert_array_equal(l2, lo)
        # byte 0 holds channel 0 (low nibble) and channel 1 (high nibble)
        assert rec[0, 0, 0] == codes[0, 0, 0] | (codes[0, 0, 1] << 4)
    assert [O.q4_row_bytes(d) for d in (64, 80, 96, 128)] == [48, 64, 80, 96]


def test_q4_attention_is_attention_over_dequantised_caches():
    rng = _rng(30)
    L, B, H_kv, S, D = 4, 1, 2, 20, 32
    kc, vc = _caches(rng, L, B, H_kv, S, D, layers=[1, 2])
    kq = {l: O.q4_dequantize_records(O.q4_pack(*O.q4_quantize(O.bf16_round(k.astype(np.float32)))), D)
          for l, k in kc.items()}
    vq = {l: O.q4_dequantize_records(O.q4_pack(*O.q4_quantize(O.bf16_round(v.astype(np.float32)))), D)
          for l, v in vc.items()}
    q = rng.standard_normal((B, 4, D))
    ws = {3: _weights(rng, H_kv, D)}
    got = O.decode_attn(q, 3, L, O.FUSED, kq, vq, [S], weights=ws)
    full = O.decode_attn(q, 3, L, O.FUSED, kc, vc, [S], weights=ws)
    # 4-bit noise, not a different function: close to the unquantised result
    assert np.max(np.abs(got - full)) < 0.2


# Closed-form cases of the 4-bit quantiser, worked by hand from its stated
# definition (min of the group; scale = bf16((max - min) / 15) with the
# division in fp32; code = clamp(rint((x - min) / scale), 0, 15), rint rounding
# halves to even).  [Slides] "Four-bit KV quantization is the stronger
# combination", Table 14, names 4-bit KV caches; the grouping and code are
# this library's reading.  Each case pins the step size: a divisor of 14 or
# 16 in place of 15 changes the stored scale and at least one code.
_Q4_CASES = [
    # 0, 0.5, ..., 7.5: (7.5 - 0) / 15 = 0.5 exactly, codes 0..15
    ("grid", [0.5 * j for j in range(16)], 0.5, 0.0, list(range(16))),
    # span 30 from -10: scale 2.0; (x + 10) / 2 hits many halves, which
    # round to even (7.5 -> 8, 0.5 -> 0, 14.5 -> 14, 5.5 -> 6, 6.5 -> 6,
    # 8.5 -> 8, 9.5 -> 10, 10.5 -> 10)
    ("ties", [-10, 20, 0, 5, -9, 19, 1, 2, 3, 4, 6, 7, 8, 9, 10, 11], 2.0, -10.0,
     [0, 15, 5, 8, 0, 14, 6, 6, 6, 7, 8, 8, 9, 10, 10, 10]),
    # span 1: 1/15 = 2^-4 * 1.0666..; to 8 significant bits 2^-4 * (1 + 9/128)
    # = 0.06689453125.  x / scale: 1 -> 14.95, 0.5 -> 7.47, 0.25 -> 3.74,
    # 0.75 -> 11.21, 0.125 -> 1.87, 0.375 -> 5.61, 0.625 -> 9.34, 0.875 -> 13.08
    ("inexact", [0, 1, 0.5, 0.25, 0.75, 0.125, 0.375, 0.625, 0.875, 0, 1, 0.5, 0.25, 0.75,
                 0.125, 0.375], 0.06689453125, 0.0,
     [0, 15, 7, 4, 11, 2, 6, 9, 13, 0, 15, 7, 4, 11, 2, 6]),
    # negative span 1.5 from -3: 0.1 in fp32 is 0x3DCCCCCD, which rounds up to
    # the bf16 0x3DCD = 0.10009765625.  (x + 3) / scale: 1.5 -> 14.99,
    # 0.75 -> 7.49, 1 -> 9.99, 0.5 -> 4.995, 1.25 -> 12.49, 0.25 -> 2.498,
    # 1.375 -> 13.74
    ("negative", [-3, -1.5, -2.25, -2, -2.5, -1.75, -2.75, -1.625, -3, -1.5, -2.25, -2, -2.5,
                  -1.75, -2.75, -1.625], 0.10009765625, -3.0,
     [0, 15, 7, 10, 5, 12, 2, 14, 0, 15, 7, 10, 5, 12, 2, 14]),
]


@pytest.mark.parametrize("name,x,scale,lo,codes", _Q4_CASES, ids=[c[0] for c in _Q4_CASES])
def test_q4_quantiser_closed_form_cases(name, x, scale, lo, codes):
    xs = np.asarray(x, dtype=np.float32)[None, :]
    assert np.array_equal(O.bf16_round(xs), xs), "inputs must be bf16 values"
    c, s, m = O.q4_quantize(xs)
    assert float(s[0, 0]) == scale
    assert float(m[0, 0]) == lo
    assert c[0].tolist() == codes
    # the group's max reconstructs within 15 bf16 ulps of the scale (the
    # scale's own rounding, accumulated over the 15 steps)
    ulp = 2.0 ** (np.floor(np.log2(scale)) - 7)
    assert abs((lo + 15 * scale) - max(x)) <= 15 * ulp / 2 + 1e-12
    # two groups side by side keep their own parameters
    c2, s2, m2 = O.q4_quantize(np.concatenate([xs, xs[:, ::-1]], axis=1))
    assert s2[0].tolist() == [scale, scale] and m2[0].tolist() == [lo, lo]
    assert c2[0, 16:].tolist() == codes[::-1]
