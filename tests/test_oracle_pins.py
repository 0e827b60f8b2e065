"""Pins of the CPU oracle to things other than itself: number-format definitions
checked against torch's independent casts, closed forms, invariants the method's
definition fixes, brute force on tiny inputs, and a library softmax-attention
special case.  Each test is chosen so that a plausible mistake in the oracle (a
dropped term, a wrong sign or index, a transposed operand) fails it."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import csa_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))
rng = np.random.default_rng(1234)


# ----------------------------------------------------------------------------- e4m3 / bf16
def test_e4m3_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = O.decode_e4m3(codes)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert nan.sum() == 2                         # S.1111.111 only
    assert np.array_equal(ref[~nan], ours[~nan])
    assert O.decode_e4m3(np.uint8(0x7E)) == 448.0
    assert O.decode_e4m3(np.uint8(0x01)) == 2.0 ** -9


def test_e4m3_encode_roundtrip_and_rne_against_torch():
    finite = [c for c in range(256) if not np.isnan(O.E4M3_TABLE[c])]
    vals = O.E4M3_TABLE[finite]
    back = O.encode_e4m3(vals)
    # -0 and +0 both decode to 0; everything else must round-trip exactly
    for c, b in zip(finite, back):
        if O.E4M3_TABLE[c] == 0:
            assert b in (0x00, 0x80)
        else:
            assert b == c
    x = (rng.standard_normal(20000) * 60).astype(np.float32)
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.encode_e4m3(x.astype(np.float64)), ref)


def test_e4m3_midpoints_tie_to_even_and_saturate():
    pos = [c for c in range(0x7E)]
    for c in pos:
        lo, hi = O.E4M3_TABLE[c], O.E4M3_TABLE[c + 1]
        mid = (lo + hi) / 2
        got = int(O.encode_e4m3(np.array([mid]))[0])
        assert got == (c if c % 2 == 0 else c + 1), (c, mid, got)
    assert O.encode_e4m3(np.array([500.0, -1e9, 449.0]))[0] == 0x7E
    assert O.encode_e4m3(np.array([-1e9]))[0] == 0xFE
    assert O.encode_e4m3(np.array([2.0 ** -11]))[0] == 0x00      # below half the least subnormal
    assert O.encode_e4m3(np.array([3 * 2.0 ** -11]))[0] == 0x01  # above half


def test_bf16_codec_against_torch():
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.encode_bf16(x.astype(np.float64)), ref)
    back = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.decode_bf16(ref), back)
    # midpoint between 1 and 1+2^-7 ties to even (1.0); next midpoint ties up
    assert O.encode_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80
    assert O.encode_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82


# ----------------------------------------------------------------------------- rotary embedding
def test_rope_position_zero_is_identity_and_norm_preserved():
    v = rng.standard_normal((5, 128))
    assert np.array_equal(O.rope(v, 0, 64, 10000.0), v)
    r = O.rope(v, 123457, 64, 10000.0)
    assert np.allclose(np.linalg.norm(r, axis=1), np.linalg.norm(v, axis=1), rtol=0, atol=1e-12)
    assert np.array_equal(r[:, :64], v[:, :64])       # only the last 64 dims turn


def test_rope_closed_form_pairs():
    # d_rope = 4, theta = 10000: pair 0 turns by p, pair 1 by p * 10000^(-1/2) = p / 100
    v = np.array([7.0, 1.0, 0.0, 1.0, 0.0])
    p = 3
    r = O.rope(v, p, 4, 10000.0)
    assert r[0] == 7.0
    assert np.allclose(r[1:3], [math.cos(p), math.sin(p)], atol=1e-15)
    assert np.allclose(r[3:5], [math.cos(p / 100), math.sin(p / 100)], atol=1e-15)
    # the pair is (x, y) -> (x cos - y sin, x sin + y cos)
    r2 = O.rope(np.array([0.0, 1.0]), 0.5, 2, 10000.0)
    assert np.allclose(r2, [-math.sin(0.5), math.cos(0.5)], atol=1e-15)


def test_rope_relative_position_identity():
    q = rng.standard_normal(64)
    k = rng.standard_normal(64)
    for p, pp in [(1000, 10), (1 << 20, (1 << 20) - 127), (5, 5)]:
        lhs = O.rope(q, p, 64, 10000.0) @ O.rope(k, pp, 64, 10000.0)
        rhs = O.rope(q, p - pp, 64, 10000.0) @ k
        assert abs(lhs - rhs) < 1e-9 * (1 + abs(rhs))


# ----------------------------------------------------------------------------- pooling
def test_pool_m1_is_identity():
    x = rng.standard_normal((1, 16))
    g = rng.standard_normal((1, 16))
    assert np.allclose(O.pool_block(x, g, np.array([0.3])), x[0], rtol=0, atol=1e-15)


def test_pool_equal_logits_give_mean_and_dominant_gives_copy():
    x = rng.standard_normal((4, 8))
    assert np.allclose(O.pool_block(x, np.zeros((4, 8)), np.zeros(4)), x.mean(axis=0), atol=1e-15)
    g = np.zeros((4, 8))
    g[2, :] = 100.0
    assert np.allclose(O.pool_block(x, g, np.zeros(4)), x[2], atol=1e-30 + 1e-40)
    # a dominant slot bias selects that slot in every channel
    assert np.allclose(O.pool_block(x, np.zeros((4, 8)), np.array([0, 0, 0, 200.0])), x[3])


def test_pool_m2_closed_form_and_shift_invariance():
    x = rng.standard_normal((2, 6))
    g = rng.standard_normal((2, 6))
    b = np.array([0.4, -0.7])
    l0, l1 = g[0] + b[0], g[1] + b[1]
    a0 = 1 / (1 + np.exp(-(l0 - l1)))
    assert np.allclose(O.pool_block(x, g, b), a0 * x[0] + (1 - a0) * x[1], atol=1e-14)
    # adding a constant to a channel's logits changes nothing
    assert np.allclose(O.pool_block(x, g + 5.0, b), O.pool_block(x, g, b), atol=1e-14)


def test_pool_brute_force_loops():
    m, d = 5, 7
    x = rng.standard_normal((m, d))
    g = rng.standard_normal((m, d))
    b = rng.standard_normal(m) * 0.5
    out = np.zeros(d)
    for c in range(d):
        ws = [math.exp(g[i, c] + b[i]) for i in range(m)]
        tot = sum(ws)
        out[c] = sum(ws[i] / tot * x[i, c] for i in range(m))
    assert np.allclose(O.pool_block(x, g, b), out, atol=1e-14)


# ----------------------------------------------------------------------------- quantisation
def test_quantise_scale_and_extreme_code():
    v = rng.standard_normal(448) * 3
    codes, s = O.quantise_e4m3(v)
    assert s == np.float32(np.float32(np.abs(v).max()) / np.float32(448))
    j = int(np.argmax(np.abs(v)))
    assert abs(O.decode_e4m3(codes[j])) == 448.0
    deq = O.decode_e4m3(codes) * float(s)
    # error at most half a code step (relative 2^-4) plus the subnormal floor
    assert np.all(np.abs(deq - v) <= np.abs(v) * 2.0 ** -4 + float(s) * 2.0 ** -10 + 1e-12)
    c0, s0 = O.quantise_e4m3(np.zeros(8))
    assert s0 == 1.0 and not c0.any()


def test_compress_entries_follow_block_layout():
    m, d, dr = 4, 16, 8
    T = 12
    x = rng.standard_normal((T, d))
    g = rng.standard_normal((T, d))
    b = rng.standard_normal(m)
    out = O.compress_entries(x, g, b, m, dr, 10000.0, "f32", 1, 2)
    e1 = O.rope(O.pool_block(x[4:8], g[4:8], b), 4, dr, 10000.0)
    assert np.allclose(out["kv_nope"][0], e1[:8].astype(np.float32))
    assert np.allclose(out["kv_rope"][0], e1[8:].astype(np.float32))
    e2 = O.rope(O.pool_block(x[8:12], g[8:12], b), 8, dr, 10000.0)
    assert np.allclose(out["kv_rope"][1], e2[8:].astype(np.float32))


# ----------------------------------------------------------------------------- indexer and top-k
def test_indexer_one_head_one_hot_and_negative():
    k = rng.standard_normal((50, 16))
    q = rng.standard_normal((1, 16))
    s = O.indexer_scores(q, np.array([1.0]), k)
    assert np.allclose(s, np.maximum(k @ q[0], 0))
    q3 = rng.standard_normal((3, 16))
    s3 = O.indexer_scores(q3, np.array([0.0, 1.0, 0.0]), k)
    assert np.allclose(s3, np.maximum(k @ q3[1], 0))
    assert not O.indexer_scores(-np.abs(q), np.array([1.0]), np.abs(k)).any()


def test_indexer_brute_force():
    H, dI, N = 3, 5, 9
    q = rng.standard_normal((H, dI))
    w = rng.uniform(0, 1, H)
    k = rng.standard_normal((N, dI))
    ref = [sum(w[h] * max(0.0, sum(q[h, c] * k[j, c] for c in range(dI))) for h in range(H)) for j in range(N)]
    assert np.allclose(O.indexer_scores(q, w, k), ref, atol=1e-13)


def test_topk_brute_force_with_ties():
    for trial in range(200):
        n = int(rng.integers(1, 40))
        k = int(rng.integers(1, 45))
        sc = rng.integers(0, 6, n).astype(np.float64)      # many ties
        idx, cnt = O.topk(sc, k)
        assert cnt == min(n, k)
        sel = idx[:cnt]
        assert np.all(np.diff(sel) > 0) and np.all(idx[cnt:] == -1)
        # brute force: j is selected iff fewer than k entries beat it, where
        # (score, -index) is the order
        for j in range(n):
            beaten = sum(1 for i in range(n) if sc[i] > sc[j] or (sc[i] == sc[j] and i < j))
            assert (j in set(sel.tolist())) == (beaten < k)


def test_visible_entries():
    assert O.visible_entries(3, 4) == 1
    assert O.visible_entries(2, 4) == 0
    assert O.visible_entries(4095, 4) == 1024
    assert O.visible_entries((1 << 20), 4) == (1 << 18)
    assert O.visible_entries(127, 128) == 1


# ----------------------------------------------------------------------------- attention
def _plain_attention_torch(q, kv, d):
    qt, kt = torch.from_numpy(q), torch.from_numpy(kv)
    p = torch.softmax(qt @ kt.T / math.sqrt(d), dim=-1)
    return (p @ kt).numpy(), torch.logsumexp(qt @ kt.T / math.sqrt(d), dim=-1).numpy()


def test_attention_reduces_to_library_softmax_attention():
    H, d, n = 4, 32, 20
    q = rng.standard_normal((H, d))
    ent = rng.standard_normal((n, d))
    sink = np.full(H, -np.inf)
    o, lse = O.attend(q, 0, ent, np.zeros((0, d)), np.zeros(0, np.int64), sink, 16, 10000.0)
    ro, rl = _plain_attention_torch(q, ent, d)      # position 0: rope is the identity on q
    assert np.allclose(o, ro, atol=1e-12) and np.allclose(lse, rl, atol=1e-12)


def test_attention_sink_mass_and_equal_keys():
    H, d = 3, 16
    q = rng.standard_normal((H, d))
    v = rng.standard_normal(d)
    ent = np.tile(v, (7, 1))
    sink = rng.standard_normal(H)
    o, lse = O.attend(q, 0, ent, np.zeros((0, d)), np.zeros(0, np.int64), sink, 0, 10000.0)
    p_sink = np.exp(sink - lse)
    assert np.all((p_sink > 0) & (p_sink < 1))
    assert np.allclose(o, (1 - p_sink)[:, None] * v[None, :], atol=1e-13)
    # lse brute force: log(7 exp(q.v/sqrt d) + exp(z))
    ref = np.log(7 * np.exp(q @ v / math.sqrt(d)) + np.exp(sink))
    assert np.allclose(lse, ref, atol=1e-12)


def test_attention_permutation_invariance_and_window_shift():
    H, d, dr = 2, 24, 8
    q = rng.standard_normal((H, d))
    ent = rng.standard_normal((9, d))
    sink = rng.standard_normal(H)
    perm = rng.permutation(9)
    a = O.attend(q, 50, ent, np.zeros((0, d)), np.zeros(0, np.int64), sink, dr, 10000.0)
    b = O.attend(q, 50, ent[perm], np.zeros((0, d)), np.zeros(0, np.int64), sink, dr, 10000.0)
    assert np.allclose(a[0], b[0], atol=1e-13) and np.allclose(a[1], b[1], atol=1e-13)
    # window tokens rotate at their own positions: logits depend on t - tau only,
    # so lse is unchanged when the query and its window move together
    win = rng.standard_normal((5, d))
    l1 = O.attend(q, 100, np.zeros((0, d)), win, np.arange(96, 101), sink, dr, 10000.0)[1]
    l2 = O.attend(q, 70100, np.zeros((0, d)), win, np.arange(70096, 70101), sink, dr, 10000.0)[1]
    assert np.allclose(l1, l2, atol=1e-9)
    # ...but not when only the query moves
    l3 = O.attend(q, 101, np.zeros((0, d)), win, np.arange(96, 101), sink, dr, 10000.0)[1]
    assert not np.allclose(l1, l3, atol=1e-6)


def test_csa_with_all_entries_selected_equals_hca():
    H, d, dr, m, n_win = 4, 32, 16, 4, 6
    n_e = 10
    t = n_e * m + 2
    q = rng.standard_normal((H, d))
    ent = rng.standard_normal((n_e, d))
    keys = rng.standard_normal((n_e, 8))
    qi = rng.standard_normal((2, 8))
    wi = rng.uniform(0, 1, 2)
    sink = rng.standard_normal(H)
    raw = {p: rng.standard_normal(d) for p in range(t + 1)}
    wf = lambda pos: np.array([raw[int(p)] for p in pos])
    csa = O.query_step("csa", q, t, sink, ent, wf, m, n_win, dr, 10000.0, qi, wi, keys, k=n_e + 5)
    hca = O.query_step("hca", q, t, sink, ent, wf, m, n_win, dr, 10000.0)
    assert csa["count"] == n_e
    assert np.allclose(csa["o"], hca["o"], atol=1e-13) and np.allclose(csa["lse"], hca["lse"], atol=1e-13)


def test_topk_planted_entries_win():
    H, dI, N = 8, 32, 400
    q = rng.standard_normal((H, dI))
    w = rng.uniform(0, 1, H)
    keys = rng.standard_normal((N, dI))
    dirv = (w[:, None] * q).sum(0)
    dirv /= np.linalg.norm(dirv)
    planted = rng.choice(N, 10, replace=False)
    keys[planted] += 12 * dirv
    idx, cnt = O.topk(O.indexer_scores(q, w, keys), 10)
    assert set(idx.tolist()) == set(planted.tolist())


# ----------------------------------------------------------------------------- page figures
def test_cache_layout_is_about_two_percent_of_bf16_gqa8():
    figs = json.load(open(os.path.join(HERE, "golden", "page_figures.json")))
    m_csa = figs["csa_compression_ratio"]["value"]
    m_hca = figs["hca_compression_ratio"]["value"]
    d, dr, d_idx = 512, 64, 128
    entry = (d - dr) * 1 + dr * 2 + 4            # e4m3 nope + bf16 rope + fp32 scale
    idx = d_idx + 4                               # e4m3 indexer key + scale
    csa = (entry + idx) / m_csa
    hca = entry / m_hca
    per_layer = (csa + hca) / 2                   # alternating layers
    gqa8 = 8 * 128 * 2 * 2                        # 8 kv heads x 128 dims x (K, V) x bf16
    ratio = per_layer / gqa8
    assert abs(ratio - figs["kv_cache_vs_bf16_gqa8"]["value"]) < 0.005, ratio
