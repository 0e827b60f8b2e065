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


# ----------------------------------------------------------------------------- window, paging, stored formats
def test_window_positions_hand_values():
    """The window of a query at t holds raw tokens max(0, t-W+1) .. t: the query's own
    token included, W tokens once t >= W-1."""
    assert O.window_positions(0, 128).tolist() == [0]
    assert O.window_positions(5, 128).tolist() == [0, 1, 2, 3, 4, 5]
    w = O.window_positions(200, 128)
    assert w[0] == 73 and w[-1] == 200 and len(w) == 128 and np.all(np.diff(w) == 1)
    assert O.window_positions(127, 128).tolist() == list(range(128))
    assert O.window_positions(9, 1).tolist() == [9]
    assert O.ring_slot(np.array([127, 128, 129, 300]), 128).tolist() == [127, 0, 1, 44]


def test_entry_rows_contiguous_and_paged_hand_table():
    # contiguous: sequence b owns rows [b*max_entries, (b+1)*max_entries)
    assert O.entry_rows(3, 2, 10, None, 0).tolist() == [20, 21, 22]
    # two pages of two entries per sequence, physical pages out of order
    pt = np.array([[3, 1], [0, 2]], dtype=np.int32)
    assert O.entry_rows(4, 0, 0, pt, 2).tolist() == [6, 7, 2, 3]
    assert O.entry_rows(3, 1, 0, pt, 2).tolist() == [0, 1, 4]


def test_decode_kv_scales_only_the_e4m3_dims_and_keeps_the_order():
    nope = np.array([[0x38, 0x40], [0xB8, 0x00]], dtype=np.uint8)     # 1, 2 | -1, 0
    scale = np.array([0.5, 4.0], dtype=np.float32)
    rope = np.array([[0x3F80], [0xC000]], dtype=np.uint16)             # 1 | -2 (bf16)
    got = O.decode_kv(nope, scale, rope, "e4m3")
    assert got.tolist() == [[0.5, 1.0, 1.0], [-4.0, 0.0, -2.0]]
    f = O.decode_kv(np.array([[1.5, -2.0]], np.float32), None, np.array([[7.0]], np.float32), "f32")
    assert f.tolist() == [[1.5, -2.0, 7.0]]
    k = O.decode_index_keys(np.array([[0x38, 0xC0]], np.uint8), np.array([0.25], np.float32), "e4m3")
    assert k.tolist() == [[0.25, -0.5]]


def test_e4m3_scale_subnormal_branch():
    tiny = np.finfo(np.float32).tiny
    assert O.e4m3_scale(np.array([1e-37, -3e-38])) == np.float32(1.0)    # amax/448 is subnormal
    assert O.e4m3_scale(np.array([448 * tiny])) == np.float32(tiny)      # smallest normal scale is kept
    assert O.e4m3_scale(np.array([0.0, -0.0])) == np.float32(1.0)
    assert O.e4m3_scale(np.array([-896.0, 3.0])) == np.float32(2.0)      # |.| of a negative amax


def test_compress_entries_e4m3_branch_hand_worked():
    """Two blocks of m = 2 tokens, d = 6 (4 e4m3 dims + 2 rotary dims), equal gates:
    each entry is the mean of its block.  Block 0 sits at position 0 (no turn); block
    1 at position 2 (its single rotary pair turns by 2 radians)."""
    x = np.array([[8, -2, 0, 6, 20, 0],
                  [0, 0, 0, 0, 0, 2],
                  [1, 1, 1, 1, 1, 0],
                  [1, 1, 1, 1, 1, 0]], dtype=np.float64)
    g = np.zeros_like(x)
    out = O.compress_entries(x, g, np.zeros(2), 2, 2, 10000.0, "e4m3", 0, 2)
    # block 0: mean nope [4, -1, 0, 3] -> scale fp32(4)/448 (the rotary dims [10, 1] do not
    # enter the scale); codes 448 -> 0x7E, -112 -> 0xEE, 0, 3/s just below 336 -> 320 -> 0x7A
    assert out["kv_scale"][0] == np.float32(np.float32(4.0) / np.float32(448.0))
    assert out["kv_nope"][0].tolist() == [0x7E, 0xEE, 0x00, 0x7A]
    assert out["kv_rope"][0].tolist() == [0x4120, 0x3F80]               # bf16 10, 1: not scaled
    # block 1: mean nope [1, 1, 1, 1] -> all 448; rotary pair (1, 0) at position 2
    assert out["kv_scale"][1] == np.float32(np.float32(1.0) / np.float32(448.0))
    assert out["kv_nope"][1].tolist() == [0x7E] * 4
    exp = O.encode_bf16(np.array([math.cos(2.0), math.sin(2.0)]))
    assert out["kv_rope"][1].tolist() == exp.tolist()


def test_compress_index_keys_own_bias_no_turn_own_scale():
    """Indexer keys pool with the bias they are given (here slot 1 dominates, so a key is
    its block's second token), are not rotated even at a nonzero position, and carry
    their own e4m3 scale."""
    ix = np.array([[9, 9, 9, 9],
                   [-2, 1, 0.5, 0],
                   [9, 9, 9, 9],
                   [3, -6, 1.5, 0]], dtype=np.float64)
    ig = np.zeros_like(ix)
    out = O.compress_index_keys(ix, ig, np.array([0.0, 50.0]), 2, "e4m3", 0, 2)
    s0 = np.float32(np.float32(2.0) / np.float32(448.0))
    s1 = np.float32(np.float32(6.0) / np.float32(448.0))
    assert out["idx_scale"].tolist() == [s0, s1]
    assert out["idx_key"][0].tolist() == [0xFE, 0x76, 0x6E, 0x00]       # -448, 224, 112, 0 (units of 2/448)
    assert out["idx_key"][1].tolist() == [0x76, 0xFE, 0x6E, 0x00]       # 224, -448, 112, 0
    f = O.compress_index_keys(ix, ig, np.array([0.0, 50.0]), 2, "f32", 1, 1)
    assert np.allclose(f["idx_key"][0], ix[3], rtol=0, atol=1e-12)


def test_query_step_brute_force_tiny():
    """One CSA query written out with loops: indexer scores over the visible entries,
    top-k with ties to the lower index, one softmax over the selected entries, the
    window (rotated at its positions) and the sink."""
    m, d, dr, n_win, k, theta = 2, 4, 2, 3, 2, 10000.0
    t = 9                                           # entries 0..4 visible, window 7, 8, 9
    n_e = 6
    ent = rng.standard_normal((n_e, d))
    keys = rng.standard_normal((n_e, 3))
    q = rng.standard_normal((2, d))
    qi = rng.standard_normal((2, 3))
    wi = np.array([0.7, 0.2])
    sink = np.array([0.3, -1.0])
    raw = {p: rng.standard_normal(d) for p in range(t + 1)}
    res = O.query_step("csa", q, t, sink, ent, lambda pos: np.array([raw[int(p)] for p in pos]), m, n_win, dr,
                       theta, qi, wi, keys, k=k)
    sc = [sum(wi[h] * max(0.0, sum(qi[h, c] * keys[j, c] for c in range(3))) for h in range(2)) for j in range(5)]
    order = sorted(range(5), key=lambda j: (-sc[j], j))[:k]

    def turn(v, p):
        a = p * theta ** 0.0
        return np.array([v[0], v[1], v[2] * math.cos(a) - v[3] * math.sin(a), v[2] * math.sin(a) + v[3] * math.cos(a)])

    kv = [ent[j] for j in sorted(order)] + [turn(raw[p], p) for p in (7, 8, 9)]
    for h in range(2):
        qh = turn(q[h], t)
        logits = [sum(qh[c] * v[c] for c in range(d)) / math.sqrt(d) for v in kv]
        den = sum(math.exp(x) for x in logits) + math.exp(sink[h])
        o = sum(math.exp(x) / den * v for x, v in zip(logits, kv))
        assert np.allclose(res["o"][h], o, rtol=0, atol=1e-12)
        assert abs(res["lse"][h] - math.log(den)) < 1e-12
    assert res["idx"].tolist() == sorted(order) and res["count"] == k
    assert np.allclose(res["scores"], sc, rtol=0, atol=1e-12)


def test_query_side_fp8_quantiser_hand_values():
    """The query-side FP8 variant: per head, the power of two S with max|q_h| S in
    [2^7, 2^8), then e4m3 rounding to nearest even.  q_h = (1, -0.3, 0, 0.01): S = 128,
    q S = (128, -38.4, 0, 1.28) -> e4m3 (128, -40, 0, 1.25) -> q' = (1, -0.3125, 0, 0.009765625)."""
    q = np.array([[1.0, -0.3, 0.0, 0.01],
                  [0.0, 0.0, 0.0, 0.0],
                  [-6.0, 3.0, 0.5, 2.5]])
    got = O.quantise_query_e4m3(q)
    assert got[0].tolist() == [1.0, -0.3125, 0.0, 1.25 / 128]
    assert not got[1].any()
    # head 2: max 6 -> S = 2^(8-3) = 32: 6*32 = 192 (exact), 96, 16, 80 -> all on the grid
    assert got[2].tolist() == [-6.0, 3.0, 0.5, 2.5]
    # every head lands on its scale's e4m3 grid, within half a step of q
    r = rng.standard_normal((8, 64)) * np.exp(rng.uniform(-8, 8, (8, 1)))
    qq = O.quantise_query_e4m3(r)
    for h in range(8):
        _, ex = math.frexp(np.abs(r[h]).max())
        s = 2.0 ** (8 - ex)
        assert 128 <= np.abs(r[h]).max() * s < 256
        codes = O.encode_e4m3(qq[h] * s)
        assert np.array_equal(O.decode_e4m3(codes), qq[h] * s)
        assert np.all(np.abs(qq[h] - r[h]) <= np.abs(r[h]) * 2.0 ** -4 + 2.0 ** -10 / s)


def test_window_only_layer_brute_force_and_relation_to_hca():
    """A sliding-window-only query: one softmax over the window tokens (rotated at their
    positions) and the sink, no entries -- written out with loops; and equal to HCA's
    result for a query that sees no complete block yet."""
    d, dr, n_win, theta = 4, 2, 3, 10000.0
    q = rng.standard_normal((2, d))
    sink = np.array([0.2, -0.4])
    raw = {p: rng.standard_normal(d) for p in range(12)}
    wf = lambda pos: np.array([raw[int(p)] for p in pos])

    def turn(v, p):
        return np.array([v[0], v[1], v[2] * math.cos(p) - v[3] * math.sin(p), v[2] * math.sin(p) + v[3] * math.cos(p)])

    for t in (0, 1, 11):
        res = O.query_step("swa", q, t, sink, np.zeros((0, d)), wf, 128, n_win, dr, theta)
        kv = [turn(raw[p], p) for p in range(max(0, t - n_win + 1), t + 1)]
        for h in range(2):
            qh = turn(q[h], t)
            lg = [float(qh @ v) / math.sqrt(d) for v in kv]
            den = sum(math.exp(x) for x in lg) + math.exp(sink[h])
            o = sum(math.exp(x) / den * v for x, v in zip(lg, kv))
            assert np.allclose(res["o"][h], o, rtol=0, atol=1e-12) and abs(res["lse"][h] - math.log(den)) < 1e-12
    ent = rng.standard_normal((5, d))
    a = O.query_step("swa", q, 2, sink, ent, wf, 4, n_win, dr, theta)
    b = O.query_step("hca", q, 2, sink, ent, wf, 4, n_win, dr, theta)     # t = 2 < m - 1: no entry visible
    assert np.array_equal(a["o"], b["o"]) and np.array_equal(a["lse"], b["lse"])


# ----------------------------------------------------------------------------- FP4 (e2m1) indexer keys
def test_e2m1_codec_definition_ties_and_packing():
    """OCP e2m1: sign, 2 exponent bits (bias 1), 1 mantissa bit, subnormal at exponent 0."""
    assert O.E2M1_TABLE.tolist() == [0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    for c in range(16):   # every non-zero value round-trips to its own code
        if O.E2M1_TABLE[c] != 0:
            assert O.encode_e2m1(np.array([O.E2M1_TABLE[c]]))[0] == c
    # midpoints go to the code with mantissa bit 0 (even); beyond 6 saturates
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    assert O.decode_e2m1(O.encode_e2m1(np.array(mids))).tolist() == [0, 1, 1, 2, 2, 4, 4]
    assert O.encode_e2m1(np.array([7.0, -100.0, 0.26, -0.74]))[:].tolist() == [7, 15, 1, 9]
    # two codes per byte, element 2i in the low nibble
    assert O.pack_e2m1(np.array([1, 2, 3, 4], np.uint8)).tolist() == [0x21, 0x43]
    assert O.unpack_e2m1(np.array([0x21, 0x43], np.uint8), 4).tolist() == [1, 2, 3, 4]
    assert O.e2m1_scale(np.array([-3.0, 1.0])) == np.float32(np.float32(3.0) / np.float32(6.0))
    assert O.e2m1_scale(np.zeros(4)) == np.float32(1.0)


def test_e2m1_encoders_agree():
    """The oracle's encoder (nearest of the eight magnitudes, ties to the even code) and
    the input generator's (threshold counting) are written independently; they agree."""
    from long_context_attention_05_b300 import synthetic as S
    x = (rng.standard_normal((64, 128)) * np.exp(rng.uniform(-3, 2.5, (64, 1)))).astype(np.float32)
    x[0, :14] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.75, -5, 6, 7, 0, -0.0]
    assert np.array_equal(S.to_e2m1_packed(x), O.pack_e2m1(O.encode_e2m1(x.astype(np.float64))))


def test_compress_index_keys_fp4_hand_worked():
    """One block of m = 2 with slot 1 dominant (the key is its second token):
    key (6, -3, 1, 0.2) -> scale 6/6 = 1, codes (7, 0b1101, 2, 0), packed (0xD7, 0x02)."""
    ix = np.array([[9, 9, 9, 9], [6, -3, 1, 0.2]], dtype=np.float64)
    out = O.compress_index_keys(ix, np.zeros_like(ix), np.array([0.0, 60.0]), 2, "e4m3", 0, 1, idx_dtype="e2m1")
    assert out["idx_scale"].tolist() == [1.0]
    assert out["idx_key"][0].tolist() == [0xD7, 0x02]
    dec = O.decode_index_keys(out["idx_key"], out["idx_scale"], "e4m3", "e2m1", 4)
    assert dec.tolist() == [[6.0, -3.0, 1.0, 0.0]]
