"""GPU vs oracle parity of the compressor (softmax-gated pooling fused into the
append): e4m3 entries within one code step (the two sides round from fp32 and
fp64), scales to fp32 rounding, bf16 rotary dims within one bf16 step, raw ring
copies exact, pooling state carried across calls bit-exactly."""
import numpy as np
import pytest
import torch

import harness as H
import long_context_attention_05_b300 as L
from long_context_attention_05_b300 import synthetic as S
from oracle import csa_oracle as O

pytestmark = pytest.mark.gpu


def _build(w, n_calls):
    """Feeds the workload's context tokens in n_calls equal chunks."""
    ctx = S.context_tokens(w)
    inp = S.step_inputs(w)
    cache = L.Cache.from_host(w, S.empty_cache(w))
    T = max(w.ctx)
    bounds = np.linspace(0, T, n_calls + 1).astype(int)
    pb = L.to_device(inp["pos_bias"])
    ipb = L.to_device(inp["idx_pos_bias"]) if w.kind == "csa" else None
    for a, b in zip(bounds[:-1], bounds[1:]):
        sl = {k: L.to_device(np.ascontiguousarray(v[:, a:b])) for k, v in ctx.items()}
        L.csa_compress(cache, sl["x"], sl["gate"], pb, sl.get("idx_x"), sl.get("idx_gate"), ipb)
    torch.cuda.synchronize()
    return cache, ctx, inp


def _host(cache, name):
    t = cache.t[name]
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


@pytest.mark.parametrize("m,d,d_idx,T", [(4, 512, 128, 1024 + 3), (128, 512, 0, 128 * 9 + 5), (4, 128, 64, 402),
                                         (1, 64, 16, 37)])
def test_compress_e4m3_against_oracle(m, d, d_idx, T):
    kind = "csa" if d_idx else "hca"
    w = S.Workload(name="cmp", kind=kind, mode="decode", batch=2, ctx=(T, T), m=m, d=d, d_rope=64 if d >= 128 else 16,
                   heads=1, d_idx=d_idx, heads_idx=1 if d_idx else 0, k=1, n_win=128, kv_dtype="e4m3",
                   tok_dtype="bf16", seeded_cache=False, seed=7)
    cache, ctx, inp = _build(w, 3)
    nb = T // m
    for b in range(2):
        x = O.decode_bf16(ctx["x"][b])
        g = O.decode_bf16(ctx["gate"][b])
        st = O.compress_entries(x, g, inp["pos_bias"], m, w.d_rope, w.theta, "e4m3", 0, nb)
        rows = b * w.max_entries + np.arange(nb)
        codes = _host(cache, "kv_nope")[rows]
        scale = _host(cache, "kv_scale")[rows]
        # fp32 online pooling of m tokens vs fp64: relative error of the pooled amax
        # is bounded by a few fp32 roundings per token
        assert np.all(np.abs(scale.astype(np.float64) / st["kv_scale"] - 1) <= (4 * m + 8) * 2.0 ** -24)
        dq_gpu = O.decode_e4m3(codes) * scale[:, None]
        dq_ref = O.decode_e4m3(st["kv_nope"]) * st["kv_scale"][:, None].astype(np.float64)
        # at most one e4m3 step apart (the step at the larger magnitude)
        step = np.ldexp(1.0, np.floor(np.log2(np.maximum(np.abs(dq_ref) / scale[:, None], 2 ** -6))).astype(int) - 3) \
            * scale[:, None]
        assert np.all(np.abs(dq_gpu - dq_ref) <= 1.0001 * step), "kv codes differ by more than one step"
        frac_exact = np.mean(codes == st["kv_nope"])
        assert frac_exact > 0.99, frac_exact
        rope_g = O.decode_bf16(_host(cache, "kv_rope")[rows])
        rope_r = O.decode_bf16(st["kv_rope"])
        assert np.all(np.abs(rope_g - rope_r) <= 2.0 * H.bf16_half_ulp(rope_r) + 1e-30)
        if d_idx:
            ix = O.decode_bf16(ctx["idx_x"][b])
            ig = O.decode_bf16(ctx["idx_gate"][b])
            ks = O.compress_index_keys(ix, ig, inp["idx_pos_bias"], m, "e4m3", 0, nb)
            kc = _host(cache, "idx_key")[rows]
            assert np.mean(kc == ks["idx_key"]) > 0.99
            assert np.all(np.abs(kc.astype(int) - ks["idx_key"].astype(int)) <= 1)
        # raw ring
        ring = _host(cache, "win")[b]
        for p in range(T - min(T, w.win_cap), T):
            assert np.array_equal(ring[p % w.win_cap], ctx["x"][b, p])
    assert list(cache.t["n_tokens"].cpu().numpy()) == [T, T]


def test_pool_state_carry_is_bit_exact():
    """One token per call and one call for everything must store identical bytes."""
    w = S.Workload(name="carry", kind="csa", mode="decode", batch=3, ctx=(203,) * 3, m=4, d=512, d_rope=64,
                   heads=1, d_idx=128, heads_idx=1, k=1, n_win=128, kv_dtype="e4m3", tok_dtype="bf16",
                   seeded_cache=False, seed=9)
    c1, _, _ = _build(w, 1)
    c2, _, _ = _build(w, 203)
    c3, _, _ = _build(w, 7)
    for name in ("kv_nope", "kv_scale", "kv_rope", "idx_key", "idx_scale", "win", "pool_state", "n_tokens"):
        a, b, c = _host(c1, name), _host(c2, name), _host(c3, name)
        assert np.array_equal(a, b) and np.array_equal(a, c), name


def test_compress_paged_matches_contiguous():
    base = dict(name="pg", kind="csa", mode="decode", batch=2, ctx=(900, 900), m=4, d=512, d_rope=64, heads=1,
                d_idx=128, heads_idx=1, k=1, n_win=128, kv_dtype="e4m3", tok_dtype="bf16", seeded_cache=False,
                seed=11)
    wc = S.Workload(**base)
    wp = S.Workload(**{**base, "page_size": 64, "spare_pages": 3})
    cc, _, _ = _build(wc, 2)
    cp, _, _ = _build(wp, 2)
    pt = cp.t["page_table"].cpu().numpy()
    for b in range(2):
        n = 225
        rc = b * wc.max_entries + np.arange(n)
        rp = pt[b, np.arange(n) // 64].astype(np.int64) * 64 + np.arange(n) % 64
        for name in ("kv_nope", "kv_scale", "kv_rope", "idx_key", "idx_scale"):
            assert np.array_equal(_host(cc, name)[rc], _host(cp, name)[rp]), name
