"""Shared helpers of the parity tests: run one step of a workload through the
C ABI and compute the oracle's expectation for the same seeded inputs.

The oracle never sees anything the CUDA path produced: both sides start from
the arrays of long_context_attention_05_b300.synthetic.  The one direction that
does cross is oracle -> GPU (e.g. the oracle's top-k set fed to the GPU's
attention), which tests the GPU stage on exactly the oracle's input.
"""
from __future__ import annotations

import math
from typing import Dict

import numpy as np

from oracle import csa_oracle as O

# tolerances (relative to the largest |value| of the compared row)
TOL_F32 = 1e-5
TOL_LOW = 2e-3
TIE_REL = 1e-6


# ----------------------------------------------------------------------------- oracle side
def _dec_tok(a, w):
    return O.decode_tokens(a, w.tok_dtype)


def seq_entries(w, arrs, b, n):
    rows = O.entry_rows(n, b, w.max_entries, arrs.get("page_table"), w.page_size)
    sc = arrs["kv_scale"][rows] if w.kv_dtype == "e4m3" else None
    return O.decode_kv(arrs["kv_nope"][rows], sc, arrs["kv_rope"][rows], w.kv_dtype)


def seq_index_keys(w, arrs, b, n):
    rows = O.entry_rows(n, b, w.max_entries, arrs.get("page_table"), w.page_size)
    sc = arrs["idx_scale"][rows] if (w.kv_dtype == "e4m3" or w.idx_dtype == "e2m1") else None
    return O.decode_index_keys(arrs["idx_key"][rows], sc, w.kv_dtype, w.idx_dtype, w.d_idx)


def new_entries(w, inp, b, ctx):
    """Entries (decoded, float64) completed by the step's new tokens, when the
    cache holds whole blocks (seeded caches): blocks ctx/m .. (ctx+n_new)/m - 1."""
    assert ctx % w.m == 0
    nb = w.n_new // w.m
    if nb == 0:
        return np.zeros((0, w.d)), (np.zeros((0, w.d_idx)) if w.kind == "csa" else None), None
    x = _dec_tok(inp["x"][b], w)
    g = _dec_tok(inp["gate"][b], w)
    st = _compress_at(x, g, inp["pos_bias"], w, ctx // w.m, nb)
    ent = O.decode_kv(st["kv_nope"], st.get("kv_scale"), st["kv_rope"], w.kv_dtype)
    keys = None
    if w.kind == "csa":
        ix = _dec_tok(inp["idx_x"][b], w)
        ig = _dec_tok(inp["idx_gate"][b], w)
        ks = O.compress_index_keys(ix, ig, inp["idx_pos_bias"], w.m, w.kv_dtype, 0, nb, idx_dtype=w.idx_dtype)
        keys = O.decode_index_keys(ks["idx_key"], ks.get("idx_scale"), w.kv_dtype, w.idx_dtype, w.d_idx)
    return ent, keys, st


def _compress_at(x, g, bias, w, j_first, nb):
    """Entries of blocks j_first .. j_first+nb-1 whose tokens are x[0:nb*m] (the
    chunk starts at token j_first*m)."""
    pad = j_first * w.m
    xx = np.concatenate([np.zeros((pad, x.shape[1])), x], axis=0)
    gg = np.concatenate([np.zeros((pad, g.shape[1])), g], axis=0)
    return O.compress_entries(xx, gg, bias, w.m, w.d_rope, w.theta, w.kv_dtype, j_first, nb)


class LazyEntries:
    """Decoded entries of one sequence, decoded on indexing (a full 1M-token cache
    does not fit in float64 at once): the seeded old entries followed by the
    entries the step completed."""

    def __init__(self, w, arrs, b, n_old, ent_new):
        self.w, self.arrs, self.b, self.n_old, self.ent_new = w, arrs, b, n_old, ent_new
        self.shape = (n_old + len(ent_new), w.d)

    def __getitem__(self, sel):
        idx = np.arange(self.shape[0])[sel]
        out = np.zeros((len(idx), self.w.d))
        old = idx < self.n_old
        if old.any():
            rows = O.entry_rows(self.n_old, self.b, self.w.max_entries, self.arrs.get("page_table"),
                                self.w.page_size)[idx[old]]
            sc = self.arrs["kv_scale"][rows] if self.w.kv_dtype == "e4m3" else None
            out[old] = O.decode_kv(self.arrs["kv_nope"][rows], sc, self.arrs["kv_rope"][rows], self.w.kv_dtype)
        if (~old).any():
            out[~old] = self.ent_new[idx[~old] - self.n_old]
        return out


def window_fn(w, arrs, inp, b, ctx):
    ring = _dec_tok(arrs["win"][b], w)
    x = _dec_tok(inp["x"][b], w)

    def f(pos):
        out = []
        for p in pos:
            p = int(p)
            out.append(x[p - ctx] if p >= ctx else ring[p % w.win_cap])
        return np.array(out).reshape(len(out), w.d)
    return f


def oracle_seeded_step(w, arrs, inp, b, i, idx_override=None, ent_cache=None):
    """Oracle result of query i (position ctx+i) of sequence b after the step
    appended w.n_new tokens to a seeded cache."""
    ctx = w.ctx[b]
    t = ctx + i
    n_old = ctx // w.m
    if ent_cache is not None and b in ent_cache:
        ent, keys = ent_cache[b]
    else:
        keys_old = seq_index_keys(w, arrs, b, n_old) if w.kind == "csa" else None
        ent_new, keys_new, _ = new_entries(w, inp, b, ctx)
        ent = LazyEntries(w, arrs, b, n_old, ent_new)
        keys = np.concatenate([keys_old, keys_new], axis=0) if w.kind == "csa" else None
        if ent_cache is not None:
            ent_cache[b] = (ent, keys)
    q = _dec_tok(inp["q"][b, i], w)
    kw = {}
    if w.kind == "csa":
        kw = dict(q_idx=_dec_tok(inp["q_idx"][b, i], w), w_idx=inp["w_idx"][b, i].astype(np.float64),
                  idx_keys=keys, k=w.k, idx_override=idx_override, q_fp8=w.q_fp8)
    res = O.query_step(w.kind, q, t, inp["sink"].astype(np.float64), ent, window_fn(w, arrs, inp, b, ctx), w.m,
                       w.n_win, w.d_rope, w.theta, **kw)
    res["n_old"] = n_old
    if w.kind == "csa":
        res["slack"] = score_slack(w, kw["q_idx"], kw["w_idx"], keys, n_old, res["n_vis"])
    return res


def score_slack(w, q_idx, w_idx, keys, n_old, n_vis):
    """Per-entry allowance on indexer scores of entries the step itself
    compressed (j >= n_old): each side quantised those keys from its own pooled
    values (fp32 on the GPU, fp64 here), so an e4m3 code may differ by one step
    and the scale by (4m+8) fp32 roundings.  Zero for seeded entries."""
    slack = np.zeros(n_vis)
    if n_vis <= n_old or w.kv_dtype != "e4m3":
        return slack
    k = keys[n_old:n_vis]
    a = np.abs(k)
    if w.idx_dtype == "e2m1":   # one e2m1 step: 0.5 below 2, 1 below 4, 2 above (scale-relative)
        s = np.maximum(a.max(axis=1, keepdims=True) / 6.0, 1e-30)
        v = a / s
        step = np.where(v < 2, 0.5, np.where(v < 4, 1.0, 2.0)) * s
    else:
        # one e4m3 step at each element's magnitude (scale-relative), in value units
        s = np.maximum(a.max(axis=1, keepdims=True) / 448.0, 1e-30)
        v = a / s
        step = np.where(v >= 2.0 ** -6, np.ldexp(1.0, (np.floor(np.log2(np.maximum(v, 2.0 ** -6))) - 3).astype(int)),
                        2.0 ** -9) * s
    dk = step + a * (4 * w.m + 8) * 2.0 ** -24
    slack[n_old:] = (np.abs(q_idx) @ dk.T).T @ np.abs(w_idx)
    return slack


# ----------------------------------------------------------------------------- comparisons
def row_rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.maximum(np.abs(ref).max(axis=-1), 1e-30)
    return np.abs(got - ref).max(axis=-1) / den


def bf16_half_ulp(ref):
    a = np.abs(np.asarray(ref, np.float64))
    e = np.floor(np.log2(np.maximum(a, 1e-38)))
    return np.ldexp(1.0, (e - 8).astype(int))


def check_rows(got, ref, tol, out_bf16=False, what="", extra=0.0):
    """Per row: |got - ref| <= tol * max_row|ref| (+ half a bf16 ulp of ref when
    the output is stored in bf16, + a per-element `extra` allowance)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.maximum(np.abs(ref).max(axis=-1, keepdims=True), 1e-30)
    allow = tol * den + (bf16_half_ulp(ref) if out_bf16 else 0.0) + extra
    bad = np.abs(got - ref) > allow
    worst = float(row_rel_err(got, ref).max()) if got.size else 0.0
    assert not bad.any(), f"{what}: {int(bad.sum())} elements outside tolerance; worst row rel err {worst:.3e}"
    return worst


def check_topk(gpu_idx, gpu_cnt, ref_idx, ref_cnt, ref_scores, what="", slack=None):
    """Index sets must match except for near-ties: every index in one set but not
    the other must have an oracle score within TIE_REL of the oracle's k-th score
    (widened by the entry's quantisation slack for entries the step compressed)."""
    assert int(gpu_cnt) == int(ref_cnt), f"{what}: count {gpu_cnt} != {ref_cnt}"
    g = np.asarray(gpu_idx)[: int(gpu_cnt)]
    assert np.all(np.diff(g) > 0), f"{what}: indices not strictly ascending"
    assert np.all(np.asarray(gpu_idx)[int(gpu_cnt):] == -1), f"{what}: padding is not -1"
    r = np.asarray(ref_idx)[: int(ref_cnt)]
    gs, rs = set(g.tolist()), set(r.tolist())
    diff = (gs - rs) | (rs - gs)
    if not diff:
        return 0
    kth = min(ref_scores[j] for j in rs)
    jk = min(rs, key=lambda j: (ref_scores[j], -j))
    sl = (lambda j: 0.0) if slack is None else (lambda j: float(slack[j]))
    for j in diff:
        assert abs(ref_scores[j] - kth) <= TIE_REL * abs(kth) + sl(j) + sl(jk), \
            f"{what}: index {j} differs (score {ref_scores[j]!r}, k-th {kth!r})"
    return len(diff) // 2


def bf16_tensor_to_np(t):
    import torch
    return t.float().cpu().numpy().astype(np.float64) if t.dtype == torch.bfloat16 else t.cpu().numpy().astype(np.float64)


# ----------------------------------------------------------------------------- GPU side (through the C ABI)
def gpu_inputs(w, inp):
    import long_context_attention_05_b300 as L
    return {k: L.to_device(v) for k, v in inp.items()}


def gpu_compress(w, cache, gi):
    import long_context_attention_05_b300 as L
    L.csa_compress(cache, gi["x"], gi["gate"], gi["pos_bias"], gi.get("idx_x"), gi.get("idx_gate"),
                   gi.get("idx_pos_bias"))


def gpu_query_stages(w, cache, gi, out_dtype, ws, chained=False, idx_in=None):
    """Indexer scores + top-k (CSA) and attention for the step's queries.
    Returns host numpy arrays."""
    import torch
    import long_context_attention_05_b300 as L
    B, n_q = w.batch, w.n_new
    res = {}
    if w.kind == "csa":
        idx = torch.full((B, n_q, w.k), -7, dtype=torch.int32, device="cuda")
        cnt = torch.full((B, n_q), -7, dtype=torch.int32, device="cuda")
        if chained:
            L.csa_index_topk(cache, gi["q_idx"], gi["w_idx"], w.k, idx, cnt, ws, q_fp8=w.q_fp8)
        else:
            scores = torch.full((B * n_q, cache.entry_cap), float("nan"), dtype=torch.float32, device="cuda")
            L.csa_index_scores(cache, gi["q_idx"], gi["w_idx"], scores, ws, q_fp8=w.q_fp8)
            L.csa_topk(cache, scores, B, n_q, w.k, idx, cnt, ws)
            res["scores"] = scores
        use = idx if idx_in is None else idx_in
        out = torch.empty((B, n_q, w.heads, w.d), dtype=out_dtype, device="cuda")
        lse = torch.empty((B, n_q, w.heads), dtype=torch.float32, device="cuda")
        L.csa_sparse_attend(cache, gi["q"], gi["sink"], use, out, lse, ws)
        res.update(idx=idx, cnt=cnt)
    else:
        out = torch.empty((B, n_q, w.heads, w.d), dtype=out_dtype, device="cuda")
        lse = torch.empty((B, n_q, w.heads), dtype=torch.float32, device="cuda")
        L.hca_attend(cache, gi["q"], gi["sink"], out, lse, ws)
    res.update(o=out, lse=lse)
    torch.cuda.synchronize()
    return {k: (v.float().cpu().numpy() if v.dtype == torch.bfloat16 else v.cpu().numpy()) for k, v in res.items()}


def gpu_seeded_step(w, arrs, inp, out_dtype=None, chained=False):
    import torch
    import long_context_attention_05_b300 as L
    out_dtype = out_dtype or (torch.float32 if w.tok_dtype == "f32" else torch.bfloat16)
    cache = L.Cache.from_host(w, arrs)
    gi = gpu_inputs(w, inp)
    gpu_compress(w, cache, gi)
    ws = L.alloc_workspace(cache, w.batch, w.n_new, w.heads, w.k)
    res = gpu_query_stages(w, cache, gi, out_dtype, ws, chained=chained)
    res["cache"] = cache
    res["gi"] = gi
    res["ws"] = ws
    return res
