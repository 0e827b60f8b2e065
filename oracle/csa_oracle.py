"""CPU oracle of DeepSeek-V4 compressed attention (CSA / HCA) — TEST INFRASTRUCTURE.

This module exists only to check the CUDA library.  Nothing in the product path
imports it: only the tests, the package's smoke check and the benchmark's
CPU-baseline / reference leg call it.  It shares no code with the CUDA side
(no kernels, headers, tables or helpers); the only common code is the seeded
input generator, which holds none of the method's arithmetic.

Everything is computed in float64, one definition step at a time, in plain
numpy; a matmul or a sort is used as a library step where the definition is a
sum of products or an ordering.  No blocking, fusion or reordering beyond that.

What it computes.  Sources are five web write-ups of the DeepSeek-V4 report,
cited by title and section:
  [V]  "DeepSeek V4 infrastructure" (volanea.com), section "Compression only
       works if the attention path is engineered end to end"
  [B]  "DeepSeek Releases V4 with Million-Token Context Optimized for AI
       Agents" (botbeat.news), section "Summary"
  [J]  "Inside DeepSeek V4: How a Resource-Constrained Team Engineered a
       Million-Token AI Giant" (jakobijn.be), section "The Architecture:
       Hybrid Attention (CSA + HCA)"
  [S]  "DeepSeek V4: How They Crushed the Million-Token Memory Problem"
       (sameershanbhag.com), section "Two kinds of memory instead of one"
The pages give no equations; the per-step formulas below are the plainest
reading of their words.  The indexer-score formula, the per-channel gate and
all sizes are fixed by this library's specification (the pages state none).

* Compression (softmax-gated pooling with a learned positional bias, [B]
  and [S]): every
  non-overlapping block of m tokens becomes one entry.  Per channel c the
  logits are the token's gate logit plus a bias that depends only on the slot
  i in the block; a softmax over the m slots weights the token vectors.
  CSA uses m = 4, HCA m = 128.
* Partial rotary embedding ([V]):
  the last d_rope dims are rotated in consecutive pairs (2i, 2i+1) with angle
  p * theta^(-2i/d_rope).  An entry is rotated at the position of its block's
  first token; a query at its own position; a window token at its position.
* Storage ([S], the note on compression ratio times storage quantisation): e4m3 for the non-rotary dims
  with one fp32 scale per entry, bf16 for the rotary dims; the indexer key is
  e4m3 with its own scale.  (The FP32 configuration stores fp32.)
* Lightning indexer ([S]: ReLU-scored multi-head dot products; [V]): score_j = sum_h w_h *
  ReLU(q_h . k_j) over the entries the query may see; top-k keeps the k best.
* Shared-KV multi-query attention, sliding window and attention sink ([V]): one stored vector per entry or
  window token is both key and value for every head; one softmax per head over
  {selected entries} U {window tokens} U {sink}, logits scaled by 1/sqrt(d);
  the sink adds exp(z_h) to the denominator and contributes no value.
* HCA ([S]; [J], "2. The Big Picture"): the same attention over all
  entries, no selection.

Readings where the pages are silent are listed in the repository's design
notes; each function below states the one it uses.
"""
from __future__ import annotations

import math
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

# =========================================================================== number formats
E4M3_MAX = 448.0


def _e4m3_value(code: int) -> float:
    """Value of one OCP e4m3 code: sign, 4 exponent bits (bias 7), 3 mantissa
    bits; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinity."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
_E4M3_POS_CODE = {E4M3_TABLE[c]: c for c in range(0x7F)}  # finite non-negative codes


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def _round_to_precision(a: np.ndarray, sig_bits: int, min_exp: int) -> np.ndarray:
    """Round non-negative a to `sig_bits` significant bits, nearest-even, with
    exponent floor `min_exp` (gradual underflow below the smallest normal)."""
    a = np.asarray(a, dtype=np.float64)
    out = np.zeros_like(a)
    nz = a > 0
    _, ex = np.frexp(a[nz])                 # a = f * 2^ex, f in [0.5, 1)
    lead = np.maximum(ex - 1, min_exp)      # exponent of the leading bit
    quantum = np.ldexp(1.0, lead - (sig_bits - 1))
    out[nz] = np.rint(a[nz] / quantum) * quantum   # rint: ties to even count
    return out


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """float64 -> e4m3 codes: round to nearest even, saturate to +-448 (satfinite)."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    r = np.minimum(_round_to_precision(np.where(nan, 0.0, np.minimum(a, 1e300)), 4, -6), E4M3_MAX)
    codes = np.vectorize(_E4M3_POS_CODE.__getitem__, otypes=[np.uint8])(r) if r.size else r.astype(np.uint8)
    codes = np.asarray(codes, dtype=np.uint8) | np.where(sign, 0x80, 0).astype(np.uint8)
    return np.where(nan, np.uint8(0x7F), codes).astype(np.uint8)


E2M1_MAX = 6.0


def _e2m1_value(code: int) -> float:
    """Value of one OCP e2m1 (FP4) code: sign, 2 exponent bits (bias 1), 1 mantissa
    bit; exponent 0 is subnormal (m/2); no infinity or NaN."""
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * m * 0.5
    return s * (1.0 + m / 2.0) * 2.0 ** (e - 1)


E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)


def decode_e2m1(codes: np.ndarray) -> np.ndarray:
    return E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF]


def encode_e2m1(x: np.ndarray) -> np.ndarray:
    """float64 -> e2m1 codes (0..15): round to nearest, ties to the even code (the one
    with mantissa bit 0), saturating at +-6."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E2M1_MAX)
    mags = E2M1_TABLE[:8]
    dist = np.abs(a[..., None] - mags)                      # distance to each magnitude
    best = dist.min(axis=-1, keepdims=True)
    cand = dist == best                                     # one, or two at a midpoint
    even = cand & ((np.arange(8) & 1) == 0)
    code = np.where(even.any(axis=-1), np.argmax(even, axis=-1), np.argmax(cand, axis=-1)).astype(np.uint8)
    return (code | np.where(np.signbit(x) & (code > 0), 0x8, 0)).astype(np.uint8)


def unpack_e2m1(packed: np.ndarray, n: int) -> np.ndarray:
    """Two codes per byte (element 2i in the low nibble, 2i+1 in the high) -> [.., n] codes."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out[..., :n]


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit pattern -> float64 (bf16 is the upper half of an IEEE binary32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def encode_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bits, round to nearest even directly from float64."""
    x = np.asarray(x, dtype=np.float64)
    r = _round_to_precision(np.abs(x), 8, -126)
    r = np.where(np.signbit(x), -r, r)
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def decode_tokens(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Per-token inputs in storage form (fp32 array or bf16 bits) -> float64."""
    if dtype == "f32":
        return np.asarray(arr, dtype=np.float32).astype(np.float64)
    return decode_bf16(arr)


def fp32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32)


# =========================================================================== rotary embedding
def rope(v: np.ndarray, pos, d_rope: int, theta: float) -> np.ndarray:
    """Rotate the last d_rope dims of v (shape [..., d]) at integer position(s)
    pos (scalar or broadcastable to v.shape[:-1]).  Pair i = dims
    (base+2i, base+2i+1) turns by pos * theta^(-2i/d_rope), RoFormer style."""
    v = np.asarray(v, dtype=np.float64)
    out = v.copy()
    base = v.shape[-1] - d_rope
    pos = np.asarray(pos, dtype=np.float64)
    for i in range(d_rope // 2):
        ang = pos * theta ** (-2.0 * i / d_rope)
        c, s = np.cos(ang), np.sin(ang)
        a = v[..., base + 2 * i]
        b = v[..., base + 2 * i + 1]
        out[..., base + 2 * i] = a * c - b * s
        out[..., base + 2 * i + 1] = a * s + b * c
    return out


# =========================================================================== compression (a1)
def pool_block(x: np.ndarray, g: np.ndarray, bias: np.ndarray) -> np.ndarray:
    """Softmax-gated pooling of one block: x, g are [m, d], bias is [m] (one
    scalar per slot, broadcast over channels).  Per channel c:
        l_i = g_ic + bias_i,  a_i = exp(l_i) / sum_j exp(l_j),  e_c = sum_i a_i x_ic."""
    logits = np.asarray(g, np.float64) + np.asarray(bias, np.float64)[:, None]
    logits = logits - logits.max(axis=0, keepdims=True)   # shift for exp range only
    a = np.exp(logits)
    a = a / a.sum(axis=0, keepdims=True)
    return (a * np.asarray(x, np.float64)).sum(axis=0)


def e4m3_scale(v: np.ndarray) -> np.float32:
    """Per-entry scale: s = fp32(max|v|) / 448 in fp32 arithmetic; if that is
    zero or below the smallest normal fp32, s = 1."""
    amax = np.float32(np.max(np.abs(v))) if v.size else np.float32(0)
    s = np.float32(amax) / np.float32(E4M3_MAX)
    if not (s >= np.finfo(np.float32).tiny):
        s = np.float32(1.0)
    return np.float32(s)


def e2m1_scale(v: np.ndarray) -> np.float32:
    """FP4 indexer keys: s = fp32(max|v|) / 6 in fp32 arithmetic; 1 if that is zero
    or below the smallest normal fp32 (the e4m3 rule with e2m1's largest value)."""
    amax = np.float32(np.max(np.abs(v))) if v.size else np.float32(0)
    s = np.float32(amax) / np.float32(E2M1_MAX)
    if not (s >= np.finfo(np.float32).tiny):
        s = np.float32(1.0)
    return np.float32(s)


def quantise_e4m3(v: np.ndarray) -> Tuple[np.ndarray, np.float32]:
    """Codes = RNE_e4m3(v / s), saturating; dequantised value = code * s."""
    s = e4m3_scale(v)
    return encode_e4m3(np.asarray(v, np.float64) / np.float64(s)), s


def compress_entries(x: np.ndarray, g: np.ndarray, bias: np.ndarray, m: int, d_rope: int,
                     theta: float, kv_dtype: str, first_block: int, n_blocks: int
                     ) -> Dict[str, np.ndarray]:
    """KV entries j = first_block .. first_block+n_blocks-1 of one sequence from its
    token history x, g ([T, d] float64, T >= (first_block+n_blocks)*m).
    Entry j pools tokens [j*m, (j+1)*m), is rotated at position j*m, and is
    stored as e4m3 nope dims + fp32 scale + bf16 rope dims (or fp32)."""
    d = x.shape[1]
    dn = d - d_rope
    nope, scale, rp = [], [], []
    for j in range(first_block, first_block + n_blocks):
        e = pool_block(x[j * m:(j + 1) * m], g[j * m:(j + 1) * m], bias)
        e = rope(e, j * m, d_rope, theta)
        if kv_dtype == "e4m3":
            c, s = quantise_e4m3(e[:dn])
            nope.append(c)
            scale.append(s)
            rp.append(encode_bf16(e[dn:]))
        else:
            nope.append(fp32(e[:dn]))
            rp.append(fp32(e[dn:]))
    out = {"kv_nope": np.array(nope).reshape(n_blocks, dn), "kv_rope": np.array(rp).reshape(n_blocks, d_rope)}
    if kv_dtype == "e4m3":
        out["kv_scale"] = np.array(scale, dtype=np.float32)
    return out


def compress_index_keys(ix: np.ndarray, ig: np.ndarray, bias: np.ndarray, m: int, kv_dtype: str,
                        first_block: int, n_blocks: int, idx_dtype: str = "") -> Dict[str, np.ndarray]:
    """Indexer keys: the same gated pooling on the indexer-key stream, with its own
    gate logits and bias; no rotation; e4m3 + per-entry scale (or fp32).  With
    idx_dtype "e2m1" (FP4 indexer keys, [S]: "FP4 for the indexer"): codes
    RNE_e2m1(e / s), s = max|e| / 6, two codes per byte."""
    keys, scale = [], []
    for j in range(first_block, first_block + n_blocks):
        e = pool_block(ix[j * m:(j + 1) * m], ig[j * m:(j + 1) * m], bias)
        if idx_dtype == "e2m1":
            s = e2m1_scale(e)
            keys.append(pack_e2m1(encode_e2m1(e / np.float64(s))))
            scale.append(s)
        elif kv_dtype == "e4m3":
            c, s = quantise_e4m3(e)
            keys.append(c)
            scale.append(s)
        else:
            keys.append(fp32(e))
    out = {"idx_key": np.array(keys).reshape(n_blocks, -1)}
    if kv_dtype == "e4m3" or idx_dtype == "e2m1":
        out["idx_scale"] = np.array(scale, dtype=np.float32)
    return out


# =========================================================================== cache access
def entry_rows(n: int, b: int, max_entries: int, page_table: Optional[np.ndarray], page_size: int
               ) -> np.ndarray:
    """Physical rows of logical entries 0..n-1 of sequence b (contiguous: one
    stretch of max_entries rows per sequence; paged: page table lookup)."""
    j = np.arange(n, dtype=np.int64)
    if page_table is None or not page_size:
        return b * max_entries + j
    return page_table[b, j // page_size].astype(np.int64) * page_size + j % page_size


def decode_kv(nope: np.ndarray, scale: Optional[np.ndarray], rp: np.ndarray, kv_dtype: str) -> np.ndarray:
    """Stored entries -> float64 vectors [n, d]: nope = code * scale, rope = bf16."""
    if kv_dtype == "e4m3":
        return np.concatenate([decode_e4m3(nope) * np.asarray(scale, np.float64)[:, None],
                               decode_bf16(rp)], axis=1)
    return np.concatenate([np.asarray(nope, np.float64), np.asarray(rp, np.float64)], axis=1)


def decode_index_keys(keys: np.ndarray, scale: Optional[np.ndarray], kv_dtype: str, idx_dtype: str = "",
                      d_idx: int = 0) -> np.ndarray:
    if idx_dtype == "e2m1":
        return decode_e2m1(unpack_e2m1(keys, d_idx)) * np.asarray(scale, np.float64)[:, None]
    if kv_dtype == "e4m3":
        return decode_e4m3(keys) * np.asarray(scale, np.float64)[:, None]
    return np.asarray(keys, np.float64)


# =========================================================================== indexer (a2) and top-k (a3)
def visible_entries(t: int, m: int) -> int:
    """A query at position t sees entry j iff its block has ended: (j+1)*m - 1 <= t."""
    return (t + 1) // m


def quantise_query_e4m3(q_idx: np.ndarray) -> np.ndarray:
    """Query-side FP8 variant of the indexer (the write-ups call the indexer low
    precision; [S]): each head's query vector q_h is put on the e4m3 grid of a
    power-of-two scale S_h with max|q_h| * S_h in [2^7, 2^8) (RNE), and the scores
    use q_h' = e4m3(q_h * S_h) / S_h.  A zero vector stays zero.  (The power-of-two
    scale is this library's reading: multiplying by it is exact.)"""
    q = np.asarray(q_idx, np.float64)
    out = np.zeros_like(q)
    for h in range(q.shape[0]):
        amax = np.abs(q[h]).max() if q.shape[1] else 0.0
        if amax == 0:
            continue
        _, ex = math.frexp(amax)          # amax = f * 2^ex, f in [0.5, 1)
        s = 2.0 ** (8 - ex)
        out[h] = decode_e4m3(encode_e4m3(q[h] * s)) / s
    return out


def indexer_scores(q_idx: np.ndarray, w: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """score_j = sum_h w_h * ReLU(q_h . k_j).  q_idx [H_I, d_I], w [H_I], keys [N, d_I]."""
    dots = keys @ np.asarray(q_idx, np.float64).T          # [N, H_I]
    return np.maximum(dots, 0.0) @ np.asarray(w, np.float64)


def topk(scores: np.ndarray, k: int) -> Tuple[np.ndarray, int]:
    """Indices of the k largest scores; ties go to the lower index.  Returned in
    ascending index order, padded with -1 when fewer than k entries exist."""
    n = len(scores)
    order = sorted(range(n), key=lambda j: (-scores[j], j))[: min(k, n)]
    sel = np.sort(np.array(order, dtype=np.int64))
    out = np.full(k, -1, dtype=np.int32)
    out[: len(sel)] = sel
    return out, len(sel)


# =========================================================================== attention (a4, a5)
def attend(q: np.ndarray, t: int, entries: np.ndarray, window_raw: np.ndarray, window_pos: np.ndarray,
           sink: np.ndarray, d_rope: int, theta: float) -> Tuple[np.ndarray, np.ndarray]:
    """Shared-KV multi-query attention of one query token.

    q [H, d] (raw; rotated here at position t); entries [n_e, d]: stored entry
    vectors (already rotated at their block position when they were stored);
    window_raw [n_w, d]: raw window tokens, rotated here at window_pos; sink [H].
    Returns o [H, d] and lse [H] = log(sum_j exp(l_hj) + exp(z_h)).
    """
    H, d = q.shape
    qr = rope(q, t, d_rope, theta)
    win = rope(window_raw, np.asarray(window_pos), d_rope, theta) if len(window_raw) else np.zeros((0, d))
    kv = np.concatenate([np.asarray(entries, np.float64).reshape(-1, d), win], axis=0)   # keys = values
    logits = qr @ kv.T / math.sqrt(d)                        # [H, n]
    z = np.asarray(sink, np.float64)
    mx = np.maximum(logits.max(axis=1) if kv.shape[0] else np.full(H, -np.inf), z)
    e = np.exp(logits - mx[:, None])
    es = np.exp(z - mx)
    denom = e.sum(axis=1) + es
    p = e / denom[:, None]
    o = p @ kv
    lse = mx + np.log(denom)
    return o, lse


def window_positions(t: int, n_win: int) -> np.ndarray:
    """Window of a query at t: raw tokens max(0, t-n_win+1) .. t."""
    return np.arange(max(0, t - n_win + 1), t + 1, dtype=np.int64)


def ring_slot(pos: np.ndarray, win_cap: int) -> np.ndarray:
    return np.asarray(pos) % win_cap


# =========================================================================== one query of a step
def query_step(kind: str, q: np.ndarray, t: int, sink: np.ndarray, entries: np.ndarray, window_fn,
               m: int, n_win: int, d_rope: int, theta: float, q_idx: Optional[np.ndarray] = None,
               w_idx: Optional[np.ndarray] = None, idx_keys: Optional[np.ndarray] = None,
               k: int = 0, idx_override: Optional[np.ndarray] = None, q_fp8: bool = False
               ) -> Dict[str, np.ndarray]:
    """All stages for the query at position t of one sequence.

    entries / idx_keys: float64 decoded stored entries / indexer keys of the
    sequence (at least the visible ones); window_fn(positions) -> raw float64
    window tokens.  CSA: indexer scores over the visible entries, top-k, then
    attention over the selected entries + window + sink.  HCA: attention over
    all visible entries + window + sink.  SWA (sliding-window-only layer, [S]: the
    multi-token-prediction block): window + sink, no entries.  idx_override replaces the oracle's own
    top-k set in the attention stage (used to test attention on a given set).
    q_fp8 scores with the query-side FP8 variant (quantise_query_e4m3).
    """
    n_vis = visible_entries(t, m) if kind != "swa" else 0
    assert entries.shape[0] >= n_vis, "entries missing"
    res: Dict[str, np.ndarray] = {"n_vis": n_vis}
    if kind == "csa":
        scores = indexer_scores(quantise_query_e4m3(q_idx) if q_fp8 else q_idx, w_idx, idx_keys[:n_vis])
        idx, count = topk(scores, k)
        res.update(scores=scores, idx=idx, count=count)
        use = idx_override if idx_override is not None else idx
        use = use[use >= 0]
        sel = entries[use]
    else:
        sel = entries[:n_vis]
    pos = window_positions(t, n_win)
    o, lse = attend(q, t, sel, window_fn(pos), pos, sink, d_rope, theta)
    res.update(o=o, lse=lse)
    return res
