"""Seeded synthetic inputs for the CSA/HCA hot path.

This module only draws random numbers and stores them in the byte formats the
cache uses (fp32, bf16 bit patterns, e4m3 codes).  It performs none of the
attention method's arithmetic: no pooling, no rotary embedding, no
quantisation rule, no scoring.  Both the CUDA path (through the package
binding) and the CPU oracle (through the tests) read the arrays it returns, so
the two sides see identical input bytes.

Numbers come from numpy's PCG64 generator seeded with ``[seed, stream]`` so
each array has its own independent stream.  Casts to bf16 / e4m3 use torch's
CPU conversion routines (round-to-nearest-even); e4m3 inputs are clamped to
the finite range first because torch maps out-of-range values to NaN.

Directly seeded compressed caches stand in for the output of the compressor
over a long context (pooling a million tokens per sequence is not part of one
decode step).  Their per-entry e4m3 scales are drawn at random, independent of
any rule the method uses to pick scales.

Workloads follow the configurations the DeepSeek-V4 write-ups describe
(hybrid attention: CSA with 4-token compression and top-k selection, HCA with
128-token compression and dense attention; sliding window; attention sink),
with the sizes of the five benchmark configurations.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import numpy as np
import torch

E4M3_MAX = 448.0


# --------------------------------------------------------------------------- casts
def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16), round to nearest even (torch)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """float32 array -> OCP e4m3 codes (uint8), clamped to +-448 first (torch cast)."""
    x = np.clip(np.ascontiguousarray(x, dtype=np.float32), -E4M3_MAX, E4M3_MAX)
    return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def to_e2m1_packed(x: np.ndarray) -> np.ndarray:
    """float32 array [..., n] -> OCP e2m1 (FP4) codes, two per byte (element 2i in the
    low nibble), round to nearest with ties to the even code, saturating at +-6."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x)
    m = ((a > 0.25).astype(np.uint8) + (a >= 0.75) + (a > 1.25) + (a >= 1.75) + (a > 2.5) + (a >= 3.5) +
         (a > 5.0)).astype(np.uint8)
    codes = m | np.where((x < 0) & (m > 0), 8, 0).astype(np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def normal(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    return (_rng(seed, stream).standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def uniform(seed: int, stream: int, shape, lo=0.0, hi=1.0) -> np.ndarray:
    return _rng(seed, stream).uniform(lo, hi, size=shape).astype(np.float32)


# --------------------------------------------------------------------------- workloads
@dataclasses.dataclass(frozen=True)
class Workload:
    """Sizes and formats of one synthetic workload.

    kind: "csa" (indexer + top-k + sparse attention) or "hca" (dense attention).
    mode: "decode" (one new token and one query per sequence per step) or
          "prefill" (n_new tokens appended and n_new queries per sequence).
    ctx:  tokens already in each sequence's cache before the step (tuple, one per
          sequence).  Directly seeded caches need ctx to be a multiple of m.
    """

    name: str
    kind: str
    mode: str
    batch: int
    ctx: tuple
    m: int
    d: int
    d_rope: int
    heads: int
    d_idx: int
    heads_idx: int
    k: int
    n_win: int
    kv_dtype: str          # "f32" or "e4m3"
    tok_dtype: str         # dtype of per-token inputs, queries, window ring: "f32" or "bf16"
    page_size: int = 0     # entries per page; 0 = contiguous
    n_new: int = 1         # tokens appended (= queries) per sequence per step
    seeded_cache: bool = True   # False: build the cache by compressing per-token inputs
    plant_frac: float = 0.0
    seed: int = 0
    theta: float = 10000.0
    extra_entries: int = 64     # spare entry capacity per sequence for repeated steps
    spare_pages: int = 0        # spare physical pages in the pool (paged caches)
    q_fp8: bool = False         # indexer: query-side FP8 variant
    idx_dtype: str = ""         # indexer-key storage: "" (as kv_dtype) or "e2m1" (FP4)

    def __post_init__(self):
        if len(self.ctx) != self.batch:
            raise ValueError(f"{self.name}: {len(self.ctx)} context lengths for batch {self.batch}")

    @property
    def n_entries(self):
        return tuple(c // self.m for c in self.ctx)

    @property
    def win_cap(self):
        # ring must hold the window of every query of a step
        need = self.n_win + self.n_new - 1
        cap = 1
        while cap < max(need, self.m, 1):
            cap *= 2
        return max(cap, 128)

    @property
    def max_entries(self):
        return max(self.n_entries) + self.n_new // self.m + 1 + self.extra_entries

    @property
    def max_pages(self):
        if not self.page_size:
            return 0
        return -(-self.max_entries // self.page_size)

    def pages_needed(self, b):
        """Pages sequence b owns in a paged cache: its entries, the step's new ones and
        the spare capacity (the longest sequence needs max_pages)."""
        cap = self.n_entries[b] + self.n_new // self.m + 1 + self.extra_entries
        return -(-cap // self.page_size)


def config0(**kw) -> Workload:
    """Single CSA layer decode in FP32: batch 1, 4096 context tokens, m=4 (1024
    entries), d=128 (64 rope dims), 16 query heads sharing one KV, indexer 4 heads
    of dim 64, top-k 64, window 128, sink; cache built by the compressor."""
    base = dict(name="csa_decode_fp32_4k", kind="csa", mode="decode", batch=1, ctx=(4095,), m=4,
                d=128, d_rope=64, heads=16, d_idx=64, heads_idx=4, k=64, n_win=128,
                kv_dtype="f32", tok_dtype="f32", seeded_cache=False, seed=0)
    base.update(kw)
    return Workload(**base)


def config1(**kw) -> Workload:
    """Single HCA layer decode: batch 8, 131072 tokens, m=128 (1024 entries), 64
    heads d=128 with FP8 e4m3 compressed KV (64 e4m3 dims + 64 bf16 rope dims),
    bf16 queries, window 128, sink."""
    base = dict(name="hca_decode_bf16_fp8_128k", kind="hca", mode="decode", batch=8,
                ctx=(131072,) * 8, m=128, d=128, d_rope=64, heads=64, d_idx=0, heads_idx=0, k=0,
                n_win=128, kv_dtype="e4m3", tok_dtype="bf16", seed=1)
    base.update(kw)
    return Workload(**base)


def config2(**kw) -> Workload:
    """Single CSA layer decode at 1M context: batch 4, 2^20 tokens, m=4 (262144
    entries), indexer 64 heads d=128 with FP8 keys, top-k 2048, 64 heads d=512
    (448 e4m3 + 64 bf16 rope dims), window 128, sink, 1% planted entries."""
    base = dict(name="csa_decode_1m", kind="csa", mode="decode", batch=4, ctx=(1 << 20,) * 4,
                m=4, d=512, d_rope=64, heads=64, d_idx=128, heads_idx=64, k=2048, n_win=128,
                kv_dtype="e4m3", tok_dtype="bf16", plant_frac=0.01, seed=2)
    base.update(kw)
    return Workload(**base)


def config3(**kw) -> Workload:
    """CSA prefill chunk: 8192 new tokens appended to a 65536-token cache, m=4
    pooling of the new tokens, causal indexer + per-query top-2048, sparse
    attention with window 128 and sink; 64 heads d=512, indexer 64 heads d=128."""
    base = dict(name="csa_prefill_8k_on_64k", kind="csa", mode="prefill", batch=1, ctx=(65536,),
                m=4, d=512, d_rope=64, heads=64, d_idx=128, heads_idx=64, k=2048, n_win=128,
                kv_dtype="e4m3", tok_dtype="bf16", n_new=8192, seed=3, extra_entries=0)
    base.update(kw)
    return Workload(**base)


def config4_lengths(batch=32, seed=4, lo=1 << 13, hi=1 << 20, align=128):
    """Per-sequence context lengths, log-uniform in [lo, hi], rounded down to a
    multiple of `align` so every seeded cache holds whole blocks of both layers."""
    u = _rng(seed, 999).uniform(math.log(lo), math.log(hi), size=batch)
    return tuple(int(max(lo, (int(math.exp(v)) // align) * align)) for v in u)


def config4_layers(batch=32, seed=4, **kw):
    """Interleaved hybrid stack: 4 layers CSA/HCA/CSA/HCA on paged caches (64-entry
    pages in random physical order), batch 32, log-uniform context lengths."""
    ctx = kw.pop("ctx", None) or config4_lengths(batch, seed)
    layers = []
    for li, kind in enumerate(("csa", "hca", "csa", "hca")):
        common = dict(name=f"stack_l{li}_{kind}", kind=kind, mode="decode", batch=len(ctx), ctx=ctx,
                      d=512, d_rope=64, heads=64, n_win=128, kv_dtype="e4m3", tok_dtype="bf16",
                      page_size=64, seed=seed * 100 + li, spare_pages=8)
        if kind == "csa":
            common.update(m=4, d_idx=128, heads_idx=64, k=2048)
        else:
            common.update(m=128, d_idx=0, heads_idx=0, k=0)
        common.update(kw)
        layers.append(Workload(**common))
    return layers


# --------------------------------------------------------------------------- generators
# stream ids
_S_X, _S_G, _S_IX, _S_IG, _S_B, _S_IB = 1, 2, 3, 4, 5, 6
_S_Q, _S_QI, _S_W, _S_SINK = 7, 8, 9, 10
_S_NOPE, _S_SCALE, _S_ROPE, _S_IK, _S_IS, _S_RING, _S_PLANT, _S_PAGES = 11, 12, 13, 14, 15, 16, 17, 18


def _tok(x: np.ndarray, dtype: str) -> np.ndarray:
    return x if dtype == "f32" else to_bf16_bits(x)


def step_inputs(w: Workload, step: int = 0) -> Dict[str, np.ndarray]:
    """Inputs of one step: the appended tokens (KV stream and indexer-key stream with
    their gate logits), the position biases, the queries and the sink logits."""
    s = w.seed * 1000 + step
    B, n = w.batch, w.n_new
    out = {
        "x": _tok(normal(s, _S_X, (B, n, w.d)), w.tok_dtype),
        "gate": _tok(normal(s, _S_G, (B, n, w.d)), w.tok_dtype),
        "pos_bias": normal(w.seed, _S_B, (w.m,), std=0.5),
        "q": _tok(normal(s, _S_Q, (B, n, w.heads, w.d)), w.tok_dtype),
        "sink": normal(w.seed, _S_SINK, (w.heads,)),
    }
    if w.kind == "csa":
        out.update({
            "idx_x": _tok(normal(s, _S_IX, (B, n, w.d_idx)), w.tok_dtype),
            "idx_gate": _tok(normal(s, _S_IG, (B, n, w.d_idx)), w.tok_dtype),
            "idx_pos_bias": normal(w.seed, _S_IB, (w.m,), std=0.5),
            "q_idx": _tok(normal(s, _S_QI, (B, n, w.heads_idx, w.d_idx)), w.tok_dtype),
            "w_idx": uniform(s, _S_W, (B, n, w.heads_idx)),
        })
    return out


def context_tokens(w: Workload) -> Dict[str, np.ndarray]:
    """Per-token inputs of the whole context (used when the cache is built by the
    compressor rather than seeded directly)."""
    B, T = w.batch, max(w.ctx)
    out = {
        "x": _tok(normal(w.seed, 101, (B, T, w.d)), w.tok_dtype),
        "gate": _tok(normal(w.seed, 102, (B, T, w.d)), w.tok_dtype),
    }
    if w.kind == "csa":
        out["idx_x"] = _tok(normal(w.seed, 103, (B, T, w.d_idx)), w.tok_dtype)
        out["idx_gate"] = _tok(normal(w.seed, 104, (B, T, w.d_idx)), w.tok_dtype)
    return out


def _random_scales(seed, stream, shape):
    # per-entry scale in [1/32, 1/16): arbitrary, independent of the values
    return (np.float32(1.0 / 32.0) * (1.0 + uniform(seed, stream, shape))).astype(np.float32)


def seeded_cache(w: Workload, q_idx: Optional[np.ndarray] = None, w_idx: Optional[np.ndarray] = None
                 ) -> Dict[str, np.ndarray]:
    """A compressed cache filled directly with random entries (storage bytes), the
    window ring with random raw tokens and an empty pooling state.

    Returned arrays are in physical row order: contiguous caches have
    batch*max_entries rows (sequence b owns rows [b*max_entries, (b+1)*max_entries));
    paged caches have n_pages*page_size rows plus a page table [batch, max_pages]
    mapping logical page -> physical page (a seeded permutation).

    Planting (plant_frac > 0, CSA only): a seeded subset of each sequence's entries
    has its indexer key moved by +3 along the unit direction of sum_h w_h q_h of
    that sequence's first query, so a top-k selection is not arbitrary.
    """
    assert all(c % w.m == 0 for c in w.ctx), "seeded caches hold whole blocks only"
    B, d, dr = w.batch, w.d, w.d_rope
    dn = d - dr
    if w.page_size:
        n_pages, page_table = page_layout(w)
        rows = n_pages * w.page_size
    else:
        rows = B * w.max_entries
        page_table = None
    out: Dict[str, np.ndarray] = {}
    if w.kv_dtype == "e4m3":
        scale = _random_scales(w.seed, _S_SCALE, (rows,))
        nope_vals = normal(w.seed, _S_NOPE, (rows, dn))
        out["kv_nope"] = to_e4m3_codes(nope_vals / scale[:, None])
        out["kv_scale"] = scale
        out["kv_rope"] = to_bf16_bits(normal(w.seed, _S_ROPE, (rows, dr)))
    else:
        out["kv_nope"] = normal(w.seed, _S_NOPE, (rows, dn))
        out["kv_rope"] = normal(w.seed, _S_ROPE, (rows, dr))
    if w.kind == "csa":
        keys = normal(w.seed, _S_IK, (rows, w.d_idx))
        if w.plant_frac > 0:
            assert q_idx is not None and w_idx is not None
            for b in range(B):
                qh = q_idx[b, 0].astype(np.float64) if q_idx.dtype == np.float32 else \
                    _bf16_bits_to_f32(q_idx[b, 0]).astype(np.float64)
                dirv = (w_idx[b, 0].astype(np.float64)[:, None] * qh).sum(axis=0)
                dirv = (dirv / np.linalg.norm(dirv)).astype(np.float32)
                n_e = w.n_entries[b]
                n_plant = int(round(w.plant_frac * n_e))
                js = _rng(w.seed, _S_PLANT + 1000 * b).choice(n_e, size=n_plant, replace=False)
                prow = _rows_of(w, page_table, b, js)
                keys[prow] += np.float32(3.0) * dirv[None, :]
        if w.idx_dtype == "e2m1":
            # per-entry scale in [0.6, 1.2): keys ~N(0,1) land mostly inside e2m1's +-6
            iscale = (np.float32(0.6) * (1.0 + uniform(w.seed, _S_IS, (rows,)))).astype(np.float32)
            out["idx_key"] = to_e2m1_packed(keys / iscale[:, None])
            out["idx_scale"] = iscale
        elif w.kv_dtype == "e4m3":
            iscale = _random_scales(w.seed, _S_IS, (rows,))
            out["idx_key"] = to_e4m3_codes(keys / iscale[:, None])
            out["idx_scale"] = iscale
        else:
            out["idx_key"] = keys
    ring = normal(w.seed, _S_RING, (B, w.win_cap, d))
    out["win"] = _tok(ring, w.tok_dtype)
    out["pool_state"] = np.zeros((B, 3 * (d + w.d_idx)), dtype=np.float32)
    out["n_tokens"] = np.asarray(w.ctx, dtype=np.int64)
    if page_table is not None:
        out["page_table"] = page_table
    return out


def empty_cache(w: Workload) -> Dict[str, np.ndarray]:
    """Zeroed cache storage (the compressor fills it)."""
    B, d, dr = w.batch, w.d, w.d_rope
    rows = B * w.max_entries if not w.page_size else page_layout(w)[0] * w.page_size
    out: Dict[str, np.ndarray] = {}
    if w.kv_dtype == "e4m3":
        out["kv_nope"] = np.zeros((rows, d - dr), np.uint8)
        out["kv_scale"] = np.zeros((rows,), np.float32)
        out["kv_rope"] = np.zeros((rows, dr), np.uint16)
        if w.kind == "csa":
            out["idx_key"] = np.zeros((rows, w.d_idx // 2 if w.idx_dtype == "e2m1" else w.d_idx), np.uint8)
            out["idx_scale"] = np.zeros((rows,), np.float32)
    else:
        out["kv_nope"] = np.zeros((rows, d - dr), np.float32)
        out["kv_rope"] = np.zeros((rows, dr), np.float32)
        if w.kind == "csa":
            out["idx_key"] = np.zeros((rows, w.d_idx), np.float32)
    out["win"] = np.zeros((B, w.win_cap, d), np.float32 if w.tok_dtype == "f32" else np.uint16)
    out["pool_state"] = np.zeros((B, 3 * (d + w.d_idx)), dtype=np.float32)
    out["n_tokens"] = np.zeros((B,), dtype=np.int64)
    if w.page_size:
        out["page_table"] = page_layout(w)[1]
    return out


def page_layout(w: Workload):
    """Physical pages of a paged cache: sequence b owns pages_needed(b) pages, taken
    from a seeded permutation of the pool (plus spare_pages unused ones).  The page
    table is [batch, max_pages]; slots past a sequence's own pages repeat its last
    page (they are never read for data)."""
    need = [w.pages_needed(b) for b in range(w.batch)]
    n_pages = sum(need) + w.spare_pages
    perm = _rng(w.seed, _S_PAGES).permutation(n_pages).astype(np.int32)
    table = np.empty((w.batch, w.max_pages), dtype=np.int32)
    off = 0
    for b, nb in enumerate(need):
        table[b, :nb] = perm[off:off + nb]
        table[b, nb:] = perm[off + nb - 1]
        off += nb
    return n_pages, table


def _rows_of(w: Workload, page_table, b, js):
    js = np.asarray(js, dtype=np.int64)
    if page_table is None:
        return b * w.max_entries + js
    return page_table[b, js // w.page_size].astype(np.int64) * w.page_size + js % w.page_size


def _bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    # storage reinterpretation (bf16 is the top half of an fp32 pattern); used only
    # to form the planting direction above
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def cache_bytes(arrs: Dict[str, np.ndarray]) -> int:
    """Bytes of a cache's entry storage (KV and indexer keys with their scales)."""
    keys = ("kv_nope", "kv_scale", "kv_rope", "idx_key", "idx_scale")
    return int(sum(arrs[k].nbytes for k in keys if k in arrs))
