"""Reproducibility properties of the CUDA path (the write-ups stress bitwise
reproducible, batch-invariant kernels): identical bits on a rerun, for a
sequence alone versus inside a batch, and for a paged cache versus the same
entries stored contiguously."""
import numpy as np
import pytest
import torch

import harness as H
from long_context_attention_05_b300 import synthetic as S

pytestmark = pytest.mark.gpu


def _same(a, b, keys=("idx", "cnt", "o", "lse")):
    for k in keys:
        if k in a:
            assert np.array_equal(a[k], b[k], equal_nan=True), k


def _setup(w):
    inp = S.step_inputs(w)
    arrs = S.seeded_cache(w, inp.get("q_idx"), inp.get("w_idx"))
    return arrs, inp


@pytest.mark.parametrize("kind", ["csa", "hca"])
def test_rerun_is_bitwise_identical(kind):
    w = S.config2(ctx=(65536, 40000, 8192, 100000)) if kind == "csa" else S.config1(batch=3, ctx=(131072, 65536, 1024))
    arrs, inp = _setup(w)
    a = H.gpu_seeded_step(w, arrs, inp)
    b = H.gpu_seeded_step(w, arrs, inp)
    _same(a, b, ("idx", "cnt", "o", "lse", "scores"))


def _slice_batch(w, arrs, inp, b):
    """Sequence b of a contiguous seeded cache as a batch of one (same bytes)."""
    import dataclasses
    extra = w.max_entries - (w.ctx[b] // w.m + w.n_new // w.m + 1)   # keep the batch's entry capacity
    w1 = dataclasses.replace(w, batch=1, ctx=(w.ctx[b],), extra_entries=extra)
    rows = slice(b * w.max_entries, (b + 1) * w.max_entries)
    a1 = {k: (v[rows] if k in ("kv_nope", "kv_scale", "kv_rope", "idx_key", "idx_scale") else v) for k, v in arrs.items()}
    # the single sequence keeps the batch's entry capacity
    a1["win"] = arrs["win"][b:b + 1]
    a1["pool_state"] = arrs["pool_state"][b:b + 1]
    a1["n_tokens"] = arrs["n_tokens"][b:b + 1]
    i1 = {k: (v[b:b + 1] if v.ndim >= 2 and v.shape[0] == w.batch else v) for k, v in inp.items()}
    return w1, a1, i1


@pytest.mark.parametrize("kind", ["csa", "hca512"])
def test_batch_invariance(kind):
    """A sequence's results are the same bits alone as in a batch (top-k call, and a
    dense d = 512 call, whose splits hold four chunks)."""
    w = (S.config2(ctx=(65536, 40000, 8192, 100000), extra_entries=64) if kind == "csa"
         else S.config1(batch=4, ctx=(131072, 65536, 1024, 262144), d=512, extra_entries=64))
    arrs, inp = _setup(w)
    full = H.gpu_seeded_step(w, arrs, inp)
    for b in (0, 2, 3):
        w1, a1, i1 = _slice_batch(w, arrs, inp, b)
        assert w1.max_entries == w.max_entries
        one = H.gpu_seeded_step(w1, a1, i1)
        for k in ("idx", "cnt", "o", "lse"):
            if k in full and full[k] is not None:
                assert np.array_equal(one[k][0], full[k][b]), (b, k)


def test_paged_equals_contiguous():
    import dataclasses
    w = S.config2(batch=3, ctx=(65536, 40000, 8192), extra_entries=64)
    arrs, inp = _setup(w)
    cont = H.gpu_seeded_step(w, arrs, inp)
    wp = dataclasses.replace(w, page_size=64, spare_pages=5)
    n_pages = w.batch * wp.max_pages + wp.spare_pages
    perm = np.random.default_rng(5).permutation(n_pages).astype(np.int32)
    pt = perm[: w.batch * wp.max_pages].reshape(w.batch, wp.max_pages)
    ap = dict(arrs)
    for name in ("kv_nope", "kv_scale", "kv_rope", "idx_key", "idx_scale"):
        src = arrs[name]
        dst = np.zeros((n_pages * 64,) + src.shape[1:], dtype=src.dtype)
        for b in range(w.batch):
            n = w.max_entries
            j = np.arange(wp.max_pages * 64)
            j = j[j < n]
            dst[pt[b, j // 64].astype(np.int64) * 64 + j % 64] = src[b * w.max_entries + j]
        ap[name] = dst
    ap["page_table"] = pt
    paged = H.gpu_seeded_step(wp, ap, inp)
    _same(cont, paged)


def test_padded_key_list_is_bitwise_identical():
    """The window comes first in a row's key list, so padding the selected entries with
    absent (-1) slots adds only chunks and splits of absent keys, whose partials weigh
    exactly zero: the same bits for k = 512 and the same list padded to 640 and 1024."""
    import long_context_attention_05_b300 as L
    w = S.config2(ctx=(65536, 40000, 8192, 100000), k=512)
    arrs, inp = _setup(w)
    base = H.gpu_seeded_step(w, arrs, inp, chained=True)
    cache, gi, ws0 = base["cache"], base["gi"], base["ws"]
    idx = torch.from_numpy(base["idx"]).cuda()
    outs = []
    for k in (512, 640, 1024):
        pad = torch.full((w.batch, 1, k), -1, dtype=torch.int32, device="cuda")
        pad[:, :, :512] = idx
        ws = L.alloc_workspace(cache, w.batch, 1, w.heads, k)
        out = torch.empty((w.batch, 1, w.heads, w.d), dtype=torch.float32, device="cuda")
        lse = torch.empty((w.batch, 1, w.heads), dtype=torch.float32, device="cuda")
        L.csa_sparse_attend(cache, gi["q"], gi["sink"], pad, out, lse, ws)
        torch.cuda.synchronize()
        outs.append((out.cpu().numpy(), lse.cpu().numpy()))
    for k, (o, l) in zip((640, 1024), outs[1:]):
        assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1]), k


@pytest.mark.parametrize("d", [128, 512])
def test_dense_rows_do_not_depend_on_the_entry_capacity(d):
    """HCA's split plan covers the cache's entry capacity; splits past a row's keys do
    nothing, so the capacity (and the split count it gives) leaves the bits unchanged.
    d = 512 takes four 64-key chunks per split, d = 128 two."""
    import dataclasses
    w = S.config1(batch=3, ctx=(131072, 65536, 1024), d=d)
    arrs, inp = _setup(w)
    a = H.gpu_seeded_step(w, arrs, inp)
    w2 = dataclasses.replace(w, extra_entries=w.extra_entries + 3000)
    rows2 = w2.max_entries
    a2 = dict(arrs)
    for name in ("kv_nope", "kv_scale", "kv_rope"):
        src = arrs[name]
        dst = np.zeros((w.batch * rows2,) + src.shape[1:], dtype=src.dtype)
        for b in range(w.batch):
            dst[b * rows2:b * rows2 + w.max_entries] = src[b * w.max_entries:(b + 1) * w.max_entries]
        a2[name] = dst
    b2 = H.gpu_seeded_step(w2, a2, inp)
    _same(a, b2)
