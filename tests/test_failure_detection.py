"""Failure detection of the bounded device waits, without a GPU fault.

The tensor-core indexer's mbarrier waits give up after a bounded number of polls:
the kernel records CSA_ERR_TIMEOUT in the status word, lets the copies and MMAs it
already issued finish, frees its tensor memory and returns, so the context stays
usable.  The test hook CSA_DEBUG_STARVE_INDEXER makes the producer issue no key
copies (the full barrier of the first key tile is a flag nothing sets) and
CSA_DEBUG_WAIT_LIMIT shortens the waits, so a small call runs a wait out.  The
top-k that follows sees the status word and reports count -1 for every row; a
clean call afterwards gives the normal result."""
import ctypes

import numpy as np
import pytest
import torch

import long_context_attention_05_b300 as L
from long_context_attention_05_b300 import synthetic as S


def test_debug_knobs_are_validated():
    lib = L.lib()
    assert lib.csa_debug_set(99, 0) == 1 and "unknown debug knob" in lib.csa_last_error().decode()
    assert lib.csa_debug_set(L.CSA_DEBUG_WAIT_LIMIT, -5) == 1
    assert lib.csa_debug_set(L.CSA_DEBUG_WAIT_LIMIT, 0) == 0
    assert lib.csa_debug_set(L.CSA_DEBUG_STARVE_INDEXER, 0) == 0
    assert lib.csa_static_status(None, None) == 1


def _setup():
    w = S.config2(ctx=(65536, 40000, 8192, 30000), k=512)
    inp = S.step_inputs(w)
    arrs = S.seeded_cache(w, inp["q_idx"], inp["w_idx"])
    cache = L.Cache.from_host(w, arrs)
    gi = {k: L.to_device(x) for k, x in inp.items()}
    ws = L.alloc_workspace(cache, w.batch, 1, w.heads, w.k)
    return w, cache, gi, ws


def _outs(w):
    return (torch.full((w.batch, 1, w.k), 7, dtype=torch.int32, device="cuda"),
            torch.full((w.batch, 1), 7, dtype=torch.int32, device="cuda"))


class _Starved:
    """Sets the failure injection for the duration of a with-block (always restored)."""

    def __enter__(self):
        L.debug_set(L.CSA_DEBUG_WAIT_LIMIT, 4096)
        L.debug_set(L.CSA_DEBUG_STARVE_INDEXER, 1)

    def __exit__(self, *a):
        L.debug_set(L.CSA_DEBUG_STARVE_INDEXER, 0)
        L.debug_set(L.CSA_DEBUG_WAIT_LIMIT, 0)


@pytest.mark.gpu
def test_indexer_wait_runs_out_and_reports_timeout():
    w, cache, gi, ws = _setup()
    ref_idx, ref_cnt = _outs(w)
    L.csa_index_topk(cache, gi["q_idx"], gi["w_idx"], w.k, ref_idx, ref_cnt, ws)
    torch.cuda.synchronize()
    assert L.device_status(ws) == 0 and int(ref_cnt.min()) == w.k
    with _Starved():
        idx, cnt = _outs(w)
        L.csa_index_topk(cache, gi["q_idx"], gi["w_idx"], w.k, idx, cnt, ws)
        torch.cuda.synchronize()
    assert L.device_status(ws) == L.STATUS_CODES["TIMEOUT"]
    assert torch.all(cnt == -1) and torch.all(idx == -1)
    # the status word was cleared by the read; the context is usable and the call is exact again
    idx, cnt = _outs(w)
    L.csa_index_topk(cache, gi["q_idx"], gi["w_idx"], w.k, idx, cnt, ws)
    torch.cuda.synchronize()
    assert L.device_status(ws) == 0
    assert torch.equal(idx, ref_idx) and torch.equal(cnt, ref_cnt)


@pytest.mark.gpu
def test_status_word_is_sticky_for_the_separate_top_k():
    """A failed scores call leaves the status word set: a top-k given that workspace
    reports -1 counts until the word is read (and so cleared)."""
    w, cache, gi, ws = _setup()
    scores = torch.zeros((w.batch, cache.entry_cap), dtype=torch.float32, device="cuda")
    with _Starved():
        L.csa_index_scores(cache, gi["q_idx"], gi["w_idx"], scores, ws)
    idx, cnt = _outs(w)
    L.csa_topk(cache, scores, w.batch, 1, w.k, idx, cnt, ws)
    torch.cuda.synchronize()
    assert torch.all(cnt == -1)
    assert L.device_status(ws) == L.STATUS_CODES["TIMEOUT"]
    L.csa_index_scores(cache, gi["q_idx"], gi["w_idx"], scores, ws)
    L.csa_topk(cache, scores, w.batch, 1, w.k, idx, cnt, ws)
    torch.cuda.synchronize()
    assert L.device_status(ws) == 0 and int(cnt.min()) == w.k


@pytest.mark.gpu
def test_static_entry_point_reports_timeout():
    w, cache, gi, ws = _setup()
    ref_idx, ref_cnt = _outs(w)
    L.csa_index_topk(cache, gi["q_idx"], gi["w_idx"], w.k, ref_idx, ref_cnt, ws)
    with _Starved():
        idx, cnt = _outs(w)
        L.csa_index_topk_static(cache, gi["q_idx"], gi["w_idx"], w.k, idx, cnt)
        torch.cuda.synchronize()
    assert L.static_status() == L.STATUS_CODES["TIMEOUT"]
    assert torch.all(cnt == -1)
    idx, cnt = _outs(w)
    L.csa_index_topk_static(cache, gi["q_idx"], gi["w_idx"], w.k, idx, cnt)
    torch.cuda.synchronize()
    assert L.static_status() == 0
    assert torch.equal(idx, ref_idx) and torch.equal(cnt, ref_cnt)
