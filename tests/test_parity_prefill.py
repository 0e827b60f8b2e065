"""GPU vs oracle parity of a prefill chunk: n_new tokens pooled into new
entries, causal indexer scoring and per-query top-k, sparse attention with the
window and the sink, for every query of the chunk (small chunk) or a seeded
sample of query rows (the full 8192-token chunk on a 65536-token cache)."""
import numpy as np
import pytest
import torch

import harness as H
from long_context_attention_05_b300 import synthetic as S
from test_parity_decode import _check_step, _seeded

pytestmark = pytest.mark.gpu


def test_c3_geometry_small_chunk_all_rows():
    w = S.config3(ctx=(4096,), n_new=256, k=128)
    arrs, inp = _seeded(w)
    res = H.gpu_seeded_step(w, arrs, inp)
    _check_step(w, arrs, inp, res, H.TOL_LOW, what="c3 small")
    # the chunk appended 64 entries and advanced n_tokens
    assert int(res["cache"].t["n_tokens"][0]) == 4096 + 256


def test_c3_chunk_not_block_aligned_and_short_rows():
    # a query near the chunk start sees fewer than k entries
    w = S.config3(ctx=(64,), n_new=130, k=40)
    arrs, inp = _seeded(w)
    res = H.gpu_seeded_step(w, arrs, inp)
    _check_step(w, arrs, inp, res, H.TOL_LOW, what="c3 ragged")
    assert res["cnt"][0, 0] == 16 and res["cnt"][0, -1] == 40


def test_c3_full_chunk_sampled_rows():
    w = S.config3()
    arrs, inp = _seeded(w)
    res = H.gpu_seeded_step(w, arrs, inp)
    rng = np.random.default_rng(3)
    rows = list(range(16)) + list(range(w.n_new - 16, w.n_new)) + sorted(rng.choice(np.arange(16, w.n_new - 16), 32,
                                                                                      replace=False).tolist())
    ties = _check_step(w, arrs, inp, res, H.TOL_LOW, rows=[(0, i) for i in rows], what="c3 full")
    print(f"c3 full: near-tie flips {ties} over {len(rows)} sampled rows")
