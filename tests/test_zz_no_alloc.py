"""csa_index_topk_static: the index + top-k entry point for callers that cannot
allocate device memory (an engine that has reserved all memory for its own
pool, a plugin interface without an allocator, a loop where cudaMalloc's
synchronisation is not acceptable).  Its scratch is a fixed device array inside
the library, so the caller passes only inputs and outputs.

Checked through the C ABI against csa_index_topk (the workspace variant) on the
same inputs, on two calls in a row with different queries: the selected
indices and counts must be identical (the same kernels run; only the scratch
location differs).  Also checks that a request larger than the fixed scratch
is refused with a clear error.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import harness as H
import long_context_attention_05_b300 as L
from long_context_attention_05_b300 import synthetic as S

pytestmark = pytest.mark.gpu


def _setup(w):
    inp = S.step_inputs(w)
    arrs = S.seeded_cache(w, inp.get("q_idx"), inp.get("w_idx"))
    cache = L.Cache.from_host(w, arrs)
    gi = H.gpu_inputs(w, inp)
    H.gpu_compress(w, cache, gi)
    return cache


def test_static_scratch_matches_workspace_variant_on_consecutive_calls():
    w = S.config2(ctx=(65536, 40000, 131072, 8192), k=1024)
    cache = _setup(w)
    B = w.batch
    ws = L.alloc_workspace(cache, B, 1, w.heads, w.k)
    for call in range(2):
        q = S.step_inputs(w, step=10 + call)          # different queries on each call
        q_idx, w_idx = L.to_device(q["q_idx"]), L.to_device(q["w_idx"])
        ref_idx = torch.full((B, 1, w.k), -7, dtype=torch.int32, device="cuda")
        ref_cnt = torch.full((B, 1), -7, dtype=torch.int32, device="cuda")
        L.csa_index_topk(cache, q_idx, w_idx, w.k, ref_idx, ref_cnt, ws)
        got_idx = torch.full((B, 1, w.k), -9, dtype=torch.int32, device="cuda")
        got_cnt = torch.full((B, 1), -9, dtype=torch.int32, device="cuda")
        L.csa_index_topk_static(cache, q_idx, w_idx, w.k, got_idx, got_cnt)
        torch.cuda.synchronize()
        assert torch.equal(got_cnt, ref_cnt), call
        assert torch.equal(got_idx, ref_idx), call
        assert int(got_cnt.min()) == w.k


def test_static_scratch_refuses_oversized_requests():
    w = S.config2(batch=8, ctx=(4096,) * 8)
    cache = _setup(w)
    # claim a larger entry capacity: 8 rows x 270000 entries x 4 bytes of scores exceed
    # the 8 MiB scratch, so the call must refuse before launching anything
    cache.struct.max_entries = 270000
    assert 256 + 8 * 270000 * 4 > L.STATIC_SCRATCH_BYTES
    idx = torch.empty((8, 1, w.k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((8, 1), dtype=torch.int32, device="cuda")
    q = S.step_inputs(w)
    with pytest.raises(RuntimeError, match="static scratch holds"):
        L.csa_index_topk_static(cache, L.to_device(q["q_idx"]), L.to_device(q["w_idx"]), w.k, idx, cnt)
