"""The fused indexer + top-k call.  When the tensor-core indexer runs, it also counts
each query row's scores per 13-bit key prefix, and the row-split top-k finds the bin
of the k-th largest score from those counts instead of building its own histogram.
The selection must equal the separate calls' (same scores, exact selection either
way), on repeated calls (the top-k leaves the counts zeroed), and when the workspace
starts out holding garbage or counts that do not match the scores (the top-k checks
the counts against the keys and takes its radix passes over the row instead)."""
import numpy as np
import pytest
import torch

import long_context_attention_05_b300 as L
from long_context_attention_05_b300 import synthetic as S

pytestmark = pytest.mark.gpu


def _setup(w):
    inp = S.step_inputs(w)
    arrs = S.seeded_cache(w, inp.get("q_idx"), inp.get("w_idx"))
    cache = L.Cache.from_host(w, arrs)
    gi = {k: L.to_device(x) for k, x in inp.items()}
    ws = L.alloc_workspace(cache, w.batch, w.n_new, w.heads, w.k)
    return cache, gi, ws


def _outs(w):
    idx = torch.full((w.batch, w.n_new, w.k), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((w.batch, w.n_new), -7, dtype=torch.int32, device="cuda")
    return idx, cnt


def _separate(w, cache, gi, ws, want_scores=False):
    idx, cnt = _outs(w)
    scores = torch.empty((w.batch * w.n_new, cache.entry_cap), dtype=torch.float32, device="cuda")
    L.csa_index_scores(cache, gi["q_idx"], gi["w_idx"], scores, ws)
    L.csa_topk(cache, scores, w.batch, w.n_new, w.k, idx, cnt, ws)
    torch.cuda.synchronize()
    if want_scores:
        return (idx.cpu().numpy(), cnt.cpu().numpy()), scores.cpu().numpy()
    return idx.cpu().numpy(), cnt.cpu().numpy()


def _align256(n):
    return (n + 255) // 256 * 256


def _hist_view(w, cache, ws):
    """The per-row prefix counts in the workspace, reached into through the layout:
    the top-k area is the workspace's last bytes, 256-byte aligned; it starts with
    rows x 8192 counts, then 4 counter words and 2048 digit counts per row, 16 bytes
    per 8192-entry part and row, and min(8192, k + 4096) list entries of 8 bytes per
    part and row."""
    rows = w.batch * w.n_new
    parts = -(-cache.entry_cap // 8192)
    area = (rows * 8192 * 4 + _align256(rows * 2052 * 4) + _align256(rows * parts * 16)
            + rows * parts * min(8192, w.k + 4096) * 8)
    off = (ws.numel() - area) // 256 * 256
    return ws[off:off + rows * 8192 * 4].view(torch.int32).view(rows, 8192)


def _fused(w, cache, gi, ws):
    idx, cnt = _outs(w)
    L.csa_index_topk(cache, gi["q_idx"], gi["w_idx"], w.k, idx, cnt, ws)
    torch.cuda.synchronize()
    assert L.device_status(ws) == 0
    return idx.cpu().numpy(), cnt.cpu().numpy()


def _same(a, b, what):
    assert np.array_equal(a[1], b[1]), f"{what}: counts differ"
    assert np.array_equal(a[0], b[0]), f"{what}: indices differ in {int((a[0] != b[0]).sum())} places"


@pytest.mark.parametrize("ctx", [(65536, 40000, 8192, 30000), (1 << 20,) * 4])
def test_fused_matches_separate_on_repeated_calls(ctx):
    w = S.config2(ctx=ctx)
    cache, gi, ws = _setup(w)
    ref = _separate(w, cache, gi, ws)
    for rep in range(3):
        _same(_fused(w, cache, gi, ws), ref, f"call {rep}")


def test_fused_with_garbage_workspace():
    w = S.config2(ctx=(262144, 131072, 65536, 200000))
    cache, gi, ws = _setup(w)
    ref = _separate(w, cache, gi, ws)
    g = torch.Generator(device="cuda").manual_seed(5)
    ws[256:] = torch.randint(0, 256, (ws.numel() - 256,), dtype=torch.uint8, device="cuda", generator=g)
    _same(_fused(w, cache, gi, ws), ref, "garbage workspace")
    _same(_fused(w, cache, gi, ws), ref, "call after it")


def test_fused_with_counts_of_another_call():
    """Counts left in the workspace (as a fused call whose top-k never ran would leave
    them): the indexer adds the real counts on top, the total no longer equals the
    number of scores, and the top-k selects over the whole row instead."""
    w = S.config2(ctx=(131072,) * 4)
    cache, gi, ws = _setup(w)
    ref = _separate(w, cache, gi, ws)
    hist = _hist_view(w, cache, ws)
    hist.zero_()
    hist[:, 5000] = 131072 // 4   # all of each row's entries in one bin
    _same(_fused(w, cache, gi, ws), ref, "counts of another call")
    assert int(hist.abs().sum()) == 0, "the top-k leaves the counts zeroed"


def _prefix_counts(scores, n):
    """Per-row counts of the top 13 bits of the order-preserving image of each score."""
    bits = scores[:, :n].copy().view(np.uint32)
    keys = np.where(bits & 0x80000000, ~bits, bits | 0x80000000).astype(np.uint32)
    return np.stack([np.bincount(r >> 19, minlength=8192) for r in keys]).astype(np.int64)


@pytest.mark.parametrize("kind", ["shifted", "overflow"])
def test_fused_with_counts_that_total_n_but_lie(kind):
    """Counts planted so that, once the indexer has added the real ones, each row's
    total is exactly its number of scores but the bins are wrong.  "shifted": k
    counts moved from the lowest bin to the highest, so the top-k's threshold bin is
    one that holds no key.  "overflow": the threshold bin claims 100 keys near the
    bottom of the key range while every key lies at or above it, so each CTA's list
    outgrows its block.  The CTAs' own counts disagree with the histogram either
    way: the selection must still be exact and the counts left zeroed."""
    w = S.config2(ctx=(131072,) * 4)
    cache, gi, ws = _setup(w)
    ref, scores = _separate(w, cache, gi, ws, want_scores=True)
    n = 131072 // 4
    true = _prefix_counts(scores, n)
    if kind == "shifted":
        want = true.copy()
        want[:, 8191] += w.k
        want[:, 0] -= w.k
    else:
        assert true[:, :2].sum() == 0   # every key's prefix is at least 2
        want = np.zeros_like(true)
        want[:, 2] = w.k - 1
        want[:, 1] = 100
        want[:, 0] = n - (w.k - 1) - 100
    planted = ((want - true) & 0xFFFFFFFF).astype(np.uint32).view(np.int32)
    hist = _hist_view(w, cache, ws)
    hist.copy_(torch.from_numpy(planted))
    _same(_fused(w, cache, gi, ws), ref, f"counts that lie ({kind})")
    assert int(hist.abs().sum()) == 0, "the top-k leaves the counts zeroed"
    _same(_fused(w, cache, gi, ws), ref, f"call after counts that lie ({kind})")


def test_fused_paged_ragged_stack_layer():
    ctx = (8192, 12800, 20480, 9088, 8320)
    w = [x for x in S.config4_layers(ctx=ctx) if x.kind == "csa"][0]
    cache, gi, ws = _setup(w)
    ref = _separate(w, cache, gi, ws)
    for rep in range(2):
        _same(_fused(w, cache, gi, ws), ref, f"paged call {rep}")


@pytest.mark.parametrize("kind", ["equal", "two_levels"])
def test_fused_crowded_threshold_bin(kind):
    """Identical keys (every score equal) or two key values (the upper one on ~30% of
    the entries): the threshold prefix bin holds far more than the candidate list,
    so the fused top-k takes its radix passes (and still leaves the counts zeroed)."""
    w = S.config2(ctx=(65536, 40000, 65536, 30000), k=1024)
    inp = S.step_inputs(w)
    arrs = S.seeded_cache(w, inp["q_idx"], inp["w_idx"])
    shape = arrs["idx_key"].shape
    if kind == "equal":
        arrs["idx_key"] = np.full(shape, np.uint8(0x38), np.uint8)
    else:
        keys = np.full(shape, np.uint8(0x30), np.uint8)
        keys[np.random.default_rng(3).random(shape[0]) < 0.3] = np.uint8(0x38)
        arrs["idx_key"] = keys
    arrs["idx_scale"] = np.full_like(arrs["idx_scale"], 1.0 / 64.0)
    cache = L.Cache.from_host(w, arrs)
    gi = {k: L.to_device(x) for k, x in inp.items()}
    ws = L.alloc_workspace(cache, w.batch, w.n_new, w.heads, w.k)
    ref = _separate(w, cache, gi, ws)
    if kind == "equal":
        for b in range(w.batch):
            assert sorted(ref[0][b, 0].tolist()) == list(range(w.k))
    for rep in range(2):
        _same(_fused(w, cache, gi, ws), ref, f"{kind} call {rep}")


@pytest.mark.parametrize("n_new", [64, 200])
def test_fused_prefill_shaped_rows(n_new):
    """Many query rows on one sequence: 64 rows take the flat indexer grid and 4-CTA
    clusters, 200 rows (more than the SMs) one indexer CTA per row and single-CTA
    clusters; both fill and consume the prefix histograms."""
    w = S.config3(ctx=(8192,), n_new=n_new, k=256)
    cache, gi, ws = _setup(w)
    ref = _separate(w, cache, gi, ws)
    for rep in range(2):
        _same(_fused(w, cache, gi, ws), ref, f"prefill rows {n_new} call {rep}")
