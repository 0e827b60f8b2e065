"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/csa.h declares, and rejects bad arguments before it
touches the device."""
import ctypes
import os
import re

import pytest

import long_context_attention_05_b300 as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "csa.h")).read()
    return set(re.findall(r"^CSA_API\s+[\w\s\*]*?\b(\w+)\s*\(", src, re.M))


def test_library_exports_every_declared_function():
    L.lib()
    declared = _declared()
    assert declared == set(L.EXPORTS), declared ^ set(L.EXPORTS)
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert declared <= exported, declared - exported
    assert L.version() >= 100


def _struct(**kw):
    s = L.CsaCacheStruct()
    s.m, s.d, s.d_rope, s.d_idx = 4, 512, 64, 128
    s.kv_dtype, s.win_dtype, s.n_win, s.win_cap = L.CSA_E4M3, L.CSA_BF16, 128, 128
    s.page_size, s.max_pages, s.max_entries, s.rope_theta = 0, 0, 1000, 10000.0
    fake = 1 << 20   # never dereferenced: every call below fails validation first or only sizes
    for n in ("kv_nope", "kv_scale", "kv_rope", "idx_key", "idx_scale", "win", "pool_state", "n_tokens"):
        setattr(s, n, fake)
    for k, v in kw.items():
        setattr(s, k, v)
    return s


def test_workspace_size_and_geometry_checks():
    lib = L.lib()
    s = _struct()
    n = lib.csa_workspace_size(ctypes.byref(s), 4, 1, 64, 2048)
    # scores for 4 rows x 1000 entries, and split partials of the decode attention
    assert n >= 256 + 4 * 1000 * 4
    chunks = -(-(2048 + 128) // 64)            # tensor-core attention: 64-key chunks, 2 per split
    splits = -(-chunks // 2)
    assert n >= 256 + 4 * splits * 64 * 512 * 4
    assert lib.csa_workspace_size(ctypes.byref(_struct(d=500)), 4, 1, 64, 2048) == 0
    assert lib.csa_workspace_size(ctypes.byref(_struct(d_idx=100)), 4, 1, 64, 2048) == 0
    assert lib.csa_workspace_size(ctypes.byref(_struct(win_cap=64)), 4, 1, 64, 2048) == 0
    assert lib.csa_workspace_size(None, 4, 1, 64, 2048) == 0


@pytest.mark.parametrize("field,value,code", [
    ("m", 0, 1), ("d_rope", 62, 1), ("kv_dtype", 7, 1), ("win_dtype", L.CSA_E4M3, 1),
    ("kv_nope", None, 1), ("kv_scale", None, 1), ("idx_key", None, 1), ("kv_nope", (1 << 20) + 8, 1),
    ("d_idx", 96, 2), ("n_win", 0, 1), ("rope_theta", 0.5, 1),
])
def test_invalid_cache_rejected(field, value, code):
    lib = L.lib()
    s = _struct(**{field: value})
    st = lib.csa_index_topk(ctypes.byref(s), 1, 1, 1 << 20, L.CSA_BF16, 1 << 20, 64, 2048, 1 << 20, 1 << 20,
                            1 << 20, 1 << 30, None)
    assert st == code, lib.csa_last_error()
    assert lib.csa_last_error()


def test_invalid_call_arguments_rejected():
    lib = L.lib()
    s = ctypes.byref(_struct())
    big = 1 << 30
    assert lib.csa_compress(s, 0, 1, 1, 1, 1, 1, 1, 1, L.CSA_BF16, None) == 1
    assert lib.csa_compress(s, 1, 1, 1, 1, 1, 1, 1, 1, L.CSA_F32, None) == 1      # dtype != ring dtype
    assert lib.csa_compress(s, 1, 1, 1, 1, None, 1, 1, 1, L.CSA_BF16, None) == 1  # missing indexer stream
    assert lib.csa_index_topk(s, 1, 1, 1 << 20, L.CSA_BF16, 1 << 20, 64, 0, 1 << 20, 1 << 20, 1 << 20, big, None) == 1
    assert lib.csa_index_topk(s, 1, 1, 1 << 20, L.CSA_BF16, 1 << 20, 64, 2048, 1 << 20, 1 << 20, None, big, None) == 3
    assert lib.csa_index_topk(s, 1, 1, 1 << 20, L.CSA_BF16, 1 << 20, 64, 2048, 1 << 20, 1 << 20, 1 << 20, 16,
                              None) == 3
    assert lib.csa_index_topk(s, 1, 1, 1 << 20, L.CSA_BF16, 1 << 20, 64, 2048, 1 << 20, 1 << 20, (1 << 20) + 16,
                              big, None) == 3   # workspace alignment
    assert lib.csa_index_scores(s, 1, 1, 1 << 20, L.CSA_BF16, 1 << 20, 64, 1 << 20, 10, None, 0, None) == 1
    assert lib.csa_sparse_attend(s, 1, 1, 1 << 20, L.CSA_BF16, 200, 1 << 20, 1 << 20, 2048, 1 << 20, L.CSA_BF16,
                                 None, 1 << 20, big, None) == 2
    assert lib.csa_sparse_attend(s, 1, 1, 1 << 20, L.CSA_E4M3, 64, 1 << 20, 1 << 20, 2048, 1 << 20, L.CSA_BF16,
                                 None, 1 << 20, big, None) == 1
    assert lib.csa_sparse_attend(s, 1, 1, 1 << 20, L.CSA_BF16, 64, 1 << 20, None, 2048, 1 << 20, L.CSA_BF16,
                                 None, 1 << 20, big, None) == 1
    assert lib.hca_attend(s, 1, 1, 1 << 20, L.CSA_BF16, 64, None, 1 << 20, L.CSA_BF16, None, 1 << 20, big,
                          None) == 1
    # window ring too small for a prefill of 200 queries
    assert lib.hca_attend(s, 1, 200, 1 << 20, L.CSA_BF16, 64, 1 << 20, 1 << 20, L.CSA_BF16, None, 1 << 20, big,
                          None) == 1
    assert lib.csa_device_status(None, None, None) == 1


def _align256(n):
    return (n + 255) // 256 * 256


def _expected_workspace(batch, n_q, heads, k, d=512, n_win=128, entry_cap=1000):
    """The workspace layout written out: a 256-byte header; from it, the scores of the
    indexer (rows x entry capacity) or the attention's split partials, whichever is
    larger; then, for decode-sized calls (rows <= 256) with a top-k, the top-k area at
    the end: per-row histograms of 8192 score-key prefixes, and the row-split top-k's
    per-row counters (4 words) and digit counts (2048 words), per-part slots (16 bytes
    per 8192-entry part) and per-part lists of min(8192, k + 4096) (index, key)
    entries of 8 bytes."""
    rows = batch * n_q
    chunks = -(-(k + n_win) // 64)              # tensor-core attention: 64-key chunks
    splits = -(-chunks // 2) if n_q == 1 else 1  # decode: two chunks per split
    parts = rows * splits * heads
    part_bytes = (_align256(parts * d * 4) + _align256(parts * 2 * 4)) if splits > 1 else 0
    need = max(256 + _align256(rows * entry_cap * 4), 256 + part_bytes)
    area = 0
    if rows <= 256:
        tk_parts = -(-entry_cap // 8192)
        area = rows * 8192 * 4
        if k + 4096 <= 8192:
            area += (_align256(rows * 2052 * 4) + _align256(rows * tk_parts * 16)
                     + rows * tk_parts * min(8192, k + 4096) * 8)
    return _align256(need) + area


@pytest.mark.parametrize("batch,n_q", [(4, 1), (32, 1), (256, 1), (257, 1), (2, 300)])
def test_workspace_layout_reserves_prefix_histograms_for_decode_sized_calls(batch, n_q):
    lib = L.lib()
    s = _struct()
    got = lib.csa_workspace_size(ctypes.byref(s), batch, n_q, 64, 2048)
    assert got == _expected_workspace(batch, n_q, 64, 2048)


def test_split_plan_does_not_depend_on_the_batch():
    """The attention's split count per row depends only on the key-list capacity, so
    a row's reduction order (and its bits) cannot change with the rest of the batch:
    the partials grow exactly linearly with the batch."""
    lib = L.lib()
    s = _struct(max_entries=10)   # tiny scores: the partials set the size
    area = lambda b: b * 8192 * 4 + _align256(b * 2052 * 4) + _align256(b * 16) + b * (2048 + 4096) * 8
    sizes = [lib.csa_workspace_size(ctypes.byref(s), b, 1, 64, 2048) - area(b) for b in (1, 2, 3, 8)]
    per_row = [(sizes[i] - 256) for i in range(4)]
    assert all(abs(per_row[i] / (1, 2, 3, 8)[i] - per_row[0]) < 512 for i in range(4))


@pytest.mark.parametrize("d,cps", [(512, 4), (256, 4), (128, 2)])
def test_dense_wide_decode_takes_four_chunks_per_split(d, cps):
    """A dense decode call (every visible entry, no top-k list: k = 0) with d >= 256 puts
    four 64-key chunks in a split, narrower dense calls two: the d-wide partials such a
    call writes per split are what the merge reads back.  The plan depends on the call's
    kind and the cache's d and capacity only (never the batch)."""
    lib = L.lib()
    s = _struct(d=d, max_entries=1000)
    chunks = -(-(1000 + 128) // 64)
    splits = -(-chunks // cps)
    for batch in (1, 3):
        parts = batch * splits * 64
        want = 256 + _align256(parts * d * 4) + _align256(parts * 2 * 4)
        assert lib.csa_workspace_size(ctypes.byref(s), batch, 1, 64, 0) == want
