"""FP4 (e2m1) indexer keys ("FP4 for the indexer": the pages' own indexer
precision): the compressor quantises the indexer stream to e2m1 with a per-entry
scale; the tensor-core indexer streams the packed keys (64 bytes per entry instead
of 128) and a converter warpgroup turns them into the e4m3 tiles the MMA reads; the
CUDA-core indexer decodes them directly.  Everything against the oracle's own e2m1
codec."""
import dataclasses

import numpy as np
import pytest
import torch

import harness as H
import long_context_attention_05_b300 as L
from long_context_attention_05_b300 import synthetic as S
from oracle import csa_oracle as O
from test_parity_decode import _check_step, _seeded

pytestmark = pytest.mark.gpu


def test_compress_fp4_index_keys_against_oracle():
    T = 4 * 700 + 3
    w = S.Workload(name="cmp4", kind="csa", mode="decode", batch=2, ctx=(T, T), m=4, d=128, d_rope=64, heads=1,
                   d_idx=128, heads_idx=1, k=1, n_win=128, kv_dtype="e4m3", tok_dtype="bf16", seeded_cache=False,
                   seed=9, idx_dtype="e2m1")
    ctx = S.context_tokens(w)
    inp = S.step_inputs(w)
    cache = L.Cache.from_host(w, S.empty_cache(w))
    bounds = np.linspace(0, T, 4).astype(int)
    for a, b in zip(bounds[:-1], bounds[1:]):
        sl = {k: L.to_device(np.ascontiguousarray(v[:, a:b])) for k, v in ctx.items()}
        L.csa_compress(cache, sl["x"], sl["gate"], L.to_device(inp["pos_bias"]), sl["idx_x"], sl["idx_gate"],
                       L.to_device(inp["idx_pos_bias"]))
    torch.cuda.synchronize()
    nb = T // 4
    for b in range(2):
        ks = O.compress_index_keys(O.decode_bf16(ctx["idx_x"][b]), O.decode_bf16(ctx["idx_gate"][b]),
                                   inp["idx_pos_bias"], 4, "e4m3", 0, nb, idx_dtype="e2m1")
        rows = b * w.max_entries + np.arange(nb)
        got_codes = cache.t["idx_key"][rows].cpu().numpy()
        got_scale = cache.t["idx_scale"][rows].cpu().numpy()
        assert got_codes.shape == (nb, 64)
        assert np.all(np.abs(got_scale.astype(np.float64) / ks["idx_scale"] - 1) <= (4 * 4 + 8) * 2.0 ** -24)
        dq = O.decode_index_keys(got_codes, got_scale, "e4m3", "e2m1", 128)
        ref = O.decode_index_keys(ks["idx_key"], ks["idx_scale"], "e4m3", "e2m1", 128)
        step = np.where(np.abs(ref) / ks["idx_scale"][:, None] < 2, 0.5, 2.0) * ks["idx_scale"][:, None]
        assert np.all(np.abs(dq - ref) <= step * (1 + 1e-6)), "more than one e2m1 step apart"
        same = (O.unpack_e2m1(got_codes, 128) == O.unpack_e2m1(ks["idx_key"], 128)).mean()
        assert same > 0.99, same


@pytest.mark.parametrize("heads_idx", [64, 48])
def test_fp4_indexer_against_oracle(heads_idx):
    """64 heads: tensor-core kernel (raw ring + converter); 48: CUDA-core kernel."""
    w = S.config2(ctx=(8192, 20000, 4096, 131072), heads_idx=heads_idx, k=512, idx_dtype="e2m1")
    arrs, inp = _seeded(w)
    assert arrs["idx_key"].shape[1] == 64
    res = H.gpu_seeded_step(w, arrs, inp)
    _check_step(w, arrs, inp, res, H.TOL_LOW, what=f"fp4 h={heads_idx}")
    fused = H.gpu_seeded_step(w, arrs, inp, chained=True)
    assert np.array_equal(fused["idx"], res["idx"]) and np.array_equal(fused["o"], res["o"])


def test_fp4_paged_stack_layer_and_full_context():
    ctx = (8192, 12800, 20480, 9088, 8320)
    w = dataclasses.replace([x for x in S.config4_layers(ctx=ctx) if x.kind == "csa"][0], idx_dtype="e2m1")
    arrs, inp = _seeded(w)
    res = H.gpu_seeded_step(w, arrs, inp, chained=True)
    _check_step(w, arrs, inp, res, H.TOL_LOW, what="fp4 paged")
    w = S.config2(idx_dtype="e2m1")
    arrs, inp = _seeded(w)
    res = H.gpu_seeded_step(w, arrs, inp, chained=True)
    ties = _check_step(w, arrs, inp, res, H.TOL_LOW, what="fp4 1M")
    print(f"fp4 1M: near-tie flips {ties}")
    assert np.all(res["cnt"][:, 0] == w.k)
