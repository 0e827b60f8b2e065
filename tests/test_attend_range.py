"""Input range of the tensor-core attention: the bf16 window tokens and rotary dims
and the e4m3 entries' per-entry scales may hold any finite magnitude.  The kernel
scales every key by powers of two before it rounds to f16, so magnitudes far
outside f16's range (|x| > 65504, or below its normal range 2^-14) keep their
precision.

Each sequence of the batch gets its own magnitude a: its window ring, the new
token, its entries' rotary dims and e4m3 scales are multiplied by a and its query
by 1/a, so the logits stay well conditioned while every stored key operand is far
from 1.  Compared with the oracle on the same stored bytes (the outputs scale
with a; the tolerance is relative to each row's largest value)."""
import numpy as np
import pytest
import torch

import harness as H
from long_context_attention_05_b300 import synthetic as S
from test_parity_decode import _check_step

pytestmark = pytest.mark.gpu

MAGS = (1e5, 1e-6, 3e4, 2e-5)


def _scaled(w, arrs, inp, mags):
    a = {k: v.copy() for k, v in arrs.items()}
    i = {k: v.copy() for k, v in inp.items()}
    f32 = H.O.decode_bf16
    for b, m in enumerate(mags):
        a["win"][b] = S.to_bf16_bits((f32(arrs["win"][b]) * m).astype(np.float32))
        i["x"][b] = S.to_bf16_bits((f32(inp["x"][b]) * m).astype(np.float32))
        i["q"][b] = S.to_bf16_bits((f32(inp["q"][b]) / m).astype(np.float32))
        rows = b * w.max_entries + np.arange(w.max_entries)
        a["kv_rope"][rows] = S.to_bf16_bits((f32(arrs["kv_rope"][rows]) * m).astype(np.float32))
        a["kv_scale"][rows] = (arrs["kv_scale"][rows] * np.float32(m)).astype(np.float32)
    return a, i


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_csa_keys_far_outside_f16_range(out):
    w = S.config2(batch=4, ctx=(8192, 4096, 20000, 65536), k=512)
    inp = S.step_inputs(w)
    arrs = S.seeded_cache(w, inp["q_idx"], inp["w_idx"])
    arrs, inp = _scaled(w, arrs, inp, MAGS)
    assert np.abs(H.O.decode_bf16(arrs["win"][0])).max() > 1e5   # beyond f16's largest finite value
    res = H.gpu_seeded_step(w, arrs, inp, torch.bfloat16 if out == "bf16" else torch.float32, chained=True)
    assert np.all(np.isfinite(res["o"])) and np.all(np.isfinite(res["lse"]))
    _check_step(w, arrs, inp, res, H.TOL_LOW, what=f"range {out}", out_bf16=(out == "bf16"))


def test_hca_keys_far_outside_f16_range():
    w = S.config1(batch=4, ctx=(131072, 16384, 65536, 8192))
    inp = S.step_inputs(w)
    arrs = S.seeded_cache(w)
    arrs, inp = _scaled(w, arrs, inp, MAGS)
    res = H.gpu_seeded_step(w, arrs, inp, torch.float32)
    assert np.all(np.isfinite(res["o"]))
    _check_step(w, arrs, inp, res, H.TOL_LOW, what="hca range", out_bf16=False)
