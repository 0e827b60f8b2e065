"""The sliding-window-only layer (the multi-token-prediction block's attention) and
prefill of a long prompt in chunks, on the GPU through the C ABI.

SWA: a ring seeded with raw tokens, one appended token per sequence, and the
attention over the window and the sink, compared with the oracle per row (bf16 d=512
on the tensor-core kernel, fp32 d=128 on the CUDA-core kernel), contexts shorter and
longer than the window.

Chunked prefill: the same prompt prefilled in one call and in chunks of 256, 300 and
1 tokens gives bitwise identical outputs, indices and lse (every query row is
computed the same way); the one-shot result is compared with the oracle on sampled
rows, for two sequences."""
import numpy as np
import pytest
import torch

import harness as H
import long_context_attention_05_b300 as L
from long_context_attention_05_b300 import synthetic as S
from oracle import csa_oracle as O

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt", ["bf16_d512", "f32_d128"])
def test_window_only_layer(fmt):
    B, W, cap = 4, 128, 128
    d, heads, dt = (512, 64, "bf16") if fmt == "bf16_d512" else (128, 16, "f32")
    ctx = (1000, 5, 127, 70000)
    rng_seed = 7
    ring = S.normal(rng_seed, 1, (B, cap, d))
    x = S.normal(rng_seed, 2, (B, 1, d))
    q = S.normal(rng_seed, 3, (B, 1, heads, d))
    sink = S.normal(rng_seed, 4, (heads,))
    enc = (lambda a: a) if dt == "f32" else S.to_bf16_bits
    ring_s, x_s, q_s = enc(ring), enc(x), enc(q)
    tens = {"win": L.to_device(ring_s), "n_tokens": L.to_device(np.asarray(ctx, np.int64))}
    cache = L.Cache(m=1, d=d, d_rope=64, d_idx=0, kv_dtype=L.CSA_E4M3, win_dtype=L.CSA_F32 if dt == "f32" else L.CSA_BF16,
                    n_win=W, win_cap=cap, max_entries=0, rope_theta=10000.0, tensors=tens)
    L.swa_append(cache, L.to_device(x_s))
    n = L.swa_workspace_size(cache, B, 1, heads)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out = torch.empty((B, 1, heads, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, 1, heads), dtype=torch.float32, device="cuda")
    L.swa_attend(cache, L.to_device(q_s), L.to_device(sink), out, lse, ws)
    torch.cuda.synchronize()
    assert list(tens["n_tokens"].cpu().numpy()) == [c + 1 for c in ctx]
    dec = (lambda a: np.asarray(a, np.float64)) if dt == "f32" else O.decode_bf16
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    tol = H.TOL_F32 if dt == "f32" else H.TOL_LOW
    for b in range(B):
        t = ctx[b]
        r_ring, r_x = dec(ring_s[b]), dec(x_s[b, 0])
        wf = lambda pos: np.array([r_x if int(p) == t else r_ring[int(p) % cap] for p in pos]).reshape(len(pos), d)
        ref = O.query_step("swa", dec(q_s[b, 0]), t, sink.astype(np.float64), np.zeros((0, d)), wf, 1, W, 64, 10000.0)
        H.check_rows(o[b, 0], ref["o"], tol, what=f"swa {fmt} b={b}")
        assert np.all(np.abs(l[b, 0] - ref["lse"]) <= tol * np.maximum(1, np.abs(ref["lse"])))


def _prefill_setup(w):
    inp = S.step_inputs(w)
    arrs = S.seeded_cache(w, inp["q_idx"], inp["w_idx"])
    return arrs, inp


def test_chunked_prefill_equals_one_shot_and_the_oracle():
    w = S.config3(batch=2, ctx=(4096, 2048), n_new=600, k=128)
    arrs, inp = _prefill_setup(w)
    one = H.gpu_seeded_step(w, arrs, inp, torch.float32, chained=True)
    for chunk in (256, 300, 1):
        cache = L.Cache.from_host(w, arrs)
        gi = H.gpu_inputs(w, inp)
        out = torch.empty((w.batch, w.n_new, w.heads, w.d), dtype=torch.float32, device="cuda")
        lse = torch.empty((w.batch, w.n_new, w.heads), dtype=torch.float32, device="cuda")
        L.csa_prefill_chunked(cache, chunk, gi["x"], gi["gate"], gi["pos_bias"], gi["idx_x"], gi["idx_gate"],
                              gi["idx_pos_bias"], gi["q_idx"], gi["w_idx"], gi["q"], gi["sink"], w.k, out, lse)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), one["o"]), chunk
        assert np.array_equal(lse.cpu().numpy(), one["lse"]), chunk
        assert list(cache.t["n_tokens"].cpu().numpy()) == [c + w.n_new for c in w.ctx]
    from test_parity_decode import _check_step
    rows = [(0, 0), (0, 1), (0, 255), (0, 256), (0, 599), (1, 0), (1, 300), (1, 599)]
    _check_step(w, arrs, inp, one, H.TOL_LOW, rows=rows, what="chunked prefill", out_bf16=False)
