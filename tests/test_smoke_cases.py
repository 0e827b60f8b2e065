"""The cases the smoke entry point runs are well formed (one context length per
row) and the oracle computes them; the GPU side of smoke() is exercised on a GPU."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import __graft_entry__ as G  # noqa: E402
import harness as H  # noqa: E402
from long_context_attention_05_b300 import synthetic as S  # noqa: E402


def test_smoke_cases_are_consistent_and_the_oracle_runs_them():
    for w in G.smoke_workloads():
        assert len(w.ctx) == w.batch, w.name
        inp = S.step_inputs(w)
        arrs = S.seeded_cache(w, inp.get("q_idx"), inp.get("w_idx"))
        for b in range(w.batch):
            ref = H.oracle_seeded_step(w, arrs, inp, b, 0)
            assert np.isfinite(ref["o"]).all()
