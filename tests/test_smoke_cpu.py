"""The host half of __graft_entry__.smoke() on the CPU: every smoke case draws its
inputs and gets the oracle's decode output, and the tolerance check accepts the
reference itself and rejects a perturbed copy."""
import numpy as np

import __graft_entry__ as G
from long_context_hybrid_02_b300 import synth


def test_smoke_cases_cover_both_kernel_families():
    ws = G.smoke_workloads()
    assert {w.dtype for w in ws} == {"f32", "bf16"}
    assert any(w.dtype == "bf16" and w.d == 512 and w.H % 64 == 0 for w in ws)


def test_smoke_reference_runs_for_every_case():
    for w in G.smoke_workloads():
        tok, qry = synth.make_tokens(w, "cpu"), synth.make_queries(w, "cpu")
        for b in range(w.B):
            o, lse = G.smoke_reference(w, tok, qry, b)
            assert o.shape == (w.H, w.d) and lse.shape == (w.H,)
            assert np.isfinite(o).all() and np.isfinite(lse).all()
            assert G.smoke_excess(o, o, w.dtype) <= 0
            bad = o.copy()
            bad[0, 0] += 1.0
            assert G.smoke_excess(bad, o, w.dtype) > 0
