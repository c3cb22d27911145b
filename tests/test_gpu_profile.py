"""Per-phase profiling of the indexer call (GPU): same results with and without it."""
import pytest
import torch

import dsa_indexer_cross_gb300 as D
from dsa_indexer_cross_gb300 import synth

from gpu_cases import run_indexer

pytestmark = pytest.mark.gpu


def test_profiled_indexer_call_reports_phases_and_keeps_results():
    w = synth.WORKLOADS["tiny"]
    geo = synth.geometry(w)
    L = synth.layer_inputs(w, geo, 0, device="cuda")
    idx_plain, _, bits = run_indexer(w, geo, L)
    assert bits == 0
    D.dsa_profile_enable(True)
    try:
        idx_prof, _, bits = run_indexer(w, geo, L)
        ms = D.dsa_profile_indexer_last()
    finally:
        D.dsa_profile_enable(False)
    assert bits == 0
    assert torch.equal(idx_plain, idx_prof)
    assert len(ms) == 4 and all(m >= 0.0 for m in ms)
    assert ms[2] > 0.0                    # the score kernel ran
    assert sum(ms) < 1000.0
