"""bench.py's algorithmic work per launch (the roofline numerators), counted independently.

The selected rows must be what the oracle's top-k actually returns (min(k, L_t) per query),
and the FLOP and byte counts must follow from them and from the tensor shapes.
"""
import numpy as np

import bench
from dsa_indexer_cross_gb300 import synth
from oracle import dsa_oracle as O


def test_roofline_counts_match_the_oracle_selection_on_tiny():
    w = synth.WORKLOADS["tiny"]
    geo = synth.geometry(w)
    L = synth.layer_inputs(w, geo, 0, device="cpu", with_attn=False)
    idx = O.indexer_topk(synth.to_f64(L["q_idx"]), synth.to_f64(L["k_idx"]), synth.to_f64(L["w"]), geo.q_pos,
                         geo.k_pos, geo.ks, geo.ke, w.rope_dim, w.theta, w.topk)
    selected = int((idx >= 0).sum())
    R = bench.roofline_numbers(w, geo)
    assert R["rows"] == selected
    pairs = sum(int(geo.ke[t] - geo.ks[t]) for t in range(w.n_q))
    assert R["pairs"] == pairs
    assert R["attn_flops"] == 2.0 * selected * w.n_heads * (w.d_qk + w.d_v)
    scored = sum(int(geo.ke[t] - geo.ks[t]) for t in range(w.n_q) if geo.ke[t] - geo.ks[t] > w.topk)
    assert R["idx_flops"] == 2.0 * scored * w.n_heads_idx * w.head_dim_idx
    assert R["idx_flops_causal"] == 2.0 * pairs * w.n_heads_idx * w.head_dim_idx
    gathered = selected * w.d_qk * 2 + w.n_q * w.n_heads * (w.d_qk + w.d_v) * 2 + w.n_q * w.topk * 4
    assert R["attn_gathered"] == gathered


def test_prefill_4k_selected_pairs():
    # causal prefill of 4096 tokens with k = 2048: rows t < 2048 select their whole prefix
    # (t + 1 keys), the rest select k
    w = synth.WORKLOADS["prefill_4k"]
    R = bench.roofline_numbers(w, synth.geometry(w))
    assert R["rows"] == sum(t + 1 for t in range(2048)) + 2048 * 2048 == 6_292_480
    assert R["attn_flops"] == 2.0 * 6_292_480 * 16 * 1088


def test_traffic_figure_is_keyed_to_its_sources(tmp_path, monkeypatch):
    """The captured DRAM traffic is reported only while the kernel and planner sources are the
    ones it was captured from; a layout-only change keeps it, any other change drops it."""
    csrc = tmp_path / "dsa_indexer_cross_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("int f(int x) {\n  return x + 1;\n}\n")
    (csrc / "p.cu").write_text("int g() { return 2; }\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench._src_sha(("k.cu", "p.cu"))
    monkeypatch.setitem(bench.MEASURED_TRAFFIC, ("kern", "wl"), (123.0, ("k.cu", "p.cu"), sha, "a capture"))
    assert bench.traffic_for("kern", "wl")[0] == 123.0
    (csrc / "k.cu").write_text("int f(int x)\n{\n    return x + 1;   \n}\n")   # layout only
    assert bench.traffic_for("kern", "wl")[0] == 123.0
    (csrc / "p.cu").write_text("int g() { return 3; }\n")
    nbytes, why = bench.traffic_for("kern", "wl")
    assert nbytes is None and "changed since the capture" in why
    assert bench.traffic_for("other", "wl")[0] is None
