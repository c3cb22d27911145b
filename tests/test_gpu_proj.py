"""GPU parity of the indexer's input projections (dsa_indexer_projections) against the oracle.

fp32 accumulation on the tensor cores, rounded once to bf16 for q_idx and k_idx: within the
standard error bound of an fp32 sum of K products (K 2^-23 sum |a b|) plus two bf16 spacings
(three for k_idx, whose LayerNorm statistics are fp32, with the bound scaled by |gamma| / std);
w in fp32 within twice the accumulation bound.  Shapes span several token tiles with a
ragged tail, several K blocks, narrow (4-head) and wide (64 x 128) index heads.
"""
import math

import numpy as np
import pytest
import torch

import dsa_indexer_cross_gb300 as D
from dsa_indexer_cross_gb300 import synth
from gpu_cases import DEV
from oracle import dsa_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dsa_indexer_cross_gb300.build import build
    build()
    assert torch.cuda.is_available()


def _ulp(ref: np.ndarray) -> np.ndarray:
    """bf16 spacing (8 significant bits) at |ref|."""
    return 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 7)


@pytest.mark.parametrize("T,Dh,Dq,H,d", [(300, 256, 192, 64, 128), (77, 128, 64, 4, 64), (1, 64, 128, 32, 128)])
def test_projections_match_oracle(T, Dh, Dq, H, d):
    g = torch.Generator(device=DEV)
    g.manual_seed(T * 7 + H)
    rn = lambda *s: torch.randn(s, generator=g, device=DEV, dtype=torch.float32)
    x = (rn(T, Dh) * 0.5).to(torch.bfloat16)
    ql = (rn(T, Dq) * 0.5).to(torch.bfloat16)
    wq = (rn(H * d, Dq) / math.sqrt(Dq)).to(torch.bfloat16)
    wk = (rn(d, Dh) / math.sqrt(Dh)).to(torch.bfloat16)
    wp = (rn(H, Dh) / math.sqrt(Dh)).to(torch.bfloat16)
    gamma = 1.0 + 0.1 * rn(d)
    beta = 0.1 * rn(d)
    q_idx = torch.empty((T, H, d), dtype=torch.bfloat16, device=DEV)
    k_idx = torch.empty((T, d), dtype=torch.bfloat16, device=DEV)
    w = torch.empty((T, H), dtype=torch.float32, device=DEV)
    ws = D.dsa_indexer_projections(D.ProjDesc(T, Dh, Dq, H, d, 1e-6), x, ql, wq, wk, gamma, beta, wp, q_idx, k_idx, w)
    assert D.dsa_workspace_status(ws) == 0
    f = synth.to_f64
    q_ref, k_ref, w_ref = O.indexer_projections(f(x), f(ql), f(wq), f(wk), f(gamma), f(beta), f(wp), H, d, 1e-6)
    # fp32 accumulation of K products: |error| <= K u sum_i |a_i b_i| (standard GEMM bound),
    # then one rounding to bf16 on each side (two bf16 spacings)
    gam = lambda A, B: np.abs(A) @ np.abs(B).T
    u = 2.0 ** -23   # allows the accumulator to truncate rather than round
    q_bound = (2 * _ulp(q_ref).reshape(T, H * d) + Dq * u * gam(f(ql), f(wq))).reshape(T, H, d)
    assert np.all(np.abs(f(q_idx) - q_ref) <= q_bound)
    # the key's accumulation error passes through the LayerNorm scale (|gamma| / std), plus two
    # bf16 spacings for the fp32 statistics and the final rounding
    y = f(x) @ f(wk).T
    rstd = 1.0 / np.sqrt(y.var(axis=1, keepdims=True) + 1e-6)
    k_bound = 3 * _ulp(k_ref) + 4 * np.abs(f(gamma)) * rstd * Dh * u * gam(f(x), f(wk)).max(axis=1, keepdims=True)
    assert np.all(np.abs(f(k_idx) - k_ref) <= k_bound)
    w_bound = 2 * Dh * u * gam(f(x), f(wp)) + 1e-30
    assert np.all(np.abs(f(w) - w_ref) <= w_bound)
