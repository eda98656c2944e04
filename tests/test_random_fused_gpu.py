"""Seeded random calls of the fused score -> select path (GPU only).

Sixteen calls of topk_index_topk_fused, each drawn from a fixed seed: query
count T (a multiple of 4), key count S (a multiple of 128), K, the valid
lengths (causal, uniform, or with empty and short queries mixed in), the
weights (positive, or of both signs so that scores and thresholds go
negative), and the sampling tier.  The fused call gates every score it
writes against the query's tau1 and selects from the survivors (xllm-io
LiteTopK review, "二、核心思想" and "详细方法"; thresholds and certification
as in PaperDaily 问题二).  Its scores must equal topk_index_scores' bit for
bit, and every row must pass the oracle's checker on those scores and equal
the oracle's set where its boundary is untied.
"""
import numpy as np
import pytest
import torch

from exact_top_sparse_gb300 import synth
from tests.test_parity_gpu import verify

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
CASES = 16


@pytest.fixture(scope="module")
def ets():
    import __graft_entry__ as g
    g.build()
    import exact_top_sparse_gb300 as m
    return m


def draw(i):
    g = np.random.default_rng(3000 + i)
    T = int(g.choice([4, 8, 36, 128, 260]))
    S = 128 * int(g.choice([8, 96, 160, 512, 1024, 2048]))
    K = int(g.choice([1, 64, 1000, 2048, 4096]))
    lens_kind = str(g.choice(["causal", "uniform", "mixed"]))
    signed = bool(g.random() < 0.3)
    stride = int(g.choice([64, 128, 256, 512]))
    rho0 = float(np.round(g.uniform(1.0, 3.0), 2))
    rho1 = float(np.round(rho0 + g.uniform(0.0, 0.75), 2))
    return dict(T=T, S=S, K=K, lens_kind=lens_kind, signed=signed, stride=stride, rho0=rho0,
                rho1=rho1, seed=4000 + i)


@pytest.mark.parametrize("i", range(CASES))
def test_random_fused_case(ets, i):
    c = draw(i)
    T, S, K = c["T"], c["S"], c["K"]
    g = np.random.default_rng(c["seed"])
    q, k, w, lens = synth.index_inputs(T, S, seed=c["seed"], device=DEV)
    if c["signed"]:
        w = w * 2.0 - 0.125
    if c["lens_kind"] == "uniform":
        lens = torch.from_numpy(g.integers(1, S + 1, T).astype(np.int32))
    elif c["lens_kind"] == "mixed":
        lv = g.integers(0, S + 1, T).astype(np.int32)
        lv[g.random(T) < 0.15] = 0
        short = g.random(T) < 0.25
        lv[short] = g.integers(0, 2 * K + 2, int(short.sum()))
        lens = torch.from_numpy(np.minimum(lv, S).astype(np.int32))
    old = ets.get_params()
    try:
        ets.set_params(stride=c["stride"], rho0=c["rho0"], rho1=c["rho1"], long_len=0)
        dl = lens.to(DEV)
        scores, idx, dg = ets.topk_index_topk_fused(q, k, w, dl, K, diag=True)
        plain = ets.topk_index_scores(q, k, w, row_lens=dl)
        torch.cuda.synchronize()
        assert ets.index_read_status() == 0, c
        assert torch.equal(scores, plain), c
        verify(scores, lens, K, idx)
        assert not np.any(dg["flags"] & (ets.FLAG_INTERNAL | ets.FLAG_TIMEOUT)), c
    finally:
        ets.set_params(**old)
