"""Fused score -> select (GPU only).

topk_index_topk_fused moves the selection's proposal and certification into
the score stage: a first score pass over the fixed-stride sample of the keys
gives each query's tau0 and tau1, and the full score pass appends every score
>= tau1 to that query's candidates while it writes the row (the xllm-io
review of LiteTopK, sections "核心思想" and "详细方法": gate the scores while
they are produced; PaperDaily section 问题二 for the thresholds).  The result
must be the exact Top-K of the scores the call wrote: every row passes the
oracle's checker on those scores and equals the oracle's set where the
boundary is untied.  The scores themselves must equal, bit for bit, what
topk_index_scores writes for the same inputs (the gate does not touch them).
Rows whose candidates cannot certify them (C(tau1) < K, or more candidates
than the area holds) are forced here and must come out exact as well.
"""
import numpy as np
import pytest
import torch

from exact_top_sparse_gb300 import synth
from tests.test_parity_gpu import verify

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def ets():
    import __graft_entry__ as g
    g.build()
    import exact_top_sparse_gb300 as m
    return m


@pytest.fixture
def params(ets):
    old = ets.get_params()
    yield ets
    ets.set_params(**old)


def _check(ets, q, k, w, lens, K, diag=True):
    dl = lens.to(DEV)
    scores, idx, dg = ets.topk_index_topk_fused(q, k, w, dl, K, diag=True)
    plain = ets.topk_index_scores(q, k, w, row_lens=dl)
    torch.cuda.synchronize()
    assert ets.index_read_status() == 0
    assert torch.equal(scores, plain)
    verify(scores, lens, K, idx)
    assert not np.any(dg["flags"] & (ets.FLAG_INTERNAL | ets.FLAG_TIMEOUT))
    return scores, idx, dg


@pytest.mark.parametrize("T,S", [(64, 65536), (256, 131072), (2048, 262144)])
def test_fused_equals_the_oracle_on_its_scores(ets, T, S):
    q, k, w, lens = synth.index_inputs(T, S, seed=T + 7, device=DEV)
    _, _, dg = _check(ets, q, k, w, lens, 2048)
    sampled = dg["path"] >= ets.PATH_TAU0
    # most rows are served from their candidates (tau0 path)
    assert (dg["path"] == ets.PATH_TAU0).sum() >= 0.9 * sampled.sum()


def test_fused_short_rows_sentinels_and_unsampled(ets):
    """Valid lengths from 0 to S: sentinel rows (len <= K), rows below the
    sampling minimum (exact path on the written row) and sampled rows."""
    T, S = 48, 32768
    q, k, w, _ = synth.index_inputs(T, S, seed=9, device=DEV)
    lens = torch.tensor([0, 1, 2047, 2048, 2049, 3000, 5000, 12287, 12288, 12289, 20000, S]
                        + [S - 700 * i for i in range(T - 12)], dtype=torch.int32)
    _, _, dg = _check(ets, q, k, w, lens, 2048)
    assert set(dg["path"][:4].tolist()) == {ets.PATH_SENTINEL}
    assert dg["path"][4] == ets.PATH_DIRECT and dg["path"][11] >= ets.PATH_TAU0


def test_fused_underfilled_rows_recover_from_the_written_row(params):
    """Targets at K itself on a coarse stride: about half the rows admit
    fewer than K scores (tau1 path or exact recovery over the written row)."""
    ets = params
    ets.set_params(stride=1024, rho0=1.0, rho1=1.0, long_len=0)
    T, S = 128, 65536
    q, k, w, lens = synth.index_inputs(T, S, seed=21, device=DEV)
    _, _, dg = _check(ets, q, k, w, lens, 2048)
    assert (dg["path"] == ets.PATH_RECOVERY).sum() > 0
    assert (dg["path"] == ets.PATH_TAU0).sum() > 0


def test_fused_overflowing_rows_reread_the_written_row(ets):
    """All weights zero: every valid score is 0, so every one is admitted and
    rows longer than the candidate area overflow; any K indices are right."""
    T, S = 16, 65536
    q, k, w, lens = synth.index_inputs(T, S, seed=4, device=DEV)
    w.zero_()
    _, _, dg = _check(ets, q, k, w, lens, 2048)
    assert np.all(dg["flags"][lens.numpy() > 16384] & ets.FLAG_OVERFLOW)


@pytest.mark.parametrize("K", [1, 100, 4096])
def test_fused_other_k(ets, K):
    T, S = 32, 65536
    q, k, w, lens = synth.index_inputs(T, S, seed=K, device=DEV)
    _check(ets, q, k, w, lens, K)


def test_fused_graph_replay_with_new_queries(ets):
    T, S = 64, 65536
    q, k, w, lens = synth.index_inputs(T, S, seed=33, device=DEV)
    dl = lens.to(DEV)
    scores = torch.empty((T, S), dtype=torch.float32, device=DEV)
    out = torch.empty((T, 2048), dtype=torch.int32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ets.topk_index_topk_fused(q, k, w, dl, 2048, scores=scores, out=out, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ets.topk_index_topk_fused(q, k, w, dl, 2048, scores=scores, out=out, stream=s)
    q2, _, w2, _ = synth.index_inputs(T, S, seed=34, device=DEV)
    q.copy_(q2)
    w.copy_(w2)
    out.fill_(-7)
    g.replay()
    s.synchronize()
    verify(scores, lens, 2048, out)
    assert torch.equal(scores, ets.topk_index_scores(q, k, w, row_lens=dl))


def test_fused_argument_errors(ets):
    lib = ets.load_library()
    q, k, w, lens = synth.index_inputs(4, 256, seed=1, device=DEV)
    dl = lens.to(DEV)
    sc = torch.empty((4, 256), dtype=torch.float32, device=DEV)
    out = torch.empty((4, 16), dtype=torch.int32, device=DEV)
    args = [q.data_ptr(), k.data_ptr(), w.data_ptr(), 4, 256, 64, 128, dl.data_ptr(),
            sc.data_ptr(), 256, 16, out.data_ptr(), None, None]
    assert lib.topk_index_topk_fused(*args) == 0
    torch.cuda.synchronize()
    no_lens = list(args); no_lens[7] = None
    assert lib.topk_index_topk_fused(*no_lens) == -1
    big_k = list(args); big_k[10] = 5000
    assert lib.topk_index_topk_fused(*big_k) == -6
    bad_s = list(args); bad_s[4] = 200
    assert lib.topk_index_topk_fused(*bad_s) == -8
