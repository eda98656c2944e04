"""Indexer-score stage on the tensor cores against the CPU oracle (GPU only).

The kernel evaluates eq. (1) of the xllm-io LiteTopK review ("核心公式"),
I[t][s] = sum_j w[t][j] * ReLU(q[t][j] . k[s]), from bfloat16 q and k with
FP32 accumulation; the oracle evaluates the same sums in double from the
same bfloat16 values.

Tolerance.  Let M = sum_j |w_tj| * sum_d |q_tjd * k_sd| and u = 2^-24 (FP32
unit roundoff).  Each product q_tjd * k_sd of two bfloat16 values (8
significant bits each) is exact in FP32.  Recursive FP32 summation of the 128
products of a head errs by at most 127 rounding errors, each no larger than
the running sum of magnitudes: |fl(dot_j) - dot_j| <= 127 * e * sum_d |p_d|,
with e = u for round-to-nearest and e = 2u for an accumulator that truncates
(the tensor core's internal order and rounding are not IEEE round-to-nearest
per step, so 2u is assumed).  ReLU adds no error and does not enlarge one;
the product with w_tj adds one rounding (u) and the FP32 sum over 64 heads
at most 63 more (u each), all relative to M at most.  First order:
|gpu - exact| <= (127 * 2 + 1 + 63) * u * M = 318 * 2^-24 * M < 2^-15.68 * M.
The test admits |gpu - oracle| <= 2^-14 * M + 1e-30: a margin of 3.2 over
that worst case (5.4 if the tensor core rounded to nearest), and the oracle's
own double-precision error is below 2^-45 * M.  The bound is a worst case;
typical errors are far smaller.  The causal suffix (s >= row_lens[t]) must be
exactly -inf.  The chained Top-K is exact
on the scores the GPU produced: it must pass the oracle's set contract on
those scores and equal the oracle's set wherever the boundary is untied.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_top_sparse_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
TOL = 2.0 ** -14


@pytest.fixture(scope="module")
def ets():
    import __graft_entry__ as g
    g.build()
    import exact_top_sparse_gb300 as m
    return m


def check_pairs(q, k, w, got, ts, ss):
    val, mag = oracle.index_scores(synth.bf16_bits(q), synth.bf16_bits(k), w.cpu().numpy(), ts, ss)
    g = got[torch.as_tensor(ts, device=got.device), torch.as_tensor(ss, device=got.device)]
    g = g.double().cpu().numpy()
    err = np.abs(g - val)
    bad = np.nonzero(err > TOL * mag + 1e-30)[0]
    assert bad.size == 0, "pairs %s: gpu %s oracle %s" % (
        list(zip(np.asarray(ts)[bad[:4]], np.asarray(ss)[bad[:4]])), g[bad[:4]], val[bad[:4]])
    return float((err / np.maximum(mag, 1e-30)).max())


@pytest.mark.parametrize("T,S", [(4, 128), (8, 1024), (12, 33024)])
def test_every_pair_small(ets, T, S):
    q, k, w, lens = synth.index_inputs(T, S, seed=T + S, device=DEV)
    got = ets.topk_index_scores(q, k, w)
    torch.cuda.synchronize()
    ts, ss = np.meshgrid(np.arange(T), np.arange(S), indexing="ij")
    check_pairs(q, k, w, got, ts.ravel(), ss.ravel())


def test_several_units_and_causal_mask(ets):
    # 2 key chunks per query block (the second one partial), 10 query blocks
    T, S = 40, 65536 + 4096
    q, k, w, lens = synth.index_inputs(T, S, seed=3, device=DEV)
    dl = lens.to(DEV)
    got = ets.topk_index_scores(q, k, w, row_lens=dl)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    ts = rng.integers(0, T, 6000)
    ss = np.minimum(rng.integers(0, S, 6000), lens.numpy()[ts] - 1)
    ts = np.concatenate([ts, np.arange(T), np.arange(T)])
    ss = np.concatenate([ss, np.zeros(T, np.int64), lens.numpy() - 1])
    check_pairs(q, k, w, got, ts, ss)
    cols = torch.arange(S, device=DEV)
    masked = cols[None, :] >= dl[:, None]
    assert bool(torch.isneginf(got[masked]).all())
    assert bool(torch.isfinite(got[~masked]).all())


def test_short_valid_lengths_skip_tiles(ets):
    """Query blocks whose valid lengths end early compute only the tiles they
    need; the rest of each row, and rows of length 0, are exactly -inf."""
    T, S = 48, 8192
    q, k, w, _ = synth.index_inputs(T, S, seed=8, device=DEV)
    lens = torch.tensor([0, 0, 0, 0] + [1, 2, 127, 128] + [129, 300, 1000, 4096]
                        + [8192 - 5 * i for i in range(36)], dtype=torch.int32)
    dl = lens.to(DEV)
    got = ets.topk_index_scores(q, k, w, row_lens=dl)
    torch.cuda.synchronize()
    ts, ss = [], []
    for t in range(T):
        L = int(lens[t])
        if L > 0:
            cols = np.unique(np.concatenate([np.arange(min(L, 40)), np.arange(max(0, L - 40), L)]))
            ts.append(np.full(cols.size, t)); ss.append(cols)
    check_pairs(q, k, w, got, np.concatenate(ts), np.concatenate(ss))
    cols = torch.arange(S, device=DEV)
    masked = cols[None, :] >= dl[:, None]
    assert bool(torch.isneginf(got[masked]).all()) and bool(torch.isfinite(got[~masked]).all())


def test_full_size_scores_sampled(ets):
    """T = 2048 queries over S = 262144 keys (the chain's configuration):
    sampled pairs against the oracle, the causal suffix everywhere."""
    T, S = 2048, 262144
    q, k, w, lens = synth.index_inputs(T, S, seed=11, device=DEV)
    dl = lens.to(DEV)
    got = ets.topk_index_scores(q, k, w, row_lens=dl)
    torch.cuda.synchronize()
    assert ets.index_read_status() == 0
    rng = np.random.default_rng(2)
    ts = rng.integers(0, T, 4000)
    ss = np.minimum(rng.integers(0, S, 4000), lens.numpy()[ts] - 1)
    check_pairs(q, k, w, got, ts, ss)
    cols = torch.arange(S, device=DEV)
    for r0 in range(0, T, 256):
        blk = got[r0:r0 + 256]
        masked = cols[None, :] >= dl[r0:r0 + 256, None]
        assert bool(torch.isneginf(blk[masked]).all()) and bool(torch.isfinite(blk[~masked]).all())


@pytest.mark.parametrize("T,S", [(64, 65536), (2048, 262144)])
def test_chained_topk_is_exact_on_the_scores(ets, T, S):
    q, k, w, lens = synth.index_inputs(T, S, seed=T, device=DEV)
    dl = lens.to(DEV)
    scores, idx = ets.topk_index_topk(q, k, w, dl, 2048)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, T - 1], np.random.default_rng(4).integers(0, T, 30)]))
    xs = scores[torch.as_tensor(rows, device=DEV)].cpu().numpy()
    v = oracle.compare(xs, lens.numpy()[rows], 2048, idx[torch.as_tensor(rows, device=DEV)].cpu().numpy())
    assert not v["check"].any() and not v["set_mismatch"].any()
    # the selected scores themselves agree with the oracle
    sel = idx[torch.as_tensor(rows[:4], device=DEV)].cpu().numpy()
    ts = np.repeat(rows[:4], 64)
    ss = sel[:, :64].ravel()
    check_pairs(q, k, w, scores, ts, ss)


def test_graph_replay_of_the_chain(ets):
    T, S = 64, 32768
    q, k, w, lens = synth.index_inputs(T, S, seed=5, device=DEV)
    dl = lens.to(DEV)
    scores = torch.empty((T, S), dtype=torch.float32, device=DEV)
    out = torch.empty((T, 2048), dtype=torch.int32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ets.topk_index_topk(q, k, w, dl, 2048, scores=scores, out=out, stream=s)  # workspace
    s.synchronize()
    ref = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ets.topk_index_topk(q, k, w, dl, 2048, scores=scores, out=out, stream=s)
    out.fill_(-7)
    scores.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.sort(dim=1).values, ref.sort(dim=1).values)


def test_shape_and_alignment_errors(ets):
    q, k, w, lens = synth.index_inputs(4, 256, seed=1, device=DEV)
    lib = ets.load_library()
    ok = lambda *a: lib.topk_index_scores(*a)
    sc = torch.empty((4, 256), dtype=torch.float32, device=DEV)
    base = [q.data_ptr(), k.data_ptr(), w.data_ptr(), 4, 256, 64, 128, None, sc.data_ptr(), 256, None]
    assert ok(*base) == 0
    torch.cuda.synchronize()
    bad_h = list(base); bad_h[5] = 32
    assert ok(*bad_h) == -8
    bad_t = list(base); bad_t[3] = 3
    assert ok(*bad_t) == -8
    bad_s = list(base); bad_s[4] = 200
    assert ok(*bad_s) == -8
    bad_ld = list(base); bad_ld[9] = 255
    assert ok(*bad_ld) == -1
    mis = list(base); mis[0] = q.data_ptr() + 2
    assert ok(*mis) == -2
