"""Per-row K on the GPU against the oracle (GPU only).

Row r selects k_r = clamp(row_k[r], 0, K_max) into the first k_r slots of an
[M, K_max] result, -1 in the rest.  Each row must pass the one-K checker at
k_r and equal the oracle's set when its boundary is untied; sampled rows
also have thresholds, counts and path compared with the oracle's stage-1/2
definition at their own targets ceil(rho * k_r).
"""
import numpy as np
import pytest
import torch

import oracle
from exact_top_sparse_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
KINDS = ["direct", "persistent", "kvsplit"]


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


def force(ets, kind, **kw):
    kinds = {"direct": ets.KIND_DIRECT, "persistent": ets.KIND_PERSISTENT,
             "kvsplit": ets.KIND_KVSPLIT, "auto": ets.KIND_AUTO}
    ets.set_params(force_kind=kinds[kind], **kw)


def verify(x, lens, ks, K_max, got):
    v = oracle.compare_per_row(x.float().cpu().numpy(), lens.cpu().numpy(), ks.cpu().numpy(),
                               K_max, got.cpu().numpy())
    bad = np.nonzero(v["check"])[0]
    assert bad.size == 0, "rows %s fail the contract: %s" % (
        bad[:8].tolist(), [oracle.CHECK_CODES[int(c)] for c in v["check"][bad[:8]]])
    assert not v["set_mismatch"].any(), np.nonzero(v["set_mismatch"])[0][:8]
    assert not v["tail"].any(), np.nonzero(v["tail"])[0][:8]
    return v


def verify_diag(ets, x, lens, ks, K_max, diag, sample_min_len=0):
    """Each sampled row's thresholds, counts and path equal the oracle's at
    the row's own K and its tier's targets ceil(rho * k_r)."""
    p = ets.get_params()
    xh, lh = x.cpu().numpy(), lens.cpu().numpy()
    kc = oracle.clamp_row_k(ks.cpu().numpy(), K_max)
    for k in np.unique(kc):
        if k == 0:
            continue
        rows = np.nonzero(kc == k)[0]
        lk = lh[rows]
        long_rows = (lk >= p["long_len"]) if p["long_len"] > 0 else np.zeros(lk.shape, bool)
        for mask, stride, r0, r1 in [(~long_rows, p["stride"], p["rho0"], p["rho1"]),
                                     (long_rows, p["long_stride"], p["long_rho0"],
                                      p["long_rho1"])]:
            if not mask.any():
                continue
            T0 = int(np.ceil(np.float64(np.float32(r0)) * k))
            T1 = max(T0, int(np.ceil(np.float64(np.float32(r1)) * k)))
            sel = rows[mask]
            ref = oracle.thresholds(xh[sel], lh[sel], int(k), stride, T0, T1, sample_min_len)
            d = diag[sel]
            assert np.array_equal(d["path"], ref["path"]), (k, sel)
            s = ref["path"] >= oracle.PATH_TAU0
            assert np.array_equal(d["tau0"][s], ref["tau"][s, 0])
            assert np.array_equal(d["tau1"][s], ref["tau"][s, 1])
            assert np.array_equal(d["count0"][s], ref["count"][s, 0])
            assert np.array_equal(d["count1"][s], ref["count"][s, 1])
    assert not np.any(diag["flags"] & (ets.FLAG_INTERNAL | ets.FLAG_TIMEOUT))


@pytest.mark.parametrize("kind", KINDS)
def test_mixed_k_every_kind(params, kind):
    """k from 0 to K_max and past both ends, on rows shorter and longer than
    k, through every kind; sampled rows with small k take the tau1 and
    recovery paths."""
    ets = params
    force(ets, kind, sample_min_len=0, kv_segments=5 if kind == "kvsplit" else 0)
    N, K_max = 45000, 4096
    ks = torch.tensor([0, 1, 7, 100, 2047, 2048, 4096, -3, 9000, 16, 3000, 2048, 64, 512, 1, 4095],
                      dtype=torch.int32)
    lens = torch.tensor([45000, 45000, 44000, 30001, 45000, 2048, 4097, 45000, 45000, 17, 2999,
                         40000, 0, 45000, 1, 45000], dtype=torch.int32)
    x = synth.indexer_rows(lens, N, seed=21, device=DEV)
    ets.read_status()
    out, dg = ets.topk_ragged_k_diag(x, lens.to(DEV), ks.to(DEV), K_max)
    torch.cuda.synchronize()
    verify(x, lens, ks, K_max, out)
    if kind != "direct":
        verify_diag(ets, x, lens, ks, K_max, dg)
    assert ets.read_status() & ets.FLAG_K_CLAMPED
    clamped = (dg["flags"] & ets.FLAG_K_CLAMPED) != 0
    assert clamped.tolist() == [bool(k < 0 or k > K_max) for k in ks.tolist()]


@pytest.mark.parametrize("kind", ["auto", "persistent", "kvsplit"])
def test_long_rows_random_k(params, kind):
    """256K-1M columns, both sampling tiers, k drawn over [1, 4096]."""
    ets = params
    if kind != "auto":
        force(ets, kind)
    N, M, K_max = 1048576, 24, 4096
    g = torch.Generator().manual_seed(5)
    ks = torch.randint(1, K_max + 1, (M,), generator=g, dtype=torch.int32)
    ks[:4] = torch.tensor([1, 2, 2048, 4096], dtype=torch.int32)
    lens = torch.randint(262144, N + 1, (M,), generator=g, dtype=torch.int32)
    lens[-1] = N
    x = synth.indexer_rows(lens, N, seed=6, device=DEV)
    out, dg = ets.topk_ragged_k_diag(x, lens.to(DEV), ks.to(DEV), K_max)
    torch.cuda.synchronize()
    verify(x, lens, ks, K_max, out)
    verify_diag(ets, x, lens, ks, K_max, dg, sample_min_len=ets.get_params()["sample_min_len"])
    del x


def test_uniform_k_matches_one_k_call(ets):
    """Every row at k = K: the same sets as the one-K call (128K causal rows,
    the operator-matrix shape)."""
    N, M, K = 131072, 512, 2048
    lens = synth.causal_lens(N, M, 3)
    x = synth.indexer_rows(lens, N, seed=33, device=DEV)
    d_lens = lens.to(DEV)
    a = ets.topk_ragged_k(x, d_lens, torch.full((M,), K, dtype=torch.int32, device=DEV), K)
    b = ets.topk_ragged(x, d_lens, K)
    torch.cuda.synchronize()
    assert torch.equal(a.sort(dim=1).values, b.sort(dim=1).values)
    verify(x, lens, torch.full((M,), K, dtype=torch.int32), K, a)


@pytest.mark.parametrize("kind", KINDS)
def test_bf16_rows_per_row_k(params, kind):
    ets = params
    force(ets, kind, sample_min_len=0, kv_segments=3 if kind == "kvsplit" else 0)
    N, K_max = 40000, 2048
    ks = torch.tensor([2048, 1, 0, 300, 2000, 2048, 5], dtype=torch.int32)
    lens = torch.tensor([40000, 40000, 40000, 39000, 1999, 33333, 6], dtype=torch.int32)
    x = synth.indexer_rows(lens, N, seed=8, device=DEV).to(torch.bfloat16)
    out = ets.topk_ragged_k(x, lens.to(DEV), ks.to(DEV), K_max)
    torch.cuda.synchronize()
    verify(x, lens, ks, K_max, out)


def test_per_row_k_in_a_graph(ets):
    """Captured once, replayed with new k values written into the same buffer."""
    N, M, K_max = 131072, 256, 2048
    lens = synth.causal_lens(N, M, 0)
    x = synth.indexer_rows(lens, N, seed=12, device=DEV)
    d_lens = lens.to(DEV)
    ks = torch.full((M,), K_max, dtype=torch.int32, device=DEV)
    out = torch.empty((M, K_max), dtype=torch.int32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ets.topk_ragged_k(x, d_lens, ks, K_max, out=out, stream=s)   # workspace before capture
    s.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        ets.topk_ragged_k(x, d_lens, ks, K_max, out=out, stream=s)
    for seed in (1, 2):
        g = torch.Generator().manual_seed(seed)
        new = torch.randint(0, K_max + 1, (M,), generator=g, dtype=torch.int32)
        ks.copy_(new)
        gr.replay()
        torch.cuda.synchronize()
        verify(x, lens, new, K_max, out)
