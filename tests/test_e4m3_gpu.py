"""FP8 E4M3 score rows through the same selector (GPU only).

Every E4M3 value is a binary32 value, so the exact Top-K of E4M3 rows is the
exact Top-K of their widened values: the oracle runs on the copy widened by
PyTorch's own float8_e4m3fn conversion, and every row must pass its set
contract, equal its set on untied rows, and (for sampled rows) reproduce its
thresholds, counts and path.  With 8 values per octave the rows are mostly
ties, which drives the all-equal frontier and the candidate overflow path.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_top_sparse_gb300 import synth
from tests.test_parity_gpu import verify, verify_diag

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
K = 2048
E4M3 = torch.float8_e4m3fn


@pytest.fixture
def params():
    import __graft_entry__ as g
    g.build()
    import exact_top_sparse_gb300 as m
    old = m.get_params()
    yield m
    m.set_params(**old)


def e4m3_rows(lens, N, seed, scale=1.0):
    """Indexer-like rows scaled, held below the largest E4M3 value (448) and
    rounded to E4M3 (the -inf suffix becomes NaN, which lies past every row's
    length and is never read)."""
    x = synth.indexer_rows(lens, N, seed=seed, device=DEV) * scale
    x = x.clamp(max=448.0).to(E4M3)
    return x, x.float()


@pytest.mark.parametrize("kind", ["auto", "direct", "persistent", "kvsplit"])
def test_e4m3_kinds_match_the_oracle(params, kind):
    ets = params
    N, M = 40960, 64
    kinds = {"auto": 0, "direct": ets.KIND_DIRECT, "persistent": ets.KIND_PERSISTENT,
             "kvsplit": ets.KIND_KVSPLIT}
    ets.set_params(force_kind=kinds[kind], sample_min_len=0 if kind != "auto" else 12288,
                   kv_segments=3 if kind == "kvsplit" else 0)
    lens = synth.causal_lens(N, M, 0, window=4096)
    lens[:3] = torch.tensor([0, 2048, 2049], dtype=torch.int32)
    x, xf = e4m3_rows(lens, N, seed=3, scale=4.0)
    got, dg = ets.topk_ragged_diag(x, lens.to(DEV), K)
    torch.cuda.synchronize()
    verify(xf, lens, K, got)
    if kind in ("persistent", "kvsplit"):
        verify_diag(ets, xf, lens, K, dg)


def test_every_pattern_in_order(params):
    """Rows holding each non-NaN E4M3 byte (both zeros, subnormals, normals up
    to 448, both signs) in shuffled order: the selection and the sorted result
    follow the values PyTorch's conversion gives those bytes."""
    ets = params
    pats = torch.tensor([b for b in range(256) if b not in (0x7F, 0xFF)], dtype=torch.uint8)
    rows = []
    g = torch.Generator().manual_seed(1)
    for _ in range(6):
        rows.append(pats[torch.randperm(pats.numel(), generator=g)])
    xb = torch.stack(rows)
    x = xb.view(E4M3).to(DEV)
    xf = xb.view(E4M3).float()
    n = pats.numel()
    lens = torch.full((6,), n, dtype=torch.int32)
    for kind in (ets.KIND_DIRECT, ets.KIND_PERSISTENT, ets.KIND_KVSPLIT):
        ets.set_params(force_kind=kind, sample_min_len=0, stride=4,
                       kv_segments=2 if kind == ets.KIND_KVSPLIT else 0)
        for k in (1, 37, 126, 127, 200):
            got = ets.topk_ragged(x, lens.to(DEV), k)
            before = got.clone()
            ets.topk_sort_rows(x, got)
            torch.cuda.synchronize()
            # the ordered form of the selected set, entry by entry (+0 and -0
            # are equal scores: the one tie, ordered by index)
            want = oracle.order(xf.numpy(), lens.numpy(), k, before.cpu().numpy())
            assert np.array_equal(got.cpu().numpy(), want), (kind, k)
            verify(xf.to(DEV), lens, k, got)


@pytest.mark.parametrize("N,M,kind", [(1048576, 16, "auto"), (1048576, 64, "persistent"),
                                      (262144, 256, "auto")])
def test_e4m3_long_rows(params, N, M, kind):
    """Long rows: the tie runs at the boundary span thousands of scores, so
    candidate counts overflow the on-chip buffer and the row is re-read."""
    ets = params
    if kind == "persistent":
        ets.set_params(force_kind=ets.KIND_PERSISTENT)
    lens = synth.causal_lens(N, M, group=0, window=M)
    x, xf = e4m3_rows(lens, N, seed=N + M, scale=8.0)
    assert not any(bool(torch.isnan(xf[r, :int(lens[r])]).any()) for r in range(M))
    got, dg = ets.topk_ragged_diag(x, lens.to(DEV), K)
    torch.cuda.synchronize()
    verify(xf, lens, K, got)
    verify_diag(ets, xf, lens, K, dg, sample_min_len=ets.get_params()["sample_min_len"])
    assert not np.any(dg["flags"] & (ets.FLAG_INTERNAL | ets.FLAG_TIMEOUT))


@pytest.mark.parametrize("N", [65537, 65551])
def test_e4m3_unaligned_rows(params, N):
    """Odd row strides: rows start at every byte offset, so the 16-byte
    aligned body is preceded and followed by up to 15 scores."""
    ets = params
    M = 20
    ets.set_params(sample_min_len=0)
    lens = torch.tensor([N - 5 * i for i in range(M)], dtype=torch.int32)
    x, xf = e4m3_rows(lens, N, seed=N, scale=2.0)
    for kind in (ets.KIND_PERSISTENT, ets.KIND_KVSPLIT):
        ets.set_params(force_kind=kind, kv_segments=5 if kind == ets.KIND_KVSPLIT else 0)
        got = ets.topk_ragged(x, lens.to(DEV), K)
        torch.cuda.synchronize()
        verify(xf, lens, K, got)


def test_e4m3_per_row_k(params):
    ets = params
    N, K_max = 131072, 4096
    ks = torch.tensor([0, 1, 5, 2048, 4096, 300, 4095, 17], dtype=torch.int32)
    lens = torch.tensor([N, N, 20000, N - 1, 100000, 4000, N, 9], dtype=torch.int32)
    x, xf = e4m3_rows(lens, N, seed=77, scale=4.0)
    out = ets.topk_ragged_k(x, lens.to(DEV), ks.to(DEV), K_max)
    torch.cuda.synchronize()
    v = oracle.compare_per_row(xf.cpu().numpy(), lens.numpy(), ks.numpy(), K_max,
                               out.cpu().numpy())
    assert not v["check"].any() and not v["set_mismatch"].any() and not v["tail"].any()
