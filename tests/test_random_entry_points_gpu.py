"""Seeded random calls through the other entry points (GPU only).

The host-buffer call (host arrays in and out, random chunk sizes, pageable
or page-locked rows), the explicit-workspace call (a caller-owned zeroed
buffer of topk_workspace_bytes), the fixed-scratch call (at most
NOALLOC_MAX_ROWS rows) and the optional row sort, each on rows drawn from a
fixed seed.  Every row must pass the oracle's checker and equal its set where
the boundary is untied (codexqa.cn article, section "什么叫精确，时间怎么量");
the sorted rows must equal the oracle's ordered form of the same selection.
"""
import numpy as np
import pytest
import torch

import oracle
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


def rows(i, M, N, K):
    g = np.random.default_rng(5000 + i)
    lens = g.integers(0, N + 1, M).astype(np.int32)
    lens[g.random(M) < 0.2] = g.integers(0, K + 2)
    lens = torch.from_numpy(np.minimum(lens, N).astype(np.int32))
    return synth.indexer_rows(lens, N, seed=6000 + i, device=DEV), lens


@pytest.mark.parametrize("i", range(6))
def test_host_buffer_random(ets, i):
    g = np.random.default_rng(i)
    N = int(g.choice([20000, 131072, 262144]))
    M = int(g.choice([5, 64, 333]))
    K = int(g.choice([1, 700, 2048]))
    x, lens = rows(i, M, N, K)
    xh = x.cpu()
    if i % 2:
        xh = xh.pin_memory()
    got = ets.topk_ragged_host(xh.numpy(), lens.numpy(), K,
                               rows_per_chunk=int(g.choice([0, 1, 7, 64])))
    v = oracle.compare(xh.numpy(), lens.numpy(), K, got)
    assert not v["check"].any() and not v["set_mismatch"].any()


@pytest.mark.parametrize("i", range(6))
def test_explicit_workspace_random(ets, i):
    g = np.random.default_rng(100 + i)
    N = int(g.choice([50000, 131072, 524288, 1048576]))
    M = int(g.choice([1, 9, 200, 700]))
    K = int(g.choice([16, 2048, 4096]))
    x, lens = rows(100 + i, M, N, K)
    ws = torch.zeros(ets.workspace_bytes(M, N, K), dtype=torch.uint8, device=DEV)
    got = ets.topk_ragged_ws(x, lens.to(DEV), K, ws)
    again = ets.topk_ragged_ws(x, lens.to(DEV), K, ws)  # the workspace resets itself
    torch.cuda.synchronize()
    verify(x, lens, K, got)
    verify(x, lens, K, again)


@pytest.mark.parametrize("i", range(4))
def test_fixed_scratch_random(ets, i):
    g = np.random.default_rng(200 + i)
    N = int(g.choice([40000, 262144, 1048576]))
    M = int(g.integers(1, ets.NOALLOC_MAX_ROWS + 1))
    K = int(g.choice([1, 2048]))
    x, lens = rows(200 + i, M, N, K)
    got = ets.topk_ragged_noalloc(x, lens.to(DEV), K)
    torch.cuda.synchronize()
    verify(x, lens, K, got)


@pytest.mark.parametrize("i", range(4))
def test_sorted_random(ets, i):
    g = np.random.default_rng(300 + i)
    N = int(g.choice([20000, 131072]))
    M = int(g.choice([3, 100]))
    K = int(g.choice([5, 2048, 4096]))
    x, lens = rows(300 + i, M, N, K)
    got = ets.topk_ragged(x, lens.to(DEV), K)
    ets.topk_sort_rows(x, got)
    torch.cuda.synchronize()
    verify(x, lens, K, got)
    gh = got.cpu().numpy()
    assert np.array_equal(gh, oracle.order(x.cpu().numpy(), lens.numpy(), K, gh))
