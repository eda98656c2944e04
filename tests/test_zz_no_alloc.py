"""The fixed-scratch entry point against the regular one (GPU only).

topk_ragged_noalloc() serves callers that may not allocate device memory
(serving processes whose allocator owns the whole GPU, plugin hosts that
forbid allocation while they run).  It keeps its scratch in one static device
array instead of a workspace the library allocates.  These tests call it
through the C ABI and compare its output with topk_ragged() on the same
inputs, on two calls in a row (the second call finds the first call's state
in the shared array), plus the size limit.  Index results admit no tolerance:
rows with an untied boundary must give the same set, every row must pass the
set contract.  This file sorts last so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from exact_top_sparse_gb300 import synth

pytestmark = pytest.mark.gpu

K = 2048
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def ets():
    import __graft_entry__ as g
    g.build()
    import exact_top_sparse_gb300 as m
    return m


def _noalloc_raw(ets, x, lens, k, out):
    """Direct C-ABI call of topk_ragged_noalloc (no Python-side allocation)."""
    lib = ets.load_library()
    s = torch.cuda.current_stream(DEV)
    return lib.topk_ragged_noalloc(x.data_ptr(), lens.data_ptr(), x.shape[0], x.shape[1], k,
                                   out.data_ptr(), ctypes.c_void_p(s.cuda_stream))


def _same_result(x, lens, k, a, b):
    xh, lh = x.cpu().numpy(), lens.cpu().numpy()
    ah, bh = a.cpu().numpy(), b.cpu().numpy()
    assert np.all(oracle.check(xh, lh, k, ah) == 0)
    assert np.all(oracle.check(xh, lh, k, bh) == 0)
    _, _, tied = oracle.boundary(xh, lh, k)
    same = np.all(np.sort(ah, axis=1) == np.sort(bh, axis=1), axis=1)
    assert np.all(same | tied), np.nonzero(~same & ~tied)[0][:8]


def test_noalloc_matches_regular_entry_point_twice(ets):
    M = ets.NOALLOC_MAX_ROWS
    cases = [
        (131072, synth.causal_lens(131072, M, group=0), 31),
        (65537, torch.tensor([65537, 2048, 2049, 100, 0] + [65537 - 997 * i for i in range(M - 5)],
                             dtype=torch.int32), 32),
    ]
    for N, lens, seed in cases:  # two calls in a row through the shared scratch
        x = synth.indexer_rows(lens, N, seed=seed, device=DEV)
        d_lens = lens.to(DEV)
        want = ets.topk_ragged(x, d_lens, K)
        got = torch.full((M, K), -7, dtype=torch.int32, device=DEV)
        rc = _noalloc_raw(ets, x, d_lens, K, got)
        torch.cuda.synchronize()
        assert rc == 0, ets.STATUS_NAMES.get(rc, rc)
        _same_result(x, lens, K, got, want)


def test_noalloc_smaller_batches_and_other_k(ets):
    for M, N, k, seed in ((7, 300000, 2048, 5), (40, 50000, 300, 6)):
        lens = torch.randint(1, N + 1, (M,), generator=torch.Generator().manual_seed(seed),
                             dtype=torch.int32)
        x = synth.indexer_rows(lens, N, seed=seed, device=DEV)
        d_lens = lens.to(DEV)
        want = ets.topk_ragged(x, d_lens, k)
        got = torch.empty((M, k), dtype=torch.int32, device=DEV)
        for _ in range(2):
            got.fill_(-7)
            assert _noalloc_raw(ets, x, d_lens, k, got) == 0
            torch.cuda.synchronize()
            _same_result(x, lens, k, got, want)


def test_noalloc_rejects_batches_over_its_limit(ets):
    M = ets.NOALLOC_MAX_ROWS + 1
    x = torch.zeros((M, 4096), dtype=torch.float32, device=DEV)
    lens = torch.full((M,), 4096, dtype=torch.int32, device=DEV)
    out = torch.empty((M, K), dtype=torch.int32, device=DEV)
    assert _noalloc_raw(ets, x, lens, K, out) == -3  # TOPK_ERR_WORKSPACE
    with pytest.raises(ets.TopKError):
        ets.topk_ragged_noalloc(x, lens, K, out=out)
