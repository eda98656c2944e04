"""The optional ordering pass (GPU only): each row of a Top-K result sorted
by score, largest first, equal scores by index, -1 sentinels last.  The set
is unchanged; the order must equal the oracle's ordered output (oracle.order)
of the same set, entry by entry."""
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


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K", [1, 7, 2048, 3000, 4096])
def test_sorted_rows(ets, dtype, K):
    N, M = 65536, 16
    lens = torch.tensor([0, 1, K - 1 if K > 1 else 1, K, K + 1] + [N - 100 * i for i in range(M - 5)],
                        dtype=torch.int32)
    x = synth.indexer_rows(lens, N, seed=K, device=DEV).to(dtype)
    got = ets.topk_ragged(x, lens.to(DEV), K)
    before = got.clone()
    ets.topk_sort_rows(x, got)
    torch.cuda.synchronize()
    xf = x.float()
    verify(xf, lens, K, got)
    assert torch.equal(got.sort(dim=1).values, before.sort(dim=1).values)
    want = oracle.order(xf.cpu().numpy(), lens.numpy(), K, before.cpu().numpy())
    assert np.array_equal(got.cpu().numpy(), want)


def test_sort_argument_errors(ets):
    lib = ets.load_library()
    x = torch.zeros((2, 64), dtype=torch.float32, device=DEV)
    out = torch.zeros((2, 8), dtype=torch.int32, device=DEV)
    assert lib.topk_sort_rows(x.data_ptr(), 2, 64, 0, out.data_ptr(), None) == -1
    assert lib.topk_sort_rows(x.data_ptr(), 2, 64, 4097, out.data_ptr(), None) == -6
    assert lib.topk_sort_rows(x.data_ptr(), 2, 64, 8, out.data_ptr() + 2, None) == -2
    assert lib.topk_sort_rows(x.data_ptr(), 0, 64, 8, out.data_ptr(), None) == 0
