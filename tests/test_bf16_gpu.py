"""bfloat16 score rows through the same selector (GPU only).

A bfloat16 widens exactly to FP32, so the exact Top-K of bfloat16 rows is the
exact Top-K of their widened values: the oracle runs on the widened copy and
every row must pass its set contract, equal its set on untied rows, and (for
sampled rows) reproduce its thresholds, counts and path.  bfloat16 rows have
many ties at the boundary (8 significant bits), which exercises the
all-equal frontier.
"""
import numpy as np
import pytest
import torch

from exact_top_sparse_gb300 import synth
from tests.test_parity_gpu import verify, verify_diag

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
K = 2048


@pytest.fixture
def params():
    import __graft_entry__ as g
    g.build()
    import exact_top_sparse_gb300 as m
    old = m.get_params()
    yield m
    m.set_params(**old)


def bf16_rows(lens, N, seed):
    x = synth.indexer_rows(lens, N, seed=seed, device=DEV).to(torch.bfloat16)
    return x, x.float()


@pytest.mark.parametrize("kind", ["auto", "direct", "persistent", "kvsplit"])
def test_bf16_kinds_match_the_oracle(params, kind):
    ets = params
    N, M = 40960, 64
    kinds = {"auto": 0, "direct": ets.KIND_DIRECT, "persistent": ets.KIND_PERSISTENT,
             "kvsplit": ets.KIND_KVSPLIT}
    ets.set_params(force_kind=kinds[kind], sample_min_len=0 if kind != "auto" else 16384,
                   kv_segments=3 if kind == "kvsplit" else 0)
    lens = synth.causal_lens(N, M, 0, window=4096)
    lens[:3] = torch.tensor([0, 2048, 2049], dtype=torch.int32)
    x, xf = bf16_rows(lens, N, seed=3)
    got, dg = ets.topk_ragged_diag(x, lens.to(DEV), K)
    torch.cuda.synchronize()
    verify(xf, lens, K, got)
    if kind in ("persistent", "kvsplit"):
        verify_diag(ets, xf, lens, K, dg)


@pytest.mark.parametrize("N,M", [(262144, 256), (1048576, 64)])
def test_bf16_long_rows_default_dispatch(params, N, M):
    ets = params
    lens = synth.causal_lens(N, M, group=0, window=M)
    x, xf = bf16_rows(lens, N, seed=N + M)
    got, dg = ets.topk_ragged_diag(x, lens.to(DEV), K)
    torch.cuda.synchronize()
    verify(xf, lens, K, got)
    verify_diag(ets, xf, lens, K, dg, sample_min_len=ets.get_params()["sample_min_len"])


@pytest.mark.parametrize("N", [65537, 65543])
def test_bf16_unaligned_rows(params, N):
    """Odd row strides: each row starts at a different 2-byte offset, so the
    16-byte aligned body is preceded and followed by up to 7 elements."""
    ets = params
    M = 24
    ets.set_params(sample_min_len=0)
    lens = torch.tensor([N - 7 * i for i in range(M)], dtype=torch.int32)
    x, xf = bf16_rows(lens, N, seed=N)
    for kind in (ets.KIND_PERSISTENT, ets.KIND_KVSPLIT, ets.KIND_DIRECT):
        ets.set_params(force_kind=kind, kv_segments=5 if kind == ets.KIND_KVSPLIT else 0)
        try:
            got = ets.topk_ragged(x, lens.to(DEV), K)
        except ets.TopKError:
            assert kind == ets.KIND_DIRECT  # the direct kernel may not fit this width
            continue
        torch.cuda.synchronize()
        verify(xf, lens, K, got)


@pytest.mark.parametrize("k", [1, 100, 4096])
def test_bf16_other_k(params, k):
    ets = params
    N, M = 131072, 32
    lens = synth.causal_lens(N, M, 0, window=M)
    x, xf = bf16_rows(lens, N, seed=k)
    got = ets.topk_ragged(x, lens.to(DEV), k)
    torch.cuda.synchronize()
    verify(xf, lens, k, got)


def test_bf16_rejects_misaligned_rows(params):
    ets = params
    lib = ets.load_library()
    x = torch.zeros((2, 4096), dtype=torch.bfloat16, device=DEV)
    lens = torch.full((2,), 4096, dtype=torch.int32, device=DEV)
    out = torch.empty((2, K), dtype=torch.int32, device=DEV)
    assert lib.topk_ragged_bf16(x.data_ptr() + 1, lens.data_ptr(), 2, 4096, K, out.data_ptr(),
                                None) == -2
