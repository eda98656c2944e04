"""Argument checks of the Python binding that run before any device work
(CPU only): host tensors, wrong dtypes and shapes are refused with TypeError,
and the element type picks the matching C entry point."""
import pytest
import torch

import exact_top_sparse_gb300 as ets


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    return ets.load_library()


def test_host_tensors_are_refused(lib):
    x = torch.zeros((2, 8), dtype=torch.float32)
    lens = torch.full((2,), 8, dtype=torch.int32)
    with pytest.raises(TypeError, match="CUDA tensor"):
        ets.topk_ragged(x, lens, 4)
    with pytest.raises(TypeError, match="CUDA tensor"):
        ets.topk_ragged_k(x, lens, torch.full((2,), 4, dtype=torch.int32), 4)
    with pytest.raises(TypeError, match="CUDA tensor"):
        ets.topk_ragged_diag(x, lens, 4)
    with pytest.raises(TypeError):
        ets.topk_sort_rows(x, torch.zeros((2, 4), dtype=torch.int32))
    q = torch.zeros((4, 64, 128), dtype=torch.bfloat16)
    k = torch.zeros((128, 128), dtype=torch.bfloat16)
    w = torch.zeros((4, 64), dtype=torch.float32)
    with pytest.raises(TypeError, match="CUDA"):
        ets.topk_index_scores(q, k, w)


class _Fake:
    def __init__(self, dtype):
        self.dtype = dtype


@pytest.mark.parametrize("dtype,name,want", [
    (torch.float32, "topk_ragged", "topk_ragged"),
    (torch.bfloat16, "topk_ragged", "topk_ragged_bf16"),
    (torch.float8_e4m3fn, "topk_ragged", "topk_ragged_e4m3"),
    (torch.float32, "topk_ragged_diag", "topk_ragged_diag"),
    (torch.bfloat16, "topk_ragged_diag", "topk_ragged_bf16_diag"),
    (torch.float8_e4m3fn, "topk_ragged_diag", "topk_ragged_e4m3_diag"),
    (torch.bfloat16, "topk_ragged_k", "topk_ragged_k_bf16"),
    (torch.float8_e4m3fn, "topk_ragged_k", "topk_ragged_k_e4m3"),
    (torch.float8_e4m3fn, "topk_sort_rows", "topk_sort_rows_e4m3"),
])
def test_element_type_picks_the_entry_point(lib, dtype, name, want):
    assert ets._pick(lib, _Fake(dtype), name) is getattr(lib, want)


def test_status_names_and_flags():
    assert ets.STATUS_NAMES[-8] == "TOPK_ERR_UNSUPPORTED_SHAPE"
    flags = [ets.FLAG_LEN_CLAMPED, ets.FLAG_OVERFLOW, ets.FLAG_RECOVERY, ets.FLAG_INTERNAL,
             ets.FLAG_TIMEOUT, ets.FLAG_K_CLAMPED]
    assert flags == [1, 2, 4, 8, 16, 32]
