"""C-ABI checks that need no GPU: the library builds, loads and exports every
entry point include/topk.h declares; host-only calls behave."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    import exact_top_sparse_gb300 as ets
    return ets.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "topk.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(topk_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_north_star_call():
    names = _declared()
    assert "topk_ragged" in names
    src = open(os.path.join(ROOT, "include", "topk.h")).read()
    assert re.search(r"int topk_ragged\(const float\* scores, const int32_t\* row_lens, "
                     r"int64_t M, int64_t N_alloc,\s+int32_t K, int32_t\* out_idx, "
                     r"struct CUstream_st\* stream\);", src)


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    import exact_top_sparse_gb300 as ets
    assert sorted(ets.EXPORTS) == names


def test_library_is_built_for_sm103a(lib):
    import subprocess
    from exact_top_sparse_gb300 import build
    out = subprocess.run(["cuobjdump", "--list-elf", build.LIB], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    assert "sm_103a" in out.stdout


def test_host_only_calls(lib):
    import exact_top_sparse_gb300 as ets
    assert ets.version() == 10300
    assert lib.topk_status_string(0) == b"ok"
    assert lib.topk_status_string(-5).startswith(b"workspace allocation")
    d = ets.default_params()
    assert d["stride"] == 256 and d["rho0"] == 2.0 and d["rho1"] == 2.25
    assert d["long_len"] == 786432 and d["long_stride"] == 512
    assert d["long_rho0"] == 2.75 and d["long_rho1"] == 3.0
    assert d["sample_min_len"] == 12288 and d["direct_max"] == 16384
    old = ets.set_params(stride=64)
    try:
        assert ets.get_params()["stride"] == 64
    finally:
        ets.set_params(**old)
    assert ets.get_params()["stride"] == old["stride"]
    for bad in ({"stride": 0}, {"rho0": 0.5}, {"rho1": 1.0}, {"force_kind": 9},
                {"sample_min_len": -1}, {"long_stride": 0}, {"long_len": -1},
                {"long_rho0": 0.5}, {"long_rho1": 2.5}):
        with pytest.raises(ets.TopKError):
            ets.set_params(**bad)
    assert ets.get_params() == old


def test_argument_errors_need_no_device(lib):
    # rejected on the host before any CUDA call
    vp = ctypes.c_void_p
    assert lib.topk_ragged(None, None, -1, 10, 4, None, None) == -1
    assert lib.topk_ragged(None, None, 1, 10, 0, None, None) == -1
    assert lib.topk_ragged(None, None, 1, 10, 4097, None, None) == -6
    assert lib.topk_ragged(None, None, 0, 10, 4, None, None) == 0  # M == 0 is a no-op
    assert lib.topk_ragged(vp(16), vp(16), 1, 10, 4, None, None) == -1  # null out
    assert lib.topk_ragged(vp(18), vp(16), 1, 10, 4, vp(16), None) == -2  # misaligned scores
    assert lib.topk_ragged_ws(vp(16), vp(16), 1, 10, 4, vp(16), None, 0, None) == -1
    assert lib.topk_ragged_ws(vp(16), vp(16), 1, 10, 4, vp(16), vp(100), 1 << 20, None) == -2
    assert lib.topk_workspace_bytes(0, 10, 4) == 0
    # per-row K: null row_k, K_max out of range, misaligned row_k
    assert lib.topk_ragged_k(vp(16), vp(16), None, 1, 10, 4, vp(16), None) == -1
    assert lib.topk_ragged_k(vp(16), vp(16), vp(16), 1, 10, 0, vp(16), None) == -1
    assert lib.topk_ragged_k(vp(16), vp(16), vp(16), 1, 10, 4097, vp(16), None) == -6
    assert lib.topk_ragged_k(vp(16), vp(16), vp(18), 1, 10, 4, vp(16), None) == -2
    assert lib.topk_ragged_k(None, None, None, 0, 10, 4, None, None) == 0
    assert lib.topk_ragged_k_bf16(vp(16), vp(16), None, 1, 10, 4, vp(16), None) == -1
    assert lib.topk_ragged_k_diag(vp(16), vp(16), vp(16), 1, 10, 4, vp(16), None, None) == -1


def test_no_device_is_an_error_code_not_a_crash(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import exact_top_sparse_gb300 as ets
    with pytest.raises(ets.TopKError):
        ets.plan(8, 16384, 2048)
