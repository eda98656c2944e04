"""Every row of every workload compared with the oracle (GPU only).

The set contract (codexqa.cn article, section "什么叫精确，时间怎么量") is
checked on every row of the full-size workloads, not on a sample: every row
must pass the oracle's checker, every row whose boundary is untied must equal
the oracle's set exactly, and every sampled row must reproduce the oracle's
tau0, tau1, C(tau0), C(tau1) and path.  Rows are copied to the host and
compared in chunks of at most 2 GiB of scores.

Workloads (synthetic indexer-like rows, see exact_top_sparse_gb300.synth):
  * the operator matrix (section "20 个形状都最快"): 128K, 256K, 512K and 1M
    columns, the whole 8192-row causal window in one call, and one further
    group size per width, under the default planner;
  * the width sweep 16K..64K x M in {64 .. 4096} (section "采样不是处处都该开");
  * the stride sweep s in {16, 64, 128, 256} at 32K and 256K columns;
  * decode-style calls of one and two full-length rows at 128K and 1M;
  * bfloat16 and FP8 E4M3 rows of the 8192-row window at 128K and 1M;
  * every Top-K call of the 245K-token prefill trace (section "框架轨迹").
"""
import numpy as np
import pytest
import torch

from exact_top_sparse_gb300 import synth, trace
from tests.test_parity_gpu import run, verify, verify_diag

pytestmark = pytest.mark.gpu

K = 2048
DEV = torch.device("cuda", 0)
CHUNK_BYTES = 2 << 30


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


def verify_every_row(ets, x, lens, k, got, dg=None):
    """verify() (and verify_diag() with diagnostics) on all rows of one call,
    in chunks.  The direct kernel samples no row, so under its plan every
    row longer than k is expected on the direct path."""
    M, N = x.shape
    step = max(1, min(M, CHUNK_BYTES // max(1, N * x.element_size())))
    sml = ets.get_params()["sample_min_len"]
    if ets.plan(M, N, k)["kind"] == "direct":
        sml = N + 1
    for r0 in range(0, M, step):
        r1 = min(M, r0 + step)
        verify(x[r0:r1], lens[r0:r1], k, got[r0:r1])
        if dg is not None:
            verify_diag(ets, x[r0:r1], lens[r0:r1], k, dg[r0:r1], sample_min_len=sml)


def _release(*ts):
    for t in ts:
        del t
    torch.cuda.empty_cache()


@pytest.mark.parametrize("N,M_other,group_other", [(131072, 2048, 2), (262144, 1024, 5),
                                                   (524288, 4096, 1), (1048576, 512, 11)])
def test_operator_matrix_every_row(ets, N, M_other, group_other):
    """The 8192-row window in one call (the benchmark's batch at 1M), then one
    group of another size; every row against the oracle, with thresholds."""
    lens = synth.causal_lens(N, 8192, 0)
    x = synth.indexer_rows(lens, N, seed=7, device=DEV)
    got, dg = run(ets, x, lens, diag=True)
    verify_every_row(ets, x, lens, K, got, dg)
    assert not np.any(dg["flags"] & (ets.FLAG_INTERNAL | ets.FLAG_TIMEOUT))
    # the group of M_other rows, taken from the same window
    r0 = group_other * M_other
    ls = lens[r0:r0 + M_other]
    xs = x[r0:r0 + M_other]
    got, dg = run(ets, xs, ls, diag=True)
    verify_every_row(ets, xs, ls, K, got, dg)
    _release(x, xs, got)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("N", [131072, 1048576])
def test_narrow_rows_every_row(ets, dtype, N):
    """bfloat16 and FP8 E4M3 rows of the 8192-row causal window (the
    sampler-warp kernel serves every narrow row), every row against the
    oracle run on PyTorch's own widening of the same values, with thresholds,
    counts and paths."""
    M = 8192
    lens = synth.causal_lens(N, M, 0)
    x = synth.indexer_rows(lens, N, seed=13, device=DEV)
    x = x.to(torch.bfloat16) if dtype == "bf16" else (x * 4.0).clamp(max=448.0).to(
        torch.float8_e4m3fn)
    got, dg = run(ets, x, lens, diag=True)
    assert not np.any(dg["flags"] & (ets.FLAG_INTERNAL | ets.FLAG_TIMEOUT))
    step = max(1, CHUNK_BYTES // (N * 4))
    for r0 in range(0, M, step):
        r1 = min(M, r0 + step)
        xf = x[r0:r1].float()
        verify(xf, lens[r0:r1], K, got[r0:r1])
        verify_diag(ets, xf, lens[r0:r1], K, dg[r0:r1])
        del xf
    _release(x, got)


@pytest.mark.parametrize("N", [16384, 24576, 32768, 40960, 49152, 57344, 65536])
def test_width_sweep_every_cell(ets, N):
    """Config-4 widths x every M of the sweep under the default planner."""
    for M in (64, 128, 256, 512, 1024, 2048, 4096):
        window = max(M, 8192)
        lens = synth.causal_lens(N, M, group=window // M - 1, window=window)
        x = synth.indexer_rows(lens, N, seed=N // 1024 + 3 * M, device=DEV)
        got, dg = run(ets, x, lens, diag=True)
        verify_every_row(ets, x, lens, K, got, dg)
        _release(x, got)


@pytest.mark.parametrize("stride", [16, 64, 128, 256])
@pytest.mark.parametrize("N,M", [(32768, 2048), (262144, 512)])
def test_stride_sweep_every_row(params, stride, N, M):
    ets = params
    ets.set_params(stride=stride)
    lens = synth.causal_lens(N, M, group=0)
    x = synth.indexer_rows(lens, N, seed=stride + N // 4096, device=DEV)
    got, dg = run(ets, x, lens, diag=True)
    verify_every_row(ets, x, lens, K, got, dg)
    assert np.all(dg["path"] >= ets.PATH_TAU0)  # every row of these widths is sampled
    _release(x, got)


@pytest.mark.parametrize("N", [131072, 1048576])
@pytest.mark.parametrize("M", [1, 2])
def test_decode_shape(ets, N, M):
    """A decode step: one or two full-length rows, default planner."""
    lens = torch.tensor([N, N - 777][:M], dtype=torch.int32)
    x = synth.indexer_rows(lens, N, seed=M * 31 + N % 97, device=DEV)
    got, dg = run(ets, x, lens, diag=True)
    verify_every_row(ets, x, lens, K, got, dg)
    _release(x, got)


def test_trace_245k_every_call(ets):
    """All 26 Top-K calls of the 245K-token prefill trace, on the score rows
    the benchmark replays; every row of every call against the oracle."""
    tokens = 245 * 1024
    calls = trace.calls(tokens)
    assert len(calls) == 26
    buf = synth.trace_scores(trace.WORKSPACE_FLOATS, seed=17, device=DEV)
    lens_all = torch.arange(1, tokens + 1, dtype=torch.int32)
    paths = np.zeros(5, np.int64)
    for c in calls:
        x = buf[:c.rows * c.width].view(c.rows, c.width)
        lens = lens_all[c.row0:c.row0 + c.rows]
        got, dg = run(ets, x, lens, diag=True)
        verify_every_row(ets, x, lens, K, got, dg)
        paths += np.bincount(dg["path"], minlength=5)
        del got
    assert paths[ets.PATH_TAU0] > 0
    _release(buf)
