"""Parity of the CUDA selector with the CPU oracle (GPU only).

Every result must pass the oracle's set-contract checker on every row, and
must equal the oracle's set exactly on every row whose boundary is untied
(index work: bit-exact, no tolerance).  Sampled rows also have their
thresholds tau0/tau1, counts C(tau0)/C(tau1) and path compared with the
oracle's definition of stage 1 and 2, exactly.
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


@pytest.fixture
def params(ets):
    old = ets.get_params()
    yield ets
    ets.set_params(**old)


def verify(x, lens, K, got, rows=None):
    """Checker on every row plus exact equality on untied rows."""
    if rows is not None:
        rows = torch.as_tensor(rows)
        x, lens, got = x[rows.to(x.device)], lens[rows.to(lens.device)], got[rows.to(got.device)]
    xh = x.cpu().numpy()
    lh = lens.cpu().numpy()
    gh = got.cpu().numpy()
    v = oracle.compare(xh, lh, K, gh)
    bad = np.nonzero(v["check"])[0]
    assert bad.size == 0, "rows %s fail the contract: %s" % (
        bad[:8].tolist(), [oracle.CHECK_CODES[int(c)] for c in v["check"][bad[:8]]])
    mism = np.nonzero(v["set_mismatch"])[0]
    assert mism.size == 0, "untied rows %s differ from the oracle set" % mism[:8].tolist()
    return v


def sampling_tiers(p, lens, K):
    """(row mask, stride, T0, T1) of the two sampling tiers under params p:
    rows of at least long_len elements (when long_len > 0) use the long_*
    stride and targets, the others the base ones; T = ceil(rho * K) with rho
    read as FP32, as the library computes it."""
    lh = np.asarray(lens)
    def target(rho):
        return int(np.ceil(np.float64(np.float32(rho)) * K))
    long_rows = (lh >= p["long_len"]) if p["long_len"] > 0 else np.zeros(lh.shape, bool)
    return [(~long_rows, p["stride"], target(p["rho0"]), target(p["rho1"])),
            (long_rows, p["long_stride"], target(p["long_rho0"]), target(p["long_rho1"]))]


def oracle_thresholds(p, xh, lh, K, sample_min_len):
    """The oracle's stage-1/2 quantities, each row under its own tier."""
    M = lh.shape[0]
    ref = {"tau": np.zeros((M, 2), np.float32), "count": np.zeros((M, 2), np.int64),
           "rank": np.zeros((M, 2), np.int64), "path": np.zeros(M, np.int32)}
    for mask, stride, T0, T1 in sampling_tiers(p, lh, K):
        if not mask.any():
            continue
        part = oracle.thresholds(xh[mask], lh[mask], K, stride, T0, T1, sample_min_len)
        for k in ref:
            ref[k][mask] = part[k]
    return ref


def verify_diag(ets, x, lens, K, diag, rows=None, sample_min_len=0):
    """Thresholds, counts and path of sampled rows equal the oracle's."""
    p = ets.get_params()
    if rows is not None:
        x, lens, diag = x[rows], lens[rows], diag[rows]
    ref = oracle_thresholds(p, x.cpu().numpy(), lens.cpu().numpy(), K, sample_min_len)
    sampled = ref["path"] >= oracle.PATH_TAU0
    assert np.array_equal(diag["path"][sampled], ref["path"][sampled])
    assert np.array_equal(diag["tau0"][sampled], ref["tau"][sampled, 0])
    assert np.array_equal(diag["tau1"][sampled], ref["tau"][sampled, 1])
    assert np.array_equal(diag["count0"][sampled], ref["count"][sampled, 0])
    assert np.array_equal(diag["count1"][sampled], ref["count"][sampled, 1])
    assert np.array_equal(diag["path"][~sampled], ref["path"][~sampled])
    assert not np.any(diag["flags"] & (ets.FLAG_INTERNAL | ets.FLAG_TIMEOUT))
    return ref


def run(ets, x, lens, K=K, diag=False):
    d_lens = lens.to(DEV)
    if diag:
        out, dg = ets.topk_ragged_diag(x, d_lens, K)
    else:
        out, dg = ets.topk_ragged(x, d_lens, K), None
    torch.cuda.synchronize()
    return out, dg


# ------------------------------------------------------------------ config 1
@pytest.mark.parametrize("seed", [0, 1, 2, 3])
@pytest.mark.parametrize("kind", ["auto", "persistent", "kvsplit"])
def test_tiny_config(params, seed, kind):
    ets = params
    N = 16384
    lens = synth.tiny_lens(seed, M=8, N_alloc=N, K=K)
    x = synth.indexer_rows(lens, N, seed=seed, device=DEV)
    kinds = {"auto": ets.KIND_AUTO, "persistent": ets.KIND_PERSISTENT, "kvsplit": ets.KIND_KVSPLIT}
    ets.set_params(force_kind=kinds[kind], sample_min_len=0 if kind != "auto" else 16384,
                   kv_segments=4 if kind == "kvsplit" else 0)
    got, dg = run(ets, x, lens, diag=True)
    verify(x, lens, K, got)
    if kind != "auto":
        verify_diag(ets, x, lens, K, dg)
    else:
        assert set(dg["path"].tolist()) <= {ets.PATH_SENTINEL, ets.PATH_DIRECT}


# ------------------------------------------------------------- configs 2 / 3
@pytest.mark.parametrize("group", [0, 15])
@pytest.mark.parametrize("kind", ["auto", "persistent"])
def test_128k_operator_matrix_group(params, group, kind):
    ets = params
    N, M = 131072, 512
    if kind == "persistent":
        ets.set_params(force_kind=ets.KIND_PERSISTENT)
    lens = synth.causal_lens(N, M, group)
    x = synth.indexer_rows(lens, N, seed=100 + group, device=DEV)
    got, dg = run(ets, x, lens, diag=True)
    verify(x, lens, K, got)
    verify_diag(ets, x, lens, K, dg, sample_min_len=ets.get_params()["sample_min_len"])


@pytest.mark.parametrize("N,M", [(262144, 1024), (524288, 512), (1048576, 512)])
def test_long_rows_default_dispatch(ets, N, M):
    lens = synth.causal_lens(N, M, group=8192 // M - 1)
    x = synth.indexer_rows(lens, N, seed=N + M, device=DEV)
    got, dg = run(ets, x, lens, diag=True)
    verify(x, lens, K, got)
    verify_diag(ets, x, lens, K, dg, sample_min_len=ets.get_params()["sample_min_len"])
    del x


@pytest.mark.parametrize("kind", ["auto", "persistent", "kvsplit"])
def test_rows_longer_than_the_matrix(params, kind):
    """4M-column rows (past the operator matrix): the long sampling tier, the
    KV-split's many segments, and the sampler's on-chip key buffer."""
    ets = params
    N, M = 4 * 1048576, 12
    if kind != "auto":
        ets.set_params(force_kind=ets.KIND_PERSISTENT if kind == "persistent" else ets.KIND_KVSPLIT)
    lens = torch.tensor([N, N - 1, N - 3, 3 * 1048576 + 5, 2 * 1048576 + 1, 1048576, 800000,
                         N - 12345, 4095, 2049, 1, N], dtype=torch.int32)
    x = synth.indexer_rows(lens, N, seed=44, device=DEV)
    got, dg = run(ets, x, lens, diag=True)
    verify(x, lens, K, got)
    verify_diag(ets, x, lens, K, dg, sample_min_len=ets.get_params()["sample_min_len"])
    del x


# ------------------------------------------------------------------ config 4
@pytest.mark.parametrize("N", [16384, 24576, 32768, 40960, 49152, 57344, 65536])
@pytest.mark.parametrize("M", [64, 512])
def test_width_sweep(ets, N, M):
    lens = synth.causal_lens(N, M, group=0, window=min(8192, 64 * M))
    x = synth.indexer_rows(lens, N, seed=N // 1024 + M, device=DEV)
    got, _ = run(ets, x, lens)
    verify(x, lens, K, got)


@pytest.mark.parametrize("kind", ["persistent", "kvsplit"])
def test_two_sampling_tiers_in_one_batch(params, kind):
    """Rows on both sides of long_len in one call: each is sampled with its
    own tier's stride and targets."""
    ets = params
    N, M = 65536, 96
    ets.set_params(sample_min_len=0, long_len=40000, long_stride=96, long_rho0=1.7,
                   long_rho1=2.6, stride=40, rho0=1.25, rho1=1.5,
                   force_kind=ets.KIND_PERSISTENT if kind == "persistent" else ets.KIND_KVSPLIT)
    lens = torch.randint(20000, N + 1, (M,), generator=torch.Generator().manual_seed(12),
                         dtype=torch.int32)
    lens[:2] = torch.tensor([40000, 39999], dtype=torch.int32)
    x = synth.indexer_rows(lens, N, seed=12, device=DEV)
    got, dg = run(ets, x, lens, diag=True)
    verify(x, lens, K, got)
    verify_diag(ets, x, lens, K, dg)
    tiers = sampling_tiers(ets.get_params(), lens.numpy(), K)
    assert tiers[0][0].sum() > 10 and tiers[1][0].sum() > 10


@pytest.mark.parametrize("stride", [16, 64, 128, 256])
@pytest.mark.parametrize("kind", ["persistent", "kvsplit"])
def test_stride_sweep_sampled(params, stride, kind):
    ets = params
    N, M = 65536, 256
    ets.set_params(stride=stride, sample_min_len=0,
                   force_kind=ets.KIND_PERSISTENT if kind == "persistent" else ets.KIND_KVSPLIT)
    lens = synth.causal_lens(N, M, group=0, window=8192)
    x = synth.indexer_rows(lens, N, seed=stride, device=DEV)
    got, dg = run(ets, x, lens, diag=True)
    verify(x, lens, K, got)
    verify_diag(ets, x, lens, K, dg)


@pytest.mark.parametrize("kind", ["direct", "persistent", "kvsplit"])
def test_bf16_grid_ties(params, kind):
    ets = params
    N, M = 65536 if kind != "direct" else 32768, 128
    kinds = {"direct": ets.KIND_DIRECT, "persistent": ets.KIND_PERSISTENT,
             "kvsplit": ets.KIND_KVSPLIT}
    ets.set_params(force_kind=kinds[kind], sample_min_len=0)
    lens = synth.causal_lens(N, M, group=0, window=4096)
    x = synth.to_bf16_grid(synth.indexer_rows(lens, N, seed=5, device=DEV))
    got, dg = run(ets, x, lens, diag=True)
    v = verify(x, lens, K, got)
    assert v["tied"].mean() > 0.5
    if kind != "direct":
        verify_diag(ets, x, lens, K, dg)


@pytest.mark.parametrize("kind", ["direct", "persistent", "kvsplit"])
def test_uniform_rows(params, kind):
    ets = params
    N, M = 49152, 96
    kinds = {"direct": ets.KIND_DIRECT, "persistent": ets.KIND_PERSISTENT,
             "kvsplit": ets.KIND_KVSPLIT}
    ets.set_params(force_kind=kinds[kind], sample_min_len=0)
    lens = synth.causal_lens(N, M, group=0, window=96 * 64)
    x = synth.uniform_rows(lens, N, seed=9, device=DEV)
    got, dg = run(ets, x, lens, diag=True)
    verify(x, lens, K, got)
    if kind != "direct":
        verify_diag(ets, x, lens, K, dg)


@pytest.mark.parametrize("kind", ["persistent", "kvsplit"])
def test_forced_paths_tau1_recovery_overflow(params, kind):
    """Rows built so the proposal underfills (tau1 path, exact recovery in one
    band pass or in two passes) or overfills past the on-chip buffer (spill
    area, overflow); every row must still be exact."""
    ets = params
    # the rows are built for stride 128 and targets 1.5K / 1.75K
    ets.set_params(sample_min_len=0, kv_segments=7 if kind == "kvsplit" else 0,
                   force_kind=ets.KIND_PERSISTENT if kind == "persistent" else ets.KIND_KVSPLIT,
                   stride=128, rho0=1.5, rho1=1.75, long_len=0)
    L = 65536
    lens = torch.full((1,), L, dtype=torch.int32)
    rows = [
        synth.strided_high_rows(lens, L, seed=1, stride=128, n_top=26, n_mid=2100),   # tau1
        synth.strided_high_rows(lens, L, seed=2, stride=128, n_top=40, n_mid=2100),   # recovery
        synth.strided_high_rows(lens, L, seed=3, stride=128, n_top=0, n_mid=20000,
                                on_grid=False),                                       # overflow
        synth.strided_high_rows(lens, L, seed=4, stride=128, n_top=10, n_mid=3000),   # tau0
        synth.strided_high_rows(lens, L, seed=5, stride=128, n_top=0, n_mid=9000,
                                on_grid=False),                                       # spill
        synth.strided_high_rows(lens, L, seed=6, stride=128, n_top=80, n_mid=2100),   # recovery,
    ]                                                                                  # two passes
    x = torch.cat(rows).to(DEV)
    lens6 = torch.full((6,), L, dtype=torch.int32)
    got, dg = run(ets, x, lens6, diag=True)
    verify(x, lens6, K, got)
    ref = verify_diag(ets, x, lens6, K, dg)
    assert ref["path"].tolist() == [ets.PATH_TAU1, ets.PATH_RECOVERY, ets.PATH_TAU0,
                                    ets.PATH_TAU0, ets.PATH_TAU0, ets.PATH_RECOVERY]
    assert dg["flags"][1] & ets.FLAG_RECOVERY and dg["flags"][5] & ets.FLAG_RECOVERY
    assert dg["flags"][2] & ets.FLAG_OVERFLOW
    # more candidates than the on-chip buffer holds, fewer than the spill area adds
    assert 6144 < dg["count1"][4] <= 16384 and not dg["flags"][4] & ets.FLAG_OVERFLOW


@pytest.mark.parametrize("kind", ["direct", "persistent", "kvsplit"])
def test_constant_rows(params, kind):
    ets = params
    N, M = 40000, 6
    kinds = {"direct": ets.KIND_DIRECT, "persistent": ets.KIND_PERSISTENT,
             "kvsplit": ets.KIND_KVSPLIT}
    ets.set_params(force_kind=kinds[kind], sample_min_len=0, kv_segments=3)
    lens = torch.tensor([40000, 2049, 2048, 5000, 39999, 12345], dtype=torch.int32)
    x = synth.constant_rows(lens, N, 3.25, device=DEV)
    got, _ = run(ets, x, lens)
    verify(x, lens, K, got)


# ---------------------------------------------------------------- edge cases
def test_empty_batch_and_zero_width(ets):
    x = torch.empty((0, 100), dtype=torch.float32, device=DEV)
    out = ets.topk_ragged(x, torch.empty(0, dtype=torch.int32, device=DEV), K)
    assert out.shape == (0, K)
    x = torch.empty((3, 0), dtype=torch.float32, device=DEV)
    out = ets.topk_ragged(x, torch.tensor([0, 5, -2], dtype=torch.int32, device=DEV), 16)
    torch.cuda.synchronize()
    assert bool((out == -1).all())


@pytest.mark.parametrize("kind", ["direct", "persistent", "kvsplit"])
def test_clamped_lengths_and_status(params, kind):
    ets = params
    kinds = {"direct": ets.KIND_DIRECT, "persistent": ets.KIND_PERSISTENT,
             "kvsplit": ets.KIND_KVSPLIT}
    ets.set_params(force_kind=kinds[kind], sample_min_len=0)
    N = 40000
    raw = torch.tensor([-7, 10 ** 9, 100, N], dtype=torch.int32)
    lens = raw.clamp(0, N)
    x = synth.indexer_rows(lens, N, seed=4, device=DEV)
    ets.read_status()
    got, dg = run(ets, x, raw, diag=True)
    verify(x, lens, K, got)
    assert ets.read_status() & ets.FLAG_LEN_CLAMPED
    assert dg["flags"][0] & ets.FLAG_LEN_CLAMPED and dg["flags"][1] & ets.FLAG_LEN_CLAMPED
    assert not dg["flags"][2] & ets.FLAG_LEN_CLAMPED


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["persistent", "kvsplit"])
def test_unsampled_rows_staged_and_streamed(params, kind, dtype):
    """Rows below sample_min_len on the persistent and KV-split kernels: the
    ones whose scores fit the 48 KB candidate buffer (12288 FP32 or 24576
    bfloat16 values) are loaded once and selected on chip, longer ones
    stream through the ring; lengths straddle that limit, K and the row
    lengths straddle each other."""
    ets = params
    ets.set_params(force_kind=ets.KIND_PERSISTENT if kind == "persistent" else ets.KIND_KVSPLIT,
                   sample_min_len=1 << 20, kv_segments=3 if kind == "kvsplit" else 0)
    N = 40000
    lens = torch.tensor([2049, 2500, 4096, 8191, 12287, 12288, 12289, 20000, 24575, 24576, 24577,
                         40000, 2048, 0, 9999, 31111], dtype=torch.int32)
    x = synth.indexer_rows(lens, N, seed=17, device=DEV)
    if dtype == "bf16":
        x = x.to(torch.bfloat16)
    got, dg = ets.topk_ragged_diag(x, lens.to(DEV), K)
    torch.cuda.synchronize()
    verify(x.float(), lens, K, got)
    assert set(dg["path"].tolist()) <= {ets.PATH_SENTINEL, ets.PATH_DIRECT}
    assert not np.any(dg["flags"] & (ets.FLAG_INTERNAL | ets.FLAG_TIMEOUT))
    # a short K over the same rows: boundary well inside the row
    got = ets.topk_ragged(x, lens.to(DEV), 5)
    torch.cuda.synchronize()
    verify(x.float(), lens, 5, got)


@pytest.mark.parametrize("k", [1, 7, 2048, 4096])
@pytest.mark.parametrize("kind", ["direct", "persistent", "kvsplit"])
def test_other_k(params, k, kind):
    ets = params
    kinds = {"direct": ets.KIND_DIRECT, "persistent": ets.KIND_PERSISTENT,
             "kvsplit": ets.KIND_KVSPLIT}
    ets.set_params(force_kind=kinds[kind], sample_min_len=0)
    N, M = 45000, 5
    lens = torch.tensor([45000, k, k + 1, 30001, 4097], dtype=torch.int32)
    x = synth.indexer_rows(lens, N, seed=k, device=DEV)
    got, _ = run(ets, x, lens, K=k)
    verify(x, lens, k, got)


@pytest.mark.parametrize("kind", ["direct", "persistent", "kvsplit"])
def test_unaligned_rows(params, kind):
    """Rows that start off 16-byte boundaries (odd N_alloc, offset base)."""
    ets = params
    kinds = {"direct": ets.KIND_DIRECT, "persistent": ets.KIND_PERSISTENT,
             "kvsplit": ets.KIND_KVSPLIT}
    ets.set_params(force_kind=kinds[kind], sample_min_len=0)
    N, M = 40001, 9
    lens = torch.tensor([40001, 40000, 39999, 39998, 2049, 3000, 12345, 40001, 20001],
                        dtype=torch.int32)
    base = torch.empty(M * N + 3, dtype=torch.float32, device=DEV)
    x = base[1:1 + M * N].view(M, N)
    x.copy_(synth.indexer_rows(lens, N, seed=77, device=DEV))
    assert x.data_ptr() % 16 != 0
    got, _ = run(ets, x, lens)
    verify(x, lens, K, got)


def test_explicit_workspace(ets):
    N, M = 131072, 64
    lens = synth.causal_lens(N, M, 0, window=8192)
    x = synth.indexer_rows(lens, N, seed=12, device=DEV)
    need = ets.workspace_bytes(M, N, K)
    assert need > 0
    small = torch.zeros(max(256, need - 256), dtype=torch.uint8, device=DEV)
    with pytest.raises(ets.TopKError) as e:
        ets.topk_ragged_ws(x, lens.to(DEV), K, small)
    assert e.value.code == -3
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    for _ in range(2):
        got = ets.topk_ragged_ws(x, lens.to(DEV), K, ws)
        torch.cuda.synchronize()
        verify(x, lens, K, got)


@pytest.mark.parametrize("N,M", [(131072, 512), (131072, 2048), (1048576, 256)])
def test_cuda_graph_replay(ets, N, M):
    """Capture once, replay with new scores and lengths written in place."""
    lens = synth.causal_lens(N, M, 0, window=max(M, 8192 if N > 8192 else M))
    x = synth.indexer_rows(lens, N, seed=1, device=DEV)
    d_lens = lens.to(DEV)
    out = torch.empty((M, K), dtype=torch.int32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ets.topk_ragged(x, d_lens, K, out=out)  # creates the workspace before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ets.topk_ragged(x, d_lens, K, out=out)
    for rep in range(3):
        lens2 = (lens - 37 * rep).clamp(min=0)
        x.copy_(synth.indexer_rows(lens2, N, seed=50 + rep, device=DEV))
        d_lens.copy_(lens2.to(DEV))
        out.fill_(-5)
        g.replay()
        torch.cuda.synchronize()
        verify(x, lens2, K, out)


def test_capture_without_workspace_is_refused(ets):
    N, M = 131072, 64
    x = torch.zeros((M, N), dtype=torch.float32, device=DEV)
    lens = torch.full((M,), N, dtype=torch.int32, device=DEV)
    out = torch.empty((M, K), dtype=torch.int32, device=DEV)
    ets.plan(M, N, K)  # device set-up happens outside the capture
    s = torch.cuda.Stream()  # a stream the library has never seen
    lib = ets.load_library()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        g.capture_begin()
        try:
            rc = lib.topk_ragged(x.data_ptr(), lens.data_ptr(), M, N, K, out.data_ptr(),
                                 ctypes.c_void_p(s.cuda_stream))
        finally:
            g.capture_end()
    assert rc == -5


def test_host_buffer_api(ets):
    N, M = 131072, 300
    lens = synth.causal_lens(N, M, 0, window=600)
    x = synth.indexer_rows(lens, N, seed=21, device=DEV).cpu().numpy()
    got = ets.topk_ragged_host(x, lens.numpy(), K, rows_per_chunk=64)
    v = oracle.compare(x, lens.numpy(), K, got)
    assert not v["check"].any() and not v["set_mismatch"].any()


def test_plan_kinds(ets):
    assert ets.plan(8, 16384, K)["kind"] == "direct"
    assert ets.plan(8192, 1048576, K)["kind"] == "persistent"
    p = ets.plan(512, 1048576, K)
    assert p["kind"] == "kvsplit" and p["segments"] > 1
    sms = p["sm_count"]
    assert ets.plan(512, 131072, K)["kind"] == "persistent"   # short rows: split only when tiny
    assert ets.plan(512, 524288, K)["kind"] == "persistent"
    assert ets.plan(512, 786432, K)["kind"] == "kvsplit"
    assert ets.plan(sms // 4, 131072, K)["kind"] == "kvsplit"
    assert ets.plan(4 * sms, 1048576, K)["kind"] == "persistent"


# ------------------------------------------------------------ sampler warp
@pytest.mark.parametrize("order", ["rising", "falling", "ties"])
def test_sampler_warp_thresholds_on_ordered_rows(ets, order):
    """Rows narrower than 512K FP32 elements run the sampler-warp kernel: one
    warp ranks the next row's samples while the others stream the current
    row, keeping the r1 largest sample keys in a list sorted across its
    lanes.  Rows whose scores rise along the row make every sample enter that
    list, falling rows make none after the first, and rows of a few values
    make most samples tie with the list's smallest key; tau0, tau1, the
    counts and the path must still equal the oracle's on every sampled row
    (more rows than CTAs, so most rows are prepared by a sampler warp)."""
    assert ets.plan(1024, 65536, K)["kind"] == "persistent"
    N, M = 65536, 1024
    lens = torch.full((M,), N, dtype=torch.int32) - torch.arange(M, dtype=torch.int32) * 16
    g = torch.Generator().manual_seed(71)
    base = torch.arange(N, dtype=torch.float32) / N
    if order == "rising":
        x = base.repeat(M, 1) + torch.rand((M, N), generator=g) * 1e-3
    elif order == "falling":
        x = base.flip(0).repeat(M, 1) + torch.rand((M, N), generator=g) * 1e-3
    else:
        x = torch.randint(0, 6, (M, N), generator=g).to(torch.float32)
    x = x.to(DEV)
    out, dg = run(ets, x, lens, diag=True)
    verify(x, lens, K, out)
    verify_diag(ets, x, lens, K, dg)


# ------------------------------------------------------ infinities in the rows
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["auto", "persistent", "kvsplit"])
def test_infinities_inside_the_valid_prefix(params, kind, dtype):
    """+inf and -inf are ordinary scores inside a row's valid prefix (the key
    transform keeps the IEEE order), in FP32 and bfloat16 rows: some rows carry a few +inf and many -inf,
    one row is all -inf (every score ties), one is all +inf, one has exactly K
    +inf (they are the answer), one has -inf everywhere but K - 1 finite
    scores.  Every row must pass the checker and equal the oracle's set
    where untied; sampled rows reproduce the oracle's thresholds."""
    ets = params
    kinds = {"auto": ets.KIND_AUTO, "persistent": ets.KIND_PERSISTENT,
             "kvsplit": ets.KIND_KVSPLIT}
    ets.set_params(force_kind=kinds[kind], kv_segments=3 if kind == "kvsplit" else 0)
    N, M = 65536, 640 if kind != "kvsplit" else 48
    lens = synth.causal_lens(N, M, 0, window=M * (8192 // M))
    x = synth.indexer_rows(lens, N, seed=91, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(92)
    r = torch.rand(x.shape, generator=g, device=DEV)
    x = torch.where(r < 0.001, torch.full_like(x, float("inf")), x)
    x = torch.where((r > 0.5) & (r < 0.51), torch.full_like(x, float("-inf")), x)
    L0 = int(lens[0])
    x[0, :L0] = float("-inf")
    x[1, :int(lens[1])] = float("inf")
    x[2, : 3 * K : 3] = float("inf")
    x[3, :int(lens[3])] = float("-inf")
    x[3, 100:100 + K - 1] = 1.0
    # the causal suffix stays -inf
    for i in range(4):
        x[i, int(lens[i]):] = float("-inf")
    if dtype == "bf16":
        x = x.to(torch.bfloat16)  # +-inf are bfloat16 values too
    out, dg = run(ets, x, lens, diag=True)
    xf = x.float()
    verify(xf, lens, K, out)
    verify_diag(ets, xf, lens, K, dg)
