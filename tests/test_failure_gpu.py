"""Failure detection without a GPU fault (GPU only).

Every wait in the kernels is bounded: after its limit it gives up, flags the
row (TOPK_FLAG_TIMEOUT in the device status word) and switches the other
waits of the same launch to fail fast, so a lost copy ends the launch instead
of hanging the GPU.  topk_check_wait_timeout() runs the kernels' own wait
routine on a barrier that nothing completes, with a short limit; the status
word must report the timeout, the context must stay usable, and the give-up
must stay with the launch that gave up: later calls of every kind are exact
whether or not the status word was read in between.
"""
import time

import numpy as np
import pytest
import torch

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


def test_bounded_wait_gives_up_and_reports(ets):
    lib = ets.load_library()
    ets.read_status()          # clear what earlier calls left (e.g. informational path bits)
    t0 = time.time()
    assert lib.topk_check_wait_timeout(20_000_000, None) == 0     # 20 ms
    flags = ets.read_status()                                      # syncs the stream
    assert flags & ets.FLAG_TIMEOUT
    assert time.time() - t0 < 10.0
    # re-armed: a normal selection runs and reports nothing
    N, M = 65536, 64
    lens = synth.causal_lens(N, M, 0, window=4096)
    x = synth.indexer_rows(lens, N, seed=1, device=DEV)
    got = ets.topk_ragged(x, lens.to(DEV), 2048)
    torch.cuda.synchronize()
    verify(x, lens, 2048, got)
    assert ets.read_status() & (ets.FLAG_TIMEOUT | ets.FLAG_INTERNAL) == 0


@pytest.mark.parametrize("kind", ["kvsplit", "direct", "persistent"])
def test_timeout_stays_with_its_launch(ets, kind):
    """A wait that gave up in one launch does not make later launches fail:
    without reading the status word, a KV-split, a direct and a persistent
    call right after the probe are exact and flag no row."""
    lib = ets.load_library()
    old = ets.get_params()
    kinds = {"direct": ets.KIND_DIRECT, "persistent": ets.KIND_PERSISTENT,
             "kvsplit": ets.KIND_KVSPLIT}
    try:
        ets.set_params(force_kind=kinds[kind], sample_min_len=0, kv_segments=4)
        N, M = 16384, 8
        lens = synth.tiny_lens(3, M=M, N_alloc=N, K=2048)
        x = synth.indexer_rows(lens, N, seed=3, device=DEV)
        assert lib.topk_check_wait_timeout(20_000_000, None) == 0     # 20 ms, not read
        got, dg = ets.topk_ragged_diag(x, lens.to(DEV), 2048)
        torch.cuda.synchronize()
        verify(x, lens, 2048, got)
        assert not np.any(dg["flags"] & (ets.FLAG_TIMEOUT | ets.FLAG_INTERNAL))
        assert ets.read_status() & ets.FLAG_TIMEOUT                   # the probe's own report
    finally:
        ets.set_params(**old)


def test_wait_probe_rejects_bad_limits(ets):
    lib = ets.load_library()
    assert lib.topk_check_wait_timeout(0, None) == -1
    assert lib.topk_check_wait_timeout(20_000_000_000, None) == -1
