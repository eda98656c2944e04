"""Failure detection without a GPU fault (GPU only).

Every wait in the kernels is bounded: after its limit it gives up, flags the
row (TOPK_FLAG_TIMEOUT in the device status word) and switches the other
waits to fail fast, so a lost copy ends the launch instead of hanging the
GPU.  topk_check_wait_timeout() runs the kernels' own wait routine on a
barrier that nothing completes, with a short limit; the status word must
report the timeout, reading it must re-arm the kernels, and the context must
stay usable for a normal selection afterwards.
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


def test_wait_probe_rejects_bad_limits(ets):
    lib = ets.load_library()
    assert lib.topk_check_wait_timeout(0, None) == -1
    assert lib.topk_check_wait_timeout(20_000_000_000, None) == -1
