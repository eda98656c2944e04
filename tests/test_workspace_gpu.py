"""Lifetime and initialisation of the library's cached workspaces (GPU only).

The library allocates one workspace per (device, stream) and grows it when a
larger call arrives.  A CUDA graph captured earlier on that stream keeps the
old address, so a grown-out workspace must stay allocated until
topk_release_workspaces().  A new workspace is zero-filled on the call's own
stream, ahead of the kernels that read it, which matters on streams that do
not synchronise with the legacy default stream.  The host-buffer call keeps
per-device buffers that two host threads must not use at once.
"""
import ctypes
import threading

import numpy as np
import pytest
import torch

import oracle
from exact_top_sparse_gb300 import synth
from tests.test_parity_gpu import verify

pytestmark = pytest.mark.gpu

K = 2048
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def ets():
    import __graft_entry__ as g
    g.build()
    import exact_top_sparse_gb300 as m
    return m


class _PtrAttr(ctypes.Structure):
    """struct cudaPointerAttributes of the CUDA 13 runtime (driver_types.h),
    reserved tail included: the call writes all of it."""
    _fields_ = [("type", ctypes.c_int), ("device", ctypes.c_int),
                ("devicePointer", ctypes.c_void_p), ("hostPointer", ctypes.c_void_p),
                ("reserved", ctypes.c_long * 8)]


def _is_live_device_allocation(addr: int) -> bool:
    """cudaPointerGetAttributes: a live device allocation reports
    cudaMemoryTypeDevice (2); freed memory reports unregistered (0)."""
    rt = ctypes.CDLL("libcudart.so.13")
    assert ctypes.sizeof(_PtrAttr) == 88
    rt.cudaPointerGetAttributes.argtypes = [ctypes.POINTER(_PtrAttr), ctypes.c_void_p]
    rt.cudaPointerGetAttributes.restype = ctypes.c_int
    a = _PtrAttr()
    rc = rt.cudaPointerGetAttributes(ctypes.byref(a), ctypes.c_void_p(addr))
    return rc == 0 and a.type == 2


def test_grown_workspace_stays_allocated_for_a_captured_graph(ets):
    s = torch.cuda.Stream(device=DEV)
    # a small call (KV-split, about 10 MB of workspace), then a capture of it
    N1, M1 = 131072, 64
    l1 = synth.causal_lens(N1, M1, 0, window=8192)
    x1 = synth.indexer_rows(l1, N1, seed=61, device=DEV)
    d1 = l1.to(DEV)
    o1 = torch.empty((M1, K), dtype=torch.int32, device=DEV)
    with torch.cuda.stream(s):
        ets.topk_ragged(x1, d1, K, out=o1)
    s.synchronize()
    p1, b1 = ets.cached_workspace(DEV, s)
    assert p1 != 0 and b1 > 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ets.topk_ragged(x1, d1, K, out=o1)
    # an eager call on the same stream that needs a larger workspace
    N2, M2 = 524288, 400
    l2 = synth.causal_lens(N2, M2, 0, window=8000)
    x2 = synth.indexer_rows(l2, N2, seed=62, device=DEV)
    with torch.cuda.stream(s):
        o2 = ets.topk_ragged(x2, l2.to(DEV), K)
    s.synchronize()
    p2, b2 = ets.cached_workspace(DEV, s)
    assert p2 != p1 and b2 > b1
    verify(x2, l2, K, o2)
    # the graph's workspace is still a live allocation (checked on the host
    # before anything replays the graph) ...
    assert _is_live_device_allocation(p1)
    # ... so the graph replays correctly with new data written in place
    x1.copy_(synth.indexer_rows(l1, N1, seed=63, device=DEV))
    o1.fill_(-5)
    g.replay()
    s.synchronize()
    verify(x1, l1, K, o1)


def test_new_workspace_is_zeroed_on_the_calls_stream(ets):
    """A fresh workspace on a non-blocking stream, over memory that held
    nonzero bytes just before (filled, freed back to the driver): the queue
    counters must read zero, so every row of the result is served."""
    junk = torch.full((1 << 28,), -1, dtype=torch.int32, device=DEV)  # 1 GiB of 0xFF
    torch.cuda.synchronize()
    del junk
    torch.cuda.empty_cache()
    s = torch.cuda.Stream(device=DEV)  # a stream the library has not seen
    assert ets.cached_workspace(DEV, s) == (0, 0)
    N, M = 65536, 2048
    lens = synth.causal_lens(N, M, 0)
    x = synth.indexer_rows(lens, N, seed=64, device=DEV)
    d = lens.to(DEV)
    assert ets.plan(M, N, K)["kind"] == "persistent"
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        got = torch.full((M, K), -7, dtype=torch.int32, device=DEV)
        ets.topk_ragged(x, d, K, out=got)
    s.synchronize()
    verify(x, lens, K, got)


def test_host_buffer_call_from_two_threads(ets):
    """Two host threads calling the host-buffer form at once take turns on
    the device's buffers; both results are exact."""
    N = 131072
    jobs = []
    for i, M in enumerate((96, 160)):
        lens = synth.causal_lens(N, M, 0, window=M * 4)
        x = synth.indexer_rows(lens, N, seed=70 + i, device=DEV).cpu().numpy()
        jobs.append((x, lens.numpy()))
    results = [None, None]
    errors = []

    def work(i):
        try:
            x, l = jobs[i]
            results[i] = ets.topk_ragged_host(x, l, K, rows_per_chunk=32)
        except Exception as e:  # reported below
            errors.append(e)

    th = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not errors, errors
    for (x, l), got in zip(jobs, results):
        v = oracle.compare(x, l, K, got)
        assert not v["check"].any() and not v["set_mismatch"].any()
