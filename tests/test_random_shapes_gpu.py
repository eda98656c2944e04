"""Seeded random shapes against the oracle (GPU only).

Forty calls, each drawn from a fixed seed: row width, row count, K, element
type (FP32, bfloat16, E4M3), execution kind (the planner's choice or one
forced), sampling tier (stride 64 to 1024, targets rho0 in [1.0, 3.0] with
rho1 up to 0.75 above), the sampling minimum, ragged lengths (causal,
uniform, or with empty and short rows mixed in) and, for some FP32 calls,
per-row K.  Every row of every call must pass the oracle's checker (codexqa.cn
article, section "什么叫精确，时间怎么量") and equal the oracle's set where its
boundary is untied; sampled rows must reproduce the oracle's tau0, tau1,
C(tau0), C(tau1) and path.  The draws cover the corners that fixed cases
visit one at a time: sample ranks near the sampler warp's limit of 32, rows
just above and below the sampling minimum, odd strides, ragged tails, mixed
narrow and wide rows in one call.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_top_sparse_gb300 import synth
from tests.test_parity_gpu import verify, verify_diag

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
CASES = 40


@pytest.fixture(scope="module")
def ets():
    import __graft_entry__ as g
    g.build()
    import exact_top_sparse_gb300 as m
    return m


def draw(i):
    """Case i: every choice from one seeded generator."""
    g = np.random.default_rng(1000 + i)
    N = int(g.choice([8192, 20000, 40960, 65536, 100000, 131072, 262144, 393216, 524288]))
    M = int(g.choice([1, 3, 17, 64, 300, 700, 1300]))
    if N * M > (1 << 28):  # at most 1 GiB of FP32 scores per call
        M = max(1, (1 << 28) // N)
    K = int(g.choice([1, 16, 100, 1000, 2048, 3000, 4096]))
    dtype = str(g.choice(["f32", "f32", "bf16", "e4m3"]))
    kind = str(g.choice(["auto", "auto", "persistent", "kvsplit"]))
    stride = int(g.choice([64, 128, 256, 384, 512, 1024]))
    rho0 = float(np.round(g.uniform(1.0, 3.0), 2))
    rho1 = float(np.round(rho0 + g.uniform(0.0, 0.75), 2))
    sml = int(g.choice([0, 4096, 12288, 30000]))
    lens_kind = str(g.choice(["causal", "uniform", "mixed"]))
    per_row_k = dtype == "f32" and g.random() < 0.25
    return dict(N=N, M=M, K=K, dtype=dtype, kind=kind, stride=stride, rho0=rho0, rho1=rho1,
                sml=sml, lens_kind=lens_kind, per_row_k=per_row_k, seed=2000 + i)


def lengths(c):
    g = np.random.default_rng(c["seed"])
    N, M = c["N"], c["M"]
    if c["lens_kind"] == "causal":
        return synth.causal_lens(N, M, 0, window=M * max(1, min(N, 8192) // M))
    if c["lens_kind"] == "uniform":
        return torch.from_numpy(g.integers(N // 2, N + 1, M).astype(np.int32))
    lens = g.integers(0, N + 1, M).astype(np.int32)
    lens[g.random(M) < 0.1] = 0
    short = g.random(M) < 0.2
    lens[short] = g.integers(0, 2 * c["K"] + 2, int(short.sum()))
    return torch.from_numpy(np.minimum(lens, N).astype(np.int32))


@pytest.mark.parametrize("i", range(CASES))
def test_random_case(ets, i):
    c = draw(i)
    old = ets.get_params()
    kinds = {"auto": ets.KIND_AUTO, "persistent": ets.KIND_PERSISTENT,
             "kvsplit": ets.KIND_KVSPLIT}
    try:
        ets.set_params(force_kind=kinds[c["kind"]], stride=c["stride"], rho0=c["rho0"],
                       rho1=c["rho1"], long_len=0, sample_min_len=c["sml"])
        lens = lengths(c)
        x = synth.indexer_rows(lens, c["N"], seed=c["seed"], device=DEV)
        if c["dtype"] == "bf16":
            x = x.to(torch.bfloat16)
        elif c["dtype"] == "e4m3":
            x = (x * 4.0).clamp(max=448.0).to(torch.float8_e4m3fn)
        dl = lens.to(DEV)
        if c["per_row_k"]:
            g = np.random.default_rng(c["seed"] + 1)
            rk = torch.from_numpy(g.integers(0, c["K"] + 1, c["M"]).astype(np.int32))
            got = ets.topk_ragged_k(x, dl, rk.to(DEV), c["K"])
            torch.cuda.synchronize()
            v = oracle.compare_per_row(x.cpu().numpy(), lens.numpy(), rk.numpy(), c["K"],
                                       got.cpu().numpy())
            assert not v["check"].any(), c
            assert not v["set_mismatch"].any(), c
            assert not v["tail"].any(), c
        else:
            got, dg = ets.topk_ragged_diag(x, dl, c["K"])
            torch.cuda.synchronize()
            xf = x.float() if c["dtype"] != "f32" else x
            verify(xf, lens, c["K"], got)
            sml = c["sml"]
            if ets.plan(c["M"], c["N"], c["K"])["kind"] == "direct" and c["kind"] == "auto":
                sml = c["N"] + 1  # the direct kernel samples no row
            verify_diag(ets, xf, lens, c["K"], dg, sample_min_len=sml)
            assert not np.any(dg["flags"] & (ets.FLAG_INTERNAL | ets.FLAG_TIMEOUT)), c
    finally:
        ets.set_params(**old)
