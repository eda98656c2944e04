"""CPU checks of the seeded input generators (shapes, lengths, suffix, recipe)."""
import numpy as np
import torch

import oracle
from exact_top_sparse_gb300 import synth


def test_causal_lengths():
    lens = synth.causal_lens(131072, 512, group=3)
    assert lens.dtype == torch.int32 and lens.numel() == 512
    j0 = 3 * 512
    assert int(lens[0]) == 131072 - 8192 + j0 + 1
    assert torch.all(lens[1:] - lens[:-1] == 1)
    assert int(synth.causal_lens(131072, 8192)[-1]) == 131072


def test_tiny_lengths_force_short_rows():
    for seed in range(5):
        lens = synth.tiny_lens(seed)
        assert lens.numel() == 8
        assert int((lens <= 2048).sum()) >= 2
        assert int(lens.min()) >= 512 and int(lens.max()) <= 16384


def test_indexer_rows_recipe_and_suffix():
    lens = torch.tensor([1000, 5000, 0, 20000], dtype=torch.int32)
    x = synth.indexer_rows(lens, 20000, seed=11)
    assert x.shape == (4, 20000) and x.dtype == torch.float32
    for r, L in enumerate(lens.tolist()):
        assert torch.all(torch.isinf(x[r, L:]) & (x[r, L:] < 0))
        assert torch.all(torch.isfinite(x[r, :L]))
    body = x[3, :20000]
    assert 25 < float(body.median()) < 35
    # a long upper tail: more mass far above the body than a normal would give
    # (a normal body alone would put ~0.6 of 20000 entries 4 sigma above the
    # median; the exponential tail puts ~7.6 there)
    assert int((body > float(body.median()) + 10).sum()) > 3
    # deterministic for a seed
    assert torch.equal(x, synth.indexer_rows(lens, 20000, seed=11))


def test_bf16_grid_creates_boundary_ties():
    lens = torch.full((4,), 30000, dtype=torch.int32)
    x = synth.to_bf16_grid(synth.indexer_rows(lens, 30000, seed=2))
    _, _, tied = oracle.boundary(x.numpy(), lens.numpy(), 2048)
    assert tied.all()


def test_strided_rows_drive_the_intended_paths():
    # len 10000, stride 128 -> r0 = 25, r1 = 29 at K = 2048 (targets 3072/3584)
    L, s, K = 10000, 128, 2048
    lens = torch.full((1,), L, dtype=torch.int32)
    tau1 = synth.strided_high_rows(lens, L, seed=1, stride=s, n_top=27, n_mid=2048)
    rec = synth.strided_high_rows(lens, L, seed=2, stride=s, n_top=40, n_mid=2048)
    over = synth.strided_high_rows(torch.full((1,), 65536, dtype=torch.int32), 65536, seed=3,
                                   stride=s, n_top=0, n_mid=20000, on_grid=False)
    p = [oracle.thresholds(x.numpy(), np.array([x.shape[1]], np.int32), K, s, 3072, 3584, 0)
         for x in (tau1, rec, over)]
    assert p[0]["path"][0] == oracle.PATH_TAU1
    assert p[1]["path"][0] == oracle.PATH_RECOVERY
    assert p[2]["path"][0] == oracle.PATH_TAU0 and p[2]["count"][0, 1] > 20000


def test_recovery_rows_take_one_pass_or_fall_back():
    """The library's recovery first tries the band between tau1 and a lower
    threshold tau2 of the same view (target 2 * T1).  Row `one` (40 lifted
    grid values) has enough scores above tau2 for that band to finish the
    row; row `two` (80 lifted values) does not, so the two-pass selection
    runs.  Both rows underfill tau1."""
    L, s, K, T1 = 65536, 128, 2048, 3584
    lens = torch.full((1,), L, dtype=torch.int32)
    one = synth.strided_high_rows(lens, L, seed=2, stride=s, n_top=40, n_mid=2100)
    two = synth.strided_high_rows(lens, L, seed=6, stride=s, n_top=80, n_mid=2100)
    for x, enough in ((one, True), (two, False)):
        xh, lh = x.numpy(), np.array([L], np.int32)
        p1 = oracle.thresholds(xh, lh, K, s, 3072, T1, 0)
        p2 = oracle.thresholds(xh, lh, K, s, 2 * T1, 2 * T1, 0)
        assert p1["path"][0] == oracle.PATH_RECOVERY
        assert (p2["count"][0, 1] >= K) == enough

