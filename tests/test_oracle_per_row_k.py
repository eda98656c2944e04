"""Pins of the oracle's per-row-K selection (CPU only).

Per-row K composes the one-K set contract (codexqa.cn, section
"什么叫精确，时间怎么量") row by row: row r holds the Top-k_r of its valid
prefix in its first k_r slots and -1 after them.  Pinned here by brute force
(a full sort in plain Python) on tiny rows, by its closed forms (k = 0 gives
a row of -1, k = K_max is the one-K result) and by the verdict catching
planted mistakes.
"""
import numpy as np
import pytest

import oracle

K_MAX = 24


def brute(row, L, k, K_max):
    """Full sort by (score descending, index ascending) of the first L scores."""
    out = [-1] * K_max
    if k == 0:
        return out
    if L <= k:
        out[:L] = list(range(L))
        return out
    order = sorted(range(L), key=lambda i: (-float(row[i]), i))[:k]
    out[:k] = sorted(order)
    return out


def tiny_case(seed, M=40, N=64, distinct=True):
    rng = np.random.default_rng(seed)
    if distinct:
        x = np.stack([rng.permutation(N).astype(np.float32) - 20.0 for _ in range(M)])
    else:
        x = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    lens = rng.integers(0, N + 1, size=M).astype(np.int32)
    ks = rng.integers(-4, K_MAX + 6, size=M).astype(np.int32)
    ks[:4] = [0, 1, K_MAX, K_MAX + 9]
    lens[:4] = [N, N, N, N]
    return x, lens, ks


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_brute_force_untied(seed):
    x, lens, ks = tiny_case(seed)
    got = oracle.topk_per_row(x, lens, ks, K_MAX, threads=2)
    kc = np.clip(ks, 0, K_MAX)
    for r in range(x.shape[0]):
        assert got[r].tolist() == brute(x[r], int(lens[r]), int(kc[r]), K_MAX), r


def test_closed_forms():
    x, lens, _ = tiny_case(5)
    M = x.shape[0]
    zero = oracle.topk_per_row(x, lens, np.zeros(M, np.int32), K_MAX)
    assert np.all(zero == -1)
    neg = oracle.topk_per_row(x, lens, np.full(M, -7, np.int32), K_MAX)
    assert np.all(neg == -1)
    full = oracle.topk_per_row(x, lens, np.full(M, K_MAX, np.int32), K_MAX)
    assert np.array_equal(full, oracle.topk(x, lens, K_MAX))
    over = oracle.topk_per_row(x, lens, np.full(M, 10 * K_MAX, np.int32), K_MAX)
    assert np.array_equal(over, full)


@pytest.mark.parametrize("seed", [3, 4])
def test_verdict_accepts_any_tie_choice(seed):
    x, lens, ks = tiny_case(seed, distinct=False)
    kc = np.clip(ks, 0, K_MAX)
    # brute force breaks ties by lowest index; flip it to highest index, which
    # is just as correct under the contract
    got = np.full((x.shape[0], K_MAX), -1, np.int32)
    for r in range(x.shape[0]):
        L, k = int(lens[r]), int(kc[r])
        if k == 0:
            continue
        if L <= k:
            got[r, :L] = np.arange(L)[::-1]
            continue
        order = sorted(range(L), key=lambda i: (-float(x[r, i]), -i))[:k]
        got[r, :k] = order
    v = oracle.compare_per_row(x, lens, ks, K_MAX, got)
    assert not v["check"].any() and not v["set_mismatch"].any() and not v["tail"].any()


def test_verdict_catches_planted_mistakes():
    x, lens, ks = tiny_case(7)
    lens[:] = x.shape[1]
    ks[:] = 8
    good = oracle.topk_per_row(x, lens, ks, K_MAX)
    v = oracle.compare_per_row(x, lens, ks, K_MAX, good)
    assert not v["check"].any() and not v["set_mismatch"].any() and not v["tail"].any()
    # a selected index swapped for the row's smallest score
    bad = good.copy()
    bad[0, 0] = int(np.argmin(x[0]))
    v = oracle.compare_per_row(x, lens, ks, K_MAX, bad)
    assert v["check"][0] == 4 or v["check"][0] == 2
    # a valid index written past k_r
    bad = good.copy()
    bad[1, 8] = 0
    v = oracle.compare_per_row(x, lens, ks, K_MAX, bad)
    assert v["tail"][1] and not v["tail"][0]
    # one slot short: the row's k_r-th slot left at -1
    bad = good.copy()
    bad[2, 7] = -1
    v = oracle.compare_per_row(x, lens, ks, K_MAX, bad)
    assert v["check"][2] == 3
