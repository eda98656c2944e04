"""Pins of the oracle's ordered output (CPU only).

oracle.order lists an index row by score, largest first, equal scores by
smaller index first, -1 sentinels last (the contract leaves the order free;
this is the library's optional ordered output).  Pinned by hand-derived golden
cases (tests/golden/order_cases.txt), by numpy's argsort on rows of distinct
values (where the order is unique) and by its invariants on tie-heavy rows.
"""
import os

import numpy as np
import pytest

import oracle
from tests.conftest import GOLDEN


def _cases():
    blocks = open(os.path.join(GOLDEN, "order_cases.txt")).read().split("\n\n")
    out = []
    for b in blocks:
        lines = [ln for ln in b.strip().splitlines() if ln and not ln.startswith("#")]
        if not lines or not lines[0].startswith("case"):
            continue
        d = {}
        for ln in lines:
            key, _, rest = ln.partition(" ")
            d[key] = rest.strip()
        out.append(d)
    return out


ORDER_CASES = _cases()


@pytest.mark.parametrize("case", ORDER_CASES, ids=[c["case"] for c in ORDER_CASES])
def test_golden_order_cases(case):
    K = int(case["K"])
    v = np.array([float(t) for t in case["scores"].split()], dtype=np.float32)
    idx = np.array([int(t) for t in case["idx"].split()], dtype=np.int32)
    want = np.array([int(t) for t in case["ordered"].split()], dtype=np.int32)
    got = oracle.order(v[None, :], np.array([v.size]), K, idx[None, :])
    assert got[0].tolist() == want.tolist()


def test_distinct_values_follow_argsort():
    rng = np.random.default_rng(5)
    for _ in range(200):
        L = int(rng.integers(1, 80))
        K = int(rng.integers(1, L + 3))
        v = rng.permutation(L).astype(np.float32) * np.float32(0.5) - np.float32(7.0)
        n = min(K, L)
        sel = rng.choice(L, size=n, replace=False).astype(np.int32)
        row = np.full(K, -1, np.int32)
        row[rng.permutation(K)[:n]] = sel
        want = np.full(K, -1, np.int32)
        want[:n] = sel[np.argsort(-v[sel])]
        got = oracle.order(v[None, :], np.array([L]), K, row[None, :])
        assert got[0].tolist() == want.tolist()


def test_invariants_on_tied_rows():
    rng = np.random.default_rng(6)
    M, N, K = 40, 300, 64
    v = rng.integers(0, 6, size=(M, N)).astype(np.float32)
    lens = rng.integers(0, N + 1, size=M).astype(np.int32)
    idx = oracle.topk(v, lens, K)
    for r in range(M):
        rng.shuffle(idx[r])
    got = oracle.order(v, lens, K, idx)
    for r in range(M):
        g = got[r]
        n = int((idx[r] >= 0).sum())
        assert sorted(g.tolist()) == sorted(idx[r].tolist())     # same entries
        assert np.all(g[n:] == -1) and np.all(g[:n] >= 0)         # sentinels last
        s = v[r, g[:n]]
        assert np.all(s[:-1] >= s[1:])                            # scores non-increasing
        eq = s[:-1] == s[1:]
        assert np.all(g[:n][:-1][eq] < g[:n][1:][eq])             # ties by smaller index


def test_rejects_an_index_outside_its_row():
    v = np.zeros((1, 8), np.float32)
    with pytest.raises(ValueError):
        oracle.order(v, np.array([4]), 2, np.array([[1, 5]], np.int32))
    with pytest.raises(ValueError):
        oracle.order(v, np.array([4]), 2, np.array([[1, -3]], np.int32))
