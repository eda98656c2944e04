"""Pins for the CPU oracle: each check rests on something other than the oracle.

* hand-built cases with hand-derived answers (tests/golden/contract_cases.txt,
  from the set contract);
* brute force: Python's sort of (-score, index) on every tiny row;
* a library third opinion: torch.topk on untied rows;
* closed forms: the len <= K sentinel rule; thresholds on monotone rows
  (tests/golden/threshold_cases.txt);
* invariants: certification soundness (C(tau0) >= K implies the K-th largest
  score reaches tau0), nesting (tau1 <= tau0, C(tau1) >= C(tau0));
* mutation: every kind of contract break planted in a correct answer must be
  rejected by the checker.
"""
import os
import random

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import GOLDEN


def _parse_contract_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "contract_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest, "pad": 0}
                cases.append(cur)
            elif key == "why":
                continue
            elif key == "K":
                cur["K"] = int(rest)
            elif key == "pad":
                cur["pad"] = int(rest)
            elif key == "scores":
                cur["scores"] = [float(x) for x in rest.split()] if rest else []
            elif key in ("must", "tie", "oracle"):
                cur[key] = [] if rest.strip() in ("", "-") else [int(x) for x in rest.split()]
            elif key == "take":
                cur["take"] = int(rest)
    return cases


CONTRACT_CASES = _parse_contract_cases()


def _row(case):
    vals = case["scores"] + [float("-inf")] * case["pad"]
    if not vals:
        vals = [float("-inf")]
    x = np.array([vals], dtype=np.float32)
    lens = np.array([len(case["scores"])], dtype=np.int32)
    return x, lens


@pytest.mark.parametrize("case", CONTRACT_CASES, ids=[c["name"] for c in CONTRACT_CASES])
def test_golden_contract_cases(case):
    x, lens = _row(case)
    K = case["K"]
    got = oracle.topk(x, lens, K)[0]
    assert got.tolist() == case["oracle"]
    # every answer that keeps `must` and `take` members of `tie` passes the checker
    L = len(case["scores"])
    sentinels = [-1] * max(0, K - L)
    tie = case["tie"]
    for trial in range(10):
        rng = random.Random(trial)
        pick = rng.sample(tie, case["take"]) if tie else []
        ans = case["must"] + pick
        rng.shuffle(ans)
        ans = ans + sentinels
        assert len(ans) == K
        codes = oracle.check(x, lens, K, np.array([ans], dtype=np.int32))
        assert codes[0] == 0, (case["name"], ans)
    # the boundary tie flag agrees with the hand derivation
    if L > K:
        _, _, tied = oracle.boundary(x, lens, K)
        assert bool(tied[0]) == (len(tie) > case["take"] > 0)


def _brute(vals, L, K):
    if L <= K:
        return list(range(L)) + [-1] * (K - L)
    order = sorted(range(L), key=lambda i: (-vals[i], i))
    return sorted(order[:K])


@pytest.mark.parametrize("dist", ["continuous", "few_values", "with_inf"])
def test_brute_force_tiny_rows(dist):
    rng = np.random.default_rng(12345 + len(dist))
    N = 64
    rows, lens, Ks = [], [], []
    for L in range(0, N + 1):
        for K in (1, 2, 3, 7, L - 1, L, L + 1, L + 2):
            if K < 1:
                continue
            if dist == "continuous":
                v = rng.standard_normal(N).astype(np.float32)
            elif dist == "few_values":
                v = rng.integers(0, 4, N).astype(np.float32)
            else:
                v = rng.choice(np.array([-np.inf, -1.0, 0.0, -0.0, 1.0, np.inf], np.float32), N)
            rows.append(v)
            lens.append(L)
            Ks.append(K)
    # oracle calls take one K; group rows by K
    for K in sorted(set(Ks)):
        sel = [i for i, k in enumerate(Ks) if k == K]
        x = np.stack([rows[i] for i in sel])
        ln = np.array([lens[i] for i in sel], dtype=np.int32)
        got = oracle.topk(x, ln, K)
        for j, i in enumerate(sel):
            assert got[j].tolist() == _brute(rows[i].tolist(), lens[i], K)
        assert np.all(oracle.check(x, ln, K, got) == 0)


def test_torch_topk_agrees_on_untied_rows():
    rng = np.random.default_rng(7)
    M, N, K = 16, 5000, 300
    x = rng.standard_normal((M, N)).astype(np.float32) * 3 + 30
    lens = rng.integers(K + 1, N + 1, M).astype(np.int32)
    got = oracle.topk(x, lens, K)
    _, _, tied = oracle.boundary(x, lens, K)
    for r in range(M):
        if tied[r]:
            continue
        ref = torch.topk(torch.from_numpy(x[r, :lens[r]].copy()), K, sorted=False).indices
        assert sorted(ref.tolist()) == got[r].tolist()


@pytest.mark.parametrize("L", [0, 1, 2047, 2048, 2049])
def test_sentinel_rule_closed_form(L):
    K, N = 2048, 4096
    x = np.random.default_rng(L).standard_normal((1, N)).astype(np.float32)
    got = oracle.topk(x, np.array([L], np.int32), K)[0]
    if L <= K:
        assert got.tolist() == list(range(L)) + [-1] * (K - L)
    else:
        assert len(set(got.tolist())) == K and -1 not in got


def test_row_lens_are_clamped():
    K, N = 4, 10
    x = np.arange(N, dtype=np.float32)[None, :].repeat(3, 0)
    lens = np.array([-5, 1000, 3], dtype=np.int32)
    got = oracle.topk(x, lens, K)
    assert got[0].tolist() == [-1] * 4          # clamped to 0
    assert got[1].tolist() == [6, 7, 8, 9]      # clamped to N
    assert got[2].tolist() == [0, 1, 2, -1]


def test_boundary_values_match_sorted_row():
    rng = np.random.default_rng(3)
    M, N, K = 8, 777, 100
    x = rng.integers(0, 50, (M, N)).astype(np.float32)
    lens = rng.integers(K + 1, N + 1, M).astype(np.int32)
    kth, kth1, tied = oracle.boundary(x, lens, K)
    for r in range(M):
        s = np.sort(x[r, :lens[r]])[::-1]
        assert kth[r] == s[K - 1] and kth1[r] == s[K]
        assert bool(tied[r]) == (s[K - 1] == s[K])


# ---------------------------------------------------------------- checker mutations

def _base_case():
    rng = np.random.default_rng(99)
    N, K = 50, 8
    x = rng.permutation(N).astype(np.float32)[None, :]   # distinct scores
    lens = np.array([N], np.int32)
    good = oracle.topk(x, lens, K)
    assert oracle.check(x, lens, K, good)[0] == 0
    return x, lens, K, good


def test_checker_rejects_duplicate():
    x, lens, K, good = _base_case()
    bad = good.copy()
    bad[0, 1] = bad[0, 0]
    assert oracle.check(x, lens, K, bad)[0] == 2


def test_checker_rejects_out_of_range_and_negative():
    x, lens, K, good = _base_case()
    bad = good.copy()
    bad[0, 3] = lens[0]
    assert oracle.check(x, lens, K, bad)[0] == 1
    bad = good.copy()
    bad[0, 3] = -2
    assert oracle.check(x, lens, K, bad)[0] == 1


def test_checker_rejects_swapped_smaller_for_larger():
    x, lens, K, good = _base_case()
    sel = set(good[0].tolist())
    # replace the selected max with the best unselected index (strictly smaller)
    vals = x[0]
    best_out = max((i for i in range(lens[0]) if i not in sel), key=lambda i: vals[i])
    bad = good.copy()
    j = int(np.argmax(vals[bad[0]]))
    bad[0, j] = best_out
    assert oracle.check(x, lens, K, bad)[0] == 4


def test_checker_rejects_sentinel_in_long_row():
    x, lens, K, good = _base_case()
    bad = good.copy()
    bad[0, 5] = -1
    assert oracle.check(x, lens, K, bad)[0] == 3


def test_checker_rejects_missing_sentinel_and_missing_index():
    K = 6
    x = np.arange(10, dtype=np.float32)[None, :]
    lens = np.array([4], np.int32)
    ok = np.array([[3, 1, 0, 2, -1, -1]], np.int32)
    assert oracle.check(x, lens, K, ok)[0] == 0
    missing_index = np.array([[3, 1, 0, -1, -1, -1]], np.int32)
    assert oracle.check(x, lens, K, missing_index)[0] == 5
    # a fifth slot filled with an index beyond len is an out-of-range index
    extra = np.array([[3, 1, 0, 2, 4, -1]], np.int32)
    assert oracle.check(x, lens, K, extra)[0] == 1


# ---------------------------------------------------------------- thresholds

def _threshold_cases():
    out = []
    with open(os.path.join(GOLDEN, "threshold_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            left, right = line.split("|")
            name, kind, L, s, K, T0, T1 = left.split()
            r0, r1, t0, t1, c0, c1, path = right.split()
            out.append(dict(name=name, kind=kind, L=int(L), s=int(s), K=int(K), T0=int(T0),
                            T1=int(T1), r0=int(r0), r1=int(r1), t0=float(t0), t1=float(t1),
                            c0=int(c0), c1=int(c1), path=int(path)))
    return out


THR = _threshold_cases()


@pytest.mark.parametrize("c", THR, ids=[c["name"] for c in THR])
def test_threshold_closed_forms(c):
    L = c["L"]
    i = np.arange(L, dtype=np.float32)
    v = -i if c["kind"] == "dec" else i
    x = np.concatenate([v, np.full(7, -np.inf, np.float32)])[None, :]
    res = oracle.thresholds(x, np.array([L], np.int32), c["K"], c["s"], c["T0"], c["T1"], 0)
    assert res["rank"][0].tolist() == [c["r0"], c["r1"]]
    assert res["tau"][0].tolist() == [c["t0"], c["t1"]]
    assert res["count"][0].tolist() == [c["c0"], c["c1"]]
    assert res["path"][0] == c["path"]


def test_threshold_paths_hand_built_tau1_and_recovery():
    # len 10000, s = 128: n_s = 79, r0 = 25, r1 = 29 at K = 2048 (see golden file).
    L, s, K = 10000, 128, 2048
    x = np.zeros((2, L), np.float32)
    grid = np.arange(0, L, s)
    # row 0: sample j holds 100 - j, so tau0 = 76 and tau1 = 72.  2048 entries
    # off the grid hold 74.5, between the two: C(tau0) = 25 < K and
    # C(tau1) = 29 + 2048 >= K -> the nested threshold serves the row.
    x[0, grid] = 100 - np.arange(grid.size)
    off = np.setdiff1d(np.arange(L), grid)[:2048]
    x[0, off] = 74.5
    # row 1: every sample is 1, everything else 0: tau0 = tau1 = 1 and
    # C(tau1) = 79 < K -> exact recovery.
    x[1, grid] = 1.0
    res = oracle.thresholds(x, np.array([L, L], np.int32), K, s, 3072, 3584, 0)
    assert res["tau"][0].tolist() == [76.0, 72.0]
    assert res["count"][0].tolist() == [25, 29 + 2048]
    assert res["path"].tolist() == [oracle.PATH_TAU1, oracle.PATH_RECOVERY]
    assert res["count"][1].tolist() == [79, 79]


def test_threshold_paths_sentinel_and_direct():
    x = np.ones((2, 5000), np.float32)
    res = oracle.thresholds(x, np.array([100, 4000], np.int32), 2048, 128, 3072, 3584, 4096)
    assert res["path"].tolist() == [oracle.PATH_SENTINEL, oracle.PATH_DIRECT]


def test_certification_invariants_random_rows():
    rng = np.random.default_rng(5)
    M, N, K = 24, 40000, 2048
    x = (rng.standard_normal((M, N)) * 2.5 + 30).astype(np.float32)
    tail = rng.random((M, N)) < 0.002
    x[tail] = 30 + rng.exponential(6, tail.sum())
    lens = rng.integers(2 * K, N + 1, M).astype(np.int32)
    res = oracle.thresholds(x, lens, K, 128, 3072, 3584, 0)
    kth, _, _ = oracle.boundary(x, lens, K)
    tau, cnt, path = res["tau"], res["count"], res["path"]
    assert np.all(tau[:, 1] <= tau[:, 0])
    assert np.all(cnt[:, 1] >= cnt[:, 0])
    for r in range(M):
        row = x[r, :lens[r]]
        # counts by brute force
        assert cnt[r, 0] == np.count_nonzero(row >= tau[r, 0])
        # certification soundness: if C(tau) >= K the K-th largest reaches tau,
        # so the top-K set lies inside {v >= tau}
        for j in range(2):
            if cnt[r, j] >= K:
                assert kth[r] >= tau[r, j]
            else:
                assert kth[r] < tau[r, j]
        expect = 2 if cnt[r, 0] >= K else 3 if cnt[r, 1] >= K else 4
        assert path[r] == expect
