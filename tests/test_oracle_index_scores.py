"""Pins of the oracle's indexer scores (eq. (1) of the xllm-io LiteTopK
review, section "核心公式": I[t][s] = sum_j w[t][j] * ReLU(q[t][j] . k[s])).

CPU only.  The oracle is checked against hand-derived values
(tests/golden/index_score_cases.txt), the closed form of one-hot vectors,
invariances of the definition (head order, coordinate order, linearity in w)
and, on tiny integer inputs where every sum is exact, a dense matrix product.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "index_score_cases.txt")


def bf16_bits(a):
    """Raw bfloat16 patterns of float32 values that are exact in bfloat16."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "values must be exact in bfloat16"
    return (u >> 16).astype(np.uint16)


def load_golden():
    q, k, w, exp = {}, {}, {}, []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, vals = line.split(":")
        tag, *idx = head.split()
        v = [float(x) for x in vals.split()]
        if tag == "q":
            q[(int(idx[0]), int(idx[1]))] = v
        elif tag == "k":
            k[int(idx[0])] = v
        elif tag == "w":
            w[int(idx[0])] = v
        else:
            exp.append((int(idx[0]), int(idx[1]), v[0], v[1]))
    T = 1 + max(t for t, _ in q)
    H = 1 + max(j for _, j in q)
    D = len(next(iter(q.values())))
    Q = np.zeros((T, H, D), np.float32)
    for (t, j), v in q.items():
        Q[t, j] = v
    Kk = np.array([k[s] for s in sorted(k)], np.float32)
    W = np.array([w[t] for t in sorted(w)], np.float32)
    return Q, Kk, W, exp


def scores(Q, Kk, W, ts, ss):
    return oracle.index_scores(bf16_bits(Q), bf16_bits(Kk), W, ts, ss)


def test_golden_case():
    Q, Kk, W, exp = load_golden()
    ts = [e[0] for e in exp]
    ss = [e[1] for e in exp]
    val, mag = scores(Q, Kk, W, ts, ss)
    assert val.tolist() == [e[2] for e in exp]
    assert mag.tolist() == [e[3] for e in exp]


def test_one_hot_closed_form():
    # q[t][j] = a[t][j] * e_{p[t][j]},  k[s] = b[s] * e_{r[s]}:
    # q . k = a * b when p == r, else 0, so I = sum_j w * max(0, a * b * [p == r]).
    rng = np.random.default_rng(5)
    T, H, D, S = 3, 5, 8, 7
    a = rng.choice([-2.0, -1.0, -0.5, 0.5, 1.0, 4.0], size=(T, H)).astype(np.float32)
    b = rng.choice([-1.0, 0.25, 2.0, 8.0], size=S).astype(np.float32)
    p = rng.integers(0, D, size=(T, H))
    r = rng.integers(0, D, size=S)
    W = rng.choice([0.125, 0.375, 1.0], size=(T, H)).astype(np.float32)
    Q = np.zeros((T, H, D), np.float32)
    Kk = np.zeros((S, D), np.float32)
    for t in range(T):
        for j in range(H):
            Q[t, j, p[t, j]] = a[t, j]
    for s in range(S):
        Kk[s, r[s]] = b[s]
    ts, ss = np.meshgrid(np.arange(T), np.arange(S), indexing="ij")
    val, mag = scores(Q, Kk, W, ts.ravel(), ss.ravel())
    for i, (t, s) in enumerate(zip(ts.ravel(), ss.ravel())):
        want = sum(float(W[t, j]) * max(0.0, float(a[t, j]) * float(b[s]))
                   for j in range(H) if p[t, j] == r[s])
        want_mag = sum(abs(float(W[t, j])) * abs(float(a[t, j]) * float(b[s]))
                       for j in range(H) if p[t, j] == r[s])
        assert val[i] == want and mag[i] == want_mag


def _small_ints(rng, shape, lo=-4, hi=5):
    return rng.integers(lo, hi, size=shape).astype(np.float32)


def test_invariances():
    rng = np.random.default_rng(9)
    T, H, D, S = 4, 6, 16, 10
    Q, Kk = _small_ints(rng, (T, H, D)), _small_ints(rng, (S, D))
    W = rng.choice([0.5, 1.0, 2.0], size=(T, H)).astype(np.float32)
    ts, ss = np.meshgrid(np.arange(T), np.arange(S), indexing="ij")
    ts, ss = ts.ravel(), ss.ravel()
    base, _ = scores(Q, Kk, W, ts, ss)
    hp = rng.permutation(H)      # head order
    assert np.array_equal(scores(Q[:, hp], Kk, W[:, hp], ts, ss)[0], base)
    dp = rng.permutation(D)      # coordinate order
    assert np.array_equal(scores(Q[:, :, dp], Kk[:, dp], W, ts, ss)[0], base)
    assert np.array_equal(scores(Q, Kk, 2 * W, ts, ss)[0], 2 * base)   # linear in w
    assert np.all(base >= 0)     # w >= 0 and ReLU >= 0
    assert not scores(Q, Kk, np.zeros_like(W), ts, ss)[0].any()
    # every dot product negative -> every score zero
    Qn, Kn = -np.abs(Q) - 1, np.abs(Kk) + 1
    assert not scores(Qn, Kn, W, ts, ss)[0].any()


def test_dense_product_tiny():
    # integer inputs and dyadic weights: every partial sum is exact in double
    rng = np.random.default_rng(11)
    T, H, D, S = 5, 4, 32, 9
    Q, Kk = _small_ints(rng, (T, H, D)), _small_ints(rng, (S, D))
    W = rng.choice([-1.0, 0.25, 0.5, 3.0], size=(T, H)).astype(np.float32)
    ts, ss = np.meshgrid(np.arange(T), np.arange(S), indexing="ij")
    val, mag = scores(Q, Kk, W, ts.ravel(), ss.ravel())
    dots = np.einsum("thd,sd->ths", Q.astype(np.float64), Kk.astype(np.float64))
    want = np.einsum("th,ths->ts", W.astype(np.float64), np.maximum(dots, 0.0))
    absd = np.einsum("thd,sd->ths", np.abs(Q).astype(np.float64), np.abs(Kk).astype(np.float64))
    want_mag = np.einsum("th,ths->ts", np.abs(W).astype(np.float64), absd)
    assert np.array_equal(val, want.ravel()) and np.array_equal(mag, want_mag.ravel())
    assert np.all(mag >= np.abs(val))


def test_rejects_bad_pairs():
    Q, Kk, W, _ = load_golden()
    with pytest.raises(ValueError):
        scores(Q, Kk, W, [1], [0])      # t out of range
    with pytest.raises(ValueError):
        scores(Q, Kk, W, [0], [4])      # s out of range
