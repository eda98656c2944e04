"""CPU oracle for exact Top-K over ragged FP32 score rows (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg use this package.  It shares no code with the CUDA selector and
never imports it.  The arithmetic lives in ``topk_oracle.cpp`` (plain C++ with
std::nth_element); this module only marshals numpy arrays.

Sources followed (web pages on "Sample-Guided Exact Top-K Selection for
Long-Context Sparse Attention"):
  * set contract -- codexqa.cn "几何平均快 1.55 倍…腾讯怎么测精确 Top-K",
    section "什么叫精确，时间怎么量";
  * thresholds and paths -- PaperDaily "腾讯|长上下文稀疏注意力前K精确选择",
    section 问题二 (Fig. 4 stages 1-2), and codexqa.cn section
    "采样不是处处都该开" (stride 128, targets 1.5K / 1.75K).

  * indexer scores (the stage that produces the rows) -- xllm-io review of
    LiteTopK, section "核心公式", eq. (1).

Parity status: the selection, the boundary values and the checker are pinned
by brute force, closed forms and hand-built tie rows in tests/.  The
thresholds are pinned by closed forms on strictly monotone rows; the rank rule
itself (ceil(T * n_s / len)) is a reading of the pages, which do not print it.
Per-row K (topk_per_row) composes the one-K selection row by row and is
pinned by brute force on tiny rows and its closed forms (k = 0, k = K_max).
The ordered output (order) is pinned by a hand-derived golden case, by
numpy's argsort on rows of distinct values and by its invariants.
The indexer scores are pinned by a hand-derived case, the one-hot closed form,
invariances of eq. (1) and exact dense products on tiny integer inputs.
"""
import ctypes
import os

import numpy as np

from . import build as _build

PATH_SENTINEL = 0
PATH_DIRECT = 1
PATH_TAU0 = 2
PATH_TAU1 = 3
PATH_RECOVERY = 4

CHECK_CODES = {
    0: "ok",
    1: "index outside the valid prefix",
    2: "duplicate index",
    3: "len > K but not exactly K valid indices",
    4: "min(selected) < max(unselected)",
    5: "len <= K but valid indices are not 0..len-1",
    6: "len <= K but sentinel count != K - len",
}

_lib = None


def _bind(path):
    lib = ctypes.CDLL(path)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    lib.oracle_topk.argtypes = [vp, vp, i64, i64, i32, vp, ctypes.c_int]
    lib.oracle_topk.restype = ctypes.c_int
    lib.oracle_check.argtypes = [vp, vp, i64, i64, i32, vp, vp, ctypes.c_int]
    lib.oracle_check.restype = i64
    lib.oracle_boundary.argtypes = [vp, vp, i64, i64, i32, vp, vp, vp, ctypes.c_int]
    lib.oracle_boundary.restype = ctypes.c_int
    lib.oracle_thresholds.argtypes = [vp, vp, i64, i64, i32, i32, i32, i32, i64,
                                      vp, vp, vp, vp, ctypes.c_int]
    lib.oracle_thresholds.restype = ctypes.c_int
    lib.oracle_index_scores.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, vp, i64, vp, vp,
                                        ctypes.c_int]
    lib.oracle_index_scores.restype = ctypes.c_int
    lib.oracle_order.argtypes = [vp, vp, i64, i64, i32, vp, vp, ctypes.c_int]
    lib.oracle_order.restype = ctypes.c_int
    lib.oracle_default_threads.argtypes = []
    lib.oracle_default_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(_build.build())
    return _lib


class use_library:
    """Context manager: route every call to another build of the oracle.

    Used by the mutation tests, which compile deliberately broken copies of
    the oracle source and check that the pins reject them.
    """

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self.saved = _lib
        _lib = _bind(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _as_inputs(scores, row_lens):
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    if scores.ndim != 2:
        raise ValueError("scores must be [M, N_alloc]")
    row_lens = np.ascontiguousarray(row_lens, dtype=np.int32)
    if row_lens.shape != (scores.shape[0],):
        raise ValueError("row_lens must be [M]")
    return scores, row_lens


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def topk(scores, row_lens, K: int, threads: int = 0) -> np.ndarray:
    """Exact Top-K per row; [M, K] int32, chosen indices ascending, -1 padding."""
    scores, row_lens = _as_inputs(scores, row_lens)
    M, N = scores.shape
    out = np.empty((M, K), dtype=np.int32)
    rc = _load().oracle_topk(_p(scores), _p(row_lens), M, N, K, _p(out), threads)
    if rc != 0:
        raise ValueError("oracle_topk: bad arguments")
    return out


def check(scores, row_lens, K: int, out, threads: int = 0) -> np.ndarray:
    """Contract check of an [M, K] int32 result; per-row codes (0 = ok)."""
    scores, row_lens = _as_inputs(scores, row_lens)
    M, N = scores.shape
    out = np.ascontiguousarray(out, dtype=np.int32)
    if out.shape != (M, K):
        raise ValueError("out must be [M, K]")
    err = np.empty(M, dtype=np.int32)
    rc = _load().oracle_check(_p(scores), _p(row_lens), M, N, K, _p(out), _p(err), threads)
    if rc < 0:
        raise ValueError("oracle_check: bad arguments")
    return err


def boundary(scores, row_lens, K: int, threads: int = 0):
    """(kth, kth1, tied) per row: K-th and (K+1)-th largest scores, tie flag."""
    scores, row_lens = _as_inputs(scores, row_lens)
    M, N = scores.shape
    kth = np.empty(M, dtype=np.float32)
    kth1 = np.empty(M, dtype=np.float32)
    tied = np.empty(M, dtype=np.uint8)
    rc = _load().oracle_boundary(_p(scores), _p(row_lens), M, N, K, _p(kth), _p(kth1),
                                 _p(tied), threads)
    if rc != 0:
        raise ValueError("oracle_boundary: bad arguments")
    return kth, kth1, tied.astype(bool)


def thresholds(scores, row_lens, K: int, stride: int, target0: int, target1: int,
               sample_min_len: int, threads: int = 0):
    """Sampled thresholds, counts, ranks and path per row.

    Returns a dict with tau [M,2] float32, count [M,2] int64, rank [M,2] int64
    and path [M] int32 (PATH_* constants).
    """
    scores, row_lens = _as_inputs(scores, row_lens)
    M, N = scores.shape
    tau = np.empty((M, 2), dtype=np.float32)
    cnt = np.empty((M, 2), dtype=np.int64)
    rank = np.empty((M, 2), dtype=np.int64)
    path = np.empty(M, dtype=np.int32)
    rc = _load().oracle_thresholds(_p(scores), _p(row_lens), M, N, K, stride, target0, target1,
                                   sample_min_len, _p(tau), _p(cnt), _p(rank), _p(path), threads)
    if rc != 0:
        raise ValueError("oracle_thresholds: bad arguments")
    return {"tau": tau, "count": cnt, "rank": rank, "path": path}


def compare(scores, row_lens, K: int, got, threads: int = 0):
    """Full parity verdict of a result against the oracle.

    Every row must pass the contract checker; rows whose boundary is untied
    must equal the oracle's set exactly.  Returns a dict with per-row arrays
    ``check`` (checker codes), ``tied`` and ``set_mismatch`` (bool).
    """
    scores, row_lens = _as_inputs(scores, row_lens)
    got = np.ascontiguousarray(got, dtype=np.int32)
    codes = check(scores, row_lens, K, got, threads)
    ref = topk(scores, row_lens, K, threads)
    _, _, tied = boundary(scores, row_lens, K, threads)
    mism = np.any(np.sort(got, axis=1) != np.sort(ref, axis=1), axis=1) & ~tied
    return {"check": codes, "tied": tied, "set_mismatch": mism}


def order(scores, row_lens, K: int, idx, threads: int = 0) -> np.ndarray:
    """The ordered form of an [M, K] index result: each row's indices by score,
    largest first, equal scores by smaller index, -1 sentinels last (the
    contract leaves the order free; this is the optional ordered output).
    Raises ValueError if a row holds an index outside its valid prefix."""
    scores, row_lens = _as_inputs(scores, row_lens)
    M, N = scores.shape
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    if idx.shape != (M, K):
        raise ValueError("idx must be [M, K]")
    out = np.empty((M, K), dtype=np.int32)
    rc = _load().oracle_order(_p(scores), _p(row_lens), M, N, K, _p(idx), _p(out), threads)
    if rc != 0:
        raise ValueError("oracle_order: bad arguments or an index outside its row")
    return out


def clamp_row_k(row_k, K_max: int) -> np.ndarray:
    """Per-row K as the library under test documents it: clamp into [0, K_max]."""
    return np.clip(np.asarray(row_k, dtype=np.int64), 0, K_max)


def topk_per_row(scores, row_lens, row_k, K_max: int, threads: int = 0) -> np.ndarray:
    """Per-row K: row r holds the exact Top-k_r of its valid prefix
    (k_r = clamp(row_k[r], 0, K_max); the set contract with K = k_r) in slots
    [0, k_r) of an [M, K_max] int32 result, -1 in the other slots.  The pages
    fix one K per call; this composes the one-K definition row by row."""
    scores, row_lens = _as_inputs(scores, row_lens)
    ks = clamp_row_k(row_k, K_max)
    out = np.full((scores.shape[0], K_max), -1, dtype=np.int32)
    for k in np.unique(ks):
        if k == 0:
            continue
        rows = np.nonzero(ks == k)[0]
        out[rows, :k] = topk(scores[rows], row_lens[rows], int(k), threads)
    return out


def compare_per_row(scores, row_lens, row_k, K_max: int, got, threads: int = 0):
    """Parity verdict for a per-row-K result: each row's first k_r slots get
    the one-K verdict of ``compare`` at K = k_r; ``tail`` marks rows whose
    slots [k_r, K_max) are not all -1."""
    scores, row_lens = _as_inputs(scores, row_lens)
    got = np.ascontiguousarray(got, dtype=np.int32)
    M = scores.shape[0]
    if got.shape != (M, K_max):
        raise ValueError("got must be [M, K_max]")
    ks = clamp_row_k(row_k, K_max)
    codes = np.zeros(M, dtype=np.int32)
    tied = np.zeros(M, dtype=bool)
    mism = np.zeros(M, dtype=bool)
    tail = np.array([np.any(got[r, ks[r]:] != -1) for r in range(M)], dtype=bool)
    for k in np.unique(ks):
        if k == 0:
            continue
        rows = np.nonzero(ks == k)[0]
        v = compare(scores[rows], row_lens[rows], int(k), got[rows, :k], threads)
        codes[rows], tied[rows], mism[rows] = v["check"], v["tied"], v["set_mismatch"]
    return {"check": codes, "tied": tied, "set_mismatch": mism, "tail": tail}


def index_scores(q_bits, k_bits, w, ts, ss, threads: int = 0):
    """Indexer scores I[t, s] of eq. (1) (xllm-io LiteTopK review, "核心公式")
    at the pairs (ts[i], ss[i]), in double.

    q_bits: uint16 [T, H, D] and k_bits: uint16 [S, D], raw bfloat16 patterns;
    w: float32 [T, H].  Returns (value, magnitude), both float64 [n]:
    magnitude = sum_j |w_tj| * sum_d |q_tjd * k_sd|, the scale of the rounding
    error of a lower-precision evaluation.
    """
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.float32)
    if q_bits.ndim != 3 or k_bits.ndim != 2 or w.shape != q_bits.shape[:2]:
        raise ValueError("need q [T, H, D], k [S, D], w [T, H]")
    T, H, D = q_bits.shape
    if k_bits.shape[1] != D:
        raise ValueError("q and k disagree on D")
    ts = np.ascontiguousarray(ts, dtype=np.int64)
    ss = np.ascontiguousarray(ss, dtype=np.int64)
    if ts.shape != ss.shape or ts.ndim != 1:
        raise ValueError("ts and ss must be 1-D of one length")
    n = ts.shape[0]
    value = np.empty(n, dtype=np.float64)
    mag = np.empty(n, dtype=np.float64)
    rc = _load().oracle_index_scores(_p(q_bits), _p(k_bits), _p(w), T, k_bits.shape[0], H, D,
                                     _p(ts), _p(ss), n, _p(value), _p(mag), threads)
    if rc != 0:
        raise ValueError("oracle_index_scores: bad arguments")
    return value, mag

