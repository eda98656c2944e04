"""Seeded synthetic score rows shaped like sparse-attention indexer output.

This module only draws inputs.  It holds none of the selection arithmetic and
imports nothing else from this package, so the CUDA selector's tests and the
CPU oracle can both consume what it makes: the CUDA side reads the tensor on
the device, the oracle reads a host copy of the very same bytes.

Workload recipe (stands in for the captured Hy4-Preview indexer scores, which
are not available):
  * body  : Normal(mu_r, 2.5) with a per-row location mu_r = 30 (+ Normal(0, 1)
            jitter where asked), a concentrated body like the indexer scores the
            LiteTopK review describes (most scores in a narrow band, few far
            above it);
  * tail  : each entry independently, with probability 0.002, is replaced by
            mu_r + Exponential(mean 6);
  * suffix: columns at or beyond a row's valid length hold -inf;
  * causal ragged lengths: the last 8192 rows of a causal window at width
    N_alloc, row j of the window has length N_alloc - 8192 + j + 1, cut into
    non-overlapping groups of M rows (codexqa.cn, section "20 个形状都最快").

Generation uses torch's seeded generators on whichever device is asked for.
Values drawn on the CPU and on a GPU differ for the same seed; every
comparison therefore copies the one tensor both sides read.
"""
from typing import Optional

import torch

CAUSAL_WINDOW = 8192
BODY_MEAN = 30.0
BODY_STD = 2.5
TAIL_PROB = 0.002
TAIL_MEAN = 6.0


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def causal_lens(N_alloc: int, M: int, group: int = 0, window: int = CAUSAL_WINDOW) -> torch.Tensor:
    """Valid lengths of group `group` of M rows from the last `window` causal rows."""
    if window % M != 0 or not (0 <= group < window // M):
        raise ValueError("groups of M rows must tile the causal window")
    j = torch.arange(group * M, (group + 1) * M, dtype=torch.int64)
    lens = N_alloc - window + j + 1
    return lens.clamp(min=0, max=N_alloc).to(torch.int32)


def tiny_lens(seed: int, M: int = 8, N_alloc: int = 16384, lo: int = 512,
              K: int = 2048, n_short: int = 2) -> torch.Tensor:
    """Lengths uniform in [lo, N_alloc], with the first n_short rows forced <= K."""
    g = _gen("cpu", seed)
    lens = torch.randint(lo, N_alloc + 1, (M,), generator=g, dtype=torch.int64)
    short = torch.randint(lo, K + 1, (n_short,), generator=g, dtype=torch.int64)
    lens[:n_short] = short
    return lens.to(torch.int32)


def _mask_suffix(x: torch.Tensor, lens: torch.Tensor) -> None:
    cols = torch.arange(x.shape[1], device=x.device)
    x.masked_fill_(cols[None, :] >= lens.to(x.device, torch.int64)[:, None], float("-inf"))


def indexer_rows(lens: torch.Tensor, N_alloc: int, seed: int, device="cpu",
                 jitter: bool = True, out: Optional[torch.Tensor] = None,
                 row_chunk: int = 256) -> torch.Tensor:
    """[M, N_alloc] float32: concentrated body + sparse exponential upper tail."""
    M = int(lens.numel())
    if out is None:
        out = torch.empty((M, N_alloc), dtype=torch.float32, device=device)
    for c0 in range(0, M, row_chunk):
        c1 = min(M, c0 + row_chunk)
        g = _gen(out.device, seed * 1_000_003 + c0)
        n = c1 - c0
        mu = torch.full((n, 1), BODY_MEAN, dtype=torch.float32, device=out.device)
        if jitter:
            mu += torch.randn((n, 1), generator=g, device=out.device)
        blk = out[c0:c1]
        torch.randn((n, N_alloc), generator=g, device=out.device, out=blk)
        blk.mul_(BODY_STD).add_(mu)
        tail = torch.rand((n, N_alloc), generator=g, device=out.device) < TAIL_PROB
        ex = torch.empty((n, N_alloc), dtype=torch.float32, device=out.device)
        ex.exponential_(1.0 / TAIL_MEAN, generator=g)
        ex.add_(mu)
        blk.copy_(torch.where(tail, ex, blk))
        del tail, ex
        _mask_suffix(blk, lens[c0:c1])
    return out


TRACE_ROW = 65536


def trace_scores(n_floats: int, seed: int, device="cpu") -> torch.Tensor:
    """A flat float32 buffer of n_floats indexer-like scores for a trace
    replay: full-length rows of TRACE_ROW scores laid end to end (the body and
    tail of indexer_rows), which each Top-K call of the trace views as its own
    [rows, width] score matrix (n_floats a multiple of TRACE_ROW)."""
    if n_floats % TRACE_ROW:
        raise ValueError("n_floats must be a multiple of %d" % TRACE_ROW)
    rows = n_floats // TRACE_ROW
    buf = torch.empty(n_floats, dtype=torch.float32, device=device)
    indexer_rows(torch.full((rows,), TRACE_ROW, dtype=torch.int32), TRACE_ROW, seed=seed,
                 out=buf.view(rows, TRACE_ROW))
    return buf


def uniform_rows(lens: torch.Tensor, N_alloc: int, seed: int, device="cpu") -> torch.Tensor:
    """[M, N_alloc] float32, flat Uniform(0, 1) body with no tail, -inf suffix."""
    M = int(lens.numel())
    g = _gen(device, seed)
    x = torch.rand((M, N_alloc), generator=g, device=device, dtype=torch.float32)
    _mask_suffix(x, lens)
    return x


def to_bf16_grid(x: torch.Tensor) -> torch.Tensor:
    """Round every finite value to the bfloat16 grid (round to nearest even).

    Many scores then share a value, so the K-th and (K+1)-th largest scores of
    a row are often equal (ties at the boundary).
    """
    return x.to(torch.bfloat16).to(torch.float32)


def strided_high_rows(lens: torch.Tensor, N_alloc: int, seed: int, stride: int,
                      n_top: int, n_mid: int, on_grid: bool = True, device="cpu") -> torch.Tensor:
    """Rows whose large values sit on (or off) the positions 0, stride, 2*stride, ...

    on_grid=True (underfilling proposals): every position i*stride < len gets a
    value in [100, 101); `n_top` of those grid positions, picked at random, are
    lifted to [300, 301).  `n_mid` positions off the grid get values in
    [200, 201).  All other positions hold Uniform(0, 1).  A row sample taken on
    that grid then sees the [300, 301) and [100, 101) bands but never the
    [200, 201) band.

    on_grid=False (overfilling proposals): the grid positions hold
    Uniform(0, 1) like the body, and `n_mid` off-grid positions get values in
    [200, 201), which a sample on the grid never sees.
    """
    M = int(lens.numel())
    g = _gen("cpu", seed)
    x = torch.rand((M, N_alloc), generator=g, dtype=torch.float32)
    for r in range(M):
        L = int(lens[r])
        if L <= 0:
            continue
        grid = torch.arange(0, L, stride, dtype=torch.int64)
        off = torch.ones(L, dtype=torch.bool)
        off[grid] = False
        off_pos = torch.nonzero(off).flatten()
        if on_grid:
            x[r, grid] = 100.0 + torch.rand(grid.numel(), generator=g)
            pick = grid[torch.randperm(grid.numel(), generator=g)[:n_top]]
            x[r, pick] = 300.0 + torch.rand(pick.numel(), generator=g)
        mid = off_pos[torch.randperm(off_pos.numel(), generator=g)[:n_mid]]
        x[r, mid] = 200.0 + torch.rand(mid.numel(), generator=g)
    _mask_suffix(x, lens)
    return x.to(device)


def constant_rows(lens: torch.Tensor, N_alloc: int, value: float = 1.0, device="cpu") -> torch.Tensor:
    """Every valid score equal: any K valid indices are a correct answer."""
    M = int(lens.numel())
    x = torch.full((M, N_alloc), float(value), dtype=torch.float32, device=device)
    _mask_suffix(x, lens)
    return x


def index_inputs(T: int, S: int, seed: int, H: int = 64, D: int = 128, device="cpu"):
    """Inputs of the indexer-score stage: q [T, H, D] bfloat16 ~ N(0, 1/128),
    k [S, D] bfloat16 ~ N(0, 1), w [T, H] float32 ~ U(0, 1/8), and the causal
    valid lengths len_t = S - T + t + 1 (int32 [T], clamped to [1, S])."""
    g = _gen(device, seed)
    q = (torch.randn((T, H, D), generator=g, device=device) * (1.0 / 128.0) ** 0.5).to(torch.bfloat16)
    k = torch.randn((S, D), generator=g, device=device).to(torch.bfloat16)
    w = torch.rand((T, H), generator=g, device=device) * 0.125
    lens = (torch.arange(T, dtype=torch.int64) + (S - T + 1)).clamp(1, S).to(torch.int32)
    return q, k, w, lens


def bf16_bits(x: torch.Tensor):
    """Raw 16-bit patterns of a bfloat16 tensor as a numpy uint16 array."""
    import numpy as np
    return x.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

