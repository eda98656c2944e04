"""Host side of the per-CTA timeline diagnostic (no GPU).

The record layout is the one the -DTOPK_PHASE_TIMING build writes: per CTA
slot 0 its start, slot 1 its exit, then five slots per row (row + 1, claim,
pass start, pass end, close; the pass slots stay 0 for a row served without
sampling).  The summary must count rows per CTA, skip unsampled rows in the
pass figures and measure every time from the first CTA's start.
"""
from exact_top_sparse_gb300 import phases

SLOTS = 2 + 5 * 4


def record(start, exit_, rows):
    r = [0] * SLOTS
    r[0], r[1] = start, exit_
    for j, (row, claim, p0, p1, close) in enumerate(rows):
        r[2 + 5 * j:7 + 5 * j] = [row + 1, claim, p0, p1, close]
    return r


def test_timeline_summary_counts_and_spreads():
    t0 = 10_000_000
    us = 1000
    recs = [
        # two sampled rows
        record(t0, t0 + 80 * us, [(0, t0 + 1 * us, t0 + 10 * us, t0 + 35 * us, t0 + 40 * us),
                                  (4, t0 + 41 * us, t0 + 42 * us, t0 + 70 * us, t0 + 80 * us)]),
        # one sampled row, started 1 us later
        record(t0 + us, t0 + 45 * us, [(1, t0 + 2 * us, t0 + 11 * us, t0 + 36 * us,
                                        t0 + 44 * us)]),
        # one row served without sampling (no pass stamps)
        record(t0 + us, t0 + 5 * us, [(2, t0 + 2 * us, 0, 0, t0 + 4 * us)]),
        # a CTA that never started (grid larger than the CTAs that wrote): ignored
        [0] * SLOTS,
    ]
    flat = [v for r in recs for v in r]
    s = phases.timeline_summary("8x4", flat, len(recs), SLOTS)
    assert s["timeline_ctas"] == 3
    assert s["ctas_by_rows"] == {"1": 2, "2": 1}
    assert s["start_us"] == [0.0, 1.0, 1.0, 1.0]
    assert s["exit_us"] == [5.0, 45.0, 80.0, 80.0]
    r0 = s["row0"]
    assert r0["ctas"] == 3
    assert r0["claim_us"] == [1.0, 2.0, 2.0, 2.0]
    # the unsampled row has no pass: only the two sampled first rows count
    assert r0["before_pass_us"] == [9.0, 9.0, 9.0, 9.0]
    assert r0["pass_us"] == [25.0, 25.0, 25.0, 25.0]
    assert r0["after_pass_us"] == [5.0, 8.0, 8.0, 8.0]
    r1 = s["row1"]
    assert r1["ctas"] == 1
    assert r1["pass_us"] == [28.0, 28.0, 28.0, 28.0]
    assert "row2" not in s


def test_timeline_summary_without_persistent_launch():
    # a call planned as direct or KV-split leaves every record empty
    s = phases.timeline_summary("1048576x512", [0] * (3 * SLOTS), 3, SLOTS)
    assert s == {"shape": "1048576x512", "timeline_ctas": 0}
