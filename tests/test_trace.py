"""The synthetic serving traces reproduce the call counts the pages print
(codexqa.cn, section "框架轨迹": a 245K-token request -> 4 scheduler steps and
26 Top-K calls; 430K -> 7 steps and 71 calls), and every call respects the
workspace, the causal lengths and the score kernel's query block."""
import pytest

from exact_top_sparse_gb300 import trace


@pytest.mark.parametrize("tokens,steps,n_calls", [(245 * 1024, 4, 26), (430 * 1024, 7, 71)])
def test_printed_call_counts(tokens, steps, n_calls):
    cs = trace.calls(tokens)
    assert len(cs) == n_calls
    assert len({c.step for c in cs}) == steps


@pytest.mark.parametrize("tokens", [245 * 1024, 430 * 1024, 100000, 65536, 1])
def test_calls_cover_every_query_once(tokens):
    cs = trace.calls(tokens)
    pos = 0
    for c in cs:
        assert c.row0 == pos and c.rows > 0
        assert c.rows * c.width <= trace.WORKSPACE_FLOATS
        assert max(c.lens()) <= c.width and min(c.lens()) == c.row0 + 1
        pos += c.rows
    assert pos == tokens
    # every call but the last of its step has a whole number of query blocks
    for a, b in zip(cs, cs[1:]):
        if a.step == b.step:
            assert a.rows % trace.QUERY_BLOCK == 0


def test_rows_fall_as_width_grows():
    cs = trace.calls(430 * 1024)
    per_step = {}
    for c in cs:
        per_step.setdefault(c.step, c.rows)
    rows = [per_step[s] for s in sorted(per_step)]
    assert rows == sorted(rows, reverse=True)
    assert rows[0] == 24576 and rows[1] == 12288   # W / 65536 and W / 131072
