"""Synthetic serving traces of the score -> select chain (host logic only).

The pages describe the traces they replay (codexqa.cn, section "框架轨迹"):
prefill is cut into scheduler steps of at most 64K query tokens, and the
indexer cuts each step again so that the materialised FP32 score matrix stays
in a fixed workspace; the rows per call therefore fall roughly as 1/width.
A 245K-token request gives 4 steps and 26 Top-K calls, a 430K-token request
7 steps and 71 calls.

Reading used here (the pages print only the counts): K-suffixed sizes are
binary (245K = 250,880 tokens, 430K = 440,320, a step = 65,536 query
tokens); the workspace holds W = 1.5 * 2^30 FP32 scores; step i covers query
positions [65536 i, min(65536 (i+1), L)) and its calls use the allocated
width of the step's last position; rows per call = floor(W / width), rounded
down to a multiple of 4 (the score kernel's query block), the last call of a
step taking the rest.  Query position p sees keys 0..p (valid length p + 1).
This reproduces both printed call counts.
"""
from dataclasses import dataclass
from typing import List

STEP_TOKENS = 65536
WORKSPACE_FLOATS = 3 * (1 << 29)   # 1.5 * 2^30
QUERY_BLOCK = 4


@dataclass(frozen=True)
class Call:
    step: int
    row0: int      # first query position of the call
    rows: int
    width: int     # allocated width (row stride) of the call's score rows

    def lens(self):
        """Valid length of each row (causal: position + 1)."""
        return [self.row0 + j + 1 for j in range(self.rows)]


def calls(context_tokens: int, step_tokens: int = STEP_TOKENS,
          workspace_floats: int = WORKSPACE_FLOATS, block: int = QUERY_BLOCK) -> List[Call]:
    """The Top-K calls of one prefill of `context_tokens` tokens, in order."""
    if context_tokens <= 0 or step_tokens <= 0 or workspace_floats <= 0 or block <= 0:
        raise ValueError("sizes must be positive")
    out = []
    step = 0
    for s0 in range(0, context_tokens, step_tokens):
        s1 = min(s0 + step_tokens, context_tokens)
        width = s1
        per_call = (workspace_floats // width) // block * block
        if per_call <= 0:
            raise ValueError("workspace smaller than one query block at width %d" % width)
        for r0 in range(s0, s1, per_call):
            out.append(Call(step, r0, min(per_call, s1 - r0), width))
        step += 1
    return out
