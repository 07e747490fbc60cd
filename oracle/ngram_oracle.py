"""Oracle of the n-gram / prompt-lookup drafter.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: imported by
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg;
it shares no code with the CUDA library.

Sources (page title, section):
  [LLMI] "10.6 投机解码：为什么“先猜后验”能加速" §10.6.3 实际部署: model-free
         drafts take, from the prompt or the text generated so far, a segment
         equal to the current trailing n-gram and use the tokens that follow
         it as the draft; the framework entry bounds the n-gram between a
         minimum and a maximum length (prompt_lookup_min / prompt_lookup_max).
  [KV4]  "KV Cache 优化（四）：Speculative Decoding 投机解码" §10.2 N-gram 或前缀
         匹配: no extra network, continuous segments found in the prompt or the
         history.

Reading (the pages name no tie rule; each choice is listed in the design
notes): the longest n in [n_min, n_max] whose trailing n-gram occurs earlier
wins; among its occurrences the most recent (the largest start) is used; an
occurrence must start before the trailing n-gram itself; the draft is the up
to gamma tokens after the occurrence, never past the end of the history; no
occurrence gives an empty draft.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Sequence


@dataclass
class NgramDraft:
    tokens: List[int] = field(default_factory=list)  # the draft (at most gamma tokens)
    n: int = 0        # the matched n-gram length (0: no match)
    start: int = -1   # start of the occurrence used (-1: no match)


def ngram_draft(history: Sequence[int], n_min: int, n_max: int, gamma: int) -> NgramDraft:
    """Prompt-lookup draft for one request, by the reading above, as plain
    loops: for n from n_max down to n_min, compare the trailing n-gram with
    every earlier window from the latest start backwards; the first hit is the
    answer."""
    h = [int(x) for x in history]
    L = len(h)
    for n in range(min(n_max, L - 1), max(n_min, 1) - 1, -1):
        suffix = h[L - n:]
        for j in range(L - n - 1, -1, -1):
            if h[j:j + n] == suffix:
                first = j + n
                return NgramDraft(h[first:first + gamma], n, j)
    return NgramDraft()
