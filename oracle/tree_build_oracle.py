"""Oracle of the draft-tree builder (topKSpec / topHead), one level at a time.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: imported by
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg;
it shares no code with the CUDA library.

Source (page title, section):
  [TREE] "投机推理：小模型搭树，大模型一次验证", 树形投机怎么配置 and the three
         steps after it (第一步 / 第二步 / 第三步), and 一个真实例子：从 dump
         看三轮投机: the draft model runs once per level; level i takes
         topHead[i] parents (the root alone at level 0, afterwards the nodes
         of the previous level with the highest path probability) and gives
         each parent j the top topKSpec[i][j] tokens of its draft logits as
         children; nodes are numbered level by level (A1..A6, B11, B12, B21,
         B22, C111, C211).

Readings (listed with the other readings in the design notes): the top
tokens of a row are ranked by raw logit, ties to the lower token id; the path
probability of a node is the product of the draft's softmax (temperature 1)
along its path, compared as a sum of log-probabilities, ties to the lower
node id; the chosen parents are expanded, and get their logits rows, in
node-id order; a row holding a NaN or with no finite maximum gives no
distribution and flags the request.

The level call has the shape of one draft forward: the rows of level i are
the draft logits at that level's parents, in node-id order.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

FLAG_BAD_INPUT = 1
FLAG_BAD_ROW = 4
SELECT_MARGIN = 5e-5   # a selection whose last kept and first dropped path
                       # log-probabilities are closer than this (but not tied
                       # siblings, which compare equal in any precision) is a
                       # boundary case


@dataclass
class Level:
    node_token: List[int] = field(default_factory=list)    # the new nodes, in id order
    node_parent: List[int] = field(default_factory=list)
    node_logp: List[float] = field(default_factory=list)   # path log-probability
    next_parents: List[int] = field(default_factory=list)  # ids expanded next, ascending
    boundary: bool = False
    flags: int = 0


def top_tokens(row: np.ndarray, k: int) -> List[int]:
    """The k largest logits of a row, larger first, ties to the lower id."""
    order = np.lexsort((np.arange(len(row)), -np.asarray(row, np.float64)))
    return [int(t) for t in order[:k]]


def log_softmax(row: np.ndarray) -> np.ndarray:
    x = np.asarray(row, np.float64)
    m = x.max()
    return x - m - np.log(np.exp(x - m).sum())


def row_is_bad(row: np.ndarray) -> bool:
    x = np.asarray(row, np.float64)
    return bool(np.isnan(x).any() or not np.isfinite(x.max()))


def expand_level(rows: np.ndarray, parents: Sequence[int], parent_logp: Sequence[float],
                 ks: Sequence[int], n_before: int, n_next: int) -> Level:
    """One level of the tree for one request.

    rows[j]: the draft logits at parent j (parents in id order); ks[j]: its
    number of children.  The children get ids n_before+1 .. in parent order,
    then in rank order.  The n_next children with the highest path
    log-probability are the next level's parents, returned in id order."""
    out = Level()
    if any(row_is_bad(r) for r in rows):
        out.flags = FLAG_BAD_ROW
        return out
    for j, (p, k) in enumerate(zip(parents, ks)):
        lq = log_softmax(rows[j])
        for t in top_tokens(rows[j], k):
            out.node_token.append(t)
            out.node_parent.append(int(p))
            out.node_logp.append(float(parent_logp[j]) + float(lq[t]))
    n = len(out.node_token)
    ids = [n_before + 1 + i for i in range(n)]
    ranked = sorted(range(n), key=lambda i: (-out.node_logp[i], ids[i]))
    chosen = ranked[:n_next]
    out.next_parents = sorted(ids[i] for i in chosen)
    if 0 < n_next < n:
        a, b = ranked[n_next - 1], ranked[n_next]
        gap = out.node_logp[a] - out.node_logp[b]
        siblings_tied = gap == 0 and out.node_parent[a] == out.node_parent[b]
        out.boundary = bool(gap < SELECT_MARGIN) and not siblings_tied
    return out


@dataclass
class Tree:
    node_token: np.ndarray   # int32 [N]: node 1..N
    node_parent: np.ndarray  # int32 [N]
    node_logp: np.ndarray    # float64 [N+1]: node 0 (the root) .. N
    row_of_node: np.ndarray  # int32 [N+1], -1 = not expanded
    boundary: bool
    flags: int


def build_tree(level_rows: Sequence[np.ndarray], topKSpec, topHead) -> Tree:
    """The whole tree of one request.  level_rows[i][j] are the draft logits
    at the j-th parent (in id order) of level i, as the draft model would
    produce them once those parents are known."""
    token: List[int] = []
    parent: List[int] = []
    logp: List[float] = [0.0]
    row_of: List[int] = [0]
    parents = [0]
    boundary = False
    n_rows = 1
    for i, ks in enumerate(topKSpec):
        n_next = int(topHead[i + 1]) if i + 1 < len(topHead) else 0
        lv = expand_level(np.asarray(level_rows[i]), parents, [logp[p] for p in parents], ks,
                          len(token), n_next)
        if lv.flags:
            return Tree(np.zeros(0, np.int32), np.zeros(0, np.int32), np.zeros(1), np.zeros(1, np.int32),
                        boundary, lv.flags)
        boundary |= lv.boundary
        token += lv.node_token
        parent += lv.node_parent
        logp += lv.node_logp
        row_of += [-1] * len(lv.node_token)
        for p in lv.next_parents:
            row_of[p] = n_rows
            n_rows += 1
        parents = lv.next_parents
    return Tree(np.asarray(token, np.int32), np.asarray(parent, np.int32), np.asarray(logp),
                np.asarray(row_of, np.int32), boundary, 0)
