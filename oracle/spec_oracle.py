"""Plain fp64 CPU oracle for the speculative-decoding verify-and-commit step.

TEST INFRASTRUCTURE ONLY.  This module is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by ``bench.py``'s CPU-baseline / reference
leg, and by nothing else.  It shares no code with the CUDA library and does
not import it; the product path never calls it.

Everything is computed in float64 with numpy, one request at a time, in the
order the pages state the method.  No step is blocked, fused or reordered.

Sources (page title, section):
  [KV4]  "KV Cache 优化（四）：Speculative Decoding 投机解码"
         §4 接受和拒绝 (acceptance, residual, temperature/top-k, greedy),
         §5 一个完整例子 (bonus token), §6 KV Cache 如何配合 (commit / rollback)
  [LLMI] "10.6 投机解码：为什么“先猜后验”能加速"
         §10.6.1 无损性保证 (one round; losslessness; three-token example;
         greedy special case), §10.6.3 实际部署 (verify shape, cache
         truncation, Table 10-17 tree mask, depth positions)
  [GLOS] "投机解码" glossary, 精确接受与校正分布 (q = 0 and residual-mass
         boundary cases)
  [TREE] "投机推理：小模型搭树，大模型一次验证", sections Validation and
         接受过程：沿一条路径走 (single-path walk)

Readings where the pages leave a step open (each is listed in the design
notes): top-k selects on raw logits and keeps every tie of the k-th value;
the same transform is applied to target and draft rows; a draft token is
accepted iff u < a; a = 1 if q(d) = 0 < p(d), a = 0 if both are 0; when the
residual mass is <= eps the resample draws from the target row itself;
sampling is by inverse CDF in token-index order with a strict ">"; one
uniform per accept test plus one final uniform shared by the resample and the
bonus draw; a tree node with no logits row ends the walk with no extra token;
a tree path that breaks emits the target's argmax at the stop node.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against values the pages print, closed forms, invariants and brute force.
Readings that no page fixes (top-k tie rule, eps, "<" vs "<=", tree bonus
availability) are pinned only as readings ("parity unpinned" for the choice
itself, not for the arithmetic).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

BOUNDARY_MARGIN = 1e-5   # a uniform this close to an acceptance threshold is a boundary case
DRAW_MARGIN_REL = 3e-11  # a draw whose target u*C_total lies within
DRAW_MARGIN_ABS = 1e-12  #   REL*C_total + ABS of its token's CDF interval ends is a boundary case
DEFAULT_EPS = 1e-6       # residual-mass threshold below which the fallback is used
EPS_BAND = 0.5           # a residual mass within EPS_BAND * eps of eps is a boundary case

FLAG_BAD_INPUT = 1       # a token, parent or row index out of range: request skipped
FLAG_FALLBACK = 2        # the residual-mass fallback was used
FLAG_BAD_ROW = 4         # a row whose kept logits are all -inf (no distribution)
FLAG_EOS = 16            # the round's output was cut after an end-of-sequence token
FLAG_LIMIT = 32          # the round's output was cut at the request's remaining length


# ---------------------------------------------------------------------------
# (a1) row transform: temperature + top-k, then softmax          [KV4 §4]
# ---------------------------------------------------------------------------
def kept_set(logits: np.ndarray, top_k: int) -> np.ndarray:
    """Boolean mask of the tokens top-k keeps.

    The threshold is the k-th largest raw logit counted with multiplicity;
    every token whose logit is >= that value is kept, so ties at the
    threshold can make the kept set larger than k.  top_k <= 0 or >= V keeps
    every token.  (Reading: selection on raw logits; a positive temperature
    does not change the order.)
    """
    x = np.asarray(logits, dtype=np.float64)
    V = x.shape[0]
    if top_k <= 0 or top_k >= V:
        return np.ones(V, dtype=bool)
    theta = np.sort(x)[::-1][top_k - 1]
    return x >= theta


def kept_set_top_p(probs: np.ndarray, top_p: float) -> np.ndarray:
    """Boolean mask of the tokens top-p (nucleus) keeps from a distribution.

    KV4 §4 names top-p among the transforms whose result enters the
    acceptance rule; no page defines it further.  Reading: the smallest set
    of the most probable tokens whose total probability reaches top_p, with
    every token tied with the least probable kept one also kept (the same
    tie rule as top-k).  top_p >= 1 keeps every token.
    """
    p = np.asarray(probs, dtype=np.float64)
    if top_p >= 1.0:
        return np.ones(p.shape[0], dtype=bool)
    order = np.argsort(-p, kind="stable")
    mass = 0.0
    last = p[order[0]]
    for i in order:
        mass += p[i]
        last = p[i]
        if mass >= top_p:
            break
    return p >= last


def transform_probs(logits: np.ndarray, temperature: float, top_k: int,
                    top_p: float = 1.0) -> Optional[np.ndarray]:
    """p_i = exp((l_i - m)/T) / sum_{j kept} exp((l_j - m)/T) for kept i, else 0.

    m is the largest kept logit.  With top_p < 1 the result is then cut to
    its nucleus (kept_set_top_p) and renormalised (reading: temperature, then
    top-k, then top-p).  Returns None when every kept logit is -inf (the row
    defines no distribution).
    """
    x = np.asarray(logits, dtype=np.float64)
    keep = kept_set(x, top_k)
    m = x[keep].max()
    if not np.isfinite(m):
        return None
    e = np.zeros_like(x)
    e[keep] = np.exp((x[keep] - m) / temperature)
    p = e / e.sum()
    if top_p < 1.0:
        p = np.where(kept_set_top_p(p, top_p), p, 0.0)
        p = p / p.sum()
    return p


def greedy_argmax(logits: np.ndarray) -> int:
    """Index of the largest logit; the lowest index wins a tie."""
    x = np.asarray(logits, dtype=np.float64)
    return int(np.flatnonzero(x == x.max())[0])


# ---------------------------------------------------------------------------
# (a2) acceptance test                                   [KV4 §4, LLMI §10.6.1]
# ---------------------------------------------------------------------------
def acceptance_probability(p_d: float, q_d: float) -> float:
    """a = min(1, p(d)/q(d)); where q(d) = 0 the ratio's limit is used:
    1 if p(d) > 0, else 0 ([GLOS]: the ratio only matters where q > 0)."""
    if q_d > 0.0:
        return min(1.0, p_d / q_d)
    return 1.0 if p_d > 0.0 else 0.0


# ---------------------------------------------------------------------------
# (a3, a4) inverse-CDF draw from unnormalised weights
# ---------------------------------------------------------------------------
@dataclass
class Draw:
    token: int
    near_boundary: bool


def inverse_cdf(weights: np.ndarray, u: float, margin_rel: float = DRAW_MARGIN_REL,
                margin_abs: float = DRAW_MARGIN_ABS) -> Draw:
    """The smallest i with C_i > u * C_total, C_i = sum_{j <= i} w_j in index
    order.  Zero-weight tokens can never be chosen.  If rounding leaves no
    such i, the largest i with w_i > 0 is taken.  ``near_boundary`` is set
    when u * C_total lies within margin_rel * C_total + margin_abs of either
    end of the chosen token's CDF interval."""
    w = np.asarray(weights, dtype=np.float64)
    C = np.cumsum(w)
    total = C[-1]
    t = u * total
    hit = np.flatnonzero(C > t)
    if hit.size:
        i = int(hit[0])
    else:
        i = int(np.flatnonzero(w > 0)[-1])
    lo = C[i - 1] if i > 0 else 0.0
    hi = C[i]
    m = margin_rel * total + margin_abs
    near = (t - lo) < m or (hi - t) < m
    return Draw(i, bool(near))


# ---------------------------------------------------------------------------
# one chain round, sampled                                   [LLMI §10.6.1]
# ---------------------------------------------------------------------------
@dataclass
class ChainResult:
    n_acc: int = 0
    tokens: List[int] = field(default_factory=list)   # n_acc accepted drafts + 1 drawn
    accept_prob: Optional[np.ndarray] = None           # a_k, k = 1..gamma
    residual_mass: Optional[np.ndarray] = None         # Z_k = sum max(0, p_k - q_k)
    flags: int = 0
    boundary: bool = False                             # a decision within the margin

    @property
    def n_out(self) -> int:
        return len(self.tokens)


def verify_chain_sampled(target: np.ndarray, draft: np.ndarray, draft_tokens: np.ndarray,
                         uniforms: np.ndarray, temperature: float, top_k: int = 0,
                         eps: float = DEFAULT_EPS, margin: float = BOUNDARY_MARGIN,
                         top_p: float = 1.0) -> ChainResult:
    """One speculative-sampling round of one request (top_p < 1: the nucleus
    transform too, on both sides, as KV4 §4 asks of every processed
    distribution).

    target: [gamma+1, V] logits (p_1..p_{gamma+1}); draft: [gamma, V] logits
    (q_1..q_gamma); draft_tokens: d_1..d_gamma; uniforms: u[0..gamma-1] for the
    accept tests and u[gamma] for the one final draw (resample or bonus).

    Steps ([LLMI §10.6.1] round, [KV4 §4]): transform each row; test d_k left
    to right with probability min(1, p_k(d_k)/q_k(d_k)); at the first
    rejection draw from norm(max(0, p_k - q_k)) (from p_k itself when that
    mass is <= eps, [GLOS] stable fallback) and drop the later drafts; if
    every draft is accepted draw a bonus token from p_{gamma+1} ([KV4 §5]).
    a_k and Z_k are reported for every k as diagnostics.
    """
    target = np.asarray(target, dtype=np.float64)
    draft = np.asarray(draft, dtype=np.float64).reshape(-1, target.shape[1])
    gamma = draft.shape[0]
    V = target.shape[1]
    d = [int(x) for x in np.asarray(draft_tokens).reshape(-1)[:gamma]]
    u = np.asarray(uniforms, dtype=np.float64).reshape(-1)
    res = ChainResult()
    if any(t < 0 or t >= V for t in d):
        res.flags |= FLAG_BAD_INPUT
        return res
    P = [transform_probs(target[k], temperature, top_k, top_p) for k in range(gamma + 1)]
    Q = [transform_probs(draft[k], temperature, top_k, top_p) for k in range(gamma)]
    if any(x is None for x in P) or any(x is None for x in Q):
        res.flags |= FLAG_BAD_ROW
        return res

    a = np.array([acceptance_probability(P[k][d[k]], Q[k][d[k]]) for k in range(gamma)])
    Z = np.array([np.maximum(P[k] - Q[k], 0.0).sum() for k in range(gamma)])
    res.accept_prob, res.residual_mass = a, Z

    n_acc = gamma
    for k in range(gamma):
        if abs(u[k] - a[k]) < margin:
            res.boundary = True
        if not (u[k] < a[k]):
            n_acc = k
            break
    u_final = u[gamma]
    if n_acc < gamma:
        w = np.maximum(P[n_acc] - Q[n_acc], 0.0)
        mass = w.sum()
        if abs(mass - eps) <= EPS_BAND * eps:
            res.boundary = True
        if mass <= eps:
            w = P[n_acc]
            res.flags |= FLAG_FALLBACK
        draw = inverse_cdf(w, u_final)
    else:
        draw = inverse_cdf(P[gamma], u_final)
    res.boundary |= draw.near_boundary
    res.n_acc = n_acc
    res.tokens = d[:n_acc] + [draw.token]
    return res


# ---------------------------------------------------------------------------
# (a5) greedy chain                               [KV4 §4, LLMI §10.6.1]
# ---------------------------------------------------------------------------
def verify_chain_greedy(target: np.ndarray, draft_tokens: np.ndarray) -> ChainResult:
    """Temperature 0: d_k is accepted iff it equals the argmax of p_k; at the
    first mismatch the argmax is emitted; if every draft matches, the argmax
    of p_{gamma+1} is emitted."""
    target = np.asarray(target, dtype=np.float64)
    V = target.shape[1]
    gamma = target.shape[0] - 1
    d = [int(x) for x in np.asarray(draft_tokens).reshape(-1)[:gamma]]
    res = ChainResult()
    if any(t < 0 or t >= V for t in d):
        res.flags |= FLAG_BAD_INPUT
        return res
    g = [greedy_argmax(target[k]) for k in range(gamma + 1)]
    n_acc = gamma
    for k in range(gamma):
        if d[k] != g[k]:
            n_acc = k
            break
    res.n_acc = n_acc
    res.tokens = d[:n_acc] + [g[n_acc]]
    return res


# ---------------------------------------------------------------------------
# (a6, a7) tree: single-path greedy walk, mask, positions     [TREE, LLMI]
# ---------------------------------------------------------------------------
@dataclass
class TreeResult:
    path: List[int] = field(default_factory=list)        # accepted node ids, root excluded
    tokens: List[int] = field(default_factory=list)      # their tokens + the extra token, if any
    commit_slots: List[int] = field(default_factory=list)  # [0] + path
    mask: Optional[np.ndarray] = None                    # uint32 [N+1, W]
    pos: Optional[np.ndarray] = None                     # int64 [N+1]
    flags: int = 0

    @property
    def n_acc(self) -> int:
        return len(self.path)

    @property
    def n_out(self) -> int:
        return len(self.tokens)


def tree_mask_positions(node_parent: np.ndarray, committed_len: int):
    """Attention mask and position ids of a draft tree (root = node 0).

    Bit j of row i is set iff node j is node i or one of its ancestors, so a
    node sees only its own path ([LLMI §10.6.3], Table 10-17).  A node's
    position is committed_len + its depth (root depth 0), not its row index.
    Word w of a row holds nodes 32w .. 32w+31.
    """
    par = [int(x) for x in np.asarray(node_parent).reshape(-1)]
    n = len(par) + 1
    W = (n + 31) // 32
    anc = [{0}]
    depth = [0]
    for i in range(1, n):
        p = par[i - 1]
        anc.append(anc[p] | {i})
        depth.append(depth[p] + 1)
    mask = np.zeros((n, W), dtype=np.uint32)
    for i in range(n):
        for j in anc[i]:
            mask[i, j // 32] |= np.uint32(1 << (j % 32))
    pos = committed_len + np.asarray(depth, dtype=np.int64)
    return mask, pos


def verify_tree(logits: np.ndarray, node_token: np.ndarray, node_parent: np.ndarray,
                row_of_node: np.ndarray, committed_len: int = 0) -> TreeResult:
    """Greedy tree verification ([TREE] Validation and single-path walk).

    Start at the root.  At node v with a logits row, take the target's argmax
    t of that row and move to the child of v whose token is t (the lowest
    node id if, in a malformed tree, several are); only v's own children are
    considered, so matches on other branches never count.  Stop when no child
    matches (t is then emitted as the next token) or when v has no logits row
    (no extra token).
    """
    logits = np.asarray(logits, dtype=np.float64)
    R, V = logits.shape
    tok = [int(x) for x in np.asarray(node_token).reshape(-1)]
    par = [int(x) for x in np.asarray(node_parent).reshape(-1)]
    rows = [int(x) for x in np.asarray(row_of_node).reshape(-1)]
    N = len(tok)
    res = TreeResult()
    bad = len(par) != N or len(rows) != N + 1
    bad = bad or any(not (0 <= tok[i] < V) for i in range(N))
    bad = bad or any(not (0 <= par[i] < i + 1) for i in range(N))
    bad = bad or any(not (-1 <= r < R) for r in rows)
    if bad:
        res.flags |= FLAG_BAD_INPUT
        return res
    res.mask, res.pos = tree_mask_positions(par, committed_len)
    v = 0
    extra = None
    while True:
        r = rows[v]
        if r < 0:
            break
        t = greedy_argmax(logits[r])
        child = next((c for c in range(1, N + 1) if par[c - 1] == v and tok[c - 1] == t), None)
        if child is None:
            extra = t
            break
        res.path.append(child)
        v = child
    res.tokens = [tok[c - 1] for c in res.path] + ([] if extra is None else [extra])
    res.commit_slots = [0] + res.path
    return res


def verify_chain_batch(target: np.ndarray, draft: np.ndarray, draft_tokens: np.ndarray,
                       uniforms: np.ndarray, gammas, temperatures, top_ks, top_ps=None):
    """A batch whose requests each have their own gamma, temperature, top-k
    and top-p ([LLMI §10.6.3]: requests in one batch accept different
    lengths and start the next step at different points; per-request
    sampling settings follow the same rule per request, [KV4 §4]).

    Layout reading: the arrays are padded to gamma_max = draft_tokens.shape[1]:
    target [B, gamma_max+1, V], draft [B, gamma_max, V], uniforms
    [B, gamma_max+1]; request b uses target rows 0..gamma_b, draft rows and
    tokens 0..gamma_b-1, accept uniforms u[b][0..gamma_b-1] and u[b][gamma_b]
    for its final draw.  Temperature 0 means greedy for that request.  Each
    request is one call of the single-request rule on its own slice."""
    out = []
    B = draft_tokens.shape[0]
    for b in range(B):
        g = int(gammas[b])
        T = float(temperatures[b])
        if T == 0.0:
            out.append(verify_chain_greedy(target[b, :g + 1], draft_tokens[b, :g]))
            continue
        u = np.concatenate([uniforms[b, :g], uniforms[b, g:g + 1]])
        tp = 1.0 if top_ps is None else float(top_ps[b])
        out.append(verify_chain_sampled(target[b, :g + 1], draft[b, :g], draft_tokens[b, :g], u, T,
                                        int(top_ks[b]), top_p=tp))
    return out


# ---------------------------------------------------------------------------
# round termination: EOS and the length limit                      [KV4 §5]
# ---------------------------------------------------------------------------
def truncate_round(r: ChainResult, eos: Optional[int] = None,
                   max_new: Optional[int] = None) -> ChainResult:
    """A round emits its accepted drafts and one drawn token, but an
    end-of-sequence token or the request's length limit ends it early
    ([KV4 §5]).  Reading: the emitted tokens are cut right after the first
    `eos` (the EOS itself is emitted), then to at most `max_new` tokens (a
    limit <= 0 emits nothing); n_acc counts the accepted drafts still
    emitted.  FLAG_EOS / FLAG_LIMIT say which cut shortened the round (an
    EOS that is the last token kept also sets FLAG_EOS).  A flagged (bad)
    round is returned unchanged."""
    if r.flags & (FLAG_BAD_INPUT | FLAG_BAD_ROW):
        return r
    tokens = list(r.tokens)
    flags = r.flags
    if eos is not None:
        for i, t in enumerate(tokens):
            if t == eos:
                tokens = tokens[:i + 1]
                flags |= FLAG_EOS
                break
    if max_new is not None and len(tokens) > max(max_new, 0):
        tokens = tokens[:max(max_new, 0)]
        flags |= FLAG_LIMIT
        if eos is not None and eos not in tokens:
            flags &= ~FLAG_EOS
    return ChainResult(n_acc=min(r.n_acc, len(tokens)), tokens=tokens, accept_prob=r.accept_prob,
                       residual_mass=r.residual_mass, flags=flags, boundary=r.boundary)


# ---------------------------------------------------------------------------
# (a8) KV commit + rollback                         [KV4 §6, LLMI §10.6.3]
# ---------------------------------------------------------------------------
def chain_commit_slots(n_acc: int) -> List[int]:
    """Slots a chain round commits: slot 0 holds the K/V of the last emitted
    token x (computed by this verify forward), slots 1..n_acc the accepted
    drafts.  The drawn (resampled or bonus) token has no K/V yet: it is the
    next round's x ([KV4 §6])."""
    return list(range(n_acc + 1))


def commit_kv(cache: np.ndarray, temp_kv: np.ndarray, block_table: np.ndarray,
              slots, n_slots: int, committed_len: int, block_size: int):
    """Commit one request's accepted temporary K/V into the paged cache.

    cache: [L, 2, num_blocks, block_size, H, D]; temp_kv: [L, 2, S, H, D] of
    this request; block_table: this request's row.  Slot ``slots[i]`` is
    written at position committed_len + i in every layer, K and V alike (one
    commit boundary for all layers), then the length pointer advances by
    n_slots.  Rejected slots are simply not copied (rollback = not advancing
    past them).  If any slot id, block index or block id is out of range the
    request is left untouched and (committed_len, FLAG_BAD_INPUT) is returned.
    Returns (new_len, flags).
    """
    L, two, nb, bs, H, D = cache.shape
    S = temp_kv.shape[2]
    table = [int(x) for x in np.asarray(block_table).reshape(-1)]
    sl = [int(x) for x in np.asarray(slots).reshape(-1)[:n_slots]]
    if n_slots < 0 or len(sl) != n_slots or bs != block_size:
        return committed_len, FLAG_BAD_INPUT
    dest = []
    for i in range(n_slots):
        pos = committed_len + i
        bi = pos // block_size
        if not (0 <= sl[i] < S) or bi >= len(table) or not (0 <= table[bi] < nb):
            return committed_len, FLAG_BAD_INPUT
        dest.append((table[bi], pos % block_size))
    for i, (blk, off) in enumerate(dest):
        for layer in range(L):
            for kv in range(2):
                cache[layer, kv, blk, off] = temp_kv[layer, kv, sl[i]]
    return committed_len + n_slots, 0


def blocks_in_use(length: int, block_size: int) -> int:
    """Blocks a request of this length occupies; blocks past it may be freed
    by the caller ([LLMI §10.6.3]: paged caches release the surplus)."""
    return -(-length // block_size)


@dataclass
class InPlaceCommit:
    committed_len: int
    draft_len: Optional[int]      # None: not tracked
    blocks_in_use: Optional[int]  # None: left as it was (a flagged request)
    flags: int


def commit_in_place(committed_len: int, n_out: int, gamma: int, block_size: int,
                    draft_len: Optional[int] = None, kv_capacity: int = 0) -> InPlaceCommit:
    """Commit of a chain round whose candidates' K/V the target forward
    already wrote in place, at positions committed_len .. committed_len+gamma
    ([KV4 §6]: reserved slots and a commit-length pointer, no copy;
    [LLMI §10.6.3]: those gamma+1 positions are in the cache before the
    verify, the length is cut back past a rejection, the draft model's cache
    rolls back with it).

    The kept positions are the last emitted token and the accepted drafts,
    i.e. the first n_out candidates; the length moves past them and the
    rejected ones stay beyond it.  The draft cache's length is cut back to the
    same boundary and never raised (reading: with every draft accepted the
    draft model has not yet run on the last one).  A request whose reserved
    positions do not fit (a negative length, or past kv_capacity > 0 or
    2^31-1) is flagged FLAG_BAD_INPUT and keeps every length."""
    end = committed_len + gamma + 1
    if committed_len < 0 or end > 2**31 - 1 or (kv_capacity > 0 and end > kv_capacity):
        return InPlaceCommit(committed_len, draft_len, None, FLAG_BAD_INPUT)
    new_len = committed_len + n_out
    dl = None if draft_len is None else min(draft_len, new_len)
    return InPlaceCommit(new_len, dl, blocks_in_use(new_len, block_size), 0)
