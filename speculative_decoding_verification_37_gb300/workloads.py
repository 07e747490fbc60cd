"""Seeded synthetic inputs for the speculative-decoding verify-and-commit step.

This module only draws random numbers and lays them out in the shapes the
verify step consumes.  It holds none of the verification arithmetic: no
transform-and-softmax of a row, no acceptance test, no residual, no sampling
rule of the verifier, no argmax walk over a tree and no KV commit.  What it
does implement is the *drafter* side, which the pages treat as an input to
the verifier:

* draft tokens of a chain are drawn from the (temperature / top-k restricted)
  draft distribution with the Gumbel-max trick ("KV Cache 优化（四）" §2: the
  draft model samples each candidate from q);
* a draft tree is grown from ``topKSpec`` / ``topHead`` by picking the
  highest-path-probability parents of each level and expanding each with its
  draft top-k ("投机推理：小模型搭树，大模型一次验证", sections on the tree
  configuration and the three draft steps).

Every request draws from its own PCG64 stream, seeded by
``SeedSequence([seed, kind, request])``, so any subset of requests can be
regenerated on the host without building the whole batch.  Normals are drawn
in float32; bf16 values are the float32 values rounded to nearest-even
(torch ``.to(torch.bfloat16)``); uniforms are ``integers(0, 2**24) * 2**-24``,
which are exact in float32 and float64 and lie in [0, 1).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np
import torch

# Stream kinds (second component of the seed sequence).
SEED_DRAFT_TOKENS = 0
SEED_UNIFORMS = 1
SEED_TARGET = 2
SEED_DRAFT_NOISE = 3
SEED_TEMP_KV = 4
SEED_BLOCK_PERM = 5
SEED_GREEDY = 6
SEED_EQUAL_ROWS = 7
SEED_GUMBEL = 8

KV_SENTINEL = 0x7F7F  # bf16 bit pattern the synthetic cache is filled with


def _rng(seed: int, kind: int, index: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, kind, index])))


def uniforms24(rng: np.random.Generator, shape) -> np.ndarray:
    """U[0,1) values on the 2**-24 grid: exact in float32 and float64."""
    return (rng.integers(0, 1 << 24, size=shape, dtype=np.int64).astype(np.float64)
            * (1.0 / (1 << 24))).astype(np.float32)


# --------------------------------------------------------------------------
# workload descriptions
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class KVSpec:
    """Paged KV cache geometry: one token's K and V for all layers."""
    layers: int = 32
    heads: int = 8
    head_dim: int = 128
    block_size: int = 16
    prefix: int = 2048

    @property
    def unit_bytes(self) -> int:
        """Bytes of one (layer, K|V) unit of one token (bf16)."""
        return self.heads * self.head_dim * 2

    @property
    def token_bytes(self) -> int:
        """Bytes of one token's K and V over every layer (bf16)."""
        return self.layers * 2 * self.unit_bytes


@dataclass(frozen=True)
class ChainSpec:
    name: str
    B: int
    gamma: int
    V: int
    dtype: str                      # "bf16" or "f32"
    target_sigma: float
    temperature: float              # 0 = greedy
    top_k: int = 0                  # 0 = off
    draft_sigma: Optional[float] = None   # draft = target + N(0, draft_sigma^2)
    zipf_bias: bool = False         # add -ln(1 + v) to token v's target logit
    greedy_match_p: float = 0.8     # greedy: P(draft token == target argmax)
    equal_rows_frac: float = 0.0    # fraction of requests whose draft == target
    kv: Optional[KVSpec] = None

    @property
    def greedy(self) -> bool:
        return self.temperature == 0.0

    @property
    def esize(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def logit_bytes(self) -> int:
        rows = self.B * (self.gamma + 1) + (0 if self.greedy else self.B * self.gamma)
        return rows * self.V * self.esize


@dataclass(frozen=True)
class TreeSpec:
    name: str
    B: int
    V: int
    topKSpec: Sequence[Sequence[int]]
    topHead: Sequence[int]
    target_sigma: float = 3.0
    draft_sigma: float = 1.0
    dtype: str = "bf16"
    kv: Optional[KVSpec] = None

    @property
    def n_nodes(self) -> int:
        return int(sum(sum(level) for level in self.topKSpec))

    @property
    def n_rows(self) -> int:
        return int(sum(self.topHead))

    @property
    def esize(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def logit_bytes(self) -> int:
        return self.B * self.n_rows * self.V * self.esize


# The five workloads the verify-and-commit step is specified on.
WORKLOADS = {
    1: ChainSpec("chain-tiny B=8 g=4 V=1024 f32 T=1", B=8, gamma=4, V=1024, dtype="f32",
                 target_sigma=2.0, draft_sigma=0.7, temperature=1.0),
    2: ChainSpec("chain B=64 g=4 V=128256 bf16 T=0.8 top-k=50 + KV commit", B=64, gamma=4,
                 V=128256, dtype="bf16", target_sigma=3.0, zipf_bias=True, draft_sigma=1.0,
                 temperature=0.8, top_k=50, kv=KVSpec(prefix=2048)),
    3: ChainSpec("greedy chain B=256 g=8 V=152064 bf16", B=256, gamma=8, V=152064,
                 dtype="bf16", target_sigma=3.0, temperature=0.0, greedy_match_p=0.8),
    4: TreeSpec("tree [[6],[2,2],[1,1]]/[1,2,2] B=128 V=128256 bf16 + KV commit", B=128,
                V=128256, topKSpec=((6,), (2, 2), (1, 1)), topHead=(1, 2, 2),
                kv=KVSpec(prefix=2048)),
    5: ChainSpec("chain B=512 g=7 V=128256 f32 T=1 + KV commit", B=512, gamma=7, V=128256,
                 dtype="f32", target_sigma=3.0, draft_sigma=1.5, temperature=1.0,
                 equal_rows_frac=0.01, kv=KVSpec(prefix=4096)),
}


# --------------------------------------------------------------------------
# chain batches
# --------------------------------------------------------------------------
@dataclass
class ChainBatch:
    spec: ChainSpec
    requests: np.ndarray            # request ids held in this batch
    target: torch.Tensor            # [n*(gamma+1), V] bf16 or f32, CPU
    draft: Optional[torch.Tensor]   # [n*gamma, V] or None (greedy)
    draft_tokens: np.ndarray        # int32 [n, gamma]
    uniforms: Optional[np.ndarray]  # float32 [n, gamma+1] or None (greedy)
    equal_rows: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int64))

    @property
    def n(self) -> int:
        return len(self.requests)

    def target_f64(self, i: int) -> np.ndarray:
        g = self.spec.gamma
        return self.target[i * (g + 1):(i + 1) * (g + 1)].to(torch.float64).numpy()

    def draft_f64(self, i: int) -> np.ndarray:
        g = self.spec.gamma
        return self.draft[i * g:(i + 1) * g].to(torch.float64).numpy()


def _to_torch(x32: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x32))
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def _zipf_bias(V: int) -> np.ndarray:
    return -np.log1p(np.arange(V, dtype=np.float64))


def _gumbel_pick(rows: np.ndarray, temperature: float, top_k: int, rng: np.random.Generator):
    """Draw one token per row from softmax(row / T) restricted to the rows's top-k
    values (ties at the k-th value included) with the Gumbel-max trick."""
    n, V = rows.shape
    u = rng.random((n, V), dtype=np.float32)
    np.clip(u, np.float32(1e-30), np.float32(1.0 - 2.0 ** -24), out=u)
    g = -np.log(-np.log(u))
    scores = rows.astype(np.float32) / np.float32(temperature) + g
    if 0 < top_k < V:
        kth = np.partition(rows, V - top_k, axis=1)[:, V - top_k]
        scores = np.where(rows >= kth[:, None], scores, -np.inf)
    return scores.argmax(axis=1).astype(np.int32)


def make_chain(spec: ChainSpec, seed: int = 0, requests: Optional[Sequence[int]] = None) -> ChainBatch:
    """Build a chain workload (all requests, or the listed subset)."""
    reqs = np.arange(spec.B) if requests is None else np.asarray(requests, dtype=np.int64)
    g, V = spec.gamma, spec.V
    n = len(reqs)
    equal = np.zeros(0, np.int64)
    if spec.equal_rows_frac > 0:
        m = max(1, int(round(spec.equal_rows_frac * spec.B)))
        equal = np.sort(_rng(seed, SEED_EQUAL_ROWS).choice(spec.B, size=m, replace=False))
    bias = _zipf_bias(V).astype(np.float32) if spec.zipf_bias else None

    tgt32 = np.empty((n, g + 1, V), np.float32)
    drf32 = None if spec.greedy else np.empty((n, g, V), np.float32)
    for i, b in enumerate(reqs):
        x = _rng(seed, SEED_TARGET, b).standard_normal((g + 1, V), dtype=np.float32)
        x *= np.float32(spec.target_sigma)
        if bias is not None:
            x += bias
        tgt32[i] = x
        if drf32 is not None:
            if b in equal:
                drf32[i] = x[:g]
            else:
                e = _rng(seed, SEED_DRAFT_NOISE, b).standard_normal((g, V), dtype=np.float32)
                drf32[i] = x[:g] + np.float32(spec.draft_sigma) * e
    target = _to_torch(tgt32.reshape(n * (g + 1), V), spec.dtype)
    draft = None if drf32 is None else _to_torch(drf32.reshape(n * g, V), spec.dtype)

    tokens = np.empty((n, g), np.int32)
    unif = None if spec.greedy else np.empty((n, g + 1), np.float32)
    for i, b in enumerate(reqs):
        if spec.greedy:
            rows = target[i * (g + 1):i * (g + 1) + g].float().numpy()
            best = rows.argmax(axis=1)
            r = _rng(seed, SEED_GREEDY, b)
            hit = r.random(g) < spec.greedy_match_p
            other = (best + 1 + r.integers(0, V - 1, size=g)) % V if V > 1 else best
            tokens[i] = np.where(hit, best, other).astype(np.int32)
        else:
            rows = draft[i * g:(i + 1) * g].float().numpy()
            tokens[i] = _gumbel_pick(rows, spec.temperature, spec.top_k, _rng(seed, SEED_GUMBEL, b))
            unif[i] = uniforms24(_rng(seed, SEED_UNIFORMS, b), g + 1)
    return ChainBatch(spec, reqs, target, draft, tokens, unif, equal)


# --------------------------------------------------------------------------
# draft trees (topKSpec / topHead)
# --------------------------------------------------------------------------
@dataclass
class DraftTree:
    node_token: np.ndarray   # int32 [N]   token of node 1..N
    node_parent: np.ndarray  # int32 [N]   parent id of node 1..N (0 = root), parent < own id
    row_of_node: np.ndarray  # int32 [N+1] logits row of node 0..N, -1 = none

    @property
    def N(self) -> int:
        return len(self.node_token)


def grow_tree(draft_rows: np.ndarray, topKSpec, topHead) -> DraftTree:
    """Grow a draft tree level by level.

    Level i expands ``topHead[i]`` parents, each with ``topKSpec[i][j]``
    children: the draft's top tokens at that parent (ties to the lower token
    id).  Level 0 expands the root.  Parents of level i > 0 are the
    ``topHead[i]`` nodes of level i-1 with the highest draft path probability
    (product of the draft's softmax at temperature 1 along the path; ties to
    the lower node id).  Node ids are assigned breadth first; within a level,
    children follow their parent's id and then the draft's rank.  Each
    expanded parent gets the next logits row, in node-id order.
    ``draft_rows[r]`` are the draft logits at the parent that owns row r.
    """
    if len(topKSpec) != len(topHead) or (len(topHead) and topHead[0] != 1):
        raise ValueError("topHead must start with 1 (the root) and match topKSpec")
    token, parent, logp, row_of = [-1], [-1], [0.0], [0]
    prev_level = [0]
    next_row = 1
    for i, (ks, nh) in enumerate(zip(topKSpec, topHead)):
        if len(ks) != nh:
            raise ValueError("topKSpec[i] must have topHead[i] entries")
        if i == 0:
            parents = [0]
        else:
            ranked = sorted(prev_level, key=lambda nd: (-logp[nd], nd))[:nh]
            parents = sorted(ranked)
            for p in parents:
                row_of[p] = next_row
                next_row += 1
        level = []
        for p, k in zip(parents, ks):
            row = np.asarray(draft_rows[row_of[p]], dtype=np.float64)
            z = row - row.max()
            lq = z - np.log(np.exp(z).sum())
            order = np.argsort(-row, kind="stable")[:k]
            for t in order:
                token.append(int(t))
                parent.append(p)
                logp.append(logp[p] + float(lq[t]))
                row_of.append(-1)
                level.append(len(token) - 1)
        prev_level = level
    return DraftTree(np.asarray(token[1:], np.int32), np.asarray(parent[1:], np.int32),
                     np.asarray(row_of, np.int32))


@dataclass
class TreeBatch:
    spec: TreeSpec
    requests: np.ndarray
    logits: torch.Tensor        # [n*R, V] target logits, one row per expanded parent
    node_token: np.ndarray      # int32 [n, N]
    node_parent: np.ndarray     # int32 [n, N]
    row_of_node: np.ndarray     # int32 [n, N+1]

    @property
    def n(self) -> int:
        return len(self.requests)

    def logits_f64(self, i: int) -> np.ndarray:
        R = self.spec.n_rows
        return self.logits[i * R:(i + 1) * R].to(torch.float64).numpy()


def make_tree(spec: TreeSpec, seed: int = 0, requests: Optional[Sequence[int]] = None) -> TreeBatch:
    reqs = np.arange(spec.B) if requests is None else np.asarray(requests, dtype=np.int64)
    R, N, V, n = spec.n_rows, spec.n_nodes, spec.V, len(reqs)
    tgt32 = np.empty((n, R, V), np.float32)
    toks = np.empty((n, N), np.int32)
    pars = np.empty((n, N), np.int32)
    rows = np.empty((n, N + 1), np.int32)
    for i, b in enumerate(reqs):
        x = _rng(seed, SEED_TARGET, b).standard_normal((R, V), dtype=np.float32)
        x *= np.float32(spec.target_sigma)
        tgt32[i] = x
        e = _rng(seed, SEED_DRAFT_NOISE, b).standard_normal((R, V), dtype=np.float32)
        tree = grow_tree(x + np.float32(spec.draft_sigma) * e, spec.topKSpec, spec.topHead)
        toks[i], pars[i], rows[i] = tree.node_token, tree.node_parent, tree.row_of_node
    logits = _to_torch(tgt32.reshape(n * R, V), spec.dtype)
    return TreeBatch(spec, reqs, logits, toks, pars, rows)


def make_tree_levels(spec: TreeSpec, seed: int = 0,
                     requests: Optional[Sequence[int]] = None) -> List[torch.Tensor]:
    """Draft logits for building the trees of ``spec`` level by level: entry
    i is [n*topHead[i], V] in the spec's dtype, row b*topHead[i] + j being the
    draft's logits at parent j of level i of request b.  They are the draft
    rows ``make_tree`` grows its trees from (target rows plus draft noise,
    same seeds), so the expanded parents' rows line up with its logits rows."""
    reqs = np.arange(spec.B) if requests is None else np.asarray(requests, dtype=np.int64)
    R, V, n = spec.n_rows, spec.V, len(reqs)
    rows = np.empty((n, R, V), np.float32)
    for i, b in enumerate(reqs):
        x = _rng(seed, SEED_TARGET, b).standard_normal((R, V), dtype=np.float32)
        x *= np.float32(spec.target_sigma)
        e = _rng(seed, SEED_DRAFT_NOISE, b).standard_normal((R, V), dtype=np.float32)
        rows[i] = x + np.float32(spec.draft_sigma) * e
    out, r0 = [], 0
    for h in spec.topHead:
        out.append(_to_torch(np.ascontiguousarray(rows[:, r0:r0 + h]).reshape(n * h, V), spec.dtype))
        r0 += h
    return out


# --------------------------------------------------------------------------
# paged KV cache
# --------------------------------------------------------------------------
@dataclass
class KVBatch:
    kv: KVSpec
    B: int
    S: int                       # temporary slots per request
    temp_kv: torch.Tensor        # bf16 [B, L, 2, S, H, D] (random bit patterns)
    block_table: np.ndarray      # int32 [B, max_blocks]
    committed_len: np.ndarray    # int32 [B]
    num_blocks: int

    @property
    def max_blocks(self) -> int:
        return self.block_table.shape[1]

    def cache_shape(self):
        k = self.kv
        return (k.layers, 2, self.num_blocks, k.block_size, k.heads, k.head_dim)


def make_kv(kv: KVSpec, B: int, S: int, seed: int = 0, prefix=None, pool_factor: int = 4) -> KVBatch:
    """Temporary K/V for S slots per request plus a block table.

    The prefix's blocks all point at block 0, a shared dummy block that a
    commit never reaches.  The blocks that hold positions prefix..prefix+S-1
    are physical: drawn without replacement from a pool ``pool_factor`` times
    larger than needed, in a random order, so destination addresses scatter.
    ``prefix`` may be an int or a per-request array (default ``kv.prefix``).
    """
    bs = kv.block_size
    pre = np.full(B, kv.prefix if prefix is None else 0, np.int64)
    if prefix is not None:
        pre[:] = np.asarray(prefix, dtype=np.int64)
    first = pre // bs
    last = (pre + S - 1) // bs if S > 0 else first
    n_tail = (last - first + 1).astype(np.int64)
    max_blocks = int((pre + S + bs - 1).max() // bs) if B else 1
    max_blocks = max(max_blocks, 1)
    total_tail = int(n_tail.sum())
    pool = max(1, pool_factor * total_tail)
    perm = _rng(seed, SEED_BLOCK_PERM).permutation(pool)[:total_tail] + 1
    table = np.zeros((B, max_blocks), np.int32)
    at = 0
    for b in range(B):
        for j in range(int(n_tail[b])):
            table[b, first[b] + j] = perm[at]
            at += 1
    r = _rng(seed, SEED_TEMP_KV)
    numel = B * kv.layers * 2 * S * kv.heads * kv.head_dim
    bits = r.integers(0, 1 << 16, size=numel, dtype=np.uint16).view(np.int16)
    temp = torch.from_numpy(bits).view(torch.bfloat16).reshape(
        B, kv.layers, 2, S, kv.heads, kv.head_dim)
    return KVBatch(kv, B, S, temp, table, pre.astype(np.int32), 1 + pool)


def make_cache(batch: KVBatch, device="cpu") -> torch.Tensor:
    """A cache filled with the sentinel bit pattern."""
    return torch.full(batch.cache_shape(), KV_SENTINEL, dtype=torch.int16,
                      device=device).view(torch.bfloat16)


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = [
    "KVSpec", "ChainSpec", "TreeSpec", "WORKLOADS", "ChainBatch", "make_chain", "DraftTree",
    "grow_tree", "TreeBatch", "make_tree", "KVBatch", "make_kv", "make_cache",
    "uniforms24", "KV_SENTINEL",
]


# --------------------------------------------------------------------------
# token histories for the n-gram (prompt-lookup) drafter
# --------------------------------------------------------------------------
@dataclass
class HistorySpec:
    name: str
    B: int
    max_len: int
    vocab: int
    gamma: int
    n_min: int
    n_max: int
    copy_frac: float = 0.5   # share of segments copied from earlier in the history


# A large batch of long histories (an HBM scan of about 134 MB); the shapes
# follow the chain workloads' vocabulary and the framework's default prompt
# lookup window.
NGRAM_SPEC = HistorySpec("ngram B=1024 L<=32768 V=128256 n=1..4 g=8", B=1024, max_len=32768,
                         vocab=128256, gamma=8, n_min=1, n_max=4)


def make_histories(spec: HistorySpec, seed: int = 0, requests: Optional[Sequence[int]] = None):
    """Returns (history int32 [n, max_len] padded with -1, lengths int32 [n]).
    A history is a sequence of segments: a copy (probability copy_frac) of an
    earlier stretch of 4..64 tokens, so that n-grams recur, or 4..64 fresh
    tokens drawn uniformly from the vocabulary; the last segment is always a
    copy (the text being generated continues a passage seen before, the case
    prompt lookup serves).  Lengths are drawn in [max_len/2, max_len]."""
    idx = list(range(spec.B)) if requests is None else list(requests)
    hist = np.full((len(idx), spec.max_len), -1, dtype=np.int32)
    lens = np.zeros(len(idx), dtype=np.int32)
    for r, b in enumerate(idx):
        rng = _rng(seed, 9, b)
        L = int(rng.integers(spec.max_len // 2, spec.max_len + 1))
        h = np.empty(L, dtype=np.int32)
        at = 0
        while at < L:
            m = int(min(rng.integers(4, 65), L - at))
            last = at + m >= L
            if at >= 8 and (last or rng.random() < spec.copy_frac):
                src = int(rng.integers(0, at - min(m, at) + 1))
                m = min(m, at - src)
                h[at:at + m] = h[src:src + m]
            else:
                h[at:at + m] = rng.integers(0, spec.vocab, size=m, dtype=np.int32)
            at += m
        hist[r, :L] = h
        lens[r] = L
    return hist, lens
