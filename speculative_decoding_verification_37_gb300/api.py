"""Convenience layer over the C ABI: allocates outputs and workspaces with
torch and calls the library.  No arithmetic of the method happens here."""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, Optional, Tuple

import torch

from . import _lib as L

_WORKSPACES: Dict[Tuple, torch.Tensor] = {}


def workspace(kind: int, B: int, n: int, V: int, device) -> torch.Tensor:
    """A cached zero-filled workspace for (device, kind, B, n, V) (the size of
    some kinds depends on V).  Every call leaves it zeroed, so it is reused
    without clearing; calls that share it must be ordered on one stream.
    The cache lives as long as the process; clear_workspaces() frees it."""
    dev = torch.device(device)
    if dev.type == "cuda" and dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    key = (dev.type, dev.index, kind, B, n, V)
    ws = _WORKSPACES.get(key)
    if ws is None:
        ws = L.new_workspace(kind, B, n, V, device=dev)
        _WORKSPACES[key] = ws
    return ws


def clear_workspaces() -> None:
    """Drops every cached workspace (after the work using them has finished),
    e.g. after a timeout (SPEC_FLAG_TIMEOUT asks for a fresh workspace) or
    when batch shapes change for good."""
    _WORKSPACES.clear()


@dataclass
class ChainOut:
    n_acc: torch.Tensor                   # int32 [B]
    out_tokens: torch.Tensor              # int32 [B, gamma+1]
    n_out: torch.Tensor                   # int32 [B]
    accept_prob: Optional[torch.Tensor]   # f32 [B, gamma]
    residual_mass: Optional[torch.Tensor] # f32 [B, gamma]
    flags: torch.Tensor                   # uint32 stored as int32 [B]


def chain_workspace_kind(sampled: bool, top_k: int, V: int, residual_mass: bool = False) -> int:
    """The workspace kind that lets a chain call take its fastest path."""
    if not sampled:
        return L.SPEC_WS_CHAIN
    if 0 < top_k <= L.TOPK_FAST_MAX and top_k < V:
        return L.SPEC_WS_CHAIN_TOPK
    if (top_k == 0 or top_k >= V) and not residual_mass:
        return L.SPEC_WS_CHAIN_FULL
    return L.SPEC_WS_CHAIN


def verify_chain(target: torch.Tensor, draft_tokens: torch.Tensor, *, gamma: int,
                 temperature: float, draft: Optional[torch.Tensor] = None,
                 uniforms: Optional[torch.Tensor] = None, top_k: int = 0,
                 fallback_eps: float = 1e-6, accept_prob: bool = True,
                 residual_mass: bool = False, ws: Optional[torch.Tensor] = None,
                 committed_len: Optional[torch.Tensor] = None,
                 draft_len: Optional[torch.Tensor] = None,
                 blocks_in_use: Optional[torch.Tensor] = None, block_size: int = 0,
                 kv_capacity: int = 0, eos_token: Optional[int] = None,
                 max_new: Optional[torch.Tensor] = None, top_p: float = 0.0,
                 gamma_per_request: Optional[torch.Tensor] = None,
                 temperature_per_request: Optional[torch.Tensor] = None,
                 top_k_per_request: Optional[torch.Tensor] = None,
                 top_p_per_request: Optional[torch.Tensor] = None,
                 stream=None) -> ChainOut:
    """target [B*(gamma+1), V], draft [B*gamma, V] (bf16 or f32, rows may be
    strided), draft_tokens int32 [B, gamma], uniforms f32 [B, gamma+1].

    With committed_len (int32 [B], on the device) the call also commits the
    in-place K/V of the candidates: committed_len advances by n_out,
    draft_len (if given) is cut back to it and blocks_in_use (if given)
    follows, all on the device.  eos_token / max_new (int32 [B] on the
    device) end the round early: its output is cut right after the first
    EOS, then to max_new[b] tokens.  0 < top_p < 1 adds the nucleus after
    top-k.  The *_per_request tensors (on the device, [B]) give each request
    its own gamma (<= gamma; the arrays stay padded to gamma), temperature (0:
    greedy), top-k and top-p."""
    dev = target.device
    V = target.shape[-1]
    B = target.shape[0] // (gamma + 1)
    per_request = any(x is not None for x in (gamma_per_request, temperature_per_request,
                                               top_k_per_request, top_p_per_request))
    sampled = temperature > 0 or temperature_per_request is not None
    out = ChainOut(
        n_acc=torch.empty(B, dtype=torch.int32, device=dev),
        out_tokens=torch.full((B, gamma + 1), -1, dtype=torch.int32, device=dev),
        n_out=torch.empty(B, dtype=torch.int32, device=dev),
        accept_prob=torch.empty((B, gamma), dtype=torch.float32, device=dev)
        if (sampled and accept_prob) else None,
        residual_mass=torch.empty((B, gamma), dtype=torch.float32, device=dev)
        if (sampled and residual_mass) else None,
        flags=torch.zeros(B, dtype=torch.int32, device=dev))
    if ws is None:
        kind = L.SPEC_WS_CHAIN if per_request else chain_workspace_kind(sampled, top_k, V, residual_mass)
        ws = workspace(kind, B, gamma, V, dev)
    L.spec_verify_chain(target_logits=target, draft_tokens=draft_tokens, n_acc=out.n_acc,
                        out_tokens=out.out_tokens, n_out=out.n_out, workspace=ws, gamma=gamma,
                        temperature=temperature, draft_logits=draft, uniforms=uniforms,
                        top_k=top_k, fallback_eps=fallback_eps, accept_prob=out.accept_prob,
                        residual_mass=out.residual_mass, flags=out.flags,
                        committed_len=committed_len, draft_len=draft_len,
                        blocks_in_use=blocks_in_use, block_size=block_size,
                        kv_capacity=kv_capacity, eos_token=eos_token, max_new=max_new,
                        top_p=top_p, gamma_per_request=gamma_per_request,
                        temperature_per_request=temperature_per_request,
                        top_k_per_request=top_k_per_request, top_p_per_request=top_p_per_request,
                        stream=stream)
    return out


@dataclass
class TreeOut:
    path: torch.Tensor          # int32 [B, N]
    n_acc: torch.Tensor         # int32 [B]
    out_tokens: torch.Tensor    # int32 [B, N+1]
    n_out: torch.Tensor         # int32 [B]
    tree_mask: torch.Tensor     # int32 view of uint32 [B, N+1, W]
    pos: torch.Tensor           # int32 [B, N+1]
    commit_slots: torch.Tensor  # int32 [B, N+1]
    n_commit: torch.Tensor      # int32 [B]
    flags: torch.Tensor         # int32 [B]


def verify_tree(logits: torch.Tensor, node_token: torch.Tensor, node_parent: torch.Tensor,
                row_of_node: torch.Tensor, committed_len: torch.Tensor, *, R: int,
                ws: Optional[torch.Tensor] = None, stream=None) -> TreeOut:
    dev = logits.device
    V = logits.shape[-1]
    B = logits.shape[0] // R
    N = node_token.shape[-1]
    W = (N + 1 + 31) // 32
    i32 = dict(dtype=torch.int32, device=dev)
    out = TreeOut(path=torch.full((B, N), -1, **i32), n_acc=torch.empty(B, **i32),
                  out_tokens=torch.full((B, N + 1), -1, **i32), n_out=torch.empty(B, **i32),
                  tree_mask=torch.zeros((B, N + 1, W), **i32), pos=torch.empty((B, N + 1), **i32),
                  commit_slots=torch.full((B, N + 1), -1, **i32), n_commit=torch.empty(B, **i32),
                  flags=torch.zeros(B, **i32))
    if ws is None:
        ws = workspace(L.SPEC_WS_TREE, B, R, V, dev)
    L.spec_verify_tree(logits=logits, R=R, node_token=node_token, node_parent=node_parent,
                       row_of_node=row_of_node, path=out.path, n_acc=out.n_acc,
                       out_tokens=out.out_tokens, n_out=out.n_out, workspace=ws,
                       committed_len=committed_len, tree_mask=out.tree_mask, pos=out.pos,
                       commit_slots=out.commit_slots, n_commit=out.n_commit, flags=out.flags,
                       stream=stream)
    return out


def commit_kv(temp_kv: torch.Tensor, cache: torch.Tensor, block_table: torch.Tensor,
              n_slots: torch.Tensor, committed_len: torch.Tensor, *, block_size: int,
              slots: Optional[torch.Tensor] = None, blocks_in_use: Optional[torch.Tensor] = None,
              flags: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
              stream=None) -> None:
    """Commits in place: cache and committed_len are updated on the device."""
    if ws is None:
        ws = workspace(L.SPEC_WS_COMMIT, temp_kv.shape[0], 0, 0, temp_kv.device)
    L.spec_commit_kv(temp_kv=temp_kv, cache=cache, block_table=block_table, n_slots=n_slots,
                     committed_len=committed_len, block_size=block_size, workspace=ws,
                     slots=slots, blocks_in_use=blocks_in_use, flags=flags, stream=stream)


@dataclass
class NgramOut:
    draft_tokens: torch.Tensor   # int32 [B, gamma], -1 past n_draft
    n_draft: torch.Tensor        # int32 [B]
    match_n: torch.Tensor        # int32 [B], 0 if no match
    match_start: torch.Tensor    # int32 [B], -1 if no match
    flags: torch.Tensor          # int32 [B]


def ngram_draft(history: torch.Tensor, hist_len: torch.Tensor, *, gamma: int, n_min: int = 1,
                n_max: int = 4, stream=None) -> NgramOut:
    """Prompt-lookup drafts: history int32 [B, max_len] on the device (row b's
    first hist_len[b] tokens are its history)."""
    dev = history.device
    B = history.shape[0]
    i32 = dict(dtype=torch.int32, device=dev)
    out = NgramOut(draft_tokens=torch.empty((B, gamma), **i32), n_draft=torch.empty(B, **i32),
                   match_n=torch.empty(B, **i32), match_start=torch.empty(B, **i32),
                   flags=torch.empty(B, **i32))
    L.spec_ngram_draft(history=history, hist_len=hist_len, gamma=gamma, n_min=n_min, n_max=n_max,
                       draft_tokens=out.draft_tokens, n_draft=out.n_draft, match_n=out.match_n,
                       match_start=out.match_start, flags=out.flags, stream=stream)
    return out


class TreeBuilder:
    """Builds draft trees for B requests one level at a time on the device
    (topKSpec / topHead shape).  Between levels the caller runs the draft
    model at ``next_parents`` and passes its logits rows, in that order, to
    the next ``level`` call.  Node arrays follow the tree verify's layout:
    node_token / node_parent [B, N] (node id i at index i-1), node_logp /
    row_of_node [B, N+1] (indexed by node id, the root is 0)."""

    def __init__(self, B: int, V: int, topKSpec, topHead, device, flags: bool = True):
        if len(topKSpec) != len(topHead) or not len(topHead) or topHead[0] != 1:
            raise ValueError("topHead must start with 1 (the root) and match topKSpec")
        self.B, self.V = B, V
        self.topKSpec = [list(map(int, ks)) for ks in topKSpec]
        self.topHead = list(map(int, topHead))
        self.N = sum(sum(ks) for ks in self.topKSpec)
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.node_token = torch.full((B, self.N), -1, **i32)
        self.node_parent = torch.full((B, self.N), -1, **i32)
        self.node_logp = torch.zeros((B, self.N + 1), dtype=torch.float32, device=dev)
        self.row_of_node = torch.full((B, self.N + 1), -1, **i32)
        self.flags = torch.zeros(B, **i32) if flags else None
        self.next = [torch.empty((B, h), **i32) for h in self.topHead[1:]] + [None]
        self.ws = [workspace(L.SPEC_WS_TREE_LEVEL, B, h, V, dev) for h in self.topHead]
        self.level_index = 0

    def level(self, logits: torch.Tensor, i: Optional[int] = None, stream=None) -> Optional[torch.Tensor]:
        """Expand level i (default: the next one) from its draft rows
        [B*topHead[i], V]; returns the next level's parents [B, topHead[i+1]]
        (None after the last level)."""
        i = self.level_index if i is None else i
        H = self.topHead[i]
        n_before = sum(sum(ks) for ks in self.topKSpec[:i])
        next_row0 = sum(self.topHead[:i + 1])
        n_next = self.topHead[i + 1] if i + 1 < len(self.topHead) else 0
        L.spec_tree_level(logits=logits, H=H, k=self.topKSpec[i], n_next=n_next, n_before=n_before,
                          next_row0=next_row0, node_token=self.node_token,
                          node_parent=self.node_parent, node_logp=self.node_logp,
                          row_of_node=self.row_of_node, workspace=self.ws[i],
                          parents=None if i == 0 else self.next[i - 1],
                          next_parents=self.next[i], flags=self.flags, stream=stream)
        self.level_index = i + 1
        return self.next[i]
