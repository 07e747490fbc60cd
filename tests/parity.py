"""Comparison of the CUDA path (through the C ABI) with the fp64 oracle.

Rules (tolerances written here, used by every GPU parity test):
  * greedy and tree decisions, n_acc, emitted tokens, masks, positions and
    committed KV bytes: bit-exact;
  * accept_prob and residual_mass: |gpu - oracle| <= 1e-5 (absolute);
  * sampled decisions: identical, except requests the oracle flags as
    boundary cases (a uniform within 1e-5 of an acceptance threshold; a draw
    target u*C_total within 3e-11*C_total + 1e-12 of either end of the
    chosen token's CDF interval, the arithmetic's own error; a residual mass
    within eps/2 of eps); those are counted and must stay under 1e-4 of
    decisions (a request with a boundary case is excluded from token
    equality).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from speculative_decoding_verification_37_gb300 import api

PROB_TOL = 1e-5
BOUNDARY_RATE_MAX = 1e-4


def to_dev(batch, device="cuda"):
    tgt = batch.target.to(device)
    drf = None if batch.draft is None else batch.draft.to(device)
    tok = torch.from_numpy(batch.draft_tokens).to(device)
    unif = None if batch.uniforms is None else torch.from_numpy(batch.uniforms).to(device)
    return tgt, drf, tok, unif


def run_chain(batch, residual=True, device="cuda", target=None, draft=None):
    """Run the GPU chain verify on a ChainBatch; returns numpy outputs."""
    s = batch.spec
    tgt, drf, tok, unif = to_dev(batch, device)
    if target is not None:
        tgt = target
    if draft is not None:
        drf = draft
    out = api.verify_chain(tgt, tok, gamma=s.gamma, temperature=s.temperature, draft=drf,
                           uniforms=unif, top_k=s.top_k, residual_mass=residual)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in vars(out).items()}


def full_path_used(B, gamma, V):
    """True when the last chain call on the cached SPEC_WS_CHAIN_FULL
    workspace of this shape ran the persistent full-vocabulary kernel: it
    writes its per-slice statistics right after the plain chain workspace,
    a region no other kernel touches."""
    from speculative_decoding_verification_37_gb300 import _lib as L
    torch.cuda.synchronize()
    ws = api.workspace(L.SPEC_WS_CHAIN_FULL, B, gamma, V, "cuda")
    plain = L.spec_workspace_bytes(L.SPEC_WS_CHAIN, B, gamma, V)
    plain = (plain + 255) // 256 * 256
    return bool(ws[plain:plain + 256].any())


def oracle_chain(batch, i):
    s = batch.spec
    if s.greedy:
        return O.verify_chain_greedy(batch.target_f64(i), batch.draft_tokens[i])
    return O.verify_chain_sampled(batch.target_f64(i), batch.draft_f64(i), batch.draft_tokens[i],
                                  batch.uniforms[i].astype(np.float64), s.temperature, s.top_k)


class ChainTally:
    def __init__(self):
        self.requests = 0
        self.decisions = 0
        self.boundary = 0
        self.fallback = 0
        self.max_a_err = 0.0
        self.max_z_err = 0.0

    @property
    def boundary_rate(self):
        return self.boundary / max(1, self.decisions)


def compare_chain(batch, gpu, indices, tally: ChainTally | None = None, rows=None,
                  oracle_results=None):
    """Compare GPU outputs (dict of numpy arrays over the whole batch) with the
    oracle on the listed request indices.  ``rows[i]`` maps a batch index to
    the GPU output row (default: the same index).  ``oracle_results`` (a
    dict, filled here) keeps the oracle's result per request, so two GPU
    paths can be compared with one oracle run."""
    tally = tally or ChainTally()
    s = batch.spec
    for i in indices:
        gi = i if rows is None else rows[i]
        if oracle_results is not None and i in oracle_results:
            r = oracle_results[i]
        else:
            r = oracle_chain(batch, i)
            if oracle_results is not None:
                oracle_results[i] = r
        tally.requests += 1
        if r.flags & (O.FLAG_BAD_INPUT | O.FLAG_BAD_ROW):
            assert gpu["n_out"][gi] == 0 and gpu["n_acc"][gi] == 0, i
            assert int(gpu["flags"][gi]) & (O.FLAG_BAD_INPUT | O.FLAG_BAD_ROW), i
            continue
        tally.decisions += min(r.n_acc + 1, s.gamma) + 1
        if not s.greedy:
            if gpu.get("accept_prob") is not None:
                err = np.abs(gpu["accept_prob"][gi] - r.accept_prob).max(initial=0.0)
                tally.max_a_err = max(tally.max_a_err, float(err))
                assert err <= PROB_TOL, (i, gpu["accept_prob"][gi], r.accept_prob)
            if gpu.get("residual_mass") is not None:
                err = np.abs(gpu["residual_mass"][gi] - r.residual_mass).max(initial=0.0)
                tally.max_z_err = max(tally.max_z_err, float(err))
                assert err <= PROB_TOL, (i, gpu["residual_mass"][gi], r.residual_mass)
            if r.boundary:
                tally.boundary += 1
                continue
        n = int(gpu["n_out"][gi])
        assert int(gpu["n_acc"][gi]) == r.n_acc, (i, gpu["n_acc"][gi], r.n_acc)
        assert n == r.n_out, (i, n, r.n_out)
        assert list(gpu["out_tokens"][gi][:n]) == r.tokens, (i, gpu["out_tokens"][gi][:n], r.tokens)
        fb = bool(int(gpu["flags"][gi]) & O.FLAG_FALLBACK)
        assert fb == bool(r.flags & O.FLAG_FALLBACK), i
        tally.fallback += fb
    return tally
