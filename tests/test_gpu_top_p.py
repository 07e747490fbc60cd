"""GPU parity of the top-p (nucleus) transform against the oracle, through the
C ABI: the nucleus is cut from the top-k merge's exact kept set, on target and
draft rows alike.  Same comparison rules as every sampled test (tokens exact
away from boundary cases, a and Z within 1e-5)."""
import numpy as np
import pytest
import torch

import oracle as O
from parity import PROB_TOL, to_dev
from speculative_decoding_verification_37_gb300 import _lib as L
from speculative_decoding_verification_37_gb300 import api
from speculative_decoding_verification_37_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run_and_compare(batch, top_p, quant=None):
    s = batch.spec
    tp = float(np.float32(top_p))          # the value the kernel sees
    if quant:
        batch.target = torch.round(batch.target.float() / quant).mul(quant).to(batch.target.dtype)
        batch.draft = torch.round(batch.draft.float() / quant).mul(quant).to(batch.draft.dtype)
    tgt, drf, tok, unif = to_dev(batch)
    ws = api.workspace(L.SPEC_WS_CHAIN_TOPK, s.B, s.gamma, s.V, "cuda")
    out = api.verify_chain(tgt, tok, gamma=s.gamma, temperature=s.temperature, draft=drf,
                           uniforms=unif, top_k=s.top_k, residual_mass=False, ws=ws, top_p=tp)
    torch.cuda.synchronize()
    n_out, n_acc = out.n_out.cpu().numpy(), out.n_acc.cpu().numpy()
    toks, a = out.out_tokens.cpu().numpy(), out.accept_prob.cpu().numpy()
    flags = out.flags.cpu().numpy()
    boundary = 0
    for b in range(s.B):
        r = O.verify_chain_sampled(batch.target_f64(b), batch.draft_f64(b), batch.draft_tokens[b],
                                   batch.uniforms[b].astype(np.float64), s.temperature, s.top_k,
                                   top_p=tp)
        assert np.abs(a[b] - r.accept_prob).max() <= PROB_TOL, (b, a[b], r.accept_prob)
        if r.boundary:
            boundary += 1
            continue
        assert n_acc[b] == r.n_acc and n_out[b] == r.n_out, (b, n_acc[b], r.n_acc)
        assert toks[b][:n_out[b]].tolist() == r.tokens, (b, toks[b], r.tokens)
        assert bool(flags[b] & O.FLAG_FALLBACK) == bool(r.flags & O.FLAG_FALLBACK), b
    assert boundary <= max(1, s.B // 100)


def spec(B, gamma, V, dtype, T, top_k, sigma=3.0, draft_sigma=1.0):
    return W.ChainSpec(f"t B={B} g={gamma} V={V}", B=B, gamma=gamma, V=V, dtype=dtype,
                       target_sigma=sigma, temperature=T, top_k=top_k, draft_sigma=draft_sigma)


@pytest.mark.parametrize("case", [
    # (B, gamma, V, dtype, T, top_k, top_p)
    (48, 4, 32000, "bf16", 0.8, 50, 0.9),
    (40, 3, 5000, "f32", 1.0, 20, 0.5),
    (32, 4, 3000, "bf16", 1.0, 8, 1e-4),     # the most probable token (and its ties) only
    (32, 2, 4000, "f32", 0.7, 64, 0.999),
    (24, 5, 128256, "bf16", 0.8, 128, 0.8),
])
def test_top_p_matches_oracle(case):
    B, g, V, dt, T, k, tp = case
    batch = W.make_chain(spec(B, g, V, dt, T, k), seed=B + V)
    run_and_compare(batch, tp)


def test_top_p_with_tied_logits():
    """Logits on a 0.5 grid: ties inside the top-k set and at the nucleus cut."""
    batch = W.make_chain(spec(40, 3, 2000, "bf16", 1.0, 16, sigma=1.5, draft_sigma=0.7), seed=9)
    run_and_compare(batch, 0.7, quant=0.5)
