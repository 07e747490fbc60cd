"""GPU parity of the round's early end (EOS, length limit) against the oracle
on every chain path, through the C ABI."""
from collections import Counter

import numpy as np
import pytest
import torch

import oracle as O
from parity import oracle_chain, to_dev
from speculative_decoding_verification_37_gb300 import _lib as L
from speculative_decoding_verification_37_gb300 import api
from speculative_decoding_verification_37_gb300 import workloads as W

pytestmark = pytest.mark.gpu

STOP = O.FLAG_EOS | O.FLAG_LIMIT


def chain(B, gamma, V, dtype, T, top_k=0, sigma=2.0):
    return W.ChainSpec(f"t B={B} g={gamma} V={V}", B=B, gamma=gamma, V=V, dtype=dtype,
                       target_sigma=sigma, temperature=T, top_k=top_k, draft_sigma=0.5)


def check(batch, kind, seed, in_place=False):
    s = batch.spec
    results = [oracle_chain(batch, b) for b in range(s.B)]
    # the EOS: the token that the most requests emit, so that many rounds are cut
    seen = Counter(t for r in results if not r.flags for t in set(r.tokens))
    eos = min(seen.items(), key=lambda kv: (-kv[1], kv[0]))[0]
    rng = np.random.default_rng(seed)
    max_new = rng.integers(-1, s.gamma + 3, s.B).astype(np.int32)
    max_new[::5] = 1 << 20                                  # some requests far from the limit
    tgt, drf, tok, unif = to_dev(batch)
    ws = api.workspace(kind, s.B, s.gamma, s.V, "cuda")
    extra = {}
    if in_place:
        cl = torch.full((s.B,), 100, dtype=torch.int32, device="cuda")
        extra = dict(committed_len=cl)
    out = api.verify_chain(tgt, tok, gamma=s.gamma, temperature=s.temperature, draft=drf,
                           uniforms=unif, top_k=s.top_k, ws=ws, eos_token=eos,
                           max_new=torch.from_numpy(max_new).cuda(), **extra)
    torch.cuda.synchronize()
    n_out, n_acc = out.n_out.cpu().numpy(), out.n_acc.cpu().numpy()
    toks, flags = out.out_tokens.cpu().numpy(), out.flags.cpu().numpy()
    cut_eos = cut_lim = 0
    for b, r in enumerate(results):
        t = O.truncate_round(r, eos, int(max_new[b]))
        if r.flags & (O.FLAG_BAD_INPUT | O.FLAG_BAD_ROW) or r.boundary:
            continue
        Lb = len(t.tokens)
        assert n_out[b] == Lb and n_acc[b] == t.n_acc, (b, n_out[b], n_acc[b], t.tokens, t.n_acc)
        assert toks[b][:Lb].tolist() == t.tokens, b
        assert (toks[b][Lb:] == -1).all(), b
        assert int(flags[b]) & STOP == t.flags & STOP, (b, flags[b], t.flags)
        cut_eos += bool(t.flags & O.FLAG_EOS) and Lb < len(r.tokens)
        cut_lim += bool(t.flags & O.FLAG_LIMIT)
        if in_place:
            assert int(extra["committed_len"][b]) == 100 + Lb
    assert cut_eos > 0 and cut_lim > 0


def test_stop_greedy():
    batch = W.make_chain(chain(128, 6, 64, "bf16", 0.0), seed=1)
    check(batch, L.SPEC_WS_CHAIN, 1)


def test_stop_sampled_cluster_path():
    batch = W.make_chain(chain(96, 5, 48, "f32", 1.0), seed=2)
    check(batch, L.SPEC_WS_CHAIN, 2)


def test_stop_sampled_topk_path():
    batch = W.make_chain(chain(96, 4, 3000, "bf16", 0.8, top_k=3, sigma=3.0), seed=3)
    check(batch, L.SPEC_WS_CHAIN_TOPK, 3)


def test_stop_sampled_full_path_with_in_place_commit():
    batch = W.make_chain(chain(256, 4, 1024, "f32", 0.5, sigma=3.0), seed=4)   # 1,280 items
    check(batch, L.SPEC_WS_CHAIN_FULL, 4, in_place=True)


def test_no_stop_rule_leaves_rounds_whole():
    """Without eos_token / max_new the outputs are the whole rounds and no
    stop flag is set."""
    batch = W.make_chain(chain(32, 3, 200, "f32", 1.0), seed=5)
    tgt, drf, tok, unif = to_dev(batch)
    out = api.verify_chain(tgt, tok, gamma=3, temperature=1.0, draft=drf, uniforms=unif)
    torch.cuda.synchronize()
    for b in range(32):
        r = oracle_chain(batch, b)
        if not r.boundary:
            assert int(out.n_out[b]) == r.n_out and not int(out.flags[b]) & STOP
