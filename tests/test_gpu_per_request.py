"""GPU parity of chain verification with per-request settings, through the C
ABI, against the oracle's verify_chain_batch: every request of a batch with
its own gamma (0..gamma_max, arrays padded to gamma_max), temperature (0 =
greedy), top-k and top-p ("10.6 投机解码" §10.6.3: the requests of one batch
accept different lengths; "KV Cache 优化（四）" §4: each request's processed
distributions enter its rule).  Also top-p over the full vocabulary
(top_k = 0), which takes the exact path.  Same comparison rules as every
sampled test: tokens exact away from boundary cases, a and Z within 1e-5;
greedy requests bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle as O
from parity import PROB_TOL
from speculative_decoding_verification_37_gb300 import api
from speculative_decoding_verification_37_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def mixed_batch(B, gamma, V, dtype, seed, temps, top_ks, top_ps):
    spec = W.ChainSpec(f"mixed B={B} g={gamma} V={V}", B=B, gamma=gamma, V=V, dtype=dtype,
                       target_sigma=2.5, temperature=1.0, top_k=0, draft_sigma=1.0)
    batch = W.make_chain(spec, seed=seed)
    rng = np.random.default_rng(seed + 100)
    gam = rng.integers(0, gamma + 1, size=B).astype(np.int32)
    T = rng.choice(np.asarray(temps, np.float32), size=B)
    K = rng.choice(np.asarray(top_ks, np.int32), size=B)
    P = rng.choice(np.asarray(top_ps, np.float32), size=B)
    # greedy requests: their drafts follow the target's argmax most of the time
    tgt = batch.target.float().numpy().reshape(B, gamma + 1, V)
    for b in np.nonzero(T == 0)[0]:
        am = tgt[b, :gamma].argmax(-1)
        batch.draft_tokens[b] = np.where(rng.random(gamma) < 0.7, am, batch.draft_tokens[b])
    return batch, gam, T, K, P


def run_per_request(batch, gam, T, K, P):
    s = batch.spec
    dev = "cuda"
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    out = api.verify_chain(batch.target.to(dev), t(batch.draft_tokens), gamma=s.gamma,
                           temperature=1.0, draft=batch.draft.to(dev), uniforms=t(batch.uniforms),
                           residual_mass=True, gamma_per_request=t(gam),
                           temperature_per_request=t(T), top_k_per_request=t(K),
                           top_p_per_request=t(P))
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in vars(out).items() if v is not None}


def compare(batch, got, results, gam, T):
    """Request by request against the oracle's results; returns the number of
    boundary cases."""
    boundary = 0
    for b, r in enumerate(results):
        gb = int(gam[b])
        if r.flags & (O.FLAG_BAD_INPUT | O.FLAG_BAD_ROW):
            assert got["n_out"][b] == 0 and int(got["flags"][b]) & (O.FLAG_BAD_INPUT | O.FLAG_BAD_ROW), b
            continue
        if T[b] > 0:
            assert np.abs(got["accept_prob"][b][:gb] - r.accept_prob).max(initial=0.0) <= PROB_TOL, b
            assert np.abs(got["residual_mass"][b][:gb] - r.residual_mass).max(initial=0.0) <= PROB_TOL, b
            if r.boundary:
                boundary += 1
                continue
        n = int(got["n_out"][b])
        assert int(got["n_acc"][b]) == r.n_acc and n == r.n_out, (b, gb, T[b], got["n_acc"][b], r.n_acc)
        assert list(got["out_tokens"][b][:n]) == r.tokens, (b, got["out_tokens"][b][:n], r.tokens)
        assert bool(int(got["flags"][b]) & O.FLAG_FALLBACK) == bool(r.flags & O.FLAG_FALLBACK), b
    return boundary


def oracle_batch(batch, gam, T, K, P):
    s = batch.spec
    B, g, V = s.B, s.gamma, s.V
    tgt = batch.target.double().numpy().reshape(B, g + 1, V)   # exact: bf16 / f32 -> f64
    drf = batch.draft.double().numpy().reshape(B, g, V)
    # the ABI's "off" (0, or >= 1) is the oracle's top_p = 1
    P_oracle = np.where((P > 0) & (P < 1), P, np.float32(1.0))
    return O.verify_chain_batch(tgt, drf, batch.draft_tokens, batch.uniforms.astype(np.float64),
                                gam, T, K, P_oracle)


@pytest.mark.parametrize("case", [
    # (B, gamma, V, dtype, seed)
    (64, 4, 4096, "bf16", 1),
    (40, 6, 32000, "f32", 2),
    (48, 3, 1000, "bf16", 3),      # ragged: 1000 * 2 bytes is not a multiple of 16
])
def test_mixed_settings_match_the_batch_oracle(case):
    B, g, V, dt, seed = case
    batch, gam, T, K, P = mixed_batch(B, g, V, dt, seed, temps=[0.0, 0.5, 1.0, 1.5],
                                      top_ks=[0, 1, 20, 50, 200, V], top_ps=[0.0, 0.3, 0.9, 1.0])
    assert (T == 0).any() and (T > 0).any() and (gam == 0).any() and (gam == g).any()
    got = run_per_request(batch, gam, T, K, P)
    boundary = compare(batch, got, oracle_batch(batch, gam, T, K, P), gam, T)
    assert boundary <= max(1, B // 100)


def test_every_request_gamma_zero_and_all_greedy():
    batch, gam, T, K, P = mixed_batch(32, 3, 2048, "f32", 4, temps=[1.0], top_ks=[0], top_ps=[0.0])
    gam[:] = 0  # bonus draws only
    got = run_per_request(batch, gam, T, K, P)
    assert compare(batch, got, oracle_batch(batch, gam, T, K, P), gam, T) <= 1
    assert (got["n_acc"] == 0).all() and (got["n_out"] == 1).all()
    T[:] = 0.0  # every request greedy
    gam[:] = 3
    got = run_per_request(batch, gam, T, K, P)
    assert compare(batch, got, oracle_batch(batch, gam, T, K, P), gam, T) == 0


def test_settings_out_of_range_flag_only_their_request():
    batch, gam, T, K, P = mixed_batch(8, 3, 512, "f32", 5, temps=[1.0], top_ks=[0], top_ps=[0.0])
    gam[1] = 4            # above gamma
    T[3] = -1.0           # negative temperature
    K[5] = -2             # negative top-k
    P[6] = np.float32("nan")
    got = run_per_request(batch, gam, T, K, P)
    for b in (1, 3, 5, 6):
        assert got["n_out"][b] == 0 and int(got["flags"][b]) & O.FLAG_BAD_INPUT, b
    good = [b for b in range(8) if b not in (1, 3, 5, 6)]
    res = oracle_batch(batch, np.where(np.isin(np.arange(8), good), gam, 0), np.abs(T), np.abs(K),
                       np.nan_to_num(P))
    for b in good:
        r = res[b]
        if not r.boundary:
            assert list(got["out_tokens"][b][:got["n_out"][b]]) == r.tokens, b


@pytest.mark.parametrize("case", [
    # (B, gamma, V, dtype, T, top_p): the nucleus over the full vocabulary
    (24, 3, 128256, "bf16", 0.8, 0.9),
    (16, 4, 50000, "f32", 1.0, 0.5),
    (32, 2, 4096, "bf16", 1.2, 0.999),
])
def test_top_p_over_the_full_vocabulary(case):
    B, g, V, dt, T, tp = case
    spec = W.ChainSpec(f"t B={B} g={g} V={V}", B=B, gamma=g, V=V, dtype=dt, target_sigma=3.0,
                       temperature=T, top_k=0, draft_sigma=1.0)
    batch = W.make_chain(spec, seed=B + V)
    tp = float(np.float32(tp))
    dev = "cuda"
    out = api.verify_chain(batch.target.to(dev), torch.from_numpy(batch.draft_tokens).to(dev),
                           gamma=g, temperature=T, draft=batch.draft.to(dev),
                           uniforms=torch.from_numpy(batch.uniforms).to(dev), top_k=0, top_p=tp)
    torch.cuda.synchronize()
    got = {k: v.cpu().numpy() for k, v in vars(out).items() if v is not None}
    boundary = 0
    for b in range(B):
        r = O.verify_chain_sampled(batch.target_f64(b), batch.draft_f64(b), batch.draft_tokens[b],
                                   batch.uniforms[b].astype(np.float64), T, 0, top_p=tp)
        assert np.abs(got["accept_prob"][b] - r.accept_prob).max() <= PROB_TOL, b
        if r.boundary:
            boundary += 1
            continue
        n = int(got["n_out"][b])
        assert int(got["n_acc"][b]) == r.n_acc and n == r.n_out, (b, got["n_acc"][b], r.n_acc)
        assert list(got["out_tokens"][b][:n]) == r.tokens, b
    assert boundary <= max(1, B // 100)
