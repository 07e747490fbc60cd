"""Exact and statistical pins of the oracle's chain round (CPU only).

* Brute force (V <= 4, gamma <= 3): every draft sequence, every accept/reject
  outcome and every draw is enumerated; the oracle is evaluated at interior
  points of each outcome's uniform region, with the regions derived here from
  min(1, p/q) and the residual norm(max(0, p - q)).  The resulting exact
  output distribution must equal the target's (10.6 §10.6.1 losslessness),
  for fixed rows and for the glossary page's first-order vocab-4 chain over
  concatenated rounds.
* Closed form E[tokens/round] = (1 - a^(g+1)) / (1 - a) (10.6 §10.6.2), exact
  via enumeration and statistically on simulated rounds; Table 10-16 values.
* The glossary page's empirical experiment (vocab 4, k = 4, 1e5 tokens).
"""
import itertools
from collections import defaultdict
from functools import lru_cache

import numpy as np
import pytest

from conftest import golden
import oracle as O


def logits_of(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, dtype=np.float64))


def interior_points(lo, hi):
    """Three points strictly inside [lo, hi)."""
    w = hi - lo
    return [lo + 0.1 * w, lo + 0.5 * w, lo + 0.9 * w]


def enumerate_round(p_rows_of, q_rows_of, V, gamma):
    """Exact distribution of the oracle's emitted token tuple for one round.

    p_rows_of(d) -> [gamma+1, V] target probs for draft sequence d;
    q_rows_of(prefix) -> draft probs of the next position given the drafted prefix.
    Returns {tokens tuple: probability}; asserts that the oracle's outcome at
    every interior point is the one the region implies.
    """
    dist = defaultdict(float)
    for d in itertools.product(range(V), repeat=gamma):
        Q = [q_rows_of(d[:k]) for k in range(gamma)]
        w_d = float(np.prod([Q[k][d[k]] for k in range(gamma)])) if gamma else 1.0
        if w_d == 0.0:
            continue
        P = p_rows_of(d)
        a = [min(1.0, P[k][d[k]] / Q[k][d[k]]) for k in range(gamma)]
        tgt = np.stack([logits_of(r) for r in P])
        drf = np.stack([logits_of(r) for r in Q]) if gamma else np.zeros((0, V))
        for j in range(gamma + 1):
            pr = float(np.prod(a[:j])) * ((1.0 - a[j]) if j < gamma else 1.0)
            if pr <= 0.0:
                continue
            if j < gamma:
                w = np.maximum(np.asarray(P[j]) - np.asarray(Q[j]), 0.0)
            else:
                w = np.asarray(P[gamma], dtype=np.float64)
            w = w / w.sum()
            cdf = np.concatenate([[0.0], np.cumsum(w)])
            for x in range(V):
                if w[x] == 0.0:
                    continue
                for uf in interior_points(cdf[x], cdf[x + 1]):
                    u = [0.5 * a[k] for k in range(j)]
                    if j < gamma:
                        u.append(0.5 * (1.0 + a[j]))
                    u += [0.5] * (gamma - len(u))
                    u.append(uf)
                    r = O.verify_chain_sampled(tgt, drf, list(d), u, 1.0)
                    assert r.n_acc == j
                    assert r.tokens == list(d[:j]) + [x]
                dist[tuple(d[:j]) + (x,)] += w_d * pr * w[x]
    return dist


def random_probs(rng, V, zero_frac=0.25):
    p = rng.random(V) + 0.05
    p[rng.random(V) < zero_frac] = 0.0
    if p.sum() == 0:
        p[rng.integers(V)] = 1.0
    return p / p.sum()


@pytest.mark.parametrize("seed", range(6))
def test_bruteforce_fixed_rows_lossless_and_expected_length(seed):
    rng = np.random.default_rng(100 + seed)
    V = int(rng.integers(2, 5))
    gamma = int(rng.integers(1, 4))
    P = [random_probs(rng, V) for _ in range(gamma + 1)]
    Q = [random_probs(rng, V) for _ in range(gamma)]
    dist = enumerate_round(lambda d: P, lambda prefix: Q[len(prefix)], V, gamma)
    assert sum(dist.values()) == pytest.approx(1.0, abs=1e-12)
    first = np.zeros(V)
    for toks, pr in dist.items():
        first[toks[0]] += pr
    np.testing.assert_allclose(first, P[0], atol=1e-12)        # first token ~ p_1
    # E[tokens/round] = sum_{k=0..gamma} prod_{j<=k} alpha_j, alpha_j = sum min(p_j, q_j)
    alpha = [np.minimum(P[k], Q[k]).sum() for k in range(gamma)]
    expect = sum(np.prod(alpha[:k]) for k in range(gamma + 1))
    got = sum(len(t) * pr for t, pr in dist.items())
    assert got == pytest.approx(expect, abs=1e-12)


def test_bruteforce_vocab4_chain_concatenated_rounds():
    g = golden("vocab4_chain.json")
    TGT, DRF = np.array(g["TARGET"]), np.array(g["DRAFT"])
    V = 4
    for gamma in (1, 2, 3):
        @lru_cache(maxsize=None)
        def round_dist(state):
            def p_rows(d):
                prev = [state] + list(d)
                return [TGT[prev[k]] for k in range(gamma + 1)]

            def q_row(prefix):
                return DRF[([state] + list(prefix))[-1]]
            return dict(enumerate_round(p_rows, q_row, V, gamma))

        @lru_cache(maxsize=None)
        def stream_prob(state, seq):
            """P(the stream starting after `state` begins with seq)."""
            if not seq:
                return 1.0
            tot = 0.0
            for toks, pr in round_dist(state).items():
                n = min(len(toks), len(seq))
                if toks[:n] != seq[:n]:
                    continue
                tot += pr * (1.0 if n == len(seq) else stream_prob(toks[-1], seq[n:]))
            return tot

        for m in (1, 2, 3, 4):
            for seq in itertools.product(range(V), repeat=m):
                want, prev = 1.0, 0
                for s in seq:
                    want *= TGT[prev, s]
                    prev = s
                assert stream_prob(0, seq) == pytest.approx(want, abs=1e-12)


def test_table_10_16_closed_forms():
    g = golden("table_10_16.json")

    def tokens(a, gm):
        return (1 - a ** (gm + 1)) / (1 - a)

    for row in g["rows"]:
        E = tokens(row["alpha"], row["gamma"])
        assert round(E, 2) == pytest.approx(row["tokens_per_round"])
        assert round(E / (row["gamma"] * g["c"] + 1), 2) == pytest.approx(row["speedup"])
    w = g["worked"]
    assert round(1 - w["alpha"] ** (w["gamma"] + 1), 3) == pytest.approx(w["one_minus_alpha_pow"])
    assert w["gamma"] * g["c"] + 1 == pytest.approx(w["round_cost"])
    c2 = g["c_0_2"]
    assert round(tokens(c2["alpha"], c2["gamma"]) / (c2["gamma"] * c2["c"] + 1), 2) == c2["speedup"]
    s = g["survival"]
    assert round(s["alpha"] ** 4, 2) == s["k4"] and round(s["alpha"] ** 8, 2) == s["k8"]
    assert 1 / (1 - 0.8) == pytest.approx(g["upper_bound_alpha_0_8"])


@pytest.mark.parametrize("alpha,gamma", [(0.6, 4), (0.8, 4), (0.8, 8)])
def test_simulated_rounds_match_closed_form(alpha, gamma):
    """Rows with sum min(p, q) = alpha at every position: the mean emitted count
    over simulated rounds must be within 4 sigma of (1 - a^(g+1)) / (1 - a)."""
    V = 3
    # p = (alpha, 1 - alpha, 0), q = (1, 0, 0)  ->  sum min(p, q) = alpha
    p = np.array([alpha, 1 - alpha, 0.0])
    q = np.array([1.0, 0.0, 0.0])
    tgt = np.stack([logits_of(p)] * (gamma + 1))
    drf = np.stack([logits_of(q)] * gamma)
    rng = np.random.default_rng(7)
    n = 20000
    counts = np.empty(n)
    for i in range(n):
        u = rng.random(gamma + 1)
        counts[i] = O.verify_chain_sampled(tgt, drf, [0] * gamma, u, 1.0).n_out
    expect = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert abs(counts.mean() - expect) < 4 * counts.std() / np.sqrt(n)


def _exact_vocab4_rates(TGT, DRF, k):
    """Stationary E[accepted drafts per call] and calls per token of the
    vocab-4 chain, by enumerating one round from every start state."""
    S = TGT.shape[0]
    M = np.zeros((S, S))
    e_acc = np.zeros(S)
    e_out = np.zeros(S)
    for s in range(S):
        for d in itertools.product(range(S), repeat=k):
            prev = [s] + list(d)
            w_d = np.prod([DRF[prev[j], d[j]] for j in range(k)])
            a = [min(1.0, TGT[prev[j], d[j]] / DRF[prev[j], d[j]]) for j in range(k)]
            for j in range(k + 1):
                pr = w_d * np.prod(a[:j]) * ((1 - a[j]) if j < k else 1.0)
                if pr == 0:
                    continue
                if j < k:
                    w = np.maximum(TGT[prev[j]] - DRF[prev[j]], 0)
                else:
                    w = TGT[d[-1]] if k else TGT[s]
                w = w / w.sum()
                M[s] += pr * w
                e_acc[s] += pr * j
                e_out[s] += pr * (j + 1)
    evals, evecs = np.linalg.eig(M.T)
    pi = np.real(evecs[:, np.argmin(np.abs(evals - 1))])
    pi = pi / pi.sum()
    return float(pi @ e_acc), float(1.0 / (pi @ e_out))


@pytest.mark.slow
def test_glossary_vocab4_empirical_experiment():
    g = golden("vocab4_chain.json")
    TGT, DRF = np.array(g["TARGET"]), np.array(g["DRAFT"])
    k, length, tol = g["proposal_len"], g["tokens"], g["tolerance"]
    rng = np.random.default_rng(303)
    tl, dl = logits_of(TGT), logits_of(DRF)
    out, calls, accepted = [], 0, 0
    state = g["start_state"]
    while len(out) < length:
        d, prev = [], state
        for _ in range(k):
            t = int(rng.choice(4, p=DRF[prev]))
            d.append(t)
            prev = t
        path = [state] + d
        tgt = np.stack([tl[path[j]] for j in range(k + 1)])
        drf = np.stack([dl[path[j]] for j in range(k)])
        r = O.verify_chain_sampled(tgt, drf, d, rng.random(k + 1), 1.0)
        calls += 1
        accepted += r.n_acc
        out.extend(r.tokens[:length - len(out)])
        state = out[-1]
    counts = np.zeros((4, 4))
    prev = g["start_state"]
    for t in out:
        counts[prev, t] += 1
        prev = t
    freq = counts / counts.sum(1, keepdims=True)
    assert np.abs(freq - TGT).max() < tol
    acc_rate, calls_per_token = _exact_vocab4_rates(TGT, DRF, k)
    # the page's printed figures agree with the exact expectation ...
    assert abs(acc_rate - g["printed"]["mean_accepted_draft_tokens_per_call"]) < 0.03
    assert abs(calls_per_token - g["printed"]["target_calls_per_emitted_token"]) < 0.005
    # ... and so does this simulation
    assert abs(accepted / calls - acc_rate) < 0.03
    assert abs(calls / length - calls_per_token) < 0.005
