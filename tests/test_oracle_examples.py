"""Pins of the oracle's row transform, acceptance test and residual against the
pages' printed examples, textbook routines and identities (CPU only)."""
import numpy as np
import pytest
import scipy.special

from conftest import golden
import oracle as O


def logits_of(p):
    """Logits whose temperature-1 softmax is p (zero probabilities -> -inf)."""
    p = np.asarray(p, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.log(p)


# --- the pages' worked examples -----------------------------------------------------
def test_two_token_example_acceptance_and_output():
    g = golden("two_token_example.json")
    q, p = np.array(g["q"]), np.array(g["p"])
    tgt = np.stack([logits_of(p), logits_of(p)])          # p_1 and a bonus row
    drf = logits_of(q)[None, :]
    out = np.zeros(2)
    accepted = np.zeros(2)
    for d in (0, 1):
        # acceptance probability the oracle reports for this draft token
        r = O.verify_chain_sampled(tgt, drf, [d], [0.0, 0.5], 1.0)
        assert r.accept_prob[0] == pytest.approx(g["accept"][d], abs=1e-12)
        a = g["accept"][d]
        # accept region [0, a): evaluate inside it; reject region [a, 1)
        for u0, w in ((a / 2, a), ((1 + a) / 2, 1 - a)):
            if w == 0:
                continue
            # the final uniform is spread over the whole unit interval
            for uf in np.linspace(0.005, 0.995, 100):
                rr = O.verify_chain_sampled(tgt, drf, [d], [u0, uf], 1.0)
                out[rr.tokens[0]] += q[d] * w / 100
                if rr.n_acc == 1:
                    accepted[d] += q[d] * w / 100
    np.testing.assert_allclose(accepted, g["accepted_mass"], atol=1e-12)
    assert 1 - accepted.sum() == pytest.approx(g["reject_mass"], abs=1e-12)
    np.testing.assert_allclose(out, g["output"], atol=1e-12)


def test_three_token_example():
    g = golden("three_token_example.json")
    q, p = np.array(g["q"]), np.array(g["p"])
    tgt = np.stack([logits_of(p), logits_of(p)])
    drf = logits_of(q)[None, :]
    for d in range(3):
        r = O.verify_chain_sampled(tgt, drf, [d], [0.0, 0.5], 1.0)
        assert round(r.accept_prob[0], g["accept_decimals"]) == pytest.approx(g["accept"][d])
        # Z = sum max(0, p - q) is the rejection rate, 1 - total acceptance
        assert r.residual_mass[0] == pytest.approx(g["reject_rate"], abs=1e-12)
        assert 1 - r.residual_mass[0] == pytest.approx(g["total_acceptance"], abs=1e-12)
    # residual draw after a rejection of token 0 (the only token with a < 1)
    a0 = p[0] / q[0]
    seen = np.zeros(3)
    grid = np.linspace(0.0025, 0.9975, 200)
    for uf in grid:
        r = O.verify_chain_sampled(tgt, drf, [0], [(1 + a0) / 2, uf], 1.0)
        assert r.n_acc == 0
        seen[r.tokens[0]] += 1 / len(grid)
    np.testing.assert_allclose(seen, g["residual_normalised"], atol=1e-12)
    # output distribution: accepted mass min(p, q) plus the rejection mass times the residual
    out = np.zeros(3)
    for d in range(3):
        a = min(1.0, p[d] / q[d])
        for u0, w in ((a / 2, a), ((1 + a) / 2, 1 - a)):
            if w <= 0:
                continue
            for uf in grid:
                r = O.verify_chain_sampled(tgt, drf, [d], [u0, uf], 1.0)
                out[r.tokens[0]] += q[d] * w / len(grid)
    np.testing.assert_allclose(out, g["output"], atol=1e-12)


# --- rejection mass = total variation (10.6 §10.6.1) ---------------------------------
def test_residual_mass_is_total_variation():
    rng = np.random.default_rng(11)
    for _ in range(50):
        V = int(rng.integers(2, 40))
        T = float(rng.choice([0.5, 1.0, 2.0]))
        k = int(rng.choice([0, 1, 3, V]))
        lt, ld = rng.normal(0, 2, (2, V)), rng.normal(0, 2, (1, V))
        r = O.verify_chain_sampled(lt, ld, [0], [0.5, 0.5], T, k)
        p = O.transform_probs(lt[0], T, k)
        q = O.transform_probs(ld[0], T, k)
        tv = 0.5 * np.abs(p - q).sum()
        assert r.residual_mass[0] == pytest.approx(tv, abs=1e-12)
        assert r.residual_mass[0] == pytest.approx(1 - np.minimum(p, q).sum(), abs=1e-12)


# --- row transform ------------------------------------------------------------------
def test_softmax_matches_scipy_at_temperature_one():
    rng = np.random.default_rng(3)
    for V in (1, 2, 7, 1000):
        x = rng.normal(0, 3, V)
        np.testing.assert_allclose(O.transform_probs(x, 1.0, 0), scipy.special.softmax(x),
                                   rtol=1e-12, atol=1e-15)


def test_temperature_scaling_invariance():
    rng = np.random.default_rng(4)
    x = rng.normal(0, 2, 257)
    for T, c in ((0.7, 3.0), (1.0, 0.25), (2.0, 5.0)):
        for k in (0, 5, 50):
            np.testing.assert_allclose(O.transform_probs(c * x, T * c, k),
                                       O.transform_probs(x, T, k), rtol=1e-12, atol=1e-15)


def _topk_by_counting(x, k):
    """Token i is kept iff fewer than k logits are strictly larger than x_i."""
    x = np.asarray(x)
    if k <= 0 or k >= len(x):
        return np.ones(len(x), bool)
    return np.array([(x > v).sum() < k for v in x])


def test_topk_keeps_every_tie_at_threshold():
    rng = np.random.default_rng(5)
    for _ in range(200):
        V = int(rng.integers(1, 30))
        x = rng.integers(-3, 4, V).astype(np.float64)       # heavy ties by construction
        k = int(rng.integers(0, V + 2))
        keep = O.kept_set(x, k)
        np.testing.assert_array_equal(keep, _topk_by_counting(x, k))
        if 0 < k < V:
            assert keep.sum() >= k
        p = O.transform_probs(x, 1.3, k)
        assert np.all(p[~keep] == 0) and np.all(p[keep] > 0)
        assert p.sum() == pytest.approx(1.0, abs=1e-14)


def test_topk_example_with_planted_ties():
    x = np.array([1.0, 5.0, 3.0, 5.0, 3.0, 3.0, 0.0])
    # k = 2: the two 5.0s; k = 3: threshold 3.0, so all three 3.0s join (5 kept)
    assert O.kept_set(x, 2).tolist() == [False, True, False, True, False, False, False]
    assert O.kept_set(x, 3).tolist() == [False, True, True, True, True, True, False]
    p = O.transform_probs(x, 1.0, 3)
    e = np.exp(np.array([5.0, 3.0, 5.0, 3.0, 3.0]) - 5.0)
    np.testing.assert_allclose(p[[1, 2, 3, 4, 5]], e / e.sum(), rtol=1e-14)


def test_all_minus_inf_row_is_flagged():
    x = np.full(5, -np.inf)
    assert O.transform_probs(x, 1.0, 0) is None
    r = O.verify_chain_sampled(np.stack([x, x]), np.zeros((1, 5)), [0], [0.1, 0.1], 1.0)
    assert r.flags & O.FLAG_BAD_ROW


# --- acceptance boundary cases (glossary, 精确接受与校正分布) ---------------------------
def test_q_zero_limits():
    assert O.acceptance_probability(0.3, 0.0) == 1.0
    assert O.acceptance_probability(0.0, 0.0) == 0.0
    assert O.acceptance_probability(0.2, 0.4) == 0.5
    assert O.acceptance_probability(0.5, 0.4) == 1.0


def test_accept_iff_u_below_a():
    p = np.array([0.25, 0.75])
    q = np.array([0.5, 0.5])
    tgt = np.stack([logits_of(p), logits_of(p)])
    drf = logits_of(q)[None]
    a = 0.5
    assert O.verify_chain_sampled(tgt, drf, [0], [a - 1e-9, 0.5], 1.0).n_acc == 1
    assert O.verify_chain_sampled(tgt, drf, [0], [a, 0.5], 1.0).n_acc == 0      # u == a rejects
    # a == 1 always accepts, even at the largest uniform on the 2^-24 grid
    assert O.verify_chain_sampled(tgt, drf, [1], [1 - 2.0 ** -24, 0.5], 1.0).n_acc == 1


def test_out_of_range_draft_token_is_flagged():
    x = np.zeros((2, 4))
    r = O.verify_chain_sampled(x, x[:1], [4], [0.1, 0.1], 1.0)
    assert r.flags & O.FLAG_BAD_INPUT and r.n_out == 0
    r = O.verify_chain_greedy(x, [-1])
    assert r.flags & O.FLAG_BAD_INPUT and r.n_out == 0


# --- residual-mass fallback ---------------------------------------------------------
def test_fallback_draws_from_target_when_residual_mass_vanishes():
    V = 6
    x32 = np.array([0.1, 0.7, -0.3, 0.2, 0.05, -1.0], dtype=np.float32)
    y32 = x32.copy()
    y32[1] = np.nextafter(y32[1], np.float32(2.0))   # q = p with one fp32 logit moved one ulp
    x, y = x32.astype(np.float64), y32.astype(np.float64)
    tgt = np.stack([x, x])
    drf = y[None]
    p = O.transform_probs(x, 1.0, 0)
    q = O.transform_probs(y, 1.0, 0)
    assert p[1] < q[1]
    a = p[1] / q[1]
    assert a < 1
    Z = np.maximum(p - q, 0).sum()
    assert 0 < Z <= O.DEFAULT_EPS
    cdf = np.concatenate([[0.0], np.cumsum(p)])
    for i in range(V):
        uf = 0.5 * (cdf[i] + cdf[i + 1])
        r = O.verify_chain_sampled(tgt, drf, [1], [(1 + a) / 2, uf], 1.0)
        assert r.n_acc == 0 and r.flags & O.FLAG_FALLBACK
        assert r.tokens == [i]


def test_inverse_cdf_never_picks_zero_weight():
    w = np.array([0.0, 0.2, 0.0, 0.0, 0.3, 0.0])
    for u in np.linspace(0, 1 - 1e-12, 101):
        assert w[O.inverse_cdf(w, u).token] > 0
    assert O.inverse_cdf(w, 0.0).token == 1
    assert O.inverse_cdf(w, 0.39).token == 1
    assert O.inverse_cdf(w, 0.41).token == 4


# --- greedy is the T -> 0 special case (10.6 §10.6.1) ----------------------------------
def test_greedy_equals_sampled_rule_with_one_hot_rows():
    rng = np.random.default_rng(9)
    for _ in range(100):
        V = int(rng.integers(1, 12))
        gamma = int(rng.integers(0, 4))
        tgt = rng.integers(-2, 3, (gamma + 1, V)).astype(np.float64)   # ties on purpose
        g = [int(np.flatnonzero(r == r.max())[0]) for r in tgt]
        d = rng.integers(0, V, gamma)
        d = np.where(rng.random(gamma) < 0.6, g[:gamma], d)
        greedy = O.verify_chain_greedy(tgt, d)
        one_hot_t = np.where(np.arange(V)[None] == np.array(g)[:, None], 0.0, -np.inf)
        one_hot_d = np.where(np.arange(V)[None] == d[:, None], 0.0, -np.inf)
        u = rng.random(gamma + 1)
        sampled = O.verify_chain_sampled(one_hot_t, one_hot_d.reshape(gamma, V), d, u, 1.0)
        assert greedy.tokens == sampled.tokens and greedy.n_acc == sampled.n_acc


def test_greedy_lowest_index_tie_break():
    t = np.array([[1.0, 3.0, 3.0, 0.0], [2.0, 2.0, 2.0, 2.0]])
    assert O.verify_chain_greedy(t, [2]).tokens == [1]          # tie 1 vs 2 -> 1 wins
    assert O.verify_chain_greedy(t, [1]).tokens == [1, 0]       # accepted, bonus argmax 0


# --- round termination: EOS and the length limit (KV4 §5) ---------------------------
def _round(tokens, n_acc):
    return O.ChainResult(n_acc=n_acc, tokens=list(tokens))


def test_truncate_round_hand_cases():
    r = _round([11, 12, 13, 99], 3)                 # three accepted drafts + a drawn token
    t = O.truncate_round(r)
    assert t.tokens == [11, 12, 13, 99] and t.n_acc == 3 and t.flags == 0
    t = O.truncate_round(r, eos=12)                 # EOS among the accepted drafts
    assert t.tokens == [11, 12] and t.n_acc == 2 and t.flags == O.FLAG_EOS
    t = O.truncate_round(r, eos=99)                 # EOS is the drawn token: nothing cut
    assert t.tokens == [11, 12, 13, 99] and t.n_acc == 3 and t.flags == O.FLAG_EOS
    t = O.truncate_round(r, eos=7)                  # no EOS in the round
    assert t.tokens == [11, 12, 13, 99] and t.flags == 0
    t = O.truncate_round(r, max_new=2)              # two tokens left before the limit
    assert t.tokens == [11, 12] and t.n_acc == 2 and t.flags == O.FLAG_LIMIT
    t = O.truncate_round(r, max_new=4)              # the limit is not reached
    assert t.tokens == [11, 12, 13, 99] and t.flags == 0
    t = O.truncate_round(r, max_new=0)              # finished already
    assert t.tokens == [] and t.n_acc == 0 and t.flags == O.FLAG_LIMIT
    t = O.truncate_round(r, eos=13, max_new=2)      # the limit cuts before the EOS
    assert t.tokens == [11, 12] and t.flags == O.FLAG_LIMIT
    t = O.truncate_round(r, eos=12, max_new=3)      # the EOS cuts first
    assert t.tokens == [11, 12] and t.flags == O.FLAG_EOS
    t = O.truncate_round(_round([5], 0), eos=5)     # a rejection at once, the drawn token is EOS
    assert t.tokens == [5] and t.n_acc == 0 and t.flags == O.FLAG_EOS
    bad = O.ChainResult(flags=O.FLAG_BAD_INPUT)
    assert O.truncate_round(bad, eos=1, max_new=0) is bad


def test_truncate_round_properties():
    """On random rounds: the result is the longest prefix of the round that
    has no EOS before its last token and fits the limit, and n_acc counts the
    drafts in it."""
    rng = np.random.default_rng(3)
    for _ in range(2000):
        n_acc = int(rng.integers(0, 6))
        toks = rng.integers(0, 6, n_acc + 1).tolist()
        eos = int(rng.integers(0, 7)) if rng.random() < 0.8 else None
        lim = int(rng.integers(-1, 8)) if rng.random() < 0.6 else None
        t = O.truncate_round(_round(toks, n_acc), eos, lim)
        L = len(t.tokens)
        assert t.tokens == toks[:L]
        assert eos is None or eos not in t.tokens[:-1]
        assert lim is None or L <= max(lim, 0)
        longer = toks[:L + 1]
        if L < len(toks):
            assert (eos is not None and eos in longer[:-1]) or (lim is not None and L + 1 > max(lim, 0))
        assert t.n_acc == min(n_acc, L)


# --- top-p (nucleus) transform: a reading of KV4 §4 -----------------------------------
def test_top_p_hand_cases():
    p = np.array([0.5, 0.125, 0.25, 0.125])           # dyadic: sums are exact
    assert O.kept_set_top_p(p, 0.5).tolist() == [True, False, False, False]
    assert O.kept_set_top_p(p, 0.75).tolist() == [True, False, True, False]
    # 0.76 needs a third token; the fourth is tied with it and is kept too
    assert O.kept_set_top_p(p, 0.76).tolist() == [True, True, True, True]
    assert O.kept_set_top_p(p, 1.0).all() and O.kept_set_top_p(p, 1e-9).tolist() == [True, False, False, False]


def test_top_p_after_temperature_and_top_k():
    x = np.array([2.0, 1.0, 0.0, -1.0])
    # T = 1: the top token has 0.64 < 0.85, so two are kept; T = 0.5 sharpens
    # the row to 0.87 for the top token, which alone reaches 0.85
    assert (O.transform_probs(x, 1.0, 0, 0.85) > 0).tolist() == [True, True, False, False]
    assert (O.transform_probs(x, 0.5, 0, 0.85) > 0).tolist() == [True, False, False, False]
    # top-k first: with k = 2 the two kept tokens renormalise to 0.73 / 0.27,
    # so top-p 0.7 keeps one of them
    assert (O.transform_probs(x, 1.0, 2, 0.7) > 0).tolist() == [True, False, False, False]
    p = O.transform_probs(x, 1.0, 0, 0.85)
    assert p.sum() == pytest.approx(1.0) and p[0] / p[1] == pytest.approx(np.e)


def test_top_p_properties_random():
    """Any row: the kept mass reaches top_p, dropping the least probable kept
    tie group falls short of it, and every token more probable than a kept
    one is kept."""
    rng = np.random.default_rng(11)
    for _ in range(500):
        V = int(rng.integers(1, 30))
        p = rng.dirichlet(np.ones(V) * rng.choice([0.2, 1.0, 5.0]))
        if rng.random() < 0.3:
            p = np.round(p * 8) / 8 + 1e-3                 # planted ties
            p /= p.sum()
        tp = float(rng.uniform(0.01, 0.999))
        keep = O.kept_set_top_p(p, tp)
        assert p[keep].sum() >= tp - 1e-12
        low = p[keep].min()
        assert p[keep & (p > low)].sum() < tp
        assert not (~keep & (p > low)).any()


def test_sampled_round_with_top_p_keeps_losslessness():
    """With the nucleus transform on both sides, the round's output
    distribution is still the target's (transformed) distribution: the
    brute-force enumeration of every draft and uniform region."""
    rng = np.random.default_rng(2)
    V, T, tp = 4, 1.0, 0.8
    tgt = rng.normal(0, 1, (2, V))
    drf = rng.normal(0, 1, (1, V))
    p = O.transform_probs(tgt[0], T, 0, tp)
    q = O.transform_probs(drf[0], T, 0, tp)
    out = np.zeros(V)
    grid = (np.arange(160) + 0.5) / 160
    for d in range(V):
        if q[d] == 0:
            continue
        for u0 in grid:
            for u1 in grid:
                r = O.verify_chain_sampled(tgt, drf, np.array([d]), np.array([u0, u1]), T, 0,
                                           top_p=tp)
                out[r.tokens[0]] += q[d] / grid.size ** 2
    assert np.abs(out - p).max() < 1e-2


# --- per-request gamma / temperature / top-k / top-p (batch layout reading) ----------
def test_batch_with_per_request_settings_equals_single_requests():
    """Each request of a padded batch gives exactly the single-request result
    on its own slice; a request with gamma_b < gamma_max draws its bonus from
    target row gamma_b with uniform u[gamma_b]."""
    rng = np.random.default_rng(21)
    B, gmax, V = 6, 4, 12
    tgt = rng.normal(0, 2, (B, gmax + 1, V))
    drf = tgt[:, :gmax] + rng.normal(0, 0.5, (B, gmax, V))
    tok = rng.integers(0, V, (B, gmax))
    u = rng.random((B, gmax + 1))
    gammas = [4, 0, 2, 3, 1, 4]
    temps = [1.0, 0.7, 0.0, 1.3, 1.0, 0.5]
    ks = [0, 3, 0, 5, 0, 4]
    ps = [1.0, 1.0, 1.0, 0.8, 0.5, 0.9]
    res = O.verify_chain_batch(tgt, drf, tok, u, gammas, temps, ks, ps)
    for b in range(B):
        g = gammas[b]
        if temps[b] == 0.0:
            want = O.verify_chain_greedy(tgt[b, :g + 1], tok[b, :g])
        else:
            want = O.verify_chain_sampled(tgt[b, :g + 1], drf[b, :g], tok[b, :g],
                                          np.r_[u[b, :g], u[b, g]], temps[b], ks[b], top_p=ps[b])
        assert res[b].tokens == want.tokens and res[b].n_acc == want.n_acc
        assert 1 <= res[b].n_out <= g + 1
    # gamma 0: only the bonus draw, from target row 0 with u[0]
    p0 = O.transform_probs(tgt[1, 0], 0.7, 3)
    assert p0[res[1].tokens[0]] > 0 and res[1].n_acc == 0
