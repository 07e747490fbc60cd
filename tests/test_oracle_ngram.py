"""Pins of the n-gram / prompt-lookup drafter oracle (CPU).

The pages print no worked example, so the oracle is pinned by hand-built
cases whose answer follows from the definition, by an independent brute-force
formulation (every occurrence of every n-gram listed by a dictionary), and by
properties that any correct answer has."""
import random
from collections import defaultdict

import pytest

from oracle import ngram_draft


@pytest.mark.parametrize("hist,nmin,nmax,g,want,n,start", [
    # the trailing 2-gram [5, 6] occurred at 0; the 3-gram [8, 5, 6] did not
    ([5, 6, 7, 8, 5, 6], 1, 3, 3, [7, 8, 5], 2, 0),
    # the most recent earlier occurrence of [1, 2] starts at 3, not 0
    ([1, 2, 9, 1, 2, 8, 1, 2], 2, 2, 3, [8, 1, 2], 2, 3),
    # a longer match wins over a more recent shorter one
    ([7, 1, 2, 4, 0, 2, 9, 7, 1, 2], 1, 3, 2, [4, 0], 3, 0),
    # the continuation stops at the end of the history
    ([4, 4], 1, 2, 5, [4], 1, 0),
    # the occurrence may overlap the trailing n-gram: [3,3,3] in [3,3,3,3]
    ([3, 3, 3, 3], 1, 3, 4, [3], 3, 0),
    # nothing matches
    ([1, 2, 3, 4], 1, 3, 4, [], 0, -1),
    # below n_min nothing counts
    ([1, 2, 9, 2], 2, 3, 2, [], 0, -1),
    # gamma 0: the match is still reported
    ([5, 6, 5], 1, 2, 0, [], 1, 0),
    # a one-token history has no earlier window
    ([7], 1, 3, 2, [], 0, -1),
])
def test_hand_cases(hist, nmin, nmax, g, want, n, start):
    r = ngram_draft(hist, nmin, nmax, g)
    assert (r.tokens, r.n, r.start) == (want, n, start)


def brute(h, nmin, nmax, g):
    """Independent formulation: list every occurrence of every n-gram, then
    take the longest n whose trailing n-gram has an occurrence starting
    before it, and the largest such start."""
    L = len(h)
    occ = defaultdict(list)
    for n in range(1, L + 1):
        for j in range(0, L - n + 1):
            occ[tuple(h[j:j + n])].append(j)
    for n in sorted(range(max(nmin, 1), nmax + 1), reverse=True):
        if n > L - 1:
            continue
        starts = [j for j in occ[tuple(h[L - n:])] if j < L - n]
        if starts:
            j = max(starts)
            return h[j + n:j + n + g], n, j
    return [], 0, -1


def test_matches_brute_force_on_random_histories():
    rng = random.Random(11)
    for _ in range(600):
        L = rng.randint(1, 40)
        vocab = rng.randint(2, 6)
        h = [rng.randrange(vocab) for _ in range(L)]
        nmin = rng.randint(1, 3)
        nmax = rng.randint(nmin, 6)
        g = rng.randint(0, 6)
        r = ngram_draft(h, nmin, nmax, g)
        assert (r.tokens, r.n, r.start) == brute(h, nmin, nmax, g), (h, nmin, nmax, g)


def test_properties():
    rng = random.Random(5)
    for _ in range(300):
        L = rng.randint(2, 60)
        h = [rng.randrange(4) for _ in range(L)]
        nmin, nmax, g = 1, rng.randint(1, 5), rng.randint(1, 8)
        r = ngram_draft(h, nmin, nmax, g)
        if r.n == 0:
            # no window of any allowed length matches the trailing n-gram
            for n in range(nmin, min(nmax, L - 1) + 1):
                assert all(h[j:j + n] != h[L - n:] for j in range(L - n))
            continue
        n, j = r.n, r.start
        assert h[j:j + n] == h[L - n:] and j < L - n           # an earlier occurrence
        assert r.tokens == h[j + n:j + n + g]                   # the tokens after it
        assert len(r.tokens) == min(g, L - j - n)               # never past the end
        for n2 in range(n + 1, min(nmax, L - 1) + 1):           # nothing longer matches
            assert all(h[j2:j2 + n2] != h[L - n2:] for j2 in range(L - n2))
        assert all(h[j2:j2 + n] != h[L - n:] for j2 in range(j + 1, L - n))  # nothing more recent
