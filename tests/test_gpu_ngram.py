"""GPU parity of the n-gram (prompt-lookup) drafter against the oracle,
bit-exact, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle as O
from speculative_decoding_verification_37_gb300 import api
from speculative_decoding_verification_37_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def check(hist, lens, gamma, nmin, nmax, out, rows=None):
    for r in (range(len(lens)) if rows is None else rows):
        L = int(lens[r])
        want = O.ngram_draft(hist[r, :max(L, 0)].tolist(), nmin, nmax, gamma)
        n = int(out.n_draft[r])
        got = out.draft_tokens[r].tolist()
        assert n == len(want.tokens), (r, n, want)
        assert got[:n] == want.tokens and all(x == -1 for x in got[n:]), (r, got, want)
        assert int(out.match_n[r]) == want.n and int(out.match_start[r]) == want.start, r


def run(hist, lens, gamma, nmin, nmax):
    out = api.ngram_draft(torch.from_numpy(hist).cuda(), torch.from_numpy(lens).cuda(), gamma=gamma,
                          n_min=nmin, n_max=nmax)
    torch.cuda.synchronize()
    return type(out)(**{k: v.cpu() for k, v in vars(out).items()})


@pytest.mark.parametrize("vocab,max_len,gamma,nmin,nmax", [
    (8, 300, 5, 1, 3),        # small vocabulary: many matches, ties between starts
    (50, 2000, 8, 2, 4),
    (128256, 4096, 8, 1, 4),  # the planted copies are the matches
    (128256, 4096, 16, 3, 64),
    (3, 777, 0, 1, 2),        # gamma 0: only the match is reported
])
def test_matches_oracle(vocab, max_len, gamma, nmin, nmax):
    spec = W.HistorySpec("t", B=48, max_len=max_len, vocab=vocab, gamma=gamma, n_min=nmin, n_max=nmax)
    hist, lens = W.make_histories(spec, seed=vocab + max_len)
    out = run(hist, lens, gamma, nmin, nmax)
    check(hist, lens, gamma, nmin, nmax, out)


def test_short_bad_and_strided_histories():
    hist = np.full((6, 40), -1, dtype=np.int32)
    rows = [[], [7], [7, 7], [1, 2, 3, 1, 2], list(range(40)), [5, 6, 5, 6, 5]]
    for r, h in enumerate(rows):
        hist[r, :len(h)] = h
    lens = np.array([len(h) for h in rows], dtype=np.int32)
    out = run(hist, lens, 4, 1, 3)
    check(hist, lens, 4, 1, 3, out)
    # a wider buffer: every row starts at a stride of 53
    wide = torch.full((6, 53), 9, dtype=torch.int32)
    wide[:, :40] = torch.from_numpy(hist)
    out2 = api.ngram_draft(wide.cuda()[:, :40], torch.from_numpy(lens).cuda(), gamma=4, n_min=1, n_max=3)
    torch.cuda.synchronize()
    assert torch.equal(out2.draft_tokens.cpu(), out.draft_tokens) and torch.equal(out2.n_draft.cpu(), out.n_draft)
    # a length outside [0, stride] flags that request only
    bad = torch.from_numpy(np.array([5, -1, 41, 3, 40, 2], dtype=np.int32)).cuda()
    out3 = api.ngram_draft(torch.from_numpy(hist).cuda(), bad, gamma=4, n_min=1, n_max=3)
    torch.cuda.synchronize()
    f = out3.flags.cpu().tolist()
    assert f[1] and f[2] and not f[0] and not f[3] and not f[4]
    assert int(out3.n_draft[1]) == 0 and int(out3.n_draft[2]) == 0


def test_large_batch_sampled_requests():
    """The benchmark's batch (1,024 histories of up to 32,768 tokens): every
    request's draft length agrees with the host's rules, and 24 sampled
    requests match the oracle exactly."""
    spec = W.NGRAM_SPEC
    hist, lens = W.make_histories(spec, seed=3)
    out = run(hist, lens, spec.gamma, spec.n_min, spec.n_max)
    n = out.n_draft.numpy()
    assert ((n >= 0) & (n <= spec.gamma)).all() and (out.match_n.numpy() > 0).mean() > 0.9
    rng = np.random.default_rng(0)
    check(hist, lens, spec.gamma, spec.n_min, spec.n_max, out, rows=rng.choice(spec.B, 24, replace=False))
