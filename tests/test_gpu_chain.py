"""GPU parity of chain verification (sampled and greedy) against the oracle,
through the C ABI, on seeded inputs spanning several slices and ragged tails."""
import dataclasses
import zlib

import numpy as np
import pytest
import torch

import oracle as O
from parity import ChainTally, compare_chain, run_chain
from speculative_decoding_verification_37_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def spec(B, gamma, V, dtype, T, top_k=0, draft_sigma=1.0, sigma=2.0, zipf=False):
    return W.ChainSpec(f"t B={B} g={gamma} V={V}", B=B, gamma=gamma, V=V, dtype=dtype,
                       target_sigma=sigma, temperature=T, top_k=top_k,
                       draft_sigma=None if T == 0 else draft_sigma, zipf_bias=zipf)


SAMPLED = [
    # (B, gamma, V, dtype, T, top_k)
    (4, 4, 1, "f32", 1.0, 0),
    (3, 2, 5, "f32", 1.0, 0),
    (5, 3, 31, "bf16", 0.5, 0),
    (8, 4, 1024, "f32", 1.0, 0),
    (6, 8, 4099, "bf16", 2.0, 0),
    (4, 4, 70001, "f32", 1.0, 0),      # 5 slices (cluster of 5), ragged last slice
    (4, 4, 70001, "bf16", 0.8, 0),     # 3 slices
    (3, 0, 4099, "f32", 1.0, 0),       # gamma 0: bonus draw only
    (6, 4, 4099, "bf16", 0.8, 5),
    (6, 4, 70001, "bf16", 0.8, 50),
    (6, 3, 70001, "f32", 1.3, 50),
    (5, 4, 1024, "f32", 1.0, 1),
    (5, 4, 31, "bf16", 1.0, 31),       # top-k == V keeps everything
    (16, 2, 257, "f32", 0.7, 16),
]


@pytest.mark.parametrize("case", SAMPLED, ids=lambda c: "-".join(map(str, c)))
def test_sampled_chain_matches_oracle(case):
    B, g, V, dt, T, k = case
    batch = W.make_chain(spec(B, g, V, dt, T, k), seed=zlib.crc32(repr(case).encode()) % 1000)
    gpu = run_chain(batch)
    tally = compare_chain(batch, gpu, range(batch.n))
    assert tally.boundary <= 1


def test_sampled_chain_zipf_topk_config_like():
    s = dataclasses.replace(W.WORKLOADS[2], B=6)
    batch = W.make_chain(s, seed=5)
    compare_chain(batch, run_chain(batch), range(batch.n))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_sampled_chain_misaligned_strided_rows(dt):
    B, g, V = 4, 3, 9001
    batch = W.make_chain(spec(B, g, V, dt, 1.0, 0), seed=21)
    tgt = torch.zeros((B * (g + 1), V + 13), dtype=batch.target.dtype)
    drf = torch.zeros((B * g, V + 7), dtype=batch.draft.dtype)
    tgt[:, 3:3 + V] = batch.target
    drf[:, 5:5 + V] = batch.draft
    gpu = run_chain(batch, target=tgt.cuda()[:, 3:3 + V], draft=drf.cuda()[:, 5:5 + V])
    compare_chain(batch, gpu, range(B))


@pytest.mark.parametrize("dt,layout", [("bf16", "same-phase"), ("f32", "same-phase"),
                                       ("bf16", "phase-mismatch"), ("f32", "phase-mismatch")])
def test_sampled_topk_strided_rows(dt, layout):
    """Top-k rows inside wider buffers: equal 16-byte phases take the bulk
    copies plus scalar heads and tails; unequal phases take the exact path."""
    B, g, V, k = 4, 3, 9001, 20
    batch = W.make_chain(spec(B, g, V, dt, 0.9, k), seed=23)
    width = 9016  # a multiple of 8 elements: every row starts at the same phase
    ot, od = (3, 3) if layout == "same-phase" else (3, 6)
    tgt = torch.zeros((B * (g + 1), width), dtype=batch.target.dtype)
    drf = torch.zeros((B * g, width), dtype=batch.draft.dtype)
    tgt[:, ot:ot + V] = batch.target
    drf[:, od:od + V] = batch.draft
    gpu = run_chain(batch, target=tgt.cuda()[:, ot:ot + V], draft=drf.cuda()[:, od:od + V])
    compare_chain(batch, gpu, range(B))


@pytest.mark.parametrize("dt,k", [("bf16", 5), ("f32", 3), ("bf16", 40)])
def test_sampled_topk_with_heavy_ties(dt, k):
    """Logits on a coarse grid: many ties at the k-th value, all kept."""
    B, g, V = 5, 3, 3000
    batch = W.make_chain(spec(B, g, V, dt, 1.0, k), seed=33)
    batch.target = (torch.round(batch.target.float() * 2) / 2).to(batch.target.dtype)
    batch.draft = (torch.round(batch.draft.float() * 2) / 2).to(batch.draft.dtype)
    compare_chain(batch, run_chain(batch), range(B))


def test_draft_equal_target_and_bad_inputs():
    B, g, V = 6, 3, 5000
    batch = W.make_chain(spec(B, g, V, "f32", 1.0, 0), seed=4)
    # request 0: draft == target -> p == q, a = 1, Z = 0, all accepted, bonus drawn
    batch.draft[0:g] = batch.target[0:g]
    # request 1: an out-of-range draft token; request 2: a row of -inf logits
    batch.draft_tokens[1, 1] = V
    batch.target[2 * (g + 1) + 1] = -float("inf")
    gpu = run_chain(batch)
    compare_chain(batch, gpu, range(B))
    assert gpu["n_acc"][0] == g and gpu["residual_mass"][0].max() == 0.0
    assert gpu["flags"][1] & O.FLAG_BAD_INPUT and gpu["n_out"][1] == 0
    assert gpu["flags"][2] & O.FLAG_BAD_ROW and gpu["n_out"][2] == 0


def test_fallback_when_residual_mass_vanishes():
    """Draft = target except one low-probability token's logit raised by 5e-5:
    the residual mass (about p(d) * 5e-5) is far below eps, a = p(d)/q(d) is
    about 1 - 5e-5, and u is put halfway between a and 1, so the round
    rejects and the draw comes from p itself."""
    B, g, V = 8, 1, 600
    batch = W.make_chain(spec(B, g, V, "f32", 1.0, 0), seed=8)
    for b in range(B):
        row = batch.target[b * 2].clone()
        p = O.transform_probs(row.double().numpy(), 1.0, 0)
        d = int(np.argmin(np.abs(p - 0.002)))
        batch.draft[b] = row
        batch.draft[b, d] = row[d] + 5e-5
        batch.draft_tokens[b, 0] = d
        q = O.transform_probs(batch.draft_f64(b)[0], 1.0, 0)
        a = p[d] / q[d]
        batch.uniforms[b, 0] = np.float32(a + (1 - a) / 2)
        assert np.maximum(p - q, 0).sum() < 0.5 * O.DEFAULT_EPS
    gpu = run_chain(batch)
    t = compare_chain(batch, gpu, range(B))
    assert t.boundary == 0 and t.fallback == B


@pytest.mark.parametrize("case", [(16, 3, 1000, "bf16"), (9, 8, 152064, "bf16"), (5, 0, 7, "f32"),
                                  (7, 4, 70001, "f32"), (3, 2, 1, "bf16")])
def test_greedy_chain_bit_exact_with_ties(case):
    B, g, V, dt = case
    batch = W.make_chain(spec(B, g, V, dt, 0.0, sigma=3.0), seed=12)
    # integer-valued logits: ties at the max are common; the lowest index must win
    batch.target = torch.round(batch.target.float()).to(batch.target.dtype)
    rng = np.random.default_rng(1)
    for b in range(B):
        for k in range(g):
            row = batch.target[b * (g + 1) + k].float().numpy()
            top = np.flatnonzero(row == row.max())
            batch.draft_tokens[b, k] = top[0] if rng.random() < 0.7 else top[-1]
    gpu = run_chain(batch)
    compare_chain(batch, gpu, range(B))


def test_repeat_calls_are_deterministic_and_leave_workspace_zeroed():
    batch = W.make_chain(spec(8, 4, 20000, "bf16", 0.9, 20), seed=2)
    a = run_chain(batch)
    b = run_chain(batch)
    for key in ("n_acc", "out_tokens", "n_out", "accept_prob", "residual_mass", "flags"):
        np.testing.assert_array_equal(a[key], b[key])
    from speculative_decoding_verification_37_gb300 import api, _lib as L
    ws = api.workspace(L.SPEC_WS_CHAIN_TOPK, 8, 4, 20000, "cuda")
    torch.cuda.synchronize()
    counters = ws[256:256 + 8 * 4].view(torch.int32)
    assert int(counters.abs().sum()) == 0
