"""GPU parity of the in-place chain commit (the length advance done by the
verify call itself) against the oracle, through the C ABI, on every chain
path: greedy, the cluster sampler, the top-k candidate lists and the
persistent full-vocabulary kernel."""
import numpy as np
import pytest
import torch

import oracle as O
from parity import compare_chain, oracle_chain, to_dev
from speculative_decoding_verification_37_gb300 import _lib as L
from speculative_decoding_verification_37_gb300 import api
from speculative_decoding_verification_37_gb300 import workloads as W

pytestmark = pytest.mark.gpu

BS = 16


def lengths(B, gamma, cap, rng):
    """Committed lengths that straddle block edges, plus a few that do not
    fit (the last reserved position one past the capacity, a negative one)."""
    len0 = rng.integers(0, cap - gamma - 1, B).astype(np.int32)
    len0[: B // 8] = (BS - 1 - rng.integers(0, gamma + 1, B // 8)).clip(0)
    if B >= 4:
        len0[1] = cap - gamma - 1          # ends exactly at the capacity: fits
        len0[2] = cap - gamma              # one past: flagged
        len0[3] = -3                       # flagged
    draft = (len0 + gamma - rng.integers(0, 2, B)).astype(np.int32)
    return len0, draft


def run(batch, kind, len0, dlen0, cap):
    s = batch.spec
    tgt, drf, tok, unif = to_dev(batch)
    d = dict(dtype=torch.int32, device="cuda")
    cl = torch.from_numpy(len0).to(**d)
    dl = torch.from_numpy(dlen0).to(**d)
    blk = torch.full((s.B,), -7, **d)
    ws = api.workspace(kind, s.B, s.gamma, s.V, "cuda")
    out = api.verify_chain(tgt, tok, gamma=s.gamma, temperature=s.temperature, draft=drf,
                           uniforms=unif, top_k=s.top_k, residual_mass=kind == L.SPEC_WS_CHAIN and
                           not s.greedy, ws=ws, committed_len=cl, draft_len=dl,
                           blocks_in_use=blk, block_size=BS, kv_capacity=cap)
    torch.cuda.synchronize()
    g = {k: (None if v is None else v.cpu().numpy()) for k, v in vars(out).items()}
    return g, cl.cpu().numpy(), dl.cpu().numpy(), blk.cpu().numpy()


def check(batch, kind, seed, cap=4096):
    s = batch.spec
    rng = np.random.default_rng(seed)
    len0, dlen0 = lengths(s.B, s.gamma, cap, rng)
    gpu, cl, dl, blk = run(batch, kind, len0, dlen0, cap)
    moved = 0
    for b in range(s.B):
        r = oracle_chain(batch, b)
        c = O.commit_in_place(int(len0[b]), r.n_out, s.gamma, BS, int(dlen0[b]), cap)
        if c.flags or r.flags & (O.FLAG_BAD_INPUT | O.FLAG_BAD_ROW):
            assert gpu["n_out"][b] == 0 and int(gpu["flags"][b]) & (O.FLAG_BAD_INPUT | O.FLAG_BAD_ROW), b
            assert (cl[b], dl[b], blk[b]) == (len0[b], dlen0[b], -7), b
            continue
        # the lengths follow the GPU's own n_out (equal to the oracle's away
        # from boundary cases, checked below)
        n = int(gpu["n_out"][b])
        mine = O.commit_in_place(int(len0[b]), n, s.gamma, BS, int(dlen0[b]), cap)
        assert (cl[b], dl[b], blk[b]) == (mine.committed_len, mine.draft_len, mine.blocks_in_use), b
        if not r.boundary:
            assert (cl[b], dl[b], blk[b]) == (c.committed_len, c.draft_len, c.blocks_in_use), b
        moved += 1
    good = [b for b in range(s.B) if 0 <= len0[b] and len0[b] + s.gamma + 1 <= cap]
    compare_chain(batch, gpu, good)
    assert moved > 0
    if s.B >= 4:
        assert gpu["flags"][2] & O.FLAG_BAD_INPUT and gpu["flags"][3] & O.FLAG_BAD_INPUT
        assert cl[1] > len0[1] or gpu["flags"][1]


def chain(B, gamma, V, dtype, T, top_k=0):
    return W.ChainSpec(f"t B={B} g={gamma} V={V}", B=B, gamma=gamma, V=V, dtype=dtype,
                       target_sigma=2.0, temperature=T, top_k=top_k, draft_sigma=1.0)


def test_in_place_greedy():
    batch = W.make_chain(chain(64, 5, 5000, "bf16", 0.0), seed=1)
    batch.draft_tokens[5, 0] = -1                      # a bad request keeps its lengths
    check(batch, L.SPEC_WS_CHAIN, 1)


def test_in_place_sampled_cluster_path():
    batch = W.make_chain(chain(40, 4, 3000, "f32", 0.9), seed=2)
    check(batch, L.SPEC_WS_CHAIN, 2)


def test_in_place_sampled_topk_path():
    batch = W.make_chain(chain(48, 4, 32000, "bf16", 0.8, top_k=50), seed=3)
    assert api.chain_workspace_kind(True, 50, 32000) == L.SPEC_WS_CHAIN_TOPK
    check(batch, L.SPEC_WS_CHAIN_TOPK, 3)


def test_in_place_sampled_full_path():
    batch = W.make_chain(chain(64, 4, 16384, "f32", 1.0), seed=4)   # 64*5*16 = 5,120 slices
    batch.draft_tokens[6, 1] = 16384
    check(batch, L.SPEC_WS_CHAIN_FULL, 4)


def test_in_place_gamma_zero_and_small_capacity():
    batch = W.make_chain(chain(16, 0, 1000, "f32", 1.0), seed=5)
    check(batch, L.SPEC_WS_CHAIN, 5, cap=40)
