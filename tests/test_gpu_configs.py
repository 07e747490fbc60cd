"""GPU parity at the five workloads' full sizes: every request is checked
against the oracle; the KV commit is checked block by block on the blocks it
may touch, and every other block must still hold the sentinel.

Each workload runs in the launch configuration the benchmark times (the
same workspace kind, hence the same kernels).  Asking for residual_mass
changes the kernel on the full-vocabulary workload (the persistent path does
not write it), so workload 5 runs twice: once as the benchmark runs it, once
with the residual mass so that output is checked too."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from parity import BOUNDARY_RATE_MAX, ChainTally, compare_chain, full_path_used, run_chain
from speculative_decoding_verification_37_gb300 import _lib as L
from speculative_decoding_verification_37_gb300 import api
from speculative_decoding_verification_37_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def commit_and_check(kvb: W.KVBatch, n_slots, slots=None):
    """Commit on the GPU, then compare the touched blocks with the oracle's
    commit applied to a compacted copy of those blocks."""
    d = "cuda"
    cache = W.make_cache(kvb, device=d)
    temp = kvb.temp_kv.to(d)
    lens = torch.from_numpy(kvb.committed_len.copy()).to(d)
    ns = torch.from_numpy(np.asarray(n_slots, np.int32)).to(d)
    sl = None if slots is None else torch.from_numpy(np.ascontiguousarray(slots, np.int32)).to(d)
    api.commit_kv(temp, cache, torch.from_numpy(kvb.block_table).to(d), ns, lens,
                  block_size=kvb.kv.block_size, slots=sl)
    torch.cuda.synchronize()
    # blocks a request's commit may reach: those of positions len .. len+S-1
    bs = kvb.kv.block_size
    touched = sorted({int(kvb.block_table[b, p // bs]) for b in range(kvb.B)
                      for p in range(int(kvb.committed_len[b]), int(kvb.committed_len[b]) + kvb.S)})
    remap = {blk: i for i, blk in enumerate(touched)}
    table = np.vectorize(lambda x: remap.get(int(x), len(touched)))(kvb.block_table).astype(np.int32)
    k = kvb.kv
    small = np.full((k.layers, 2, len(touched) + 1, bs, k.heads, k.head_dim), W.KV_SENTINEL, np.int16)
    temp16 = kvb.temp_kv.view(torch.int16).numpy()
    want_len = kvb.committed_len.copy()
    for b in range(kvb.B):
        s = list(range(int(n_slots[b]))) if slots is None else list(slots[b][:int(n_slots[b])])
        want_len[b], fl = O.commit_kv(small, temp16[b], table[b], s, int(n_slots[b]),
                                      int(want_len[b]), bs)
        assert fl == 0
    got = cache.view(torch.int16)
    idx = torch.tensor(touched, device=d)
    np.testing.assert_array_equal(got.index_select(2, idx).cpu().numpy(), small[:, :, :len(touched)])
    keep = torch.ones(got.shape[2], dtype=torch.bool, device=d)
    keep[idx] = False
    assert bool((got[:, :, keep] == W.KV_SENTINEL).all())
    np.testing.assert_array_equal(lens.cpu().numpy(), want_len)


def check_chain_config(cfg, residual=True, batch=None, oracle_results=None):
    spec = W.WORKLOADS[cfg]
    batch = W.make_chain(spec, seed=0) if batch is None else batch
    gpu = run_chain(batch, residual=residual)
    tally = compare_chain(batch, gpu, range(batch.n), oracle_results=oracle_results)
    assert tally.boundary <= 1, tally.boundary
    return batch, gpu, tally


def test_config1_chain_tiny():
    batch, gpu, t = check_chain_config(1)
    assert t.requests == 8


def test_config2_chain_topk_and_commit():
    batch, gpu, t = check_chain_config(2)
    spec = batch.spec
    kvb = W.make_kv(spec.kv, spec.B, spec.gamma + 1, seed=0)
    commit_and_check(kvb, gpu["n_out"])


def test_config3_greedy_chain_bit_exact():
    batch, gpu, t = check_chain_config(3)
    assert t.boundary == 0
    rate = gpu["n_acc"].mean() / batch.spec.gamma
    assert 0.2 < rate < 0.9


def test_config4_tree_and_commit():
    spec = W.WORKLOADS[4]
    tb = W.make_tree(spec, seed=0)
    kvb = W.make_kv(spec.kv, spec.B, spec.n_nodes + 1, seed=0)
    d = "cuda"
    out = api.verify_tree(tb.logits.to(d), torch.from_numpy(tb.node_token).to(d),
                          torch.from_numpy(tb.node_parent).to(d),
                          torch.from_numpy(tb.row_of_node).to(d),
                          torch.from_numpy(kvb.committed_len).to(d), R=spec.n_rows)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in vars(out).items()}
    R = spec.n_rows
    for b in range(spec.B):
        r = O.verify_tree(tb.logits_f64(b), tb.node_token[b], tb.node_parent[b], tb.row_of_node[b],
                          committed_len=int(kvb.committed_len[b]))
        assert g["n_acc"][b] == r.n_acc and list(g["path"][b][:r.n_acc]) == r.path
        assert list(g["out_tokens"][b][:g["n_out"][b]]) == r.tokens
        np.testing.assert_array_equal(g["tree_mask"][b].view(np.uint32), r.mask)
        np.testing.assert_array_equal(g["pos"][b], r.pos)
        assert list(g["commit_slots"][b][:g["n_commit"][b]]) == r.commit_slots
    assert R == 5 and g["n_acc"].mean() > 0.3
    commit_and_check(kvb, g["n_commit"], g["commit_slots"])


def test_config5_chain_f32_equal_rows_and_commit():
    """Workload 5 (B=512, gamma=7, V=128256 fp32, 5 requests with draft ==
    target): first on the persistent full-vocabulary kernel, routed exactly as
    the benchmark routes it (SPEC_WS_CHAIN_FULL workspace, no residual_mass),
    then on the cluster kernel that also writes residual_mass; one oracle run
    serves both comparisons."""
    spec = W.WORKLOADS[5]
    batch = W.make_chain(spec, seed=0)
    assert api.chain_workspace_kind(True, spec.top_k, spec.V) == L.SPEC_WS_CHAIN_FULL
    results = {}
    _, gpu_full, t_full = check_chain_config(5, residual=False, batch=batch, oracle_results=results)
    assert full_path_used(spec.B, spec.gamma, spec.V)
    assert gpu_full["residual_mass"] is None and t_full.requests == spec.B
    _, gpu, t = check_chain_config(5, residual=True, batch=batch, oracle_results=results)
    for b in batch.equal_rows:
        assert gpu_full["n_acc"][b] == spec.gamma and gpu["n_acc"][b] == spec.gamma
        assert np.all(gpu["residual_mass"][b] == 0.0)
    kvb = W.make_kv(spec.kv, spec.B, spec.gamma + 1, seed=0)
    commit_and_check(kvb, gpu_full["n_out"])


def test_boundary_case_rate_on_many_decisions():
    """Config-1 shapes with 4096 requests: boundary cases stay under 1e-4 of
    the decisions."""
    spec = dataclasses.replace(W.WORKLOADS[1], B=4096)
    batch = W.make_chain(spec, seed=1)
    gpu = run_chain(batch, residual=False)
    t = compare_chain(batch, gpu, range(batch.n), ChainTally())
    assert t.decisions > 10000
    assert t.boundary_rate < BOUNDARY_RATE_MAX, (t.boundary, t.decisions)
