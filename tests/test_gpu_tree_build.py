"""GPU parity of the draft-tree builder (spec_tree_level, one call per level)
against the oracle, through the C ABI.

Bit-exact: children tokens and parents, the next parents, rows and flags.
Path log-probabilities: |gpu - oracle| <= 2e-5 (fp32 log-sum-exp over up to
262,144 logits, accumulated over up to three levels).  A request whose
selection the oracle marks as a boundary case (the last kept and first
dropped path log-probabilities within 5e-5, not tied siblings) is counted
and excluded from the exact comparison from that level on."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from speculative_decoding_verification_37_gb300 import api
from speculative_decoding_verification_37_gb300 import workloads as W

pytestmark = pytest.mark.gpu

LOGP_TOL = 2e-5


def build_gpu(levels, topKSpec, topHead, V, device="cuda", views=None):
    B = levels[0].shape[0] // topHead[0]
    tb = api.TreeBuilder(B, V, topKSpec, topHead, device)
    for i, rows in enumerate(levels):
        tb.level(rows.to(device) if views is None else views[i])
    torch.cuda.synchronize()
    return {k: getattr(tb, k).cpu().numpy() for k in ("node_token", "node_parent", "node_logp",
                                                      "row_of_node", "flags")}, tb


def oracle_trees(levels, topKSpec, topHead, requests):
    out = {}
    for b in requests:
        rows = [lv[b * h:(b + 1) * h].double().numpy() for lv, h in zip(levels, topHead)]
        out[b] = O.build_tree(rows, topKSpec, topHead)
    return out


def logp_close(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    same_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    return bool(np.all(same_inf | (np.abs(a - b) <= LOGP_TOL)))


def compare(gpu, trees, N):
    boundary = 0
    for b, t in trees.items():
        if t.flags:
            assert gpu["flags"][b] & t.flags, b
            continue
        assert gpu["flags"][b] == 0, b
        if t.boundary:
            boundary += 1
            continue
        np.testing.assert_array_equal(gpu["node_token"][b], t.node_token, err_msg=str(b))
        np.testing.assert_array_equal(gpu["node_parent"][b], t.node_parent, err_msg=str(b))
        np.testing.assert_array_equal(gpu["row_of_node"][b], t.row_of_node, err_msg=str(b))
        assert logp_close(gpu["node_logp"][b], t.node_logp), (b, gpu["node_logp"][b], t.node_logp)
    return boundary


def random_levels(B, V, topHead, dtype, seed, sigma=3.0, quant=None):
    g = torch.Generator().manual_seed(seed)
    out = []
    for h in topHead:
        x = torch.randn((B * h, V), generator=g) * sigma
        if quant:
            x = torch.round(x / quant) * quant
        out.append(x.to(torch.bfloat16 if dtype == "bf16" else torch.float32))
    return out


def test_page_shape_large_rows_bf16():
    s = dataclasses.replace(W.WORKLOADS[4], B=24)
    levels = W.make_tree_levels(s, seed=3)
    gpu, _ = build_gpu(levels, s.topKSpec, s.topHead, s.V)
    trees = oracle_trees(levels, s.topKSpec, s.topHead, range(s.B))
    assert compare(gpu, trees, s.n_nodes) <= 1


@pytest.mark.parametrize("case", [
    # (B, V, dtype, topKSpec, topHead)
    (20, 70001, "f32", ((4,), (3, 2, 1), (2, 2, 2)), (1, 3, 3)),   # ragged last slice
    (12, 5000, "f32", ((16,), (16, 8)), (1, 2)),                    # the 16-wide lists
    (40, 3000, "bf16", ((6,), (2, 2), (1, 1)), (1, 2, 2)),
    (64, 8, "f32", ((6,), (2, 2)), (1, 2)),                         # rows shorter than a vector pass
    (9, 262144, "bf16", ((5,), (3, 3)), (1, 2)),                    # 64 slices per row
    (33, 4096, "f32", ((1,), (1,), (1,), (1,)), (1, 1, 1, 1)),      # a chain as a tree
])
def test_levels_match_oracle(case):
    B, V, dt, spec, heads = case
    levels = random_levels(B, V, heads, dt, seed=B + V)
    gpu, _ = build_gpu(levels, spec, heads, V)
    trees = oracle_trees(levels, spec, heads, range(B))
    assert compare(gpu, trees, sum(map(sum, spec))) <= 1


def test_many_ties_and_masked_tokens():
    """Logits on a 0.5 grid (many equal values: the lower token id and the
    lower node id must win) and rows with masked (-inf) tokens, one with
    fewer finite logits than children."""
    B, V, spec, heads = 48, 3000, ((6,), (3, 3), (2, 2)), (1, 2, 2)
    levels = random_levels(B, V, heads, "bf16", seed=5, sigma=1.0, quant=0.5)
    levels[0][1, 100:] = -float("inf")
    levels[0][2, 2:] = -float("inf")                     # 2 finite logits, 6 children
    levels[1][3 * 2, : V // 2] = -float("inf")
    gpu, _ = build_gpu(levels, spec, heads, V)
    trees = oracle_trees(levels, spec, heads, range(B))
    compare(gpu, trees, sum(map(sum, spec)))
    assert sorted(gpu["node_token"][2][:2].tolist()) == [0, 1] and gpu["node_token"][2][2] == 2
    assert np.isinf(gpu["node_logp"][2][3]) and np.isfinite(gpu["node_logp"][2][2])


def test_bad_rows_and_bad_parents_flag_the_request():
    B, V, spec, heads = 8, 1000, ((4,), (2, 2)), (1, 2)
    levels = random_levels(B, V, heads, "f32", seed=9)
    levels[0][1, 17] = float("nan")
    levels[0][2, :] = -float("inf")
    levels[0][3, 5] = float("inf")
    levels[1][4 * 2 + 1, 900] = float("nan")             # request 4, level 1 only
    gpu, tb = build_gpu(levels, spec, heads, V)
    for b in (1, 2, 3):
        assert gpu["flags"][b] == O.FLAG_BAD_ROW | O.FLAG_BAD_INPUT, b   # -1 parents next level
        assert (gpu["node_token"][b] == -1).all()
    assert gpu["flags"][4] == O.FLAG_BAD_ROW
    assert (tb.next[0].cpu().numpy()[[1, 2, 3]] == -1).all()
    trees = oracle_trees(levels, spec, heads, [0, 5, 6, 7])
    compare(gpu, trees, 8)


def test_strided_misaligned_rows_and_repeat_calls():
    """Rows that start one element past a 16-byte boundary, with a row stride
    above V; then a second batch through the same cached workspaces."""
    B, V, spec, heads = 16, 9001, ((6,), (2, 2), (1, 1)), (1, 2, 2)
    for seed in (1, 2):
        levels = random_levels(B, V, heads, "bf16", seed=seed)
        views = []
        for lv in levels:
            big = torch.zeros((lv.shape[0], V + 5), dtype=lv.dtype, device="cuda")
            big[:, 1:V + 1] = lv.cuda()
            views.append(big[:, 1:V + 1])
        gpu, _ = build_gpu(levels, spec, heads, V, views=views)
        trees = oracle_trees(levels, spec, heads, range(B))
        assert compare(gpu, trees, 12) <= 1


def test_built_tree_feeds_the_tree_verify():
    """The builder's node arrays are the tree verify's input layout: verify
    the GPU-built trees against target rows and compare with the oracle."""
    s = dataclasses.replace(W.WORKLOADS[4], B=16, V=20000)
    levels = W.make_tree_levels(s, seed=2)
    gpu, tb = build_gpu(levels, s.topKSpec, s.topHead, s.V)
    target = W.make_tree(s, seed=2).logits
    cl = torch.full((s.B,), 50, dtype=torch.int32, device="cuda")
    out = api.verify_tree(target.cuda(), tb.node_token, tb.node_parent, tb.row_of_node, cl, R=s.n_rows)
    torch.cuda.synchronize()
    R = s.n_rows
    for b in range(s.B):
        r = O.verify_tree(target[b * R:(b + 1) * R].double().numpy(), gpu["node_token"][b],
                          gpu["node_parent"][b], gpu["row_of_node"][b], 50)
        assert int(out.n_acc[b]) == r.n_acc and out.out_tokens[b][:r.n_out].tolist() == r.tokens


def test_large_batch_sampled():
    """The full 128-request workload, 24 requests compared."""
    s = W.WORKLOADS[4]
    levels = W.make_tree_levels(s, seed=0)
    gpu, _ = build_gpu(levels, s.topKSpec, s.topHead, s.V)
    reqs = list(range(0, s.B, 6))[:24]
    trees = oracle_trees(levels, s.topKSpec, s.topHead, reqs)
    assert compare(gpu, trees, s.n_nodes) <= 1
