"""GPU parity of tree verification (walk, mask, positions, commit slots) and
of the paged KV commit against the oracle, through the C ABI (bit-exact)."""
import numpy as np
import pytest
import torch

import oracle as O
from conftest import golden
from speculative_decoding_verification_37_gb300 import api
from speculative_decoding_verification_37_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run_tree(logits, tok, par, rows, lens, R):
    d = "cuda"
    out = api.verify_tree(logits.to(d), torch.from_numpy(np.ascontiguousarray(tok)).to(d),
                          torch.from_numpy(np.ascontiguousarray(par)).to(d),
                          torch.from_numpy(np.ascontiguousarray(rows)).to(d),
                          torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).to(d), R=R)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in vars(out).items()}


def compare_tree(logits, tok, par, rows, lens, R, gpu):
    B = tok.shape[0]
    N = tok.shape[1]
    for b in range(B):
        r = O.verify_tree(logits[b * R:(b + 1) * R].to(torch.float64).numpy(), tok[b], par[b],
                          rows[b], committed_len=int(lens[b]))
        if r.flags:
            assert gpu["flags"][b] & O.FLAG_BAD_INPUT and gpu["n_out"][b] == 0, b
            continue
        assert gpu["flags"][b] == 0
        assert gpu["n_acc"][b] == r.n_acc, b
        assert list(gpu["path"][b][:r.n_acc]) == r.path, b
        assert gpu["n_out"][b] == r.n_out, b
        assert list(gpu["out_tokens"][b][:r.n_out]) == r.tokens, b
        assert gpu["n_commit"][b] == len(r.commit_slots)
        assert list(gpu["commit_slots"][b][:len(r.commit_slots)]) == r.commit_slots, b
        np.testing.assert_array_equal(gpu["tree_mask"][b].view(np.uint32), r.mask)
        np.testing.assert_array_equal(gpu["pos"][b], r.pos)
        assert N == len(r.mask) - 1


def test_real_dump_tree_on_gpu():
    g = golden("tree_dump_example.json")
    names = ["R"] + [n["name"] for n in g["nodes"]]
    idx = {n: i for i, n in enumerate(names)}
    tok = np.array([[n["token"] for n in g["nodes"]]], np.int32)
    par = np.array([[idx[n["parent"]] for n in g["nodes"]]], np.int32)
    parents = sorted(idx[p] for p in g["target_top1"])
    rows = np.full((1, 13), -1, np.int32)
    for r, nid in enumerate(parents):
        rows[0, nid] = r
    V = 50000
    rng = np.random.default_rng(0)
    x = rng.normal(0, 1, (5, V)).astype(np.float32)
    for r, nid in enumerate(parents):
        x[r, g["target_top1"][names[nid]]] = 10.0
    logits = torch.from_numpy(x).to(torch.bfloat16)
    gpu = run_tree(logits, tok, par, rows, [77], 5)
    assert [names[i] for i in gpu["path"][0][:gpu["n_acc"][0]]] == g["accepted_path"]
    assert list(gpu["out_tokens"][0][:gpu["n_out"][0]]) == g["accepted_tokens"]
    compare_tree(logits, tok, par, rows, [77], 5, gpu)


@pytest.mark.parametrize("V,dt", [(1000, "bf16"), (70001, "f32"), (128256, "bf16")])
def test_generated_trees_match_oracle(V, dt):
    spec = W.TreeSpec("t", B=24, V=V, topKSpec=((6,), (2, 2), (1, 1)), topHead=(1, 2, 2),
                      dtype=dt, draft_sigma=0.5)
    tb = W.make_tree(spec, seed=V % 97)
    lens = np.arange(24, dtype=np.int32) * 7 + 3
    gpu = run_tree(tb.logits, tb.node_token, tb.node_parent, tb.row_of_node, lens, spec.n_rows)
    compare_tree(tb.logits, tb.node_token, tb.node_parent, tb.row_of_node, lens, spec.n_rows, gpu)
    assert gpu["n_acc"].max() >= 1      # some paths are accepted at this draft noise


def test_wide_tree_with_ties_and_bad_requests():
    """Full top-6 over three levels (258 nodes, 43 rows, 9 mask words); logits
    with ties; a malformed request of each kind is skipped and flagged."""
    spec = W.TreeSpec("wide", B=6, V=300, topKSpec=([6], [6] * 6, [6] * 36), topHead=(1, 6, 36),
                      dtype="bf16", draft_sigma=0.3)
    tb = W.make_tree(spec, seed=3)
    logits = torch.round(tb.logits.float() * 2).to(torch.bfloat16)
    tok, par, rows = tb.node_token.copy(), tb.node_parent.copy(), tb.row_of_node.copy()
    tok[1, 5] = 300                     # token out of range
    par[2, 7] = 200                     # parent id not below own id
    rows[3, 4] = 99                     # row out of range
    lens = np.full(6, 1000, np.int32)
    gpu = run_tree(logits, tok, par, rows, lens, spec.n_rows)
    compare_tree(logits, tok, par, rows, lens, spec.n_rows, gpu)
    assert all(gpu["flags"][b] & O.FLAG_BAD_INPUT for b in (1, 2, 3))


# ---------------------------------------------------------------------------
# KV commit
# ---------------------------------------------------------------------------
def commit_on_gpu(kvb, n_slots, slots=None):
    d = "cuda"
    cache = W.make_cache(kvb, device=d)
    temp = kvb.temp_kv.to(d)
    table = torch.from_numpy(kvb.block_table).to(d)
    lens = torch.from_numpy(kvb.committed_len.copy()).to(d)
    ns = torch.from_numpy(np.asarray(n_slots, np.int32)).to(d)
    sl = None if slots is None else torch.from_numpy(np.ascontiguousarray(slots, np.int32)).to(d)
    biu = torch.zeros(kvb.B, dtype=torch.int32, device=d)
    flags = torch.zeros(kvb.B, dtype=torch.int32, device=d)
    api.commit_kv(temp, cache, table, ns, lens, block_size=kvb.kv.block_size, slots=sl,
                  blocks_in_use=biu, flags=flags)
    torch.cuda.synchronize()
    return cache, lens.cpu().numpy(), biu.cpu().numpy(), flags.cpu().numpy()


def oracle_commit(kvb, n_slots, slots=None, table=None):
    cache = W.make_cache(kvb).view(torch.int16).numpy().copy()
    temp = kvb.temp_kv.view(torch.int16).numpy()
    table = kvb.block_table if table is None else table
    lens = kvb.committed_len.copy()
    flags = np.zeros(kvb.B, np.int32)
    for b in range(kvb.B):
        sl = list(range(n_slots[b])) if slots is None else slots[b]
        lens[b], flags[b] = O.commit_kv(cache, temp[b], table[b], sl, int(n_slots[b]),
                                        int(lens[b]), kvb.kv.block_size)
    return cache, lens, flags


@pytest.mark.parametrize("seed", [0, 1])
def test_commit_small_geometry_bit_exact(seed):
    rng = np.random.default_rng(seed)
    kv = W.KVSpec(layers=3, heads=2, head_dim=8, block_size=4, prefix=0)
    B, S = 9, 6
    prefix = rng.integers(0, 30, B)
    kvb = W.make_kv(kv, B, S, seed=seed, prefix=prefix)
    n_slots = rng.integers(0, S + 1, B).astype(np.int32)
    n_slots[0] = 0
    cache, lens, biu, flags = commit_on_gpu(kvb, n_slots)
    want, wlens, wflags = oracle_commit(kvb, n_slots)
    np.testing.assert_array_equal(cache.view(torch.int16).cpu().numpy(), want)
    np.testing.assert_array_equal(lens, wlens)
    np.testing.assert_array_equal(biu, [O.blocks_in_use(int(x), 4) for x in wlens])
    assert not flags.any() and not wflags.any()


def test_commit_tree_slots_and_bad_request_skipped():
    kv = W.KVSpec(layers=2, heads=1, head_dim=16, block_size=4, prefix=0)
    B, S = 4, 13
    kvb = W.make_kv(kv, B, S, seed=5, prefix=[5, 0, 9, 3])
    slots = np.full((B, S), -1, np.int32)
    paths = [[0, 1, 7, 11], [0], [0, 2, 9], [0, 3]]
    for b, pth in enumerate(paths):
        slots[b, :len(pth)] = pth
    n = np.array([len(p) for p in paths], np.int32)
    kvb.block_table[2, (9 + 1) // 4] = kvb.num_blocks + 5          # bad block id
    cache, lens, biu, flags = commit_on_gpu(kvb, n, slots)
    want, wlens, wflags = oracle_commit(kvb, n, [list(s[:k]) for s, k in zip(slots, n)])
    np.testing.assert_array_equal(cache.view(torch.int16).cpu().numpy(), want)
    np.testing.assert_array_equal(lens, wlens)
    assert flags[2] & O.FLAG_BAD_INPUT and wflags[2] == O.FLAG_BAD_INPUT
    assert not flags[[0, 1, 3]].any()


def test_commit_real_geometry_touched_blocks_only():
    kv = W.KVSpec(prefix=2045)            # commits straddle a block edge
    B, S = 16, 5
    kvb = W.make_kv(kv, B, S, seed=2)
    n = (np.arange(B) % (S + 1)).astype(np.int32)
    cache, lens, biu, flags = commit_on_gpu(kvb, n)
    want, wlens, _ = oracle_commit(kvb, n)
    got = cache.view(torch.int16).cpu().numpy()
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(lens, wlens)
