"""Pins of the oracle's tree walk, tree mask / positions and KV commit, and of
the tree generator's sizes (CPU only)."""
import numpy as np
import pytest
import torch

from conftest import golden
import oracle as O
from speculative_decoding_verification_37_gb300 import workloads as W


def dump_tree():
    """The tree of the real dump example as (node_token, node_parent,
    row_of_node) with node ids 1..12 in the page's BFS order."""
    g = golden("tree_dump_example.json")
    names = ["R"] + [n["name"] for n in g["nodes"]]
    idx = {n: i for i, n in enumerate(names)}
    tok = np.array([n["token"] for n in g["nodes"]], np.int32)
    par = np.array([idx[n["parent"]] for n in g["nodes"]], np.int32)
    parents = sorted(idx[p] for p in g["target_top1"])
    rows = np.full(len(names), -1, np.int32)
    for r, nid in enumerate(parents):
        rows[nid] = r
    return g, names, idx, tok, par, rows, parents


def rows_with_argmax(choices, V, rng, ties_at=None):
    """Random logits rows whose argmax (lowest index on ties) is choices[r]."""
    x = rng.normal(0, 1, (len(choices), V))
    for r, c in enumerate(choices):
        x[r, c] = x[r].max() + 1.0
        if ties_at is not None and ties_at[r] is not None and ties_at[r] > c:
            x[r, ties_at[r]] = x[r, c]            # a tie at a higher index must not win
    return x


def test_real_dump_walk_follows_one_path():
    g, names, idx, tok, par, rows, parents = dump_tree()
    assert len(tok) == g["draft_nodes"] and len(parents) == g["parent_rows"]
    V = 50000
    rng = np.random.default_rng(0)
    choices = [g["target_top1"][names[nid]] for nid in parents]
    logits = rows_with_argmax(choices, V, rng)
    r = O.verify_tree(logits, tok, par, rows, committed_len=100)
    assert [names[i] for i in r.path] == g["accepted_path"]
    assert r.tokens == g["accepted_tokens"]           # C111 has no logits row: no extra token
    assert r.n_acc == g["n_accepted"]
    # summing matches across branches would have counted 5 (R, A1, A2, B11, B21 all match)
    matched_anywhere = sum(
        any(par[c - 1] == nid and tok[c - 1] == g["target_top1"][names[nid]] for c in range(1, 13))
        for nid in parents)
    assert matched_anywhere == 5 and r.n_acc != matched_anywhere
    assert r.commit_slots == [0] + [idx[n] for n in g["accepted_path"]]


def test_walk_break_emits_target_choice_and_leaf_row_gives_bonus():
    _, names, idx, tok, par, rows, parents = dump_tree()
    V = 50000
    rng = np.random.default_rng(1)
    # root's choice matches A2; A2's choice matches nothing -> emit it
    choices = {"R": 43744, "A1": 41760, "A2": 777, "B11": 22870, "B21": 22870}
    logits = rows_with_argmax([choices[names[n]] for n in parents], V, rng)
    r = O.verify_tree(logits, tok, par, rows)
    assert [names[i] for i in r.path] == ["A2"] and r.tokens == [43744, 777]
    # the root's choice matches no first-level node: zero drafts, one emitted token
    choices["R"] = 5
    logits = rows_with_argmax([choices[names[n]] for n in parents], V, rng)
    r = O.verify_tree(logits, tok, par, rows)
    assert r.path == [] and r.tokens == [5] and r.commit_slots == [0]
    # give the leaf C111 a row: the walk then ends with a bonus token from it
    rows2 = rows.copy()
    rows2[idx["C111"]] = len(parents)
    choices = {"R": 41824, "A1": 41760, "A2": 45315, "B11": 22870, "B21": 22870}
    logits = rows_with_argmax([choices[names[n]] for n in parents] + [999], V, rng)
    r = O.verify_tree(logits, tok, par, rows2)
    assert r.tokens == [41824, 41760, 22870, 999] and r.n_acc == 3


def test_walk_ties_and_duplicate_children():
    # root with children tokens [7, 3, 7]: a duplicate token goes to the lowest node id
    tok = np.array([7, 3, 7, 1], np.int32)
    par = np.array([0, 0, 0, 3], np.int32)
    rows = np.array([0, -1, -1, 1, -1], np.int32)
    x = np.zeros((2, 10))
    x[0, 7] = 2.0
    x[1, 1] = 1.0
    x[1, 4] = 1.0                                     # tie: token 1 (lower) wins
    r = O.verify_tree(x, tok, par, rows)
    assert r.path == [1] and r.tokens == [7]          # node 1 has no row: stop, no extra
    x[0, 3] = 2.0                                     # now 3 and 7 tie at the root -> 3
    r = O.verify_tree(x, tok, par, rows)
    assert r.path == [2]


def test_table_10_17_mask_and_depth_positions():
    g = golden("mask_table_10_17.json")
    order = g["order"]
    par = np.array([order.index(g["parent"][n]) for n in order[1:]], np.int32)
    mask, pos = O.tree_mask_positions(par, committed_len=37)
    want = np.array(g["mask"])
    got = np.array([[(int(mask[i, j // 32]) >> (j % 32)) & 1 for j in range(5)] for i in range(5)])
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(pos, 37 + np.array(g["depth"]))


def test_mask_words_for_trees_wider_than_32():
    # a 40-node chain: node i's row has bits 0..i over two words
    par = np.arange(40, dtype=np.int32)                # node i+1's parent is node i
    mask, pos = O.tree_mask_positions(par, 0)
    assert mask.shape == (41, 2)
    for i in range(41):
        bits = [(int(mask[i, j // 32]) >> (j % 32)) & 1 for j in range(41)]
        assert bits == [1] * (i + 1) + [0] * (40 - i)
    np.testing.assert_array_equal(pos, np.arange(41))


def test_bad_tree_inputs_flagged():
    x = np.zeros((1, 4))
    assert O.verify_tree(x, [9], [0], [0, -1]).flags & O.FLAG_BAD_INPUT       # token >= V
    assert O.verify_tree(x, [1, 2], [0, 2], [0, -1, -1]).flags & O.FLAG_BAD_INPUT  # parent not < id
    assert O.verify_tree(x, [1], [0], [3, -1]).flags & O.FLAG_BAD_INPUT       # row >= R


# --- generator: tree sizes of the tree-speculation page --------------------------------
def test_generator_tree_sizes():
    g = golden("tree_dump_example.json")
    rng = np.random.default_rng(2)
    tree = W.grow_tree(rng.normal(0, 1, (5, 1000)), g["topKSpec"], g["topHead"])
    assert tree.N == g["draft_nodes"]
    assert (tree.row_of_node >= 0).sum() == g["parent_rows"]
    assert sorted(tree.row_of_node[tree.row_of_node >= 0]) == list(range(5))
    assert np.all(tree.node_parent < np.arange(1, tree.N + 1))
    full = g["full_top6_three_levels"]
    spec = [[6], [6] * 6, [6] * 36]
    head = [1, 6, 36]
    big = W.grow_tree(rng.normal(0, 1, (sum(head), 1000)), spec, head)
    assert big.N == full["total"]
    depth = [0]
    for p in big.node_parent:
        depth.append(depth[p] + 1)
    assert [depth.count(lv) for lv in (1, 2, 3)] == full["per_level"]


def test_generator_tree_follows_page_shape():
    """Level-1 children are the draft's top-6 in rank order; the two expanded
    level-1 parents are the most probable ones (A1, A2)."""
    rng = np.random.default_rng(3)
    draft = rng.normal(0, 3, (5, 2000))
    t = W.grow_tree(draft, [[6], [2, 2], [1, 1]], [1, 2, 2])
    top6 = np.argsort(-draft[0], kind="stable")[:6]
    np.testing.assert_array_equal(t.node_token[:6], top6)
    assert t.row_of_node[1] == 1 and t.row_of_node[2] == 2
    assert list(t.node_parent[6:10]) == [1, 1, 2, 2]
    assert list(t.node_parent[10:]) == sorted(t.node_parent[10:])


# --- KV commit ---------------------------------------------------------------------
def _commit_case(seed, prefix, n_acc, S=6, bs=4, L=3, H=2, D=8):
    kv = W.KVSpec(layers=L, heads=H, head_dim=D, block_size=bs, prefix=0)
    B = len(prefix)
    batch = W.make_kv(kv, B, S, seed=seed, prefix=prefix)
    cache = W.make_cache(batch).view(torch.int16).numpy().copy()
    temp = batch.temp_kv.view(torch.int16).numpy()
    return batch, cache, temp


@pytest.mark.parametrize("seed", range(4))
def test_commit_writes_accepted_slots_at_every_layer(seed):
    rng = np.random.default_rng(seed)
    B, S, bs = 5, 6, 4
    prefix = rng.integers(0, 23, B)                    # commits straddle block edges
    n_acc = rng.integers(0, S, B)
    batch, cache, temp = _commit_case(seed, prefix, n_acc, S=S, bs=bs)
    before = cache.copy()
    lens = batch.committed_len.copy()
    for b in range(B):
        slots = O.chain_commit_slots(int(n_acc[b]))
        new_len, fl = O.commit_kv(cache, temp[b], batch.block_table[b], slots, len(slots),
                                  int(lens[b]), bs)
        assert fl == 0 and new_len == lens[b] + n_acc[b] + 1
        lens[b] = new_len
    # every logical position of every request, read back through the block table
    touched = np.zeros(cache.shape[2:4], bool)
    for b in range(B):
        for i in range(int(n_acc[b]) + 1):
            pos = int(prefix[b]) + i
            blk, off = batch.block_table[b][pos // bs], pos % bs
            np.testing.assert_array_equal(cache[:, :, blk, off], temp[b][:, :, i])
            touched[blk, off] = True
    # nothing else changed (sentinel everywhere else, including the dummy block 0)
    assert not touched[0].any()
    np.testing.assert_array_equal(cache[:, :, ~touched], before[:, :, ~touched])
    assert np.all(before == W.KV_SENTINEL)


def test_commit_tree_slots_and_rollback_by_not_advancing():
    batch, cache, temp = _commit_case(9, [5], [0], S=13, bs=4)
    slots = [0, 1, 7, 11]                              # root + a path A1, B11, C111
    new_len, fl = O.commit_kv(cache, temp[0], batch.block_table[0], slots, 4, 5, 4)
    assert fl == 0 and new_len == 9
    for i, s in enumerate(slots):
        pos = 5 + i
        np.testing.assert_array_equal(cache[:, :, batch.block_table[0][pos // 4], pos % 4],
                                      temp[0][:, :, s])
    assert O.blocks_in_use(new_len, 4) == 3


def test_commit_rejects_bad_indices_without_writing():
    batch, cache, temp = _commit_case(4, [3], [2], S=6, bs=4)
    before = cache.copy()
    table = batch.block_table[0].copy()
    table[1] = cache.shape[2]                          # block id out of range
    new_len, fl = O.commit_kv(cache, temp[0], table, [0, 1, 2], 3, 3, 4)
    assert fl == O.FLAG_BAD_INPUT and new_len == 3
    np.testing.assert_array_equal(cache, before)
    new_len, fl = O.commit_kv(cache, temp[0], batch.block_table[0], [0, 6], 2, 3, 4)  # slot >= S
    assert fl == O.FLAG_BAD_INPUT and new_len == 3
    np.testing.assert_array_equal(cache, before)
    # past the end of the block table
    new_len, fl = O.commit_kv(cache, temp[0], batch.block_table[0], [0, 1, 2, 3, 4, 5], 6,
                              batch.max_blocks * 4 - 2, 4)
    assert fl == O.FLAG_BAD_INPUT
    np.testing.assert_array_equal(cache, before)


# --- in-place chain commit -----------------------------------------------------------
def _write_in_place(cache, temp_req, table, start, n, bs):
    """The target forward's own K/V writes: candidate i at position start+i."""
    for i in range(n):
        pos = start + i
        cache[:, :, table[pos // bs], pos % bs] = temp_req[:, :, i]


def _visible(cache, table, length, bs):
    return np.stack([cache[:, :, table[p // bs], p % bs] for p in range(length)], axis=2) \
        if length else np.zeros(0)


@pytest.mark.parametrize("seed", range(6))
def test_in_place_commit_equals_the_copy_commit(seed):
    """Writing every candidate's K/V in place and advancing the length by
    n_out leaves the same visible cache as copying the accepted slots after
    the verify: the rejected candidates lie past the boundary."""
    rng = np.random.default_rng(100 + seed)
    B, bs = 4, 4
    gamma = int(rng.integers(0, 6))
    S = gamma + 1
    prefix = rng.integers(0, 21, B)
    n_acc = rng.integers(0, gamma + 1, B)
    batch, cache_copy, temp = _commit_case(seed, prefix, n_acc, S=S, bs=bs)
    cache_inpl = cache_copy.copy()
    for b in range(B):
        table = batch.block_table[b]
        len0 = int(prefix[b])
        slots = O.chain_commit_slots(int(n_acc[b]))
        new_copy, fl = O.commit_kv(cache_copy, temp[b], table, slots, len(slots), len0, bs)
        assert fl == 0
        _write_in_place(cache_inpl, temp[b], table, len0, S, bs)
        c = O.commit_in_place(len0, int(n_acc[b]) + 1, gamma, bs, draft_len=len0 + gamma)
        assert c.flags == 0 and c.committed_len == new_copy
        np.testing.assert_array_equal(_visible(cache_inpl, table, c.committed_len, bs),
                                      _visible(cache_copy, table, new_copy, bs))
        # the blocks in use cover the last kept position and nothing past its block
        assert c.blocks_in_use == (new_copy - 1) // bs + 1
        # the draft cache (fed the last emitted token and the first gamma-1
        # drafts) is cut back to the boundary, or keeps its gamma positions
        assert c.draft_len == len0 + min(int(n_acc[b]) + 1, gamma)


def test_in_place_commit_special_cases():
    # every draft accepted: gamma+1 kept, the draft cache keeps what it has
    c = O.commit_in_place(10, 5, 4, 16, draft_len=14)
    assert (c.committed_len, c.draft_len, c.blocks_in_use, c.flags) == (15, 14, 1, 0)
    # a rejection at the first draft: only the last emitted token is kept
    c = O.commit_in_place(16, 1, 4, 16, draft_len=20)
    assert (c.committed_len, c.draft_len, c.blocks_in_use) == (17, 17, 2)
    # gamma 0: the bonus round keeps one position
    assert O.commit_in_place(0, 1, 0, 8).committed_len == 1
    # reserved positions past the capacity, or a negative length: nothing moves
    for len0, cap in ((60, 64), (-1, 0)):
        c = O.commit_in_place(len0, 1, 4, 16, draft_len=7, kv_capacity=cap)
        assert (c.committed_len, c.draft_len, c.blocks_in_use, c.flags) == (len0, 7, None, O.FLAG_BAD_INPUT)
    assert O.commit_in_place(59, 5, 4, 16, kv_capacity=64).flags == 0      # ends exactly at 64
    assert O.commit_in_place(2**31 - 5, 1, 4, 16).flags == O.FLAG_BAD_INPUT
