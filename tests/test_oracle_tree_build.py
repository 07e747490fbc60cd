"""Pins of the draft-tree builder's oracle (CPU only)."""
import itertools

import numpy as np
import pytest
from scipy.special import softmax

from conftest import golden
import oracle as O
from oracle import tree_build_oracle as TB
from speculative_decoding_verification_37_gb300 import workloads as W


def row_with_top(V, tokens, rng, base=0.0):
    """A logits row whose largest values are ``tokens``, in that order."""
    x = rng.normal(base, 1.0, V)
    top = x.max()
    for r, t in enumerate(tokens):
        x[t] = top + 3.0 - 0.5 * r
    return x


def test_page_dump_example_numbering_and_rows():
    """The real dump: root top-6, A1 and A2 expanded with their top-2, B11
    and B21 with their top-1; 12 nodes numbered level by level, 5 rows."""
    g = golden("tree_dump_example.json")
    nodes = {n["name"]: n for n in g["nodes"]}
    V = 50000
    rng = np.random.default_rng(0)
    kids = {"R": ["A1", "A2", "A3", "A4", "A5", "A6"], "A1": ["B11", "B12"], "A2": ["B21", "B22"],
            "B11": ["C111"], "B21": ["C211"]}
    row = {p: row_with_top(V, [nodes[c]["token"] for c in cs], rng) for p, cs in kids.items()}
    # B11 and B21 must beat B12 and B22 on path probability: the second child
    # of each row is made much less likely than the first
    for p in ("A1", "A2"):
        row[p][nodes[kids[p][1]]["token"]] -= 2.0
    levels = [[row["R"]], [row["A1"], row["A2"]], [row["B11"], row["B21"]]]
    t = O.build_tree(levels, g["topKSpec"], g["topHead"])
    assert t.flags == 0 and not t.boundary
    names = ["R"] + [n["name"] for n in g["nodes"]]
    assert list(t.node_token) == [n["token"] for n in g["nodes"]]
    assert [names[p] for p in t.node_parent] == [n["parent"] for n in g["nodes"]]
    expanded = [names[i] for i in range(len(names)) if t.row_of_node[i] >= 0]
    assert expanded == ["R", "A1", "A2", "B11", "B21"]
    assert [t.row_of_node[names.index(n)] for n in expanded] == [0, 1, 2, 3, 4]
    assert len(t.node_token) == g["draft_nodes"] and len(expanded) == g["parent_rows"]


def test_full_expansion_blows_up_to_258_nodes():
    g = golden("tree_dump_example.json")["full_top6_three_levels"]
    rng = np.random.default_rng(1)
    V = 64
    spec = [[6], [6] * 6, [6] * 36]
    heads = [1, 6, 36]
    levels = [rng.normal(0, 2, (h, V)) for h in heads]
    t = O.build_tree(levels, spec, heads)
    per_level = [int(np.sum(t.node_parent == p)) for p in (0,)] + \
        [int(np.isin(t.node_parent, np.arange(1, 7)).sum()), int((t.node_parent > 6).sum())]
    assert per_level == g["per_level"] and len(t.node_token) == g["total"]
    assert (t.row_of_node >= 0).sum() == 1 + 6 + 36


def _check_level(rows, parents, plogp, ks, n_before, n_next, lv):
    """Properties any correct level has, from definitions other than the
    oracle's: the children are a top-k (nothing dropped is larger, or equal
    with a lower id), the path probability is the product of softmax
    probabilities, the chosen parents beat every other child."""
    i = 0
    for j, k in enumerate(ks):
        row = rows[j]
        kids = lv.node_token[i:i + k]
        assert len(set(kids)) == k
        for t in range(len(row)):
            if t in kids:
                continue
            for c in kids:
                assert row[t] < row[c] or (row[t] == row[c] and t > c)
        assert all(row[a] > row[b] or (row[a] == row[b] and a < b) for a, b in zip(kids, kids[1:]))
        prob = softmax(np.asarray(row, np.float64))
        for r, c in enumerate(kids):
            assert lv.node_parent[i + r] == parents[j]
            assert np.isclose(np.exp(lv.node_logp[i + r]), np.exp(plogp[j]) * prob[c], rtol=1e-12)
        i += k
    n = len(lv.node_token)
    ids = list(range(n_before + 1, n_before + 1 + n))
    chosen = set(lv.next_parents)
    assert len(chosen) == min(n_next, n) and lv.next_parents == sorted(chosen)
    for a in chosen:
        for b in set(ids) - chosen:
            la, lb = lv.node_logp[a - n_before - 1], lv.node_logp[b - n_before - 1]
            assert la > lb or (la == lb and a < b)


@pytest.mark.parametrize("seed", range(40))
def test_level_properties_random(seed):
    rng = np.random.default_rng(seed)
    H = int(rng.integers(1, 5))
    V = int(rng.integers(2, 40))
    ks = [int(rng.integers(1, min(V, 6) + 1)) for _ in range(H)]
    rows = rng.normal(0, 2, (H, V))
    if seed % 3 == 0:
        rows = np.round(rows * 2) / 2            # many exact ties
    if seed % 5 == 0:
        rows[0, rng.integers(0, V, 2)] = -np.inf  # masked tokens are fine
    parents = sorted(rng.choice(np.arange(1, 20), H, replace=False).tolist())
    plogp = (-rng.random(H) * 3).tolist()
    if seed % 4 == 0:
        plogp = [plogp[0]] * H                   # equal parent probabilities: ties across rows
    n_before = 20
    n_next = int(rng.integers(0, sum(ks) + 2))
    lv = O.expand_level(rows, parents, plogp, ks, n_before, n_next)
    assert lv.flags == 0
    _check_level(rows, parents, plogp, ks, n_before, n_next, lv)


def test_selection_brute_force_over_subsets():
    """Tiny levels: the chosen set is the unique subset of size n_next whose
    members all beat all non-members under (log-probability, lower id)."""
    rng = np.random.default_rng(7)
    for _ in range(200):
        H, V = 2, 5
        ks = [int(rng.integers(1, 4)), int(rng.integers(1, 4))]
        rows = np.round(rng.normal(0, 1, (H, V)) * 2) / 2
        plogp = [0.0, float(rng.choice([0.0, -0.5]))]
        n = sum(ks)
        n_next = int(rng.integers(1, n + 1))
        lv = O.expand_level(rows, [1, 2], plogp, ks, 2, n_next)
        ids = list(range(3, 3 + n))
        good = []
        for sub in itertools.combinations(ids, n_next):
            ok = all(lv.node_logp[a - 3] > lv.node_logp[b - 3] or
                     (lv.node_logp[a - 3] == lv.node_logp[b - 3] and a < b)
                     for a in sub for b in set(ids) - set(sub))
            if ok:
                good.append(list(sub))
        assert good == [lv.next_parents]


def test_bad_rows_flagged():
    rows = np.zeros((2, 8))
    rows[1, 3] = np.nan
    assert O.expand_level(rows, [0, 1], [0.0, 0.0], [1, 1], 0, 1).flags == TB.FLAG_BAD_ROW
    rows = np.full((1, 8), -np.inf)
    assert O.expand_level(rows, [0], [0.0], [2], 0, 1).flags == TB.FLAG_BAD_ROW
    rows = np.zeros((1, 8))
    rows[0, 2] = np.inf
    assert O.expand_level(rows, [0], [0.0], [2], 0, 1).flags == TB.FLAG_BAD_ROW


def test_boundary_flag_on_near_tie():
    rows = np.array([[0.0, 1e-7, -5.0]])
    lv = O.expand_level(rows, [0], [0.0], [2], 0, 1)
    assert lv.boundary and lv.next_parents == [1] and lv.node_token == [1, 0]
    lv = O.expand_level(np.array([[0.0, 0.5, -5.0]]), [0], [0.0], [2], 0, 1)
    assert not lv.boundary
    # tied siblings are decided by the node id in any precision: no boundary
    lv = O.expand_level(np.array([[0.5, 0.5, -5.0]]), [0], [0.0], [2], 0, 1)
    assert not lv.boundary and lv.next_parents == [1] and lv.node_token == [0, 1]
    # equal path probabilities under different parents are a boundary case
    lv = O.expand_level(np.array([[0.5, -5.0], [0.5, -5.0]]), [1, 2], [-1.0, -1.0], [1, 1], 2, 1)
    assert lv.boundary


@pytest.mark.parametrize("seed", range(3))
def test_host_generator_grows_the_oracle_tree(seed):
    """The seeded tree workloads (the verify inputs) have the builder's shape."""
    rng = np.random.default_rng(seed)
    spec, heads, V = ((6,), (2, 2), (1, 1)), (1, 2, 2), 300
    draft_rows = rng.normal(0, 3, (sum(heads), V)).astype(np.float32)
    g = W.grow_tree(draft_rows, spec, heads)
    lv_rows, r = [], 0
    for h in heads:
        lv_rows.append(draft_rows[r:r + h])
        r += h
    t = O.build_tree(lv_rows, spec, heads)
    np.testing.assert_array_equal(g.node_token, t.node_token)
    np.testing.assert_array_equal(g.node_parent, t.node_parent)
    np.testing.assert_array_equal(g.row_of_node, t.row_of_node)


def test_level_rows_are_the_tree_workloads_draft_rows():
    """make_tree_levels gives, level by level, the draft rows make_tree grows
    its trees from (f32, so no rounding between the two): the oracle's build
    from them is make_tree's tree."""
    import dataclasses
    s = dataclasses.replace(W.WORKLOADS[4], B=3, V=700, dtype="f32")
    levels = W.make_tree_levels(s, seed=6)
    tb = W.make_tree(s, seed=6)
    for b in range(s.B):
        rows = [lv[b * h:(b + 1) * h].double().numpy() for lv, h in zip(levels, s.topHead)]
        t = O.build_tree(rows, s.topKSpec, s.topHead)
        np.testing.assert_array_equal(t.node_token, tb.node_token[b])
        np.testing.assert_array_equal(t.node_parent, tb.node_parent[b])
        np.testing.assert_array_equal(t.row_of_node, tb.row_of_node[b])
