"""Pins for the oracle's candidate tree, mask, tokens and position ids (CPU only)."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import medusa_oracle as O

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_examples.json")))


def test_node_counts():
    for branching, n in GOLD["workload_node_counts"]["cases"]:
        assert O.node_count(branching) == n
    ex = GOLD["tree_example"]
    lay = O.tree_layout(ex["branching"])
    leaves = [n for n in range(lay["N"]) if lay["first_child"][n] == -1]
    assert len(leaves) == ex["leaf_paths"]


def _closure_mask(pairs, N):
    """The page's procedure: diagonal, (child, parent), then copy the parent's row."""
    m = np.full((N, N), -np.inf)
    for i in range(N):
        m[i, i] = 0.0
    for c, p in pairs:
        m[c, p] = 0.0
        for k in range(N):
            if m[p, k] == 0.0:
                m[c, k] = 0.0
    return m


@pytest.mark.parametrize("branching", [(3, 2, 2), (4, 3, 2, 1), (5, 3, 2, 1, 1), (2, 3, 2), (1, 1, 1, 1)])
def test_mask_three_ways(branching):
    lay = O.tree_layout(branching)
    N = lay["N"]
    mask = O.ancestor_mask(lay["parent"])
    # (1) rank-path prefixes: j is an ancestor-or-self of i iff path_j is a prefix of path_i
    brute = np.zeros((N, N), dtype=np.uint8)
    for i, j in itertools.product(range(N), range(N)):
        pi, pj = lay["paths"][i], lay["paths"][j]
        brute[i, j] = 1 if pi[:len(pj)] == pj else 0
    assert np.array_equal(mask, brute)
    # (2) the page's closure procedure on topologically ordered (child, parent) pairs
    pairs = [(c, int(lay["parent"][c])) for c in range(1, N)]
    closure = _closure_mask(pairs, N)
    assert np.array_equal(mask, (closure == 0.0).astype(np.uint8))


def test_chain_mask_is_lower_triangular():
    lay = O.tree_layout((1, 1, 1, 1, 1))
    mask = O.ancestor_mask(lay["parent"])
    assert np.array_equal(mask, np.tril(np.ones((6, 6), dtype=np.uint8)))


@pytest.mark.parametrize("branching", [(3, 2, 2), (4, 3, 2, 1), (5, 3, 2, 1, 1)])
def test_layout_closed_form(branching):
    """Level offsets: parent = off_{d-1} + t // s_d, first child = off_{d+1} + t * s_{d+1}."""
    lay = O.tree_layout(branching)
    cnt, off = [1], [0]
    for s in branching:
        off.append(off[-1] + cnt[-1])
        cnt.append(cnt[-1] * s)
    for d in range(len(branching) + 1):
        for t in range(cnt[d]):
            n = off[d] + t
            assert lay["depth"][n] == d
            if d > 0:
                s = branching[d - 1]
                assert lay["parent"][n] == off[d - 1] + t // s
                assert lay["rank"][n] == t % s
            if d < len(branching):
                assert lay["first_child"][n] == off[d + 1] + t * branching[d]
            else:
                assert lay["first_child"][n] == -1


def test_tokens_positions_and_bits():
    branching = (3, 2, 2)
    B, K = 2, 3
    rng = np.random.default_rng(0)
    topk = np.stack([np.stack([rng.permutation(100)[:3] for _ in range(K)]) for _ in range(B)])
    root = np.array([7, 42])
    L = np.array([10, 0])
    t = O.tree_build(branching, root, topk, L, L_cap=40)
    for b in range(B):
        assert t["tokens"][b, 0] == root[b]
        for n in range(1, t["N"]):
            path = O.tree_layout(branching)["paths"][n]
            assert t["tokens"][b, n] == topk[b, len(path) - 1, path[-1]]
            assert t["pos"][b, n] == L[b] + len(path)
    for i in range(t["N"]):
        for j in range(t["N"]):
            bit = (int(t["anc_bits"][i, j // 64]) >> (j % 64)) & 1
            assert bit == t["mask"][i, j]
    assert list(t["flags"]) == [0, 0]
    t2 = O.tree_build(branching, root, topk, np.array([30, 0]), L_cap=40)
    assert list(t2["flags"]) == [O.FLAG_CAPACITY, 0]
