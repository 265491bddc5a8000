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


# --------------------------------------------------------------------------- pruned trees (R13)
def test_paths_of_the_full_product_give_the_cartesian_layout():
    import itertools
    for branching in ((3, 2, 2), (4, 3, 2, 1), (2, 1, 3)):
        paths = [p for d in range(1, len(branching) + 1)
                 for p in itertools.product(*[range(s) for s in branching[:d]])]
        a = O.tree_layout(branching)
        b = O.tree_layout_from_paths(reversed(paths), branching)   # input order does not matter
        assert a["N"] == b["N"] and a["paths"] == b["paths"]
        for key in ("parent", "depth", "rank", "first_child"):
            assert np.array_equal(a[key], b[key]), key


def test_pruned_tree_by_hand():
    """Paths (0) (1) (2) (0,0) (0,2) (2,1) (0,0,1): node order, links and mask by hand."""
    paths = [(0,), (1,), (2,), (0, 0), (0, 2), (2, 1), (0, 0, 1)]
    lay = O.tree_layout_from_paths(paths, (3, 3, 2))
    assert lay["N"] == 8
    assert lay["paths"] == [(), (0,), (1,), (2,), (0, 0), (0, 2), (2, 1), (0, 0, 1)]
    assert list(lay["parent"]) == [-1, 0, 0, 0, 1, 1, 3, 4]
    assert list(lay["depth"]) == [0, 1, 1, 1, 2, 2, 2, 3]
    assert list(lay["rank"]) == [0, 0, 1, 2, 0, 2, 1, 1]
    assert list(lay["first_child"]) == [1, 4, -1, 6, 7, -1, -1, -1]
    mask = O.ancestor_mask(lay["parent"])
    want = {0: {0}, 1: {0, 1}, 2: {0, 2}, 3: {0, 3}, 4: {0, 1, 4}, 5: {0, 1, 5}, 6: {0, 3, 6}, 7: {0, 1, 4, 7}}
    for i in range(8):
        assert set(np.nonzero(mask[i])[0].tolist()) == want[i]
    # tokens: head d's candidate of the node's last rank
    topk = np.array([[[10, 11, 12], [20, 21, 22], [30, 31, -1]]])
    t = O.tree_build((3, 3, 2), np.array([99]), topk, np.array([5]), paths=paths)
    assert list(t["tokens"][0]) == [99, 10, 11, 12, 20, 22, 21, 31]
    assert list(t["pos"][0]) == [5, 6, 6, 6, 7, 7, 7, 8]


@pytest.mark.parametrize("bad", [[(0, 1)], [(3,)], [(0,), (0, 0, 0, 0)], [()]])
def test_pruned_tree_rejects_malformed_paths(bad):
    with pytest.raises(ValueError):
        O.tree_layout_from_paths(bad, (3, 2, 2))


def test_walks_stop_at_a_shallow_leaf():
    """A pruned tree whose accepted path ends at a leaf above depth K: greedy stops
    there with the target's argmax as the bonus; rejection sampling draws the bonus
    from that leaf's target distribution with the uniform of the leaf's depth."""
    paths = [(0,), (1,), (1, 0)]                 # node 1 = (0) is a leaf at depth 1 < K = 2
    t = O.tree_build((2, 1), np.array([7]), np.array([[[3, 4], [5, -1]]]), np.array([0]), paths=paths)
    V = 8
    tl = np.zeros((1, t["N"], V))
    tl[0, 0, 3] = 10.0                            # root prefers token 3 = node 1's token
    tl[0, 1, 6] = 10.0                            # node 1 prefers 6
    g = O.verify_batch(0, t, tl, K=2)
    assert g["acc"][0] == 1 and list(g["path"][0]) == [0, 1, -1] and list(g["out_tokens"][0]) == [3, 6, -1]
    z = np.zeros((1, 2, V))
    # p at the leaf = softmax(tl[1]): cdf(5) = 6/(e^10+7) ~ 2.7e-4, cdf(6) ~ 0.99995, so u = 0.5 draws 6
    # and u = 0.999999 draws 7: only the leaf's own uniform u_res[1] gives 6
    r = O.verify_batch(1, t, tl, K=2, head_logits=z, u_acc=np.array([[[0.0, 0.0], [0.0, 0.0]]]),
                       u_res=np.array([[0.999999, 0.5, 0.999999]]), T=1.0)
    assert r["acc"][0] == 1 and list(r["path"][0]) == [0, 1, -1]
    assert list(r["out_tokens"][0]) == [3, 6, -1]
