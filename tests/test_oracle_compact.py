"""Pins for the oracle's KV compaction (CPU only)."""
import numpy as np
import pytest

from oracle import medusa_oracle as O


def _cache(B, H, L_cap, D, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((B, H, L_cap, D)), rng.standard_normal((B, H, L_cap, D))


def test_nothing_accepted_keeps_the_root_only():
    Kc, Vc = _cache(1, 2, 20, 4, 0)
    path = np.array([[0, -1, -1, -1, -1]])
    K2, V2, L2, kv_map = O.kv_compact(Kc, Vc, np.array([7]), np.array([0]), path)
    assert np.array_equal(K2, Kc) and np.array_equal(V2, Vc)
    assert list(L2) == [8] and list(kv_map[0]) == [0, -1, -1, -1, -1]


def test_all_accepted_chain_is_the_identity():
    Kc, Vc = _cache(2, 3, 30, 4, 1)
    path = np.array([[0, 1, 2, 3, 4]] * 2)
    K2, V2, L2, kv_map = O.kv_compact(Kc, Vc, np.array([3, 10]), np.array([4, 4]), path)
    assert np.array_equal(K2, Kc) and np.array_equal(V2, Vc)
    assert list(L2) == [8, 15]


@pytest.mark.parametrize("seed", range(10))
def test_random_tree_paths_against_a_gather(seed):
    rng = np.random.default_rng(seed)
    branching = (4, 3, 2, 1)
    lay = O.tree_layout(branching)
    N, K = lay["N"], len(branching)
    B, H, D = 3, 2, 8
    L = rng.integers(0, 12, size=B)
    L_cap = int(L.max()) + N + 2
    Kc, Vc = _cache(B, H, L_cap, D, seed)
    acc = rng.integers(0, K + 1, size=B)
    path = np.full((B, K + 1), -1)
    for b in range(B):
        cur, path[b, 0] = 0, 0
        for r in range(1, acc[b] + 1):
            kids = O.children_of(lay["parent"], cur)
            cur = kids[rng.integers(len(kids))]
            path[b, r] = cur
    K2, V2, L2, kv_map = O.kv_compact(Kc, Vc, L, acc, path)
    for b in range(B):
        Lb = int(L[b])
        for r in range(acc[b] + 1):
            src = Lb + int(path[b, r])
            assert np.array_equal(K2[b, :, Lb + r], Kc[b, :, src])
            assert np.array_equal(V2[b, :, Lb + r], Vc[b, :, src])
        # rows outside the destination range are untouched
        keep = [x for x in range(L_cap) if not (Lb <= x <= Lb + acc[b])]
        assert np.array_equal(K2[b][:, keep], Kc[b][:, keep])
        assert L2[b] == Lb + acc[b] + 1
        assert list(kv_map[b, :acc[b] + 1]) == list(path[b, :acc[b] + 1])
        assert all(v == -1 for v in kv_map[b, acc[b] + 1:])
