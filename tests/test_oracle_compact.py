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


# --------------------------------------------------------------------------- paged cache (R15)
def _paged_case(seed, B=3, Hkv=2, D=4, P=4, N=7, pages=18):
    rng = np.random.default_rng(seed)
    L = np.array([3, 8, 5])[:B]
    bt = rng.permutation(pages)[:6 * B].reshape(B, 6)                  # every sequence owns its pages
    Kp = rng.standard_normal((pages, Hkv, P, D))
    Vp = rng.standard_normal((pages, Hkv, P, D))
    Kt = rng.standard_normal((B, Hkv, N, D))
    Vt = rng.standard_normal((B, Hkv, N, D))
    return rng, L, bt, Kp, Vp, Kt, Vt


def test_paged_rows_by_hand():
    pool = np.arange(4 * 1 * 2 * 1, dtype=float).reshape(4, 1, 2, 1)   # page p, row r -> value 2p + r
    bt = np.array([[2, 0, 3]])
    rows = O.paged_rows(pool, bt, 0, 5, 2)
    assert rows[0, :, 0].tolist() == [4, 5, 0, 1, 6]                 # pages 2, 0, 3


def test_paged_attention_equals_contiguous():
    """The paged prefix plus staged tree rows give the same output as one contiguous cache."""
    _, L, bt, Kp, Vp, Kt, Vt = _paged_case(3)
    B, Hkv, N, D, P = 3, 2, 7, 4, 4
    lay = O.tree_layout((2, 2))
    assert lay["N"] == N
    mask = O.ancestor_mask(lay["parent"])
    rng = np.random.default_rng(4)
    Q = rng.standard_normal((B, N, 4, D))
    cap = int(L.max()) + N
    Kc = np.zeros((B, Hkv, cap, D))
    Vc = np.zeros((B, Hkv, cap, D))
    for b in range(B):
        for i in range(int(L[b])):        # the definition of the layout, row by row
            Kc[b, :, i] = Kp[bt[b, i // P], :, i % P]
            Vc[b, :, i] = Vp[bt[b, i // P], :, i % P]
        Kc[b, :, L[b]:L[b] + N] = Kt[b]
        Vc[b, :, L[b]:L[b] + N] = Vt[b]
    want = O.tree_attention(Q, Kc, Vc, L, mask, 4, Hkv)
    got = O.tree_attention_paged(Q, Kp, Vp, bt, P, Kt, Vt, L, mask, 4, Hkv)
    np.testing.assert_allclose(got, want, rtol=1e-13)


def test_paged_commit_equals_logical_compaction_in_every_layer():
    """Commit into pages (two layers) = R11 compaction of the logical cache whose rows
    L_b.. hold the tree; rows outside [L_b, L_b + acc] and other pages are untouched."""
    _, L, bt, Kp, Vp, Kt, Vt = _paged_case(5)
    P, N = 4, 7
    Kp2, Vp2, Kt2, Vt2 = Kp * 2, Vp * 3, Kt - 1, Vt + 1
    acc = np.array([0, 2, 1])
    path = np.array([[0, -1, -1], [0, 1, 3], [0, 2, -1]])
    kps, vps, L2, kv_map = O.kv_commit_paged([Kp, Kp2], [Vp, Vp2], bt, P, [Kt, Kt2], [Vt, Vt2], L, acc, path)
    assert L2.tolist() == [4, 11, 7] and kv_map.tolist() == [[0, -1, -1], [0, 1, 3], [0, 2, -1]]
    for layer, (K0, Ktl, Kn) in enumerate(zip((Kp, Kp2), (Kt, Kt2), kps)):
        for b in range(3):
            cap = int(L[b]) + N
            logical = np.zeros((1, 2, cap, 4))
            logical[0, :, :L[b]] = O.paged_rows(K0, bt, b, int(L[b]), P)
            logical[0, :, L[b]:] = Ktl[b]
            want, _, _, _ = O.kv_compact(logical, logical, np.array([L[b]]), acc[b:b + 1], path[b:b + 1])
            n = int(acc[b]) + 1
            np.testing.assert_array_equal(O.paged_rows(Kn, bt, b, int(L[b]) + n, P), want[0, :, :L[b] + n])
        touched = {(int(bt[b, (L[b] + r) // P]), (L[b] + r) % P) for b in range(3) for r in range(acc[b] + 1)}
        for page in range(K0.shape[0]):
            for off in range(P):
                if (page, off) not in touched:
                    np.testing.assert_array_equal(Kn[page, :, off], K0[page, :, off])
