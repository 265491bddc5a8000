"""Pins for the oracle's Medusa heads and top-s (CPU only)."""
import math

import numpy as np
import pytest

from oracle import medusa_oracle as O


def test_silu_closed_forms():
    x = np.array([0.0, 1.0, -1.0, 2.0, 40.0, -40.0])
    got = O.silu(x)
    want = [0.0, 1.0 / (1.0 + math.exp(-1.0)), -1.0 / (1.0 + math.exp(1.0)),
            2.0 / (1.0 + math.exp(-2.0)), 40.0, -40.0 * math.exp(-40.0)]
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-15)
    # x * sigmoid(x) at a spread of points
    xs = np.linspace(-8, 8, 33)
    np.testing.assert_allclose(O.silu(xs), [v * (1.0 / (1.0 + math.exp(-v))) for v in xs], rtol=1e-13)


def test_heads_hand_example():
    """d=3, V=2, one head, non-symmetric W and a bias: every term checked by hand."""
    h = np.array([[1.0, 0.0, -1.0]])
    W = np.array([[[0.0, 0.0, 0.0],     # out 0 <- nothing
                   [1.0, 0.0, 0.0],     # out 1 <- in 0
                   [0.0, 2.0, 1.0]]])   # out 2 <- 2*in 1 + in 2
    b = np.array([[0.5, 0.0, 0.0]])
    U = np.array([[[1.0, 1.0, 1.0],
                   [2.0, 0.0, -1.0]]])
    r, z = O.medusa_heads(h, W, b, U)
    sig = lambda v: 1.0 / (1.0 + math.exp(-v))
    pre = [0.5, 1.0, -1.0]
    r_want = [1.0 + pre[0] * sig(pre[0]), 0.0 + pre[1] * sig(pre[1]), -1.0 + pre[2] * sig(pre[2])]
    np.testing.assert_allclose(r[0, 0], r_want, rtol=1e-14)
    np.testing.assert_allclose(z[0, 0], [sum(r_want), 2 * r_want[0] - r_want[2]], rtol=1e-14)


def test_zero_residual_weights_reduce_to_gemv():
    """W = 0 and b = 0 give SiLU(0) = 0, so r = h and the logits are U h."""
    rng = np.random.default_rng(1)
    B, K, d, V = 2, 3, 7, 11
    h = rng.standard_normal((B, d))
    U = rng.standard_normal((K, V, d))
    r, z = O.medusa_heads(h, np.zeros((K, d, d)), None, U)
    for b in range(B):
        for k in range(K):
            assert np.array_equal(r[b, k], h[b])
            for v in range(V):
                acc = 0.0
                for i in range(d):
                    acc += U[k, v, i] * h[b, i]
                assert abs(z[b, k, v] - acc) < 1e-12


def test_bias_enters_before_silu():
    rng = np.random.default_rng(2)
    d, V = 5, 4
    h = rng.standard_normal((1, d))
    W = rng.standard_normal((1, d, d))
    b = rng.standard_normal((1, d))
    U = rng.standard_normal((1, V, d))
    r, _ = O.medusa_heads(h, W, b, U)
    for o in range(d):
        pre = sum(W[0, o, i] * h[0, i] for i in range(d)) + b[0, o]
        assert abs(r[0, 0, o] - (h[0, o] + pre / (1 + math.exp(-pre)))) < 1e-12


def _select_top(row, s):
    """Brute force: repeatedly take the largest remaining value, lowest index first."""
    taken = []
    for _ in range(s):
        best = None
        for v in range(len(row)):
            if v in taken:
                continue
            if best is None or row[v] > row[best]:
                best = v
        taken.append(best)
    return taken


@pytest.mark.parametrize("seed", range(6))
def test_top_s_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    row = np.round(rng.standard_normal(60), 1)     # rounding forces exact ties
    for s in (1, 3, 8):
        idx, _ = O.top_s(row, s)
        assert list(idx) == _select_top(row, s)


def test_top_s_ties_to_lower_index_and_flag():
    row = np.array([0.0, 5.0, 3.0, 5.0, 1.0])
    idx, near = O.top_s(row, 2)
    assert list(idx) == [1, 3] and near
    idx, near = O.top_s(np.array([0.0, 5.0, 3.0, 4.0]), 2)
    assert list(idx) == [1, 3] and not near


def test_shared_vocab_hand_example():
    """Two heads, different residual layers, one shared vocab projection U [V][d]
    (the frozen LM-head option): each head's logits are U r_k, summed by hand."""
    h = np.array([[2.0, -1.0]])
    W = np.array([[[1.0, 0.0], [0.0, 0.0]],      # head 0: out 0 <- in 0
                  [[0.0, 0.0], [0.0, -3.0]]])    # head 1: out 1 <- -3 in 1
    U = np.array([[1.0, 2.0],
                  [0.0, -1.0],
                  [3.0, 1.0]])
    r, z = O.medusa_heads(h, W, None, U)
    sig = lambda v: 1.0 / (1.0 + math.exp(-v))
    r0 = [2.0 + 2.0 * sig(2.0), -1.0 + 0.0]
    r1 = [2.0 + 0.0, -1.0 + 3.0 * sig(3.0)]
    for k, rk in enumerate((r0, r1)):
        np.testing.assert_allclose(r[0, k], rk, rtol=1e-14)
        want = [sum(U[v][i] * rk[i] for i in range(2)) for v in range(3)]
        np.testing.assert_allclose(z[0, k], want, rtol=1e-14)


def test_shared_vocab_zero_residual_is_one_gemv_for_all_heads():
    """W = 0: every head's logits are the same U h (brute-force loops)."""
    rng = np.random.default_rng(7)
    B, K, d, V = 2, 3, 5, 6
    h = rng.standard_normal((B, d))
    U = rng.standard_normal((V, d))
    _, z = O.medusa_heads(h, np.zeros((K, d, d)), None, U)
    for b in range(B):
        want = [sum(U[v, i] * h[b, i] for i in range(d)) for v in range(V)]
        for k in range(K):
            np.testing.assert_allclose(z[b, k], want, rtol=1e-12)
