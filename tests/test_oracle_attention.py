"""Pins for the oracle's tree attention (CPU only)."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import medusa_oracle as O


def _inputs(B, N, Hq, Hkv, D, L, L_cap, seed):
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((B, N, Hq, D))
    Kc = rng.standard_normal((B, Hkv, L_cap, D))
    Vc = rng.standard_normal((B, Hkv, L_cap, D))
    return Q, Kc, Vc


@pytest.mark.parametrize("L0", [0, 1, 37])
def test_chain_tree_is_causal_attention(L0):
    """A chain tree (branching 1,...,1) is ordinary causal attention over L + N tokens."""
    branching = (1, 1, 1, 1)
    lay = O.tree_layout(branching)
    N = lay["N"]
    mask = O.ancestor_mask(lay["parent"])
    B, Hq, Hkv, D = 2, 4, 2, 16
    L = np.array([L0, L0 + 3])
    L_cap = int(L.max()) + N + 5
    Q, Kc, Vc = _inputs(B, N, Hq, Hkv, D, L, L_cap, 3)
    got = O.tree_attention(Q, Kc, Vc, L, mask, Hq, Hkv)
    G = Hq // Hkv
    for b in range(B):
        Lb = int(L[b])
        T = Lb + N
        # queries for the prefix are irrelevant; put the tree queries at the end of a causal sequence
        q = torch.zeros((Hq, T, D), dtype=torch.float64)
        q[:, Lb:, :] = torch.from_numpy(Q[b]).permute(1, 0, 2)
        k = torch.from_numpy(np.repeat(Kc[b, :, :T], G, axis=0))
        v = torch.from_numpy(np.repeat(Vc[b, :, :T], G, axis=0))
        ref = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        np.testing.assert_allclose(got[b], ref[:, Lb:, :].permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("branching", [(3, 2, 2), (4, 3, 2, 1)])
def test_tree_matches_masked_sdpa(branching):
    lay = O.tree_layout(branching)
    N = lay["N"]
    mask = O.ancestor_mask(lay["parent"])
    B, Hq, Hkv, D = 2, 8, 2, 32
    L = np.array([5, 19])
    L_cap = 19 + N + 3
    Q, Kc, Vc = _inputs(B, N, Hq, Hkv, D, L, L_cap, 4)
    got = O.tree_attention(Q, Kc, Vc, L, mask, Hq, Hkv)
    for b in range(B):
        Lb = int(L[b])
        T = Lb + N
        vis = torch.cat([torch.ones((N, Lb), dtype=torch.bool), torch.from_numpy(mask.astype(bool))], dim=1)
        for h in range(Hq):
            kv = h // (Hq // Hkv)
            q = torch.from_numpy(Q[b, :, h, :])[None]
            k = torch.from_numpy(Kc[b, kv, :T])[None]
            v = torch.from_numpy(Vc[b, kv, :T])[None]
            ref = F.scaled_dot_product_attention(q, k, v, attn_mask=vis[None])
            np.testing.assert_allclose(got[b, :, h, :], ref[0].numpy(), rtol=1e-10, atol=1e-12)


def test_lone_root_without_prefix_returns_its_value():
    mask = np.ones((1, 1), dtype=np.uint8)
    Q, Kc, Vc = _inputs(1, 1, 2, 1, 8, None, 4, 5)
    got = O.tree_attention(Q, Kc, Vc, np.array([0]), mask, 2, 1)
    for h in range(2):
        np.testing.assert_allclose(got[0, 0, h], Vc[0, 0, 0], rtol=0, atol=1e-15)


def test_two_keys_closed_form():
    """One committed key plus the root: weights e^{s_i} / (e^{s_0} + e^{s_1})."""
    mask = np.ones((1, 1), dtype=np.uint8)
    D = 4
    Q = np.array([[[[1.0, 0.0, 0.0, 0.0]]]])
    Kc = np.zeros((1, 1, 2, D)); Vc = np.zeros((1, 1, 2, D))
    Kc[0, 0, 0] = [2.0, 0, 0, 0]; Kc[0, 0, 1] = [-2.0, 0, 0, 0]
    Vc[0, 0, 0] = [1.0, 0, 0, 0]; Vc[0, 0, 1] = [0, 1.0, 0, 0]
    got = O.tree_attention(Q, Kc, Vc, np.array([1]), mask, 1, 1)
    s0, s1 = 2.0 / math.sqrt(D), -2.0 / math.sqrt(D)
    w0 = math.exp(s0) / (math.exp(s0) + math.exp(s1))
    np.testing.assert_allclose(got[0, 0, 0], [w0, 1 - w0, 0, 0], rtol=1e-14)


def test_branches_do_not_interfere():
    """Changing a node's key/value changes only the outputs of its descendants (and itself)."""
    branching = (2, 2)
    lay = O.tree_layout(branching)
    N = lay["N"]
    mask = O.ancestor_mask(lay["parent"])
    Q, Kc, Vc = _inputs(1, N, 2, 2, 8, None, 10 + N, 6)
    L = np.array([10])
    base = O.tree_attention(Q, Kc, Vc, L, mask, 2, 2)
    j = 1                                   # first depth-1 node
    Kc2, Vc2 = Kc.copy(), Vc.copy()
    Kc2[0, :, 10 + j] += 1.0
    Vc2[0, :, 10 + j] -= 2.0
    alt = O.tree_attention(Q, Kc2, Vc2, L, mask, 2, 2)
    for i in range(N):
        changed = not np.allclose(base[0, i], alt[0, i])
        assert changed == bool(mask[i, j])


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_block_partials_merge_to_the_one_pass_result(seed):
    """Attention over key blocks merged by running max and exp-sum equals one softmax over all
    keys (float64 SDPA), for random block sizes, an empty block and a block whose keys are all
    masked; the order of the blocks does not matter."""
    rng = np.random.default_rng(seed)
    D, T = 16, 300
    q = rng.standard_normal(D)
    keys = 3.0 * rng.standard_normal((T, D))
    vals = rng.standard_normal((T, D))
    visible = rng.random(T) < 0.8
    visible[200:230] = False                       # a fully masked block below
    cuts = sorted(set([0, 17, 17, 128, 200, 230, 256, T]))
    parts = [O.attention_block_partial(q, keys[a:b], vals[a:b], visible[a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
    parts.append(O.attention_block_partial(q, keys[:0], vals[:0], visible[:0]))   # an empty block
    ref = F.scaled_dot_product_attention(torch.from_numpy(q)[None, None], torch.from_numpy(keys)[None],
                                         torch.from_numpy(vals)[None],
                                         attn_mask=torch.from_numpy(visible)[None, None])[0, 0].numpy()
    np.testing.assert_allclose(O.merge_attention_partials(parts), ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(O.merge_attention_partials(parts[::-1]), ref, rtol=1e-12, atol=1e-13)


def test_two_one_key_blocks_closed_form():
    """Blocks holding one key each merge to the two-key softmax weights e^{s_i} / (e^{s_0} + e^{s_1})."""
    D = 4
    q = np.array([1.0, 0, 0, 0])
    k0, k1 = np.array([[3.0, 0, 0, 0]]), np.array([[-1.0, 0, 0, 0]])
    v0, v1 = np.array([[1.0, 0, 0, 0]]), np.array([[0, 1.0, 0, 0]])
    one = np.ones(1, dtype=bool)
    out = O.merge_attention_partials([O.attention_block_partial(q, k0, v0, one),
                                      O.attention_block_partial(q, k1, v1, one)])
    s0, s1 = 3.0 / math.sqrt(D), -1.0 / math.sqrt(D)
    w0 = math.exp(s0) / (math.exp(s0) + math.exp(s1))
    np.testing.assert_allclose(out, [w0, 1 - w0, 0, 0], rtol=1e-14)
