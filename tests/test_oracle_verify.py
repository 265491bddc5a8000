"""Pins for the oracle's acceptance walks and rejection-sampling primitives (CPU only)."""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import medusa_oracle as O
from medusa_speculative_decoding_heads_gb300.synth import philox_uniforms

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_examples.json")))


def _one_hot_logits(N, V, want, hi=5.0):
    t = np.zeros((N, V))
    for n, w in enumerate(want):
        t[n, w] = hi
    return t


def _chain_tree(K, drafts, root=9):
    branching = (1,) * K
    topk = np.array([[[d] for d in drafts]])
    return O.tree_build(branching, np.array([root]), topk, np.array([0]))


# --------------------------------------------------------------------------- greedy
def test_chain_rollback_example():
    ex = GOLD["chain_rollback"]
    drafts = ex["drafts"]
    K = len(drafts)
    tree = _chain_tree(K, drafts)
    # target predictions: after root -> 1, after 1 -> 2, after 2 -> 0 (mismatch with draft 3)
    t = _one_hot_logits(tree["N"], 16, [1, 2, ex["correction"], 4, 5])
    acc, path, out, n_out = O.verify_greedy(tree["tokens"][0], tree["parent"], t, K)
    assert acc == ex["accepted_prefix"]
    assert list(out[:n_out]) == ex["emitted"]
    assert list(path[:acc + 1]) == [0, 1, 2]
    assert all(v == -1 for v in out[n_out:])


def test_all_match_yields_K_plus_one():
    ex = GOLD["all_match_bonus"]
    K = ex["K"]
    drafts = [3, 1, 4, 1, 5]
    tree = _chain_tree(K, drafts)
    t = _one_hot_logits(tree["N"], 16, drafts + [9])
    acc, path, out, n_out = O.verify_greedy(tree["tokens"][0], tree["parent"], t, K)
    assert acc == K and n_out == ex["n_out"]
    assert list(out) == drafts + [9]


@pytest.mark.parametrize("seed", range(20))
def test_tokens_per_step_range_on_trees(seed):
    rng = np.random.default_rng(seed)
    branching = (4, 3, 2, 1)
    K = len(branching)
    V = 12
    topk = np.stack([rng.permutation(V)[:4] for _ in range(K)])[None]
    tree = O.tree_build(branching, np.array([0]), topk, np.array([0]))
    t = rng.integers(0, 3, size=(tree["N"], V)).astype(float)   # many exact ties
    acc, path, out, n_out = O.verify_greedy(tree["tokens"][0], tree["parent"], t, K)
    assert 1 <= n_out <= K + 1 and n_out == acc + 1
    # walk validity: each accepted node is a child of the previous and carries the argmax token
    for r in range(1, acc + 1):
        assert tree["parent"][path[r]] == path[r - 1]
        assert tree["tokens"][0, path[r]] == int(np.argmax(t[path[r - 1]]))
    # the stop is real: no child of the last node carries the argmax (unless a leaf)
    last = path[acc]
    if tree["depth"][last] < K:
        want = int(np.argmax(t[last]))
        assert all(tree["tokens"][0, c] != want for c in O.children_of(tree["parent"], last))
    assert out[acc] == int(np.argmax(t[last]))


def _toy_next(ctx):
    """A deterministic toy target: next token from the last two tokens."""
    return (7 * ctx[-1] + 3 * ctx[-2] + len(ctx)) % 13


def test_greedy_output_equals_target_argmax_sequence():
    """Speculative greedy decoding reproduces plain greedy decoding exactly."""
    V, branching = 13, (3, 2, 2)
    K = len(branching)
    steps = 40
    rng = np.random.default_rng(11)
    ar = [1, 2]
    while len(ar) < 2 + steps * (K + 1) + 1:
        ar.append(_toy_next(ar))
    seq = [1, 2]
    lay = O.tree_layout(branching)
    for _ in range(steps):
        if len(seq) > 2 + steps:
            break
        # drafts: per depth, the true future token with probability 0.6 among random others
        topk = np.zeros((1, K, max(branching)), dtype=np.int64)
        future = []
        c2 = list(seq)
        for k in range(K):
            nt = _toy_next(c2)
            future.append(nt)
            c2.append(nt)
        for k in range(K):
            cands = list(rng.permutation(V)[:branching[k]])
            if rng.random() < 0.6 and future[k] not in cands:
                cands[rng.integers(branching[k])] = future[k]
            topk[0, k, :branching[k]] = cands
        root = seq[-1]
        tree = O.tree_build(branching, np.array([root]), topk, np.array([0]))
        # target logits of node n: one-hot at the toy target's next token after the node's context
        t = np.zeros((tree["N"], V))
        for n in range(tree["N"]):
            chain = []
            j = n
            while j > 0:
                chain.append(int(tree["tokens"][0, j]))
                j = int(tree["parent"][j])
            ctx = seq + chain[::-1]
            t[n, _toy_next(ctx)] = 1.0
        acc, path, out, n_out = O.verify_greedy(tree["tokens"][0], tree["parent"], t, K)
        seq.extend(int(x) for x in out[:n_out])
    assert seq == ar[:len(seq)]
    assert len(seq) > 2 + steps          # speculation made progress beyond one token per step


# --------------------------------------------------------------------------- rejection sampling
def _pq(seed, V=8):
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V) * 0.7)
    return p, q


@pytest.mark.parametrize("seed", range(5))
def test_exact_enumeration_single_draft(seed):
    """sum_x q(x) [1{y=x} a(x) + (1 - a(x)) res(y)] = p(y)."""
    p, q = _pq(seed)
    V = p.shape[0]
    res = O.residual(p, q)
    final = np.zeros(V)
    for x in range(V):
        a = O.acceptance_ratio(p, q, x)
        final[x] += q[x] * a
        final += q[x] * (1 - a) * res
    np.testing.assert_allclose(final, p, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(5))
def test_exact_enumeration_two_iid_drafts_residual_carried(seed):
    p, q = _pq(seed)
    V = p.shape[0]
    final = np.zeros(V)
    for x1, x2 in itertools.product(range(V), range(V)):
        w = q[x1] * q[x2]
        a1 = O.acceptance_ratio(p, q, x1)
        final[x1] += w * a1
        p1 = O.residual(p, q)
        a2 = O.acceptance_ratio(p1, q, x2)
        final[x2] += w * (1 - a1) * a2
        final += w * (1 - a1) * (1 - a2) * O.residual(p1, q)
    np.testing.assert_allclose(final, p, rtol=0, atol=1e-12)


def test_residual_sums_to_one_and_degenerate_case():
    p, q = _pq(9)
    r = O.residual(p, q)
    assert abs(r.sum() - 1) < 1e-14 and (r >= 0).all()
    assert np.array_equal(O.residual(p, p), p)


def test_inverse_cdf_brute_force():
    rng = np.random.default_rng(4)
    w = rng.random(20)
    w[3] = 0.0
    tot = sum(w)
    for u in np.linspace(0, 0.999, 97):
        y, _ = O.inverse_cdf(w, u)
        acc, ref = 0.0, None
        for v in range(20):
            acc += w[v]
            if acc > u * tot:
                ref = v
                break
        assert y == ref and w[y] > 0


def _tree_walk_first_token(p, q, s, n, seed, T=1.0):
    """First emitted token of the tree walk, depth-1 tree whose s drafts are sampled from q.

    The logits handed to the walk are T * log(p) and T * log(q), so a walk that
    divides by T before its softmax sees exactly p and q."""
    V = p.shape[0]
    branching = (s,)
    t_log = T * np.log(p)[None].repeat(1 + s, axis=0)
    h_log = T * np.log(q)[None]
    counts = np.zeros(V)
    ks = np.arange(n)
    ud = philox_uniforms(seed, ks[:, None], np.arange(s)[None, :], 10)
    ua = philox_uniforms(seed, ks[:, None], np.arange(s)[None, :], 11)
    ur = philox_uniforms(seed, ks, np.zeros(n, dtype=np.uint32), 12)
    lay = O.tree_layout(branching)
    for i in range(n):
        drafts = [O.inverse_cdf(q, float(ud[i, j]))[0] for j in range(s)]
        tokens = np.array([0] + drafts)
        acc, path, out, n_out, _ = O.verify_rejection(
            tokens, lay["parent"], t_log, h_log, ua[i][None, :], np.array([ur[i], 0.5]), 1, T)
        counts[out[0]] += 1
    return counts / n


@pytest.mark.parametrize("s", [1, 2])
def test_monte_carlo_tree_walk_preserves_target(s):
    ex = GOLD["rs_monte_carlo"]
    p, q = _pq(21)
    emp = _tree_walk_first_token(p, q, s, ex["samples"], seed=5 + s)
    tvd = 0.5 * np.abs(emp - p).sum()
    assert tvd < ex["tvd_tolerance"]


def _rs_chain_alpha_setup(K):
    q = np.array([0.4, 0.1, 0.1, 0.1, 0.1, 0.1, 0.05, 0.05])
    p = np.array([0.3, 0.2, 0.1, 0.1, 0.1, 0.1, 0.05, 0.05])      # p(0)/q(0) = 0.75
    tree = O.tree_build((1,) * K, np.array([5]), np.zeros((1, K, 1), dtype=np.int64), np.array([0]))
    t_log = np.log(p)[None].repeat(tree["N"], axis=0)
    h_log = np.log(q)[None].repeat(K, axis=0)
    return tree, t_log, h_log


def test_expected_tokens_closed_form_and_page_numbers():
    ex = GOLD["expected_tokens"]
    e = O.expected_tokens_per_step(ex["alpha"], ex["K"])
    assert abs(e - (1 - ex["alpha"] ** (ex["K"] + 1)) / (1 - ex["alpha"])) < 1e-12
    assert round(e, 4) == ex["theory"]
    assert round(100 * (1 - 1 / ex["simulated_on_page"]), 2) == ex["fewer_forwards_pct_from_simulated"]
    assert round(100 * abs(ex["simulated_on_page"] - ex["theory"]) / ex["theory"], 2) == ex["page_relative_error_pct"]
    fb = GOLD["fewer_forwards_bullets"]
    for a, pct in zip(fb["alpha_reading"], fb["fewer_forwards_pct"]):
        assert round(100 * (1 - 1 / O.expected_tokens_per_step(a, fb["K"]))) == pct


def test_expected_tokens_simulation():
    """Chain of K=5 drafts each accepted with probability 0.75: mean tokens per step -> 3.2881."""
    ex = GOLD["expected_tokens"]
    K = ex["K"]
    tree, t_log, h_log = _rs_chain_alpha_setup(K)
    steps = 30000
    ua = philox_uniforms(77, np.arange(steps)[:, None], np.arange(K)[None, :], 0)
    ur = philox_uniforms(77, np.arange(steps)[:, None], np.arange(K + 1)[None, :], 1)
    total = 0
    for i in range(steps):
        acc, path, out, n_out, _ = O.verify_rejection(
            tree["tokens"][0], tree["parent"], t_log, h_log, ua[i][:, None], ur[i], K, 1.0)
        assert 1 <= n_out <= K + 1
        total += n_out
    mean = total / steps
    assert abs(mean - ex["theory"]) / ex["theory"] < 0.01


def test_rs_walk_accepts_everything_when_target_equals_draft_and_u_small():
    K = 3
    tree, t_log, _ = _rs_chain_alpha_setup(K)
    h_log = t_log[:K]
    acc, path, out, n_out, flags = O.verify_rejection(
        tree["tokens"][0], tree["parent"], t_log, h_log, np.full((K, 1), 0.5), np.full(K + 1, 0.1), K, 1.0)
    assert acc == K and n_out == K + 1 and flags == 0


# --------------------------------------------------------------------------- planted mistakes
def test_pins_catch_a_swapped_residual(monkeypatch):
    """A residual written as max(0, q - p) breaks the exact-enumeration pin."""
    def wrong(p, q):
        w = np.maximum(0.0, q - p)
        return w / w.sum()
    monkeypatch.setattr(O, "residual", wrong)
    p, q = _pq(0)
    res = O.residual(p, q)
    final = np.zeros(p.shape[0])
    for x in range(p.shape[0]):
        a = O.acceptance_ratio(p, q, x)
        final[x] += q[x] * a
        final += q[x] * (1 - a) * res
    assert np.abs(final - p).max() > 1e-3


def test_pins_catch_a_walk_that_forgets_the_residual(monkeypatch):
    """Testing every sibling against the original p biases the output law."""
    monkeypatch.setattr(O, "residual", lambda p, q: p)
    p, q = _pq(21)
    emp = _tree_walk_first_token(p, q, 2, 40000, seed=3)
    assert 0.5 * np.abs(emp - p).sum() > GOLD["rs_monte_carlo"]["tvd_tolerance"]


# --------------------------------------------------------------------------- temperature
# "Medusa 심층 아키텍처", section "수학적 무손실 보장": p and q are the target's and the
# draft's distributions at the sampling temperature, softmax(logits / T). The pins
# below fix the division by T without restating it: logits built as T * log(w)
# must give back w / sum(w) exactly, T -> 0 must give the argmax and T -> inf the
# uniform law, and the walk fed T * log(p) must emit p.
TEMPS = (0.5, 0.7, 1.3, 2.0)


def _softmax_t_weight_error(T):
    """max |softmax_t(T log w + c, T) - w / sum w| over a few positive weight vectors."""
    worst = 0.0
    for w in ([1.0, 2.0, 3.0, 4.0], [0.05, 0.7, 0.25], [3.0, 1.0, 1.0, 1.0, 2.0, 0.5, 0.25, 0.25]):
        w = np.array(w)
        for c in (0.0, -17.5, 40.0):              # a constant shift of every logit changes nothing
            got = O.softmax_t(T * np.log(w) + c, T)
            worst = max(worst, float(np.abs(got - w / w.sum()).max()))
    return worst


@pytest.mark.parametrize("T", TEMPS)
def test_softmax_t_recovers_weights(T):
    assert _softmax_t_weight_error(T) < 1e-14


def test_softmax_t_hand_values():
    """Two-token cases worked by hand: logits (0, ln 2) at T = 1/2 are (0, ln 4) -> (1/5, 4/5);
    at T = 2 they are (0, ln sqrt 2) -> (1/(1+sqrt 2), sqrt 2/(1+sqrt 2)); logits (0, ln 3) at
    T = 0.7 weigh 1 : 3^(1/0.7)."""
    x = np.array([0.0, math.log(2.0)])
    np.testing.assert_allclose(O.softmax_t(x, 0.5), [0.2, 0.8], rtol=0, atol=1e-15)
    r2 = math.sqrt(2.0)
    np.testing.assert_allclose(O.softmax_t(x, 2.0), [1 / (1 + r2), r2 / (1 + r2)], rtol=0, atol=1e-15)
    w = 3.0 ** (1 / 0.7)                                   # 4.797... : ln 3 / 0.7 exponentiated
    np.testing.assert_allclose(O.softmax_t(np.array([0.0, math.log(3.0)]), 0.7), [1 / (1 + w), w / (1 + w)],
                               rtol=0, atol=1e-15)


def test_softmax_t_limits():
    """T -> 0 concentrates on the largest logit; T -> inf spreads evenly."""
    x = np.array([0.3, 1.0, -2.0, 0.99, 1.0 - 1e-3])
    cold = O.softmax_t(x, 1e-5)
    assert abs(cold[1] - 1.0) < 1e-12 and cold.sum() == pytest.approx(1.0, abs=1e-15)
    hot = O.softmax_t(x, 1e6)
    np.testing.assert_allclose(hot, np.full(5, 0.2), rtol=0, atol=1e-6)
    # a lower temperature sharpens: the largest probability grows as T falls
    tops = [O.softmax_t(x, T).max() for T in (4.0, 2.0, 1.0, 0.7, 0.5)]
    assert all(a < b for a, b in zip(tops, tops[1:]))


@pytest.mark.parametrize("T", (0.7, 2.0))
@pytest.mark.parametrize("seed", range(3))
def test_exact_enumeration_tempered(T, seed):
    """The single-draft rule at temperature T on vocab 8: p and q come from logits T log p0
    and T log q0, the enumerated output law is p0 to 1e-12."""
    p0, q0 = _pq(seed)
    p = O.softmax_t(T * np.log(p0), T)
    q = O.softmax_t(T * np.log(q0), T)
    V = p0.shape[0]
    res = O.residual(p, q)
    final = np.zeros(V)
    for x in range(V):
        a = O.acceptance_ratio(p, q, x)
        final[x] += q[x] * a
        final += q[x] * (1 - a) * res
    np.testing.assert_allclose(final, p0, rtol=0, atol=1e-12)


def test_monte_carlo_tree_walk_tempered():
    """The tree walk at T = 0.7 with drafts sampled from q emits p: target and head
    logits are T log p and T log q, 150k samples, total variation below 0.01."""
    ex = GOLD["rs_monte_carlo"]
    p, q = _pq(21)
    emp = _tree_walk_first_token(p, q, 2, ex["samples"], seed=41, T=0.7)
    assert 0.5 * np.abs(emp - p).sum() < ex["tvd_tolerance"]


def test_pins_catch_a_temperature_multiplied_instead_of_divided(monkeypatch):
    """softmax(x * T) in place of softmax(x / T) fails the weight pin, the hand values and the
    tempered walk."""
    def wrong(x, T):
        y = np.asarray(x, dtype=np.float64) * T
        e = np.exp(y - y.max())
        return e / e.sum()
    monkeypatch.setattr(O, "softmax_t", wrong)
    for T in TEMPS:
        assert _softmax_t_weight_error(T) > 1e-2
    with pytest.raises(AssertionError):
        test_softmax_t_hand_values()
    p, q = _pq(21)
    emp = _tree_walk_first_token(p, q, 2, 20000, seed=43, T=0.7)
    assert 0.5 * np.abs(emp - p).sum() > GOLD["rs_monte_carlo"]["tvd_tolerance"]


def test_pins_catch_a_temperature_ignored(monkeypatch):
    """A softmax that forgets T fails the weight pin at every T != 1."""
    monkeypatch.setattr(O, "softmax_t", lambda x, T: _plain_softmax(x))
    for T in TEMPS:
        assert _softmax_t_weight_error(T) > 1e-2


def _plain_softmax(x):
    y = np.asarray(x, dtype=np.float64)
    e = np.exp(y - y.max())
    return e / e.sum()
