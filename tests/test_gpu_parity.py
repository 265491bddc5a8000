"""GPU parity: every library call against the float64 oracle on identical seeded inputs.

Integer outputs (tree arrays, tokens, positions, top-s indices, acceptance,
paths, KV map, compacted KV bytes) must match bit for bit, except where the
oracle flags a near tie that float32 may legitimately order differently.
Float outputs (head logits, attention) must satisfy
|gpu - oracle| <= tol * max(1, |oracle|) with tol = 1e-5 (float32) or 2e-2 (bf16).
"""
import numpy as np
import pytest
import torch

from medusa_speculative_decoding_heads_gb300 import binding as mb, configs, synth
from medusa_speculative_decoding_heads_gb300.configs import BF16, F32, GREEDY, REJECTION
from medusa_speculative_decoding_heads_gb300.step import DeviceStep, to_device_inputs
from oracle import medusa_oracle as O

from _helpers import (TIE_BITS, assert_close, compare_verify, f64, gpu_ready, i64, planted_greedy_logits,
                      random_topk)

pytestmark = pytest.mark.gpu

NAMES = configs.ORDER


def small(w):
    """A reduced case of workload w: same dtype, tree and batch; ragged sizes that span several tiles."""
    if w.name == "tiny_fp32":
        return w
    G = w.Hq // w.Hkv
    return configs.scaled(w, d=512, V=1000, Hq=2 * G, Hkv=2, L_range=(37, 300))


def layout(w):
    """The oracle's layout of the workload's tree (pruned or Cartesian)."""
    return O.tree_layout(w.branching) if w.tree_paths is None else O.tree_layout_from_paths(w.tree_paths, w.branching)


def oracle_tree(w, root, topk, L, L_cap):
    return O.tree_build(w.branching, np.asarray(root), np.asarray(topk), np.asarray(L), L_cap, paths=w.tree_paths)


# --------------------------------------------------------------------------- tree build
@pytest.mark.parametrize("name", NAMES + configs.PRUNED)
def test_tree_build_bit_exact(name):
    dev = gpu_ready()
    w = configs.get(name)
    rng = np.random.default_rng(1)
    L = synth.committed_lengths(3, w.B, *w.L_range)
    L_cap = synth.cache_capacity(L, w.N)
    L[-1] = L_cap - w.N + 1                      # one sequence over capacity
    root = synth.root_tokens(3, w.B, w.V)
    topk = random_topk(rng, w.B, w.K, w.s_max, w.branching, w.V)
    st = DeviceStep(w, w.modes[0], L_cap, dev)
    t_topk = torch.from_numpy(topk).to(dev)
    st.tree_build(torch.from_numpy(root).to(dev), torch.from_numpy(L).to(dev), topk=t_topk)
    torch.cuda.synchronize()
    ref = oracle_tree(w, root, topk, L, L_cap)
    assert np.array_equal(i64(st.parent), ref["parent"])
    assert np.array_equal(i64(st.depth), ref["depth"])
    assert np.array_equal(i64(st.first_child), ref["first_child"])
    assert np.array_equal(i64(st.mask), ref["mask"].astype(np.int64))
    assert np.array_equal(st.anc_bits.cpu().numpy().view(np.uint64), ref["anc_bits"])
    assert np.array_equal(i64(st.tokens), ref["tokens"])
    assert np.array_equal(i64(st.pos), ref["pos"])
    assert np.array_equal(i64(st.flags), ref["flags"])


# --------------------------------------------------------------------------- heads
def check_heads(w, si, st, rows=None):
    """Compare logits and top-s of (b, k) pairs (all when rows is None)."""
    h, W, U = f64(si.h), None, None
    pairs = rows if rows is not None else [(b, k) for b in range(w.B) for k in range(w.K)]
    z_gpu = st.logits.cpu().numpy()
    topk_gpu = st.topk.cpu().numpy()
    worst = 0.0
    checked = flagged = 0
    for k in sorted({k for _, k in pairs}):
        Wk = f64(si.W[k:k + 1])
        bk = None if si.bias is None else f64(si.bias[k:k + 1])
        Uk = f64(si.U) if w.shared_vocab else f64(si.U[k:k + 1])
        bs = sorted({b for b, kk in pairs if kk == k})
        _, z = O.medusa_heads(h[bs], Wk, bk, Uk)
        for j, b in enumerate(bs):
            worst = max(worst, assert_close(z_gpu[b, k], z[j, 0], w.dtype, f"logits b={b} k={k}"))
            idx, near = O.top_s(z[j, 0], w.branching[k])
            if near:
                flagged += 1
                continue
            checked += 1
            assert list(topk_gpu[b, k, :w.branching[k]]) == list(idx), f"top-s b={b} k={k}"
            assert all(v == -1 for v in topk_gpu[b, k, w.branching[k]:])
    assert checked > 0 and flagged <= max(1, len(pairs) // 10)
    return worst


@pytest.mark.parametrize("name", NAMES)
@pytest.mark.parametrize("with_bias", [False, True])
def test_heads_small(name, with_bias):
    dev = gpu_ready()
    w = small(configs.get(name))
    si = synth.make_step_inputs(w, seed=11, device=dev, with_bias=with_bias)
    st = DeviceStep(w, w.modes[0], si.L_cap, dev)
    st.heads(si.h, si.W, si.bias, si.U)
    torch.cuda.synchronize()
    check_heads(w, si, st)


@pytest.mark.parametrize("B", [1, 3, 9, 17, 32, 33, 70])
def test_heads_batch_tiles(B):
    """Every batch tiling of the tensor-core path (1, 2 and 4 tiles of 8) with ragged batches, and batches
    past 32 sequences (run as slices of 32, the last one ragged)."""
    dev = gpu_ready()
    w = configs.scaled(configs.get("vicuna7b_b1"), B=B, d=320, V=700, L_range=(40, 40), Hq=2, Hkv=2)
    si = synth.make_step_inputs(w, seed=B, device=dev, with_bias=True)
    st = DeviceStep(w, GREEDY, si.L_cap, dev)
    st.heads(si.h, si.W, si.bias, si.U)
    torch.cuda.synchronize()
    check_heads(w, si, st)


@pytest.mark.parametrize("base,B,d,V", [("vicuna7b_b1", 1, 320, 700), ("vicuna7b_b1", 9, 320, 700),
                                        ("vicuna7b_b1", 17, 320, 700), ("vicuna7b_b1", 32, 320, 700),
                                        ("vicuna13b_b8", 3, 320, 700), ("vicuna13b_b8", 16, 320, 700),
                                        ("vicuna13b_b8", 32, 320, 700), ("tiny_fp32", 2, None, None),
                                        ("vicuna7b_b1", 1, 128, 19585), ("vicuna7b_b1", 17, 128, 19600),
                                        ("vicuna13b_b8", 8, 192, 30000)])
def test_heads_shared_vocab(base, B, d, V):
    """One vocab projection for every head: one weight stream serving all heads' columns
    (head blocks of 16, 32 and 64 columns in MMAs of 64, 128 and 256), the per-head
    path when all heads do not fit one MMA (K = 5 with B = 32) and the float32 path.
    The larger vocabularies put more than one 128-row tile on every SM, one of them
    with V not a multiple of 4 (ragged last tile, scalar top-s loads)."""
    dev = gpu_ready()
    w0 = configs.get(base)
    kw = dict(B=B, shared_vocab=True)
    if base != "tiny_fp32":
        kw.update(d=d, V=V, L_range=(40, 40), Hq=2, Hkv=2)
    w = configs.scaled(w0, **kw)
    si = synth.make_step_inputs(w, seed=B + 100, device=dev, with_bias=True)
    assert tuple(si.U.shape) == (w.V, w.d)
    st = DeviceStep(w, w.modes[0], si.L_cap, dev)
    st.heads(si.h, si.W, si.bias, si.U)
    torch.cuda.synchronize()
    check_heads(w, si, st)


@pytest.mark.parametrize("name", NAMES[1:] + configs.SHARED)
def test_heads_full_size_sampled(name):
    dev = gpu_ready()
    w = configs.get(name)
    si = synth.make_step_inputs(configs.scaled(w, L_range=(64, 64), Hq=w.Hq // w.Hkv, Hkv=1), seed=5, device=dev)
    st = DeviceStep(w, w.modes[0], si.L_cap, dev)
    st.heads(si.h, si.W, si.bias, si.U)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    pairs = [(int(rng.integers(w.B)), k) for k in (0, w.K - 1)]
    check_heads(w, si, st, rows=pairs)


@pytest.mark.parametrize("groups", [1, 7, 37, 997])
@pytest.mark.parametrize("name", ["vicuna7b_b1", "vicuna13b_b8"])
def test_heads_topk_ties(name, groups):
    """Top-s under exact ties against the oracle's top-s: vocabulary row v of every head
    copies row v % groups, so each logit value repeats about V / groups times. The oracle
    computes the logits of the `groups` distinct rows and repeats them, so its ties are
    exact by construction, and orders by larger value first, lower index among equal
    values. A row is left out only where two *distinct* values at the top-s boundary lie
    closer than the oracle's near-tie band. Few groups put more tied entries at the
    threshold than the shortlist holds (the exact per-thread path); many groups take the
    shortlist path."""
    dev = gpu_ready()
    w = configs.scaled(configs.get(name), d=128, V=5000, L_range=(40, 40), Hq=2, Hkv=2)
    si = synth.make_step_inputs(w, seed=groups, device=dev)
    U = si.U.clone()
    src = torch.arange(w.V, device=dev) % groups
    U[:] = U[:, src]
    st = DeviceStep(w, w.modes[0], si.L_cap, dev)
    st.heads(si.h, si.W, si.bias, U)
    torch.cuda.synchronize()
    _, zg = O.medusa_heads(f64(si.h), f64(si.W), None if si.bias is None else f64(si.bias), f64(U[:, :groups]))
    z = zg[:, :, np.arange(w.V) % groups]
    topk = st.topk.cpu().numpy()
    checked = 0
    for b in range(w.B):
        for k in range(w.K):
            s = w.branching[k]
            want, _ = O.top_s(z[b, k], s)
            # distinct values reaching the top s, and the next one below them
            distinct = np.unique(z[b, k])[::-1]
            last = z[b, k, want[-1]]
            n_in = int(np.searchsorted(-distinct, -last, side="right"))
            edge = distinct[:n_in + 1]
            if np.any(edge[:-1] - edge[1:] < O.TOPK_TIE * np.maximum(1.0, np.abs(edge[:-1]))):
                continue
            checked += 1
            assert list(topk[b, k, :s]) == list(want), f"b={b} k={k}"
            assert all(v == -1 for v in topk[b, k, s:])
    assert checked >= (w.B * w.K + 1) // 2


# --------------------------------------------------------------------------- attention
def check_attention(w, si, O_gpu, pairs):
    tree = layout(w)
    mask = O.ancestor_mask(tree["parent"])
    G = w.Hq // w.Hkv
    worst = 0.0
    for b, kv in pairs:
        Lb = int(si.L[b])
        q = f64(si.Q[b:b + 1, :, kv * G:(kv + 1) * G])
        kc = f64(si.Kc[b:b + 1, kv:kv + 1, :Lb + w.N])
        vc = f64(si.Vc[b:b + 1, kv:kv + 1, :Lb + w.N])
        ref = O.tree_attention(q, kc, vc, np.array([Lb]), mask, G, 1)
        got = f64(O_gpu[b:b + 1, :, kv * G:(kv + 1) * G])
        worst = max(worst, assert_close(got, ref, w.dtype, f"attention b={b} kv={kv}"))
    return worst


def run_attention(w, si, dev):
    st = DeviceStep(w, w.modes[0], si.L_cap, dev)
    st.tree_build(torch.from_numpy(si.root_token).to(dev), torch.from_numpy(si.L).to(dev),
                  topk=torch.zeros((w.B, w.K, w.s_max), dtype=torch.int32, device=dev))
    st.tree_attention(si.Q, si.Kc, si.Vc, torch.from_numpy(si.L).to(dev))
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("name", NAMES + configs.PRUNED)
def test_attention_small_all_heads(name):
    dev = gpu_ready()
    w = small(configs.get(name))
    si = synth.make_step_inputs(w, seed=21, device=dev)
    st = run_attention(w, si, dev)
    check_attention(w, si, st.O, [(b, kv) for b in range(w.B) for kv in range(w.Hkv)])


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("L0", [0, 1, 31, 32, 33, 127, 128, 129, 511])
def test_attention_edge_lengths(L0, D):
    """Empty prefix, a single key, tile boundaries of every kernel (32/64/128-key tiles)."""
    dev = gpu_ready()
    w = configs.scaled(configs.get("gqa7b_b32"), B=2, d=64, V=64, L_range=(L0, L0), D=D)
    si = synth.make_step_inputs(w, seed=L0, device=dev)
    st = run_attention(w, si, dev)
    check_attention(w, si, st.O, [(b, kv) for b in range(w.B) for kv in range(w.Hkv)])


@pytest.mark.parametrize("name,D", [("tiny_fp32", None), ("vicuna7b_b1", 128), ("gqa7b_b32", 128),
                                    ("gqa7b_b32", 64)])
@pytest.mark.parametrize("Lmax", [100, 900])
def test_attention_invalid_sequences_get_zeros(name, D, Lmax):
    """A sequence with L_b < 0 or L_b + N > L_cap gets O = 0 (the header's contract), on every
    attention kernel (float32, tcgen05 with and without leftover rows, mma.sync at D = 64) with
    one KV range and with several; the valid sequences still match the oracle."""
    dev = gpu_ready()
    base = configs.get(name)
    G = base.Hq // base.Hkv
    kw = dict(B=4, d=64, V=64, Hq=2 * G, Hkv=2, L_range=(Lmax // 2, Lmax))
    if D is not None:
        kw["D"] = D
    w = configs.scaled(base, **kw)
    si = synth.make_step_inputs(w, seed=Lmax + (D or 0), device=dev)
    L = si.L.copy()
    L[1] = si.L_cap - w.N + 1   # one row past the capacity
    L[2] = -1
    st = DeviceStep(w, w.modes[0], si.L_cap, dev)
    Ld = torch.from_numpy(L).to(dev)
    st.tree_build(torch.from_numpy(si.root_token).to(dev), Ld,
                  topk=torch.zeros((w.B, w.K, w.s_max), dtype=torch.int32, device=dev))
    st.O = torch.full_like(si.Q, float("nan"))
    st.tree_attention(si.Q, si.Kc, si.Vc, Ld)
    torch.cuda.synchronize()
    O_gpu = st.O.cpu()
    assert torch.count_nonzero(O_gpu[1:3]).item() == 0, "invalid sequences must get O = 0"
    si.L = L
    check_attention(w, si, O_gpu, [(b, kv) for b in (0, 3) for kv in range(w.Hkv)])


@pytest.mark.parametrize("G", [1, 5])
@pytest.mark.parametrize("L0", [0, 1, 127, 128, 129])
def test_attention_edge_lengths_without_leftover_rows(L0, G):
    """The tcgen05 kernel without leftover rows (G = 1: one 65-row Q tile; G = 5: 325 rows in
    Q tiles of 128, 128 and 69 rows) at the prefix lengths around a key tile: no prefix, a
    one-key prefix tile ahead of the tree tile, one and two full tiles."""
    dev = gpu_ready()
    w = configs.scaled(configs.get("gqa7b_b32"), B=2, d=64, V=64, L_range=(L0, L0), Hq=2 * G, Hkv=2)
    si = synth.make_step_inputs(w, seed=L0 + G, device=dev)
    st = run_attention(w, si, dev)
    check_attention(w, si, st.O, [(b, kv) for b in range(w.B) for kv in range(w.Hkv)])


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("Hq,Hkv,branching", [(32, 16, (4, 3, 2, 1)), (40, 8, (4, 3, 2, 1)), (64, 8, (4, 3, 2, 1)),
                                              (32, 8, (2, 2, 2)), (32, 8, (6, 4, 4))])
def test_attention_gqa_groups(Hq, Hkv, branching, D):
    """Query-row tiles of 128 over N nodes x G heads: G = 2, 5, 8 with the 65-node tree
    (2, 3, 5 tiles per KV head, ragged last tiles), a 15-node tree (one partial tile) and a
    127-node tree (two mask words per node, 4 tiles); single and split KV ranges (B = 1 and 6);
    head dims 128 (tcgen05) and 64 (mma.sync)."""
    dev = gpu_ready()
    for B, L_range in ((1, (700, 700)), (6, (0, 900))):
        w = configs.scaled(configs.get("gqa7b_b32"), B=B, d=64, V=64, Hq=Hq, Hkv=Hkv, branching=branching,
                           L_range=L_range, D=D)
        si = synth.make_step_inputs(w, seed=Hq + Hkv + B, device=dev)
        st = run_attention(w, si, dev)
        check_attention(w, si, st.O, [(b, kv) for b in range(w.B) for kv in (0, Hkv // 2, Hkv - 1)])


@pytest.mark.parametrize("G,branching", [(3, (6, 6)), (5, (5, 4)), (7, (6, 5)), (6, (7, 2)), (7, (6, 2)),
                                        (6, (8, 7)), (3, (4, 2, 2, 1)), (8, (4, 3))])
def test_attention_every_leftover_size(G, branching):
    """Query rows per KV head = 128 * MT + R for R = 1..8 (the rows past the full tiles ride with
    the MT full-tile CTAs on interleaved key tiles): single and split KV ranges, an empty prefix."""
    dev = gpu_ready()
    for B, L_range in ((1, (700, 700)), (5, (0, 400))):
        w = configs.scaled(configs.get("gqa7b_b32"), B=B, d=64, V=64, Hq=2 * G, Hkv=2, branching=branching,
                           L_range=L_range)
        si = synth.make_step_inputs(w, seed=G * 10 + len(branching) + B, device=dev)
        st = run_attention(w, si, dev)
        check_attention(w, si, st.O, [(b, kv) for b in range(w.B) for kv in range(w.Hkv)])


@pytest.mark.parametrize("name", NAMES[1:])
def test_attention_full_size_sampled(name):
    dev = gpu_ready()
    w = configs.get(name)
    si = synth.make_step_inputs(configs.scaled(w, d=64, V=64), seed=7, device=dev)
    st = run_attention(w, si, dev)
    rng = np.random.default_rng(3)
    pairs = [(int(rng.integers(w.B)), int(rng.integers(w.Hkv))) for _ in range(3)] + [(w.B - 1, w.Hkv - 1)]
    check_attention(w, si, st.O, pairs)


# --------------------------------------------------------------------------- verify
def greedy_case(w, dev, seed):
    rng = np.random.default_rng(seed)
    L = synth.committed_lengths(seed, w.B, *w.L_range)
    L_cap = synth.cache_capacity(L, w.N)
    root = synth.root_tokens(seed, w.B, w.V)
    topk = random_topk(rng, w.B, w.K, w.s_max, w.branching, w.V)
    tree = oracle_tree(w, root, topk, L, L_cap)
    tl = synth.target_logits(w, seed, device=dev)
    depths = planted_greedy_logits(tl, tree, seed, w.K)
    return L, L_cap, root, topk, tree, tl, depths


@pytest.mark.parametrize("name", NAMES + configs.PRUNED)
def test_verify_greedy_bit_exact(name):
    dev = gpu_ready()
    w = configs.scaled(configs.get(name), B=max(configs.get(name).B, 12), target_corr=0.0)
    L, L_cap, root, topk, tree, tl, depths = greedy_case(w, dev, seed=5)
    st = DeviceStep(w, GREEDY, L_cap, dev)
    st.tree_build(torch.from_numpy(root).to(dev), torch.from_numpy(L).to(dev), topk=torch.from_numpy(topk).to(dev))
    st.verify(tl)
    torch.cuda.synchronize()
    ref = O.verify_batch(GREEDY, tree, f64(tl), w.K)
    for key in ("acc", "path", "out_tokens", "n_out"):
        assert np.array_equal(i64(getattr(st, key)), ref[key]), key
    assert np.array_equal(i64(st.flags), np.zeros(w.B))
    assert (ref["acc"] >= np.array(depths)).all()
    assert len(set(ref["acc"].tolist())) > 1


@pytest.mark.parametrize("V", [3001, 13, 16])
def test_verify_greedy_ragged_vocab(V):
    """Vocabularies that are not a multiple of 8 (one entry at a time) and the smallest ones;
    planted paths of every depth, B = 24."""
    dev = gpu_ready()
    w = configs.scaled(configs.get("vicuna13b_b8"), B=24, V=V, target_corr=0.0, modes=(GREEDY,))
    L, L_cap, root, topk, tree, tl, depths = greedy_case(w, dev, seed=V)
    st = DeviceStep(w, GREEDY, L_cap, dev)
    st.tree_build(torch.from_numpy(root).to(dev), torch.from_numpy(L).to(dev), topk=torch.from_numpy(topk).to(dev))
    st.verify(tl)
    torch.cuda.synchronize()
    ref = O.verify_batch(GREEDY, tree, f64(tl), w.K)
    for key in ("acc", "path", "out_tokens", "n_out"):
        assert np.array_equal(i64(getattr(st, key)), ref[key]), key


@pytest.mark.parametrize("name", ["vicuna7b_b1", "vicuna33b_b16"])
def test_repeated_calls_share_workspace(name):
    """A workspace carries nothing from one call into the next: the same heads
    and greedy-verify calls, issued three times on one workspace (the last time
    after a heads call on other inputs), give identical results."""
    dev = gpu_ready()
    w = configs.scaled(configs.get(name), d=256, V=3000, L_range=(40, 40), Hq=2, Hkv=2, target_corr=0.0)
    si = synth.make_step_inputs(w, seed=3, device=dev)
    L, L_cap, root, topk, tree, tl, depths = greedy_case(w, dev, seed=9)
    st = st2 = DeviceStep(w, GREEDY, L_cap, dev)
    outs = []
    for rep in range(3):
        if rep == 2:   # other inputs through the same workspace first
            st.heads(si.h * 0.5, si.W, si.bias, si.U)
        st.heads(si.h, si.W, si.bias, si.U)
        st2.tree_build(torch.from_numpy(root).to(dev), torch.from_numpy(L).to(dev),
                       topk=torch.from_numpy(topk).to(dev))
        st2.verify(tl)
        torch.cuda.synchronize()
        outs.append((st.topk.cpu().numpy().copy(), i64(st2.acc).copy(), i64(st2.out_tokens).copy()))
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert np.array_equal(a, b)
    ref = O.verify_batch(GREEDY, tree, f64(tl), w.K)
    assert np.array_equal(outs[-1][1], ref["acc"]) and np.array_equal(outs[-1][2], ref["out_tokens"])


def rs_case(w, dev, seed, sigma_head=2.0):
    """Stand-in head logits (float32) and correlated target logits, identical for both sides."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    z = torch.randn((w.B, w.K, w.V), generator=gen, device=dev) * sigma_head
    L = synth.committed_lengths(seed, w.B, *w.L_range)
    L_cap = synth.cache_capacity(L, w.N)
    root = synth.root_tokens(seed, w.B, w.V)
    topk, _ = O.heads_top_s(z.double().cpu().numpy(), w.branching)
    tree = oracle_tree(w, root, topk.astype(np.int32), L, L_cap)
    corr = configs.scaled(w, target_corr=max(w.target_corr, 0.8))
    tl = synth.target_logits(corr, seed, device=dev, zhat=z, depth=tree["depth"])
    u_acc, u_res = synth.uniforms_for_step(seed, w.B, w.K, w.s_max)
    return L, L_cap, root, topk.astype(np.int32), tree, tl, z, u_acc, u_res


@pytest.mark.parametrize("name,T", [("tiny_fp32", 1.0), ("vicuna13b_b8", 1.0), ("gqa7b_b32", 0.7),
                                    ("vicuna7b_b1", 0.5), ("vicuna33b_b16", 1.3),
                                    ("vicuna13b_b8_pruned64", 1.0), ("vicuna7b_b1_pruned64", 0.7)])
def test_verify_rejection_decisions(name, T):
    dev = gpu_ready()
    w = configs.scaled(configs.get(name), temperature=T)
    if w.B < 16:
        w = configs.scaled(w, B=16)
    total_acc = 0
    for seed in (1, 2):
        L, L_cap, root, topk, tree, tl, z, u_acc, u_res = rs_case(w, dev, seed)
        st = DeviceStep(w, REJECTION, L_cap, dev)
        st.tree_build(torch.from_numpy(root).to(dev), torch.from_numpy(L).to(dev),
                      topk=torch.from_numpy(topk).to(dev))
        st.verify(tl, torch.from_numpy(u_acc).to(dev), torch.from_numpy(u_res).to(dev), head_logits=z)
        torch.cuda.synchronize()
        ref, _ = compare_verify(st, REJECTION, tree, f64(tl), w.K, head_logits=f64(z), u_acc=u_acc, u_res=u_res,
                                T=T, what=f"{name} T={T} seed={seed}")
        total_acc += int(ref["acc"].sum())
    assert total_acc > 0


# The walk runs on a cluster of 8 / 4 / 2 / 1 CTAs per sequence depending on B
# (one 256-thread CTA per SM), but on enough CTAs that each slice fits 32 entries
# per thread (full vocabularies with large batches: more CTAs than one wave);
# vocabulary slices of unequal length, rows read 8 entries at a time or one at a
# time (V % 8 != 0).
@pytest.mark.parametrize("B,V", [(8, 1000), (40, 4096), (80, 3001), (160, 2048), (40, 32000), (80, 32000),
                                 (160, 32768), (24, 32000)])
def test_verify_rejection_cluster_sizes(B, V):
    dev = gpu_ready()
    w = configs.scaled(configs.get("gqa7b_b32"), B=B, V=V, temperature=0.9, L_range=(16, 64))
    L, L_cap, root, topk, tree, tl, z, u_acc, u_res = rs_case(w, dev, seed=3)
    st = DeviceStep(w, REJECTION, L_cap, dev)
    st.tree_build(torch.from_numpy(root).to(dev), torch.from_numpy(L).to(dev), topk=torch.from_numpy(topk).to(dev))
    st.verify(tl, torch.from_numpy(u_acc).to(dev), torch.from_numpy(u_res).to(dev), head_logits=z)
    torch.cuda.synchronize()
    compare_verify(st, REJECTION, tree, f64(tl), w.K, head_logits=f64(z), u_acc=u_acc, u_res=u_res,
                   T=w.temperature, what=f"B={B} V={V}")


# --------------------------------------------------------------------------- compaction
@pytest.mark.parametrize("name", NAMES)
def test_kv_compact_bit_exact(name):
    dev = gpu_ready()
    w = small(configs.get(name))
    si = synth.make_step_inputs(w, seed=9, device=dev)
    rng = np.random.default_rng(9)
    tree = layout(w)
    acc = rng.integers(0, w.K + 1, size=w.B).astype(np.int32)
    acc[0] = 0
    acc[-1] = w.K
    path = np.full((w.B, w.K + 1), -1, dtype=np.int32)
    for b in range(w.B):
        cur = 0
        path[b, 0] = 0
        for r in range(1, acc[b] + 1):
            kids = O.children_of(tree["parent"], cur)
            cur = kids[int(rng.integers(len(kids)))]
            path[b, r] = cur
    L = si.L.copy()
    raw = lambda t: t.cpu().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).numpy()
    k0, v0 = raw(si.Kc), raw(si.Vc)
    st = DeviceStep(w, w.modes[0], si.L_cap, dev)
    st.acc.copy_(torch.from_numpy(acc))
    st.path.copy_(torch.from_numpy(path))
    Ld = torch.from_numpy(L).to(dev)
    st.kv_compact(si.Kc, si.Vc, Ld)
    torch.cuda.synchronize()
    kr, vr, Lr, kv_map = O.kv_compact(k0, v0, L, acc, path)
    assert np.array_equal(raw(si.Kc), kr) and np.array_equal(raw(si.Vc), vr)
    assert np.array_equal(i64(Ld), Lr) and np.array_equal(i64(st.kv_map), kv_map)


@pytest.mark.parametrize("name", ["tiny_fp32", "vicuna33b_b16", "gqa7b_b32"])
def test_kv_compact_leaves_invalid_sequences(name):
    """Sequences with L_b < 0 or L_b + N > L_cap are left unchanged (the header's contract):
    cache rows and length bit-exact, kv_map -1; the other sequences match the oracle."""
    dev = gpu_ready()
    base = configs.get(name)
    hkv = 2 if base.Hkv < 8 else 8               # 8 KV heads: the compaction cluster's full width
    w = configs.scaled(base, B=5, d=64, V=64, Hq=hkv * (base.Hq // base.Hkv), Hkv=hkv, L_range=(20, 300))
    si = synth.make_step_inputs(w, seed=41, device=dev)
    rng = np.random.default_rng(41)
    tree = layout(w)
    acc, path = random_paths(tree, w.K, w.B, rng)
    acc[1], acc[3] = w.K, w.K                    # full paths on the two invalid sequences
    for b in (1, 3):
        cur, path[b, 0] = 0, 0
        for r in range(1, w.K + 1):
            kids = O.children_of(tree["parent"], cur)
            cur = kids[-1]
            path[b, r] = cur
    L = si.L.copy()
    L[1] = si.L_cap - w.N + 1   # over capacity
    L[3] = -1
    raw = lambda t: t.cpu().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).numpy()
    k0, v0 = raw(si.Kc), raw(si.Vc)
    st = DeviceStep(w, w.modes[0], si.L_cap, dev)
    st.acc.copy_(torch.from_numpy(acc))
    st.path.copy_(torch.from_numpy(path))
    Ld = torch.from_numpy(L).to(dev)
    st.kv_compact(si.Kc, si.Vc, Ld)
    torch.cuda.synchronize()
    k1, v1, L1, kv_map = raw(si.Kc), raw(si.Vc), i64(Ld), i64(st.kv_map)
    for b in (1, 3):
        assert np.array_equal(k1[b], k0[b]) and np.array_equal(v1[b], v0[b]), f"sequence {b} changed"
        assert L1[b] == L[b] and (kv_map[b] == -1).all()
    ok = np.array([0, 2, 4])
    kr, vr, Lr, mr = O.kv_compact(k0[ok], v0[ok], L[ok], acc[ok], path[ok])
    assert np.array_equal(k1[ok], kr) and np.array_equal(v1[ok], vr)
    assert np.array_equal(L1[ok], Lr) and np.array_equal(kv_map[ok], mr)


def random_paths(tree, K, B, rng):
    """acc uniform in 0..K with sequence 0 at acc = 0 and the last at acc = K; a random descent."""
    acc = rng.integers(0, K + 1, size=B).astype(np.int32)
    acc[0], acc[-1] = 0, K
    path = np.full((B, K + 1), -1, dtype=np.int32)
    for b in range(B):
        cur = 0
        path[b, 0] = 0
        for r in range(1, acc[b] + 1):
            kids = O.children_of(tree["parent"], cur)
            cur = kids[int(rng.integers(len(kids)))]
            path[b, r] = cur
    return acc, path


@pytest.mark.parametrize("name,B", [("vicuna33b_b16", 4), ("gqa7b_b32", 3), ("vicuna33b_b16", 16), ("gqa7b_b32", 32)])
def test_kv_compact_full_kv_heads(name, B):
    """Compaction at the workloads' own KV-head counts, which every full-size step takes: 52 heads
    split over an 8-CTA cluster (uneven ranges of 6 and 7 heads) and 8 heads over 8 CTAs, at the
    full committed lengths (8192; 4096..16384). Small batches compare the whole cache with the
    oracle; the full batches compare the tree region of every sequence with the oracle and check
    on the device that no byte outside it changed."""
    dev = gpu_ready()
    w = configs.scaled(configs.get(name), B=B, d=64, V=64)
    si = synth.make_step_inputs(w, seed=B + 40, device=dev)
    rng = np.random.default_rng(B + 41)
    acc, path = random_paths(layout(w), w.K, w.B, rng)
    raw = lambda t: t.view(torch.int16)
    L = si.L.copy()
    full = w.B > 4
    if full:
        k_before, v_before = raw(si.Kc).clone(), raw(si.Vc).clone()
        region = lambda t, b: t[b, :, int(L[b]):int(L[b]) + w.N].cpu().numpy()
        k0 = [region(raw(si.Kc), b) for b in range(w.B)]
        v0 = [region(raw(si.Vc), b) for b in range(w.B)]
    else:
        k0, v0 = raw(si.Kc).cpu().numpy(), raw(si.Vc).cpu().numpy()
    st = DeviceStep(w, w.modes[0], si.L_cap, dev)
    st.acc.copy_(torch.from_numpy(acc))
    st.path.copy_(torch.from_numpy(path))
    Ld = torch.from_numpy(L).to(dev)
    st.kv_compact(si.Kc, si.Vc, Ld)
    torch.cuda.synchronize()
    if not full:
        kr, vr, Lr, kv_map = O.kv_compact(k0, v0, L, acc, path)
        assert np.array_equal(raw(si.Kc).cpu().numpy(), kr) and np.array_equal(raw(si.Vc).cpu().numpy(), vr)
    else:
        # the oracle on each sequence's tree region (committed length 0 there), then the rest untouched
        Lr = np.zeros(w.B, dtype=np.int64)
        kv_map = np.full((w.B, w.K + 1), -1, dtype=np.int64)
        for b in range(w.B):
            kr, vr, lr, m = O.kv_compact(k0[b][None], v0[b][None], np.zeros(1, dtype=np.int64), acc[b:b + 1],
                                         path[b:b + 1])
            assert np.array_equal(region(raw(si.Kc), b), kr[0]) and np.array_equal(region(raw(si.Vc), b), vr[0]), b
            Lr[b] = int(L[b]) + int(lr[0])
            kv_map[b] = m[0]
            k_before[b, :, int(L[b]):int(L[b]) + w.N] = raw(si.Kc)[b, :, int(L[b]):int(L[b]) + w.N]
            v_before[b, :, int(L[b]):int(L[b]) + w.N] = raw(si.Vc)[b, :, int(L[b]):int(L[b]) + w.N]
        assert torch.equal(k_before, raw(si.Kc)) and torch.equal(v_before, raw(si.Vc))
    assert np.array_equal(i64(Ld), Lr) and np.array_equal(i64(st.kv_map), kv_map)


# --------------------------------------------------------------------------- paged cache
def paged_layout(si, w, P, seed):
    """The committed rows of si.Kc/Vc moved into a shuffled page pool, the tree rows staged."""
    rng = np.random.default_rng(seed)
    cap = -(-si.L_cap // P) * P
    max_pages = cap // P
    num_pages = w.B * max_pages + 3
    bt = rng.permutation(num_pages)[:w.B * max_pages].reshape(w.B, max_pages).astype(np.int32)
    Kc, Vc = si.Kc.cpu(), si.Vc.cpu()
    Kp = torch.zeros((num_pages, w.Hkv, P, w.D), dtype=Kc.dtype)
    Vp = torch.zeros_like(Kp)
    for b in range(w.B):
        for i in range(int(si.L[b])):
            Kp[bt[b, i // P], :, i % P] = Kc[b, :, i]
            Vp[bt[b, i // P], :, i % P] = Vc[b, :, i]
    Kt = torch.stack([Kc[b, :, int(si.L[b]):int(si.L[b]) + w.N] for b in range(w.B)])
    Vt = torch.stack([Vc[b, :, int(si.L[b]):int(si.L[b]) + w.N] for b in range(w.B)])
    return cap, num_pages, bt, Kp, Vp, Kt, Vt


@pytest.mark.parametrize("name,P", [("vicuna7b_b1", 128), ("vicuna7b_b1", 256), ("gqa7b_b32", 128),
                                    ("vicuna13b_b8", 256), ("vicuna7b_b1_pruned64", 128)])
def test_attention_paged(name, P):
    """Tree attention with the committed rows in a shuffled page pool and the tree rows
    staged: the oracle's attention over the same logical cache (lengths 0, one page,
    ragged; one or several KV splits)."""
    dev = gpu_ready()
    w0 = configs.get(name)
    G = w0.Hq // w0.Hkv
    w = configs.scaled(w0, B=5 if w0.B > 1 else 1, d=256, V=1000, Hq=2 * G, Hkv=2, L_range=(0, 700))
    si = synth.make_step_inputs(w, seed=P + 3, device=dev)
    if w.B > 1:
        si.L[0], si.L[1] = 0, P      # empty prefix; exactly one page
    cap, num_pages, bt, Kp, Vp, Kt, Vt = paged_layout(si, w, P, seed=P)
    st = DeviceStep(w, w.modes[0], cap, dev)
    Ld = torch.from_numpy(si.L).to(dev)
    st.tree_build(torch.from_numpy(si.root_token).to(dev), Ld,
                  topk=torch.zeros((w.B, w.K, w.s_max), dtype=torch.int32, device=dev))
    O_gpu = torch.empty_like(si.Q)
    mb.tree_attention_paged(st.cfg, si.Q, Kp.to(dev), Vp.to(dev), num_pages, P, torch.from_numpy(bt).to(dev),
                            Kt.to(dev), Vt.to(dev), Ld, st.anc_bits, O_gpu, st.workspace)
    torch.cuda.synchronize()
    mask = O.ancestor_mask(layout(w)["parent"])
    pairs = [(b, h) for b in range(w.B) for h in range(w.Hq)]
    ref = O.tree_attention_paged(f64(si.Q), f64(Kp), f64(Vp), bt, P, f64(Kt), f64(Vt), si.L, mask, w.Hq, w.Hkv,
                                 pairs=pairs)
    assert_close(f64(O_gpu), ref, w.dtype, "paged attention")


@pytest.mark.parametrize("n_layers,P", [(1, 128), (3, 256)])
def test_kv_commit_paged_bit_exact(n_layers, P):
    """The accepted path's staged rows land at logical rows L_b.. of every layer's pages."""
    dev = gpu_ready()
    w = configs.scaled(configs.get("vicuna13b_b8"), d=256, V=1000, Hq=4, Hkv=4, L_range=(100, 900))
    si = synth.make_step_inputs(w, seed=77, device=dev)
    cap, num_pages, bt, _, _, _, _ = paged_layout(si, w, P, seed=5)
    rng = np.random.default_rng(6)
    raw = lambda shape: rng.integers(-30000, 30000, size=shape).astype(np.int16)   # bf16 bit patterns
    Kp = [raw((num_pages, w.Hkv, P, w.D)) for _ in range(n_layers)]
    Vp = [raw((num_pages, w.Hkv, P, w.D)) for _ in range(n_layers)]
    Kt = [raw((w.B, w.Hkv, w.N, w.D)) for _ in range(n_layers)]
    Vt = [raw((w.B, w.Hkv, w.N, w.D)) for _ in range(n_layers)]
    tree = layout(w)
    acc = rng.integers(0, w.K + 1, size=w.B).astype(np.int32)
    acc[0], acc[-1] = 0, w.K
    path = np.full((w.B, w.K + 1), -1, dtype=np.int32)
    for b in range(w.B):
        cur = 0
        path[b, 0] = 0
        for r in range(1, acc[b] + 1):
            kids = O.children_of(tree["parent"], cur)
            cur = kids[int(rng.integers(len(kids)))]
            path[b, r] = cur
    L = si.L.astype(np.int32).copy()
    L[2] = cap - w.N + 1                      # no room: left as it is
    to_dev = lambda arrs: torch.from_numpy(np.stack(arrs)).to(dev)
    Kpd, Vpd, Ktd, Vtd = to_dev(Kp), to_dev(Vp), to_dev(Kt), to_dev(Vt)
    st = DeviceStep(w, w.modes[0], cap, dev)
    Ld = torch.from_numpy(L).to(dev)
    mb.kv_commit_paged(st.cfg, Kpd, Vpd, P, torch.from_numpy(bt).to(dev), Ktd, Vtd, n_layers, Kp[0].size,
                       Kt[0].size, Ld, torch.from_numpy(acc).to(dev), torch.from_numpy(path).to(dev), st.kv_map)
    torch.cuda.synchronize()
    ok = np.array([0 <= L[b] and L[b] + w.N <= cap for b in range(w.B)])
    assert not ok[2] and ok.sum() == w.B - 1
    # the oracle on the sequences with room (each owns its pages, so the others are untouched)
    kps, vps, L_ok, map_ok = O.kv_commit_paged(Kp, Vp, bt[ok], P, [k[ok] for k in Kt], [v[ok] for v in Vt],
                                               L[ok], acc[ok], path[ok])
    L2 = L.astype(np.int64).copy()
    L2[ok] = L_ok
    kv_map = np.full((w.B, w.K + 1), -1, dtype=np.int64)
    kv_map[ok] = map_ok
    assert np.array_equal(Kpd.cpu().numpy(), np.stack(kps)) and np.array_equal(Vpd.cpu().numpy(), np.stack(vps))
    assert np.array_equal(i64(Ld), L2) and np.array_equal(i64(st.kv_map), kv_map)


# --------------------------------------------------------------------------- whole step
@pytest.mark.parametrize("name", NAMES + configs.SHARED + configs.PRUNED)
def test_step_end_to_end_small(name):
    """The five calls in order on one stream against the oracle's step on the same inputs."""
    dev = gpu_ready()
    w = small(configs.get(name))
    if w.B < 8:
        w = configs.scaled(w, B=8)
    check_step(w, dev)


def _limit_cases():
    base = configs.scaled(configs.get("vicuna7b_b1"), B=8, d=512, V=1000, Hq=8, Hkv=2, L_range=(37, 300),
                          modes=(GREEDY, REJECTION), temperature=0.9)
    paths = configs.pruned_paths(8, 8, 127)
    br = tuple(1 + max(p[e] for p in paths if len(p) > e) for e in range(8))
    return {
        # 128 nodes (the most the library takes) over 8 heads (the most heads): two full ancestor words,
        # a 128-key tree tile and 4 query tiles of 128 rows per KV head
        "pruned128_k8": configs.scaled(base, name="pruned128_k8", branching=br, tree_paths=paths),
        # top-8 lists (the widest branching) at two depths: 73 nodes
        "cartesian_8x8": configs.scaled(base, name="cartesian_8x8", branching=(8, 8), Hq=4, Hkv=4),
        # a chain of 8 heads with one candidate each, 64-dim heads (the mma.sync attention)
        "chain_k8_d64": configs.scaled(base, name="chain_k8_d64", branching=(1,) * 8, D=64, Hq=6, Hkv=2),
        # more sequences than one tcgen05 heads pass takes (the heads call runs two batch slices)
        "batch40": configs.scaled(base, name="batch40", B=40, branching=(3, 2, 2)),
    }


@pytest.mark.parametrize("case", ["pruned128_k8", "cartesian_8x8", "chain_k8_d64", "batch40"])
def test_step_at_limits(case):
    """The whole step at the library's limits: 128 nodes, 8 heads, top-8 lists, batches past the tcgen05 plan."""
    dev = gpu_ready()
    w = _limit_cases()[case]
    assert w.N <= 128 and w.K <= 8 and max(w.branching) <= 8
    check_step(w, dev)


def check_step(w, dev):
    for mode in w.modes:
        si = synth.make_step_inputs(w, seed=31, device=dev, with_bias=True)
        r, z = O.medusa_heads(f64(si.h), f64(si.W), f64(si.bias), f64(si.U))
        topk_ref, near = O.heads_top_s(z, w.branching)
        tree = oracle_tree(w, si.root_token, topk_ref, si.L, si.L_cap)
        if mode == REJECTION:
            tl = synth.target_logits(configs.scaled(w, target_corr=0.8), 31, device=dev,
                                     zhat=torch.from_numpy(z).float(), depth=tree["depth"])
        else:
            tl = synth.target_logits(w, 31, device=dev)
            planted_greedy_logits(tl, tree, 31, w.K)
        inp = to_device_inputs(si, tl, dev)
        Kc0, Vc0 = f64(si.Kc), f64(si.Vc)
        st = DeviceStep(w, mode, si.L_cap, dev)
        st.run(inp, write_logits=True, compact=True)
        torch.cuda.synchronize()
        assert_close(st.logits.cpu().numpy(), z, w.dtype, "logits")
        ok_b = ~near.any(axis=1)
        assert np.array_equal(i64(st.topk)[ok_b], topk_ref[ok_b])
        assert np.array_equal(i64(st.tokens)[ok_b], tree["tokens"][ok_b])
        Oref = O.tree_attention(f64(si.Q), Kc0, Vc0, si.L, tree["mask"], w.Hq, w.Hkv)
        assert_close(f64(st.O), Oref, w.dtype, "attention")
        # the oracle's walk takes the GPU's own head logits, so both sides decide on the same
        # numbers and the 1e-6 tie windows apply unchanged
        ver, _ = compare_verify(st, mode, tree, f64(tl), w.K, head_logits=f64(st.logits), u_acc=si.u_acc,
                                u_res=si.u_res, T=w.temperature, eligible=ok_b, min_compared=max(1, w.B // 2),
                                what=f"{w.name} mode={mode}")
        ok = ok_b & (ver["flags"] == 0) & ((i64(st.flags) & TIE_BITS) == 0)
        kr, vr, Lr, kv_map = O.kv_compact(Kc0, Vc0, si.L, ver["acc"], ver["path"])
        assert np.array_equal(i64(inp.L)[ok], Lr[ok]) and np.array_equal(i64(st.kv_map)[ok], kv_map[ok])
        assert np.array_equal(f64(inp.Kc)[ok], kr[ok]) and np.array_equal(f64(inp.Vc)[ok], vr[ok])
        assert ok.sum() >= max(1, w.B // 2)
