"""medusa_step_fused: the whole step as one persistent kernel, against the float64 oracle.

Every output of the five calls — head logits, top-s, the tree arrays, tokens and
position ids, tree attention, the greedy walk and the compacted cache — comes
from one cooperative launch and is checked against the oracle on the same seeded
inputs, with the tolerances of the other parity tests; its integer outputs must
also equal those of the five separate calls bit for bit.
"""
import numpy as np
import pytest
import torch

from medusa_speculative_decoding_heads_gb300 import binding as mb, configs, synth
from medusa_speculative_decoding_heads_gb300.configs import GREEDY
from medusa_speculative_decoding_heads_gb300.step import DeviceStep, to_device_inputs
from oracle import medusa_oracle as O

from _helpers import assert_close, compare_verify, f64, gpu_ready, i64, planted_greedy_logits

pytestmark = pytest.mark.gpu


def _oracle_tree(w, root, topk, L, L_cap):
    return O.tree_build(w.branching, np.asarray(root), np.asarray(topk), np.asarray(L), L_cap, paths=w.tree_paths)


def _case(name, B, **kw):
    w0 = configs.get(name)
    G = w0.Hq // w0.Hkv
    over = dict(B=B, d=512, V=1000, Hq=2 * G, Hkv=2, L_range=(37, 300), modes=(GREEDY,), target_corr=0.0)
    over.update(kw)
    return configs.scaled(w0, **over)


def run_and_check(w, dev, seed=31):
    si = synth.make_step_inputs(w, seed=seed, device=dev, with_bias=True)
    _, z = O.medusa_heads(f64(si.h), f64(si.W), f64(si.bias), f64(si.U))
    topk_ref, near = O.heads_top_s(z, w.branching)
    tree = _oracle_tree(w, si.root_token, topk_ref, si.L, si.L_cap)
    tl = synth.target_logits(w, seed, device=dev)
    planted_greedy_logits(tl, tree, seed, w.K)
    Kc0, Vc0 = f64(si.Kc), f64(si.Vc)
    # the five separate calls on a copy of the inputs, for the bit-for-bit comparison
    inp_ref = to_device_inputs(si, tl, dev)
    inp_ref.Kc, inp_ref.Vc, inp_ref.L = si.Kc.clone(), si.Vc.clone(), inp_ref.L.clone()
    ref = DeviceStep(w, GREEDY, si.L_cap, dev)
    ref.run(inp_ref, write_logits=True, compact=True)
    inp = to_device_inputs(si, tl, dev)
    st = DeviceStep(w, GREEDY, si.L_cap, dev)
    st.run_fused(inp, write_logits=True, compact=True)
    torch.cuda.synchronize()
    assert mb.poll_errors()[0] == 0
    assert_close(st.logits.cpu().numpy(), z, w.dtype, "fused logits")
    ok_b = ~near.any(axis=1)
    assert ok_b.sum() >= 1
    assert np.array_equal(i64(st.topk)[ok_b], topk_ref[ok_b]), "top-s"
    for key in ("parent", "depth", "first_child"):
        assert np.array_equal(i64(getattr(st, key)), tree[key]), key
    assert np.array_equal(i64(st.mask), tree["mask"].astype(np.int64))
    assert np.array_equal(st.anc_bits.cpu().numpy().view(np.uint64), tree["anc_bits"])
    assert np.array_equal(i64(st.tokens)[ok_b], tree["tokens"][ok_b])
    assert np.array_equal(i64(st.pos), tree["pos"])
    Oref = O.tree_attention(f64(si.Q), Kc0, Vc0, si.L, tree["mask"], w.Hq, w.Hkv)
    assert_close(f64(st.O), Oref, w.dtype, "fused attention")
    ver, _ = compare_verify(st, GREEDY, tree, f64(tl), w.K, eligible=ok_b, min_compared=1, what=f"fused {w.name}")
    ok = ok_b & (ver["flags"] == 0)
    kr, vr, Lr, kv_map = O.kv_compact(Kc0, Vc0, si.L, ver["acc"], ver["path"])
    assert np.array_equal(i64(inp.L)[ok], Lr[ok]) and np.array_equal(i64(st.kv_map)[ok], kv_map[ok])
    assert np.array_equal(f64(inp.Kc)[ok], kr[ok]) and np.array_equal(f64(inp.Vc)[ok], vr[ok])
    # the same integer results as the five separate calls, for every sequence
    for key in ("topk", "tokens", "pos", "acc", "path", "out_tokens", "n_out", "kv_map"):
        assert np.array_equal(i64(getattr(st, key)), i64(getattr(ref, key))), f"fused vs calls: {key}"
    assert np.array_equal(i64(inp.L), i64(inp_ref.L))
    assert torch.equal(inp.Kc, inp_ref.Kc) and torch.equal(inp.Vc, inp_ref.Vc)


@pytest.mark.parametrize("B", [1, 2, 3, 4])
@pytest.mark.parametrize("name", ["vicuna7b_b1", "vicuna33b_b16", "gqa7b_b32", "vicuna7b_b1_pruned64",
                                  "vicuna7b_b1_shared"])
def test_fused_step_small(name, B):
    """Cartesian (65 nodes) and pruned (64 nodes) trees, 1 and 4 query heads per KV head (two row
    blocks with a ragged tail), a shared vocab projection, ragged lengths and KV splits."""
    dev = gpu_ready()
    run_and_check(_case(name, B), dev)


def test_fused_step_limits():
    """128 nodes over 8 heads and top-8 lists at two depths, a vocabulary that is not a multiple
    of 8, an empty committed prefix."""
    dev = gpu_ready()
    base = configs.scaled(configs.get("vicuna7b_b1"), B=3, d=256, V=1003, Hq=4, Hkv=2, L_range=(0, 200),
                          modes=(GREEDY,), target_corr=0.0)
    paths = configs.pruned_paths(8, 8, 127)
    br = tuple(1 + max(p[e] for p in paths if len(p) > e) for e in range(8))
    run_and_check(configs.scaled(base, name="pruned128_k8", branching=br, tree_paths=paths), dev)
    run_and_check(configs.scaled(base, name="cartesian_8x8", branching=(8, 8)), dev)


def test_fused_step_full_size_7b():
    """The 7B-shaped step at its full size (d = 4096, V = 32000, 32 heads x 128, L = 2048)."""
    dev = gpu_ready()
    run_and_check(configs.scaled(configs.get("vicuna7b_b1"), target_corr=0.0), dev)


def test_fused_step_refuses_what_it_does_not_cover():
    dev = gpu_ready()
    for w, mode in ((configs.scaled(configs.get("vicuna7b_b1"), B=5, d=256, V=500, Hq=2, Hkv=2, L_range=(40, 40)),
                     GREEDY),
                    (configs.scaled(configs.get("vicuna7b_b1"), B=1, d=256, V=500, Hq=2, Hkv=2, L_range=(40, 40),
                                    temperature=1.0), configs.REJECTION)):
        st = DeviceStep(w, mode, 128, dev)
        si = synth.make_step_inputs(w, seed=1, device=dev)
        inp = to_device_inputs(si, synth.target_logits(configs.scaled(w, target_corr=0.0), 1, device=dev), dev)
        with pytest.raises(mb.MedusaError) as e:
            st.run_fused(inp)
        assert e.value.status == -2
