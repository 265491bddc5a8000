"""The whole step as one launch (medusa_step_graph_*): the captured graph gives exactly the
outputs of the five calls made one by one, on the same inputs and again after new inputs are
written into the same buffers, and its first step matches the float64 oracle."""
import ctypes

import numpy as np
import pytest
import torch

from medusa_speculative_decoding_heads_gb300 import binding as mb, configs, synth
from medusa_speculative_decoding_heads_gb300.configs import GREEDY, REJECTION
from medusa_speculative_decoding_heads_gb300.step import DeviceStep, to_device_inputs

from oracle import medusa_oracle as O

from _helpers import assert_close, compare_verify, f64, gpu_ready, i64, planted_greedy_logits


def test_create_checks_arguments_before_any_cuda_call():
    lib = mb.load()
    cfg = mb.make_cfg(B=2, d=64, V=100, branching=(2, 2), Hq=2, Hkv=2, D=64, L_cap=64, dtype=configs.F32, mode=GREEDY)
    out = ctypes.c_void_p()
    assert lib.medusa_step_graph_create(ctypes.byref(cfg), None, ctypes.byref(out)) == -1
    assert lib.medusa_step_graph_launch(None, None) == -1
    assert lib.medusa_step_graph_destroy(None) == -1
    bad = mb.make_cfg(B=2, d=64, V=100, branching=(9, 2), Hq=2, Hkv=2, D=64, L_cap=64, dtype=configs.F32, mode=GREEDY)
    args = mb.StepArgs()
    assert lib.medusa_step_graph_create(ctypes.byref(bad), ctypes.byref(args), ctypes.byref(out)) == -2
    assert out.value is None


def _clone(inp):
    return type(inp)(**{k: (None if v is None else v.clone()) for k, v in inp.__dict__.items()})


def _outputs(st, inp):
    names = ("topk", "tokens", "pos", "anc_bits", "mask", "acc", "path", "out_tokens", "n_out", "kv_map", "flags")
    out = {n: getattr(st, n).cpu() for n in names}
    out.update(O=st.O.cpu(), logits=st.logits.cpu(), L=inp.L.cpu(), Kc=inp.Kc.cpu(), Vc=inp.Vc.cpu())
    return out


def _targets(w, si, mode, seed, dev):
    """Independent target logits; in greedy mode a path of the oracle's tree is planted so that
    some drafts are accepted and the compaction moves rows."""
    tl = synth.target_logits(configs.scaled(w, target_corr=0.0), seed, device=dev)
    if mode == GREEDY:
        f = lambda t: t.detach().cpu().double().numpy()
        _, z = O.medusa_heads(f(si.h), f(si.W), f(si.bias), f(si.U))
        topk, _ = O.heads_top_s(z, w.branching)
        tree = O.tree_build(w.branching, si.root_token, topk, si.L, si.L_cap, paths=w.tree_paths)
        planted_greedy_logits(tl, tree, seed, w.K)
    return tl


def _check_oracle(w, mode, si, tl, st, inp, Kc0, Vc0):
    """The graph's first step against the oracle: head logits, top-s, tokens, attention, the walk
    (on the library's own head logits) and the compacted cache (Kc0, Vc0: the cache before the step)."""
    _, z = O.medusa_heads(f64(si.h), f64(si.W), f64(si.bias), f64(si.U))
    topk_ref, near = O.heads_top_s(z, w.branching)
    tree = O.tree_build(w.branching, si.root_token, topk_ref, si.L, si.L_cap, paths=w.tree_paths)
    assert_close(st.logits.cpu().numpy(), z, w.dtype, "graph logits")
    ok_b = ~near.any(axis=1)
    assert np.array_equal(i64(st.topk)[ok_b], topk_ref[ok_b]) and np.array_equal(i64(st.tokens)[ok_b],
                                                                                  tree["tokens"][ok_b])
    Oref = O.tree_attention(f64(si.Q), Kc0, Vc0, si.L, tree["mask"], w.Hq, w.Hkv)
    assert_close(f64(st.O), Oref, w.dtype, "graph attention")
    ver, _ = compare_verify(st, mode, tree, f64(tl), w.K, head_logits=f64(st.logits), u_acc=si.u_acc,
                            u_res=si.u_res, T=w.temperature, eligible=ok_b, min_compared=1, what=f"graph {w.name}")
    ok = ok_b & (ver["flags"] == 0) & ((i64(st.flags) & 3) == 0)
    kr, vr, Lr, _ = O.kv_compact(Kc0, Vc0, si.L, ver["acc"], ver["path"])
    assert np.array_equal(i64(inp.L)[ok], Lr[ok])
    assert np.array_equal(f64(inp.Kc)[ok], kr[ok]) and np.array_equal(f64(inp.Vc)[ok], vr[ok])


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny_fp32", "vicuna7b_b1", "gqa7b_b32", "vicuna13b_b8_pruned64"])
def test_graph_equals_the_five_calls(name):
    dev = gpu_ready()
    base = configs.get(name)
    w = base if name == "tiny_fp32" else configs.scaled(base, B=max(base.B, 4), d=512, V=1000,
                                                         Hq=2 * (base.Hq // base.Hkv), Hkv=2, L_range=(37, 300))
    for mode in w.modes:
        si = synth.make_step_inputs(w, seed=5, device=dev, with_bias=True)
        Kc0, Vc0 = f64(si.Kc), f64(si.Vc)   # the eager run compacts si's cache in place
        tl = _targets(w, si, mode, 5, dev)
        eager_in = to_device_inputs(si, tl, dev)
        graph_in = _clone(eager_in)
        eager = DeviceStep(w, mode, si.L_cap, dev)
        eager.run(eager_in, write_logits=True, compact=True)
        st = DeviceStep(w, mode, si.L_cap, dev)
        g = st.graph(graph_in, write_logits=True, compact=True)
        n0 = mb.launch_count()
        g.launch()
        torch.cuda.synchronize()
        assert mb.launch_count() > n0   # a replay counts its kernels
        a, b = _outputs(eager, eager_in), _outputs(st, graph_in)
        for k in a:
            assert torch.equal(a[k], b[k]), f"{name} mode {mode}: {k} differs"
        _check_oracle(w, mode, si, tl, st, graph_in, Kc0, Vc0)
        # a second step: fresh inputs written into the graph's buffers (the cache and L carry over)
        si2 = synth.make_step_inputs(w, seed=6, device=dev, with_bias=True)
        tl2 = _targets(w, si2, mode, 6, dev)
        for inp in (eager_in, graph_in):
            inp.h.copy_(si2.h)
            inp.Q.copy_(si2.Q)
            inp.target_logits.copy_(tl2)
            inp.root_token.copy_(torch.as_tensor(np.asarray(si2.root_token, dtype=np.int32), device=dev))
        eager.run(eager_in, write_logits=True, compact=True)
        g.launch()
        torch.cuda.synchronize()
        a, b = _outputs(eager, eager_in), _outputs(st, graph_in)
        for k in a:
            assert torch.equal(a[k], b[k]), f"{name} mode {mode}, second step: {k} differs"
        g.close()
