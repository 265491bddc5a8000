"""medusa_tree_attention_noalloc: tree attention without a caller workspace.

Some callers cannot allocate device memory: a serving engine that reserved
nearly all of it for its KV cache at start-up, or a plug-in whose host
framework's allocator owns every device byte. For them the library keeps tree
attention's scratch in a static device array. Through the C ABI this file
checks that two consecutive calls of that entry point give bit for bit the
output of the workspace-based entry point (both run the same kernels with the
same split of the KV range), that the output matches the float64 oracle within
the stated tolerance, and that a configuration needing more scratch than the
array holds is refused up front. It is collected last so that a failure here
never hides the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from medusa_speculative_decoding_heads_gb300 import binding as mb, configs, synth
from medusa_speculative_decoding_heads_gb300.step import cfg_for
from oracle import medusa_oracle as O

from _helpers import assert_close, f64, gpu_ready

pytestmark = pytest.mark.gpu

CASES = [
    ("vicuna7b_b1", {}),                                                 # split-KV partials over 8 splits
    ("gqa7b_b32", {"B": 4, "L_range": (300, 1500), "d": 64, "V": 64}),   # GQA, ragged lengths, leftover rows
    ("tiny_fp32", {}),                                                   # float32 path
]


def _tree_bits(w, dev):
    from medusa_speculative_decoding_heads_gb300.step import DeviceStep
    st = DeviceStep(w, w.modes[0], synth.cache_capacity(np.array([w.L_range[1]]), w.N), dev)
    st.tree_build(torch.zeros(w.B, dtype=torch.int32, device=dev), torch.zeros(w.B, dtype=torch.int32, device=dev),
                  topk=torch.zeros((w.B, w.K, w.s_max), dtype=torch.int32, device=dev))
    return st.anc_bits


@pytest.mark.parametrize("name,over", CASES)
def test_noalloc_matches_workspace_entry_point(name, over):
    dev = gpu_ready()
    w = configs.scaled(configs.get(name), **over) if over else configs.get(name)
    si = synth.make_step_inputs(configs.scaled(w, d=64, V=64), seed=4, device=dev)
    cfg = cfg_for(w, si.L_cap, w.modes[0])
    L = torch.from_numpy(si.L).to(dev)
    bits = _tree_bits(configs.scaled(w, L_range=(0, 0)), dev)
    ws = torch.empty(mb.workspace_size(cfg), dtype=torch.uint8, device=dev)
    ref = torch.empty_like(si.Q)
    mb.tree_attention(cfg, si.Q, si.Kc, si.Vc, L, bits, ref, ws)
    outs = []
    for _ in range(2):
        out = torch.full_like(si.Q, float("nan"))
        status = mb.load().medusa_tree_attention_noalloc(
            ctypes.byref(cfg), si.Q.data_ptr(), si.Kc.data_ptr(), si.Vc.data_ptr(), L.data_ptr(), bits.data_ptr(),
            out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert status == 0, mb.status_string(status)
        outs.append(out)
    torch.cuda.synchronize()
    for out in outs:
        assert torch.equal(out, ref), "no-allocation output differs from the workspace entry point"
    tree = O.tree_layout(w.branching)
    oracle_out = O.tree_attention(f64(si.Q), f64(si.Kc), f64(si.Vc), si.L, O.ancestor_mask(tree["parent"]),
                                  w.Hq, w.Hkv)
    assert_close(f64(outs[1]), oracle_out, w.dtype, f"{name} no-allocation attention vs oracle")


def test_noalloc_refuses_configurations_beyond_its_scratch():
    gpu_ready()
    w = configs.scaled(configs.get("gqa7b_b32"), B=256)
    cfg = cfg_for(w, 16448, w.modes[0])
    dummy = torch.empty(64, dtype=torch.uint8, device="cuda")
    status = mb.load().medusa_tree_attention_noalloc(
        ctypes.byref(cfg), dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
        dummy.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert status == -2   # MEDUSA_ERR_UNSUPPORTED, nothing enqueued
