"""One Medusa verify step on the GPU through the C ABI.

``DeviceStep`` owns the device buffers of one workload (inputs, outputs and the
library workspace) and enqueues the five library calls in order on one
stream: heads -> tree build -> tree attention -> verify -> KV compaction, or
captures them once as a library step graph replayed with one launch. It only
allocates tensors and marshals pointers; all arithmetic runs in libmedusa's
kernels.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from . import binding as mb
from .configs import F32, GREEDY, REJECTION, Workload


def cfg_for(w: Workload, L_cap: int, mode: int, B: Optional[int] = None) -> mb.Cfg:
    return mb.make_cfg(B=w.B if B is None else B, d=w.d, V=w.V, branching=w.branching, Hq=w.Hq, Hkv=w.Hkv,
                       D=w.D, L_cap=L_cap, dtype=w.dtype, mode=mode,
                       temperature=w.temperature if mode == REJECTION else 1.0, shared_vocab=w.shared_vocab,
                       tree_nodes=w.tree_nodes)


class DeviceStep:
    """Device-resident inputs and outputs of one step, plus the library calls."""

    def __init__(self, w: Workload, mode: int, L_cap: int, device="cuda", stream=None):
        self.w = w
        self.mode = mode
        self.cfg = cfg_for(w, L_cap, mode)
        self.dev = torch.device(device)
        self.stream = stream
        B, N, K, V, s_max = w.B, w.N, w.K, w.V, w.s_max
        i32 = dict(dtype=torch.int32, device=self.dev)
        self.logits = torch.empty((B, K, V), dtype=torch.float32, device=self.dev)
        self.topk = torch.empty((B, K, s_max), **i32)
        self.parent = torch.empty(N, **i32)
        self.depth = torch.empty(N, **i32)
        self.first_child = torch.empty(N, **i32)
        self.mask = torch.empty((N, N), dtype=torch.uint8, device=self.dev)
        self.anc_bits = torch.empty((N, 2), dtype=torch.int64, device=self.dev)
        self.tokens = torch.empty((B, N), **i32)
        self.pos = torch.empty((B, N), **i32)
        self.flags = torch.zeros(B, **i32)
        self.acc = torch.empty(B, **i32)
        self.path = torch.empty((B, K + 1), **i32)
        self.out_tokens = torch.empty((B, K + 1), **i32)
        self.n_out = torch.empty(B, **i32)
        self.kv_map = torch.empty((B, K + 1), **i32)
        self.O = None
        ws = mb.workspace_size(self.cfg)
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=self.dev)

    # ---- the five calls
    def heads(self, h, W, bias, U, write_logits: bool = True):
        mb.heads(self.cfg, h, W, bias, U, self.logits if (write_logits or self.mode == REJECTION) else None,
                 self.topk, self.workspace, self.stream)

    def tree_build(self, root_token, L, topk=None):
        mb.tree_build(self.cfg, root_token, self.topk if topk is None else topk, L, self.parent, self.depth,
                      self.first_child, self.mask, self.anc_bits, self.tokens, self.pos, self.flags, self.stream)

    def tree_attention(self, Q, Kc, Vc, L):
        if self.O is None or self.O.shape != Q.shape:
            self.O = torch.empty_like(Q)
        mb.tree_attention(self.cfg, Q, Kc, Vc, L, self.anc_bits, self.O, self.workspace, self.stream)

    def verify(self, target_logits, u_acc=None, u_res=None, head_logits=None, tokens=None):
        rs = self.mode == REJECTION
        mb.verify(self.cfg, self.tokens if tokens is None else tokens, self.parent, self.first_child,
                  target_logits, (self.logits if head_logits is None else head_logits) if rs else None,
                  u_acc if rs else None, u_res if rs else None, self.acc, self.path, self.out_tokens, self.n_out,
                  self.flags, self.workspace, self.stream)

    def kv_compact(self, Kc, Vc, L):
        mb.kv_compact(self.cfg, Kc, Vc, L, self.acc, self.path, self.kv_map, self.stream)

    def run(self, inp: "DeviceInputs", write_logits: bool = False, compact: bool = True):
        """The whole step, enqueued on the stream without host synchronisation."""
        self.heads(inp.h, inp.W, inp.bias, inp.U, write_logits=write_logits)
        self.tree_build(inp.root_token, inp.L)
        self.tree_attention(inp.Q, inp.Kc, inp.Vc, inp.L)
        self.verify(inp.target_logits, inp.u_acc, inp.u_res)
        if compact:
            self.kv_compact(inp.Kc, inp.Vc, inp.L)


    def fused_args(self, inp: "DeviceInputs", write_logits: bool = False, compact: bool = True) -> mb.StepArgs:
        """The buffers of the five calls for medusa_step_fused (greedy; no uniforms)."""
        if self.O is None or self.O.shape != inp.Q.shape:
            self.O = torch.empty_like(inp.Q)
        return mb.step_args(
            h=inp.h, W=inp.W, bias=inp.bias, U=inp.U, logits=self.logits if write_logits else None, topk=self.topk,
            root_token=inp.root_token, L=inp.L, parent=self.parent, depth=self.depth, first_child=self.first_child,
            mask=self.mask, anc_bits=self.anc_bits, tokens=self.tokens, pos=self.pos, flags=self.flags, Q=inp.Q,
            Kc=inp.Kc, Vc=inp.Vc, O=self.O, target_logits=inp.target_logits, u_acc=None, u_res=None, acc=self.acc,
            path=self.path, out_tokens=self.out_tokens, n_out=self.n_out, kv_map=self.kv_map,
            workspace=self.workspace, kv_compact=compact)

    def run_fused(self, inp: "DeviceInputs", write_logits: bool = False, compact: bool = True):
        """The whole step as one persistent kernel (medusa_step_fused)."""
        args = self.fused_args(inp, write_logits, compact)
        mb.step_fused(self.cfg, args, self.stream)
        return args

    def graph(self, inp: "DeviceInputs", write_logits: bool = False, compact: bool = True) -> mb.StepGraph:
        """The same five calls captured once as a CUDA graph over these buffers (one launch per step)."""
        rs = self.mode == REJECTION
        if self.O is None or self.O.shape != inp.Q.shape:
            self.O = torch.empty_like(inp.Q)
        return mb.StepGraph(
            self.cfg, h=inp.h, W=inp.W, bias=inp.bias, U=inp.U,
            logits=self.logits if (write_logits or rs) else None, topk=self.topk, root_token=inp.root_token,
            L=inp.L, parent=self.parent, depth=self.depth, first_child=self.first_child, mask=self.mask,
            anc_bits=self.anc_bits, tokens=self.tokens, pos=self.pos, flags=self.flags, Q=inp.Q, Kc=inp.Kc,
            Vc=inp.Vc, O=self.O, target_logits=inp.target_logits, u_acc=inp.u_acc if rs else None,
            u_res=inp.u_res if rs else None, acc=self.acc, path=self.path, out_tokens=self.out_tokens,
            n_out=self.n_out, kv_map=self.kv_map, workspace=self.workspace, kv_compact=compact)


@dataclass
class DeviceInputs:
    h: torch.Tensor
    W: torch.Tensor
    bias: Optional[torch.Tensor]
    U: torch.Tensor
    root_token: torch.Tensor
    L: torch.Tensor
    Q: torch.Tensor
    Kc: torch.Tensor
    Vc: torch.Tensor
    target_logits: torch.Tensor
    u_acc: torch.Tensor
    u_res: torch.Tensor


def to_device_inputs(si, target_logits: torch.Tensor, device="cuda") -> DeviceInputs:
    """Move a ``synth.StepInputs`` (plus target logits) to the device."""
    dev = torch.device(device)
    t = lambda x: None if x is None else x.to(dev)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    return DeviceInputs(h=t(si.h), W=t(si.W), bias=t(si.bias), U=t(si.U), root_token=i32(si.root_token),
                        L=i32(si.L), Q=t(si.Q), Kc=t(si.Kc), Vc=t(si.Vc), target_logits=t(target_logits),
                        u_acc=f32(si.u_acc), u_res=f32(si.u_res))
