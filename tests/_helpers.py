"""Shared helpers for the GPU parity tests: device setup, host copies, comparisons."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from medusa_speculative_decoding_heads_gb300 import _build, binding as mb, configs, synth
from medusa_speculative_decoding_heads_gb300.configs import F32
from oracle import medusa_oracle as O


def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    _build.build()
    mb.load()
    return torch.device("cuda")


def f64(t) -> np.ndarray:
    """Exact float64 copy of a device/host tensor (bf16 decodes exactly)."""
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float32).double().numpy()


def i64(t) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.int64)


def tol_for(dtype: int) -> float:
    """Stated tolerance: 1e-5 for float32, 2e-2 for bf16, applied as |g - o| <= tol * max(1, |o|)."""
    return 1e-5 if dtype == F32 else 2e-2


def assert_close(gpu: np.ndarray, ref: np.ndarray, dtype: int, what: str):
    tol = tol_for(dtype)
    err = np.abs(gpu - ref) / np.maximum(1.0, np.abs(ref))
    assert np.isfinite(gpu).all(), f"{what}: non-finite GPU values"
    worst = float(err.max()) if err.size else 0.0
    assert worst <= tol, f"{what}: max scaled error {worst:.3e} > {tol:.0e}"
    return worst


def random_topk(rng, B, K, s_max, branching, V):
    topk = np.full((B, K, s_max), -1, dtype=np.int32)
    for b in range(B):
        for k in range(K):
            topk[b, k, :branching[k]] = rng.choice(V, size=branching[k], replace=False)
    return topk


def planted_greedy_logits(logits: torch.Tensor, tree: dict, seed: int, K: int):
    """Boost a seeded random path so the greedy walk accepts a seeded number of drafts.

    For sequence b a depth a in 0..K and a path of a nodes are drawn (shorter if
    it reaches a leaf of a pruned tree first); the target logit of each path
    node's token is raised at its parent. Returns the planted depths.
    """
    rng = np.random.default_rng(seed)
    B = logits.shape[0]
    depths = []
    for b in range(B):
        a = int(rng.integers(0, K + 1))
        cur = 0
        nodes, toks = [], []
        for step in range(a):
            kids = O.children_of(tree["parent"], cur)
            if not kids:
                a = step
                break
            nxt = kids[int(rng.integers(len(kids)))]
            nodes.append(cur)
            toks.append(int(tree["tokens"][b, nxt]))
            cur = nxt
        synth.plant_tokens(logits, b, nodes, toks, boost=40.0)
        depths.append(a)
    return depths
