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


# A sequence whose walk the GPU flags as a near tie (|u - r| < 1e-6, or an inverse-CDF draw within
# 1e-6 of a step, in its float32 arithmetic) is excused only when the oracle, on the same inputs,
# sees a tie within this wider band: float32 ratios and prefix sums are off from float64 by a few
# units in 1e-7, far inside it. A GPU flag the oracle cannot explain is a failure.
FLAG_BAND = 1e-5
TIE_BITS = O.FLAG_RS_NEAR_TIE | O.FLAG_CDF_NEAR_TIE


def compare_verify(st, mode, tree, target_logits, K, head_logits=None, u_acc=None, u_res=None, T=1.0,
                   eligible=None, min_compared=None, what="verify"):
    """Walk outputs of a DeviceStep against the oracle's walk on the same inputs, bit for bit.

    The oracle runs with the 1e-6 windows; a sequence it flags is excluded (its n_out must
    still lie in [1, K+1]). A sequence only the GPU flags must be flagged by the oracle at
    FLAG_BAND, else the test fails. `eligible` masks out sequences excluded upstream (a
    near tie in top-s). At least `min_compared` sequences (default half the batch) must be
    compared. Returns (oracle result, number compared)."""
    B = target_logits.shape[0]
    kw = dict(head_logits=head_logits, u_acc=u_acc, u_res=u_res, T=T)
    ref = O.verify_batch(mode, tree, target_logits, K, **kw)
    band = O.verify_batch(mode, tree, target_logits, K, rs_tie=FLAG_BAND, cdf_tie=FLAG_BAND, **kw) \
        if mode == configs.REJECTION else ref
    gflags = i64(st.flags) & TIE_BITS
    n_out = i64(st.n_out)
    got = {key: i64(getattr(st, key)) for key in ("acc", "path", "out_tokens", "n_out")}
    compared = 0
    for b in range(B):
        if eligible is not None and not eligible[b]:
            continue
        if ref["flags"][b]:
            assert 1 <= n_out[b] <= K + 1, f"{what}: n_out out of range at b={b}"
            continue
        assert not gflags[b] or band["flags"][b], \
            f"{what}: GPU flagged b={b} (flags {gflags[b]}) where the oracle sees no tie within {FLAG_BAND}"
        if gflags[b]:
            continue
        for key, v in got.items():
            assert np.array_equal(v[b], ref[key][b]), f"{what}: {key} differs at b={b}"
        compared += 1
    need = max(1, B // 2) if min_compared is None else min_compared
    assert compared >= need, f"{what}: only {compared} of {B} sequences compared (need {need})"
    return ref, compared
