"""Seeded synthetic inputs for one Medusa verify step.

Both sides of every parity check (the CUDA library and the CPU oracle) take
their inputs from here; this module holds none of the method's arithmetic.

* Dense inputs (hidden state, head weights, queries, KV cache, target logits)
  are normal draws from a seeded ``torch.Generator`` on the requested device,
  rounded once to the workload's element type (bf16 round-to-nearest-even).
* The uniforms that rejection sampling consumes come from Philox4x32-10
  (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
  SC'11), written out here from its published definition: key ``(seed_lo,
  seed_hi)``, counter ``(b, slot, stream, 0)``, first output word ``x``, and
  ``u = (x >> 8) * 2**-24`` in [0, 1).
* Target logits "correlated with the head logits" are a mix of a given,
  already computed head-logit array ``zhat`` and fresh noise; the caller
  supplies ``zhat`` and the depth of every tree node.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from .configs import BF16, F32, Workload

# ---------------------------------------------------------------- Philox4x32-10
PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint32(0x9E3779B9)
PHILOX_W1 = np.uint32(0xBB67AE85)
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(ctr: np.ndarray, key) -> np.ndarray:
    """Philox4x32 with 10 rounds. ``ctr`` [..., 4] uint32, ``key`` two uint32 words."""
    c = np.array(ctr, dtype=np.uint32, copy=True)
    k0 = np.uint32(int(key[0]) & 0xFFFFFFFF)
    k1 = np.uint32(int(key[1]) & 0xFFFFFFFF)
    with np.errstate(over="ignore"):
        for rnd in range(10):
            if rnd > 0:
                k0 = (k0 + PHILOX_W0).astype(np.uint32)
                k1 = (k1 + PHILOX_W1).astype(np.uint32)
            p0 = PHILOX_M0 * c[..., 0].astype(np.uint64)
            p1 = PHILOX_M1 * c[..., 2].astype(np.uint64)
            hi0 = (p0 >> np.uint64(32)).astype(np.uint32)
            lo0 = (p0 & _MASK32).astype(np.uint32)
            hi1 = (p1 >> np.uint64(32)).astype(np.uint32)
            lo1 = (p1 & _MASK32).astype(np.uint32)
            n0 = hi1 ^ c[..., 1] ^ k0
            n2 = hi0 ^ c[..., 3] ^ k1
            c = np.stack([n0, lo1, n2, lo0], axis=-1).astype(np.uint32)
    return c


def philox_uniforms(seed: int, b: np.ndarray, slot: np.ndarray, stream: int) -> np.ndarray:
    """u in [0,1) (float32, exact) for counters (b, slot, stream, 0) under key=seed."""
    b = np.asarray(b, dtype=np.uint32)
    slot = np.asarray(slot, dtype=np.uint32)
    b, slot = np.broadcast_arrays(b, slot)
    ctr = np.stack([b, slot, np.full_like(b, stream), np.zeros_like(b)], axis=-1)
    key = np.array([seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF], dtype=np.uint32)
    x = philox4x32_10(ctr, key)[..., 0]
    return ((x >> np.uint32(8)).astype(np.float64) * 2.0 ** -24).astype(np.float32)


STREAM_U_ACC = 0
STREAM_U_RES = 1
STREAM_L = 2
STREAM_ROOT = 3


def uniforms_for_step(seed: int, B: int, K: int, s_max: int):
    """(u_acc [B][K][s_max], u_res [B][K+1]) float32: the acceptance and resampling draws."""
    bb, ss = np.meshgrid(np.arange(B), np.arange(K * s_max), indexing="ij")
    u_acc = philox_uniforms(seed, bb, ss, STREAM_U_ACC).reshape(B, K, s_max)
    bb, ss = np.meshgrid(np.arange(B), np.arange(K + 1), indexing="ij")
    u_res = philox_uniforms(seed, bb, ss, STREAM_U_RES).reshape(B, K + 1)
    return u_acc, u_res


def committed_lengths(seed: int, B: int, lo: int, hi: int) -> np.ndarray:
    """Per-sequence committed KV lengths, uniform integers in [lo, hi] (int32)."""
    if lo == hi:
        return np.full(B, lo, dtype=np.int32)
    u = philox_uniforms(seed, np.arange(B), np.zeros(B, dtype=np.uint32), STREAM_L).astype(np.float64)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int32)


def root_tokens(seed: int, B: int, V: int) -> np.ndarray:
    u = philox_uniforms(seed, np.arange(B), np.zeros(B, dtype=np.uint32), STREAM_ROOT).astype(np.float64)
    return np.minimum(np.floor(u * V), V - 1).astype(np.int32)


def cache_capacity(L: np.ndarray, N: int, align: int = 64) -> int:
    need = int(np.max(L)) + N
    return (need + align - 1) // align * align


# ---------------------------------------------------------------- dense draws
def torch_dtype(dtype: int) -> torch.dtype:
    return torch.float32 if dtype == F32 else torch.bfloat16


def normal(gen: torch.Generator, shape, sigma: float, dtype: int, device) -> torch.Tensor:
    """N(0, sigma^2) draws rounded once to the element type; drawn in slices to bound memory."""
    shape = tuple(int(s) for s in shape)
    out = torch.empty(shape, dtype=torch_dtype(dtype), device=device)
    flat = out.view(-1) if out.numel() else out
    step = 1 << 26
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        t = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
        if sigma != 1.0:
            t.mul_(sigma)
        flat[i:i + n].copy_(t)
    return out


@dataclass
class StepInputs:
    """Everything one verify step reads, on one device."""
    w: Workload
    seed: int
    h: torch.Tensor            # [B][d]
    W: torch.Tensor            # [K][d][d]   row = output feature
    bias: Optional[torch.Tensor]  # [K][d] or None
    U: torch.Tensor            # [K][V][d]   vocab projection per head
    root_token: np.ndarray     # [B] int32
    L: np.ndarray              # [B] int32
    L_cap: int
    Q: torch.Tensor            # [B][N][Hq][D]
    Kc: torch.Tensor           # [B][Hkv][L_cap][D]; tree keys at rows L_b .. L_b+N-1
    Vc: torch.Tensor           # [B][Hkv][L_cap][D]
    u_acc: np.ndarray          # [B][K][s_max] float32
    u_res: np.ndarray          # [B][K+1] float32


def make_step_inputs(w: Workload, seed: int, device="cpu", with_bias: bool = False,
                     bias_sigma: float = 0.5) -> StepInputs:
    """Seeded inputs of one step of workload ``w`` (target logits are made separately)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    B, d, V, K, N = w.B, w.d, w.V, w.K, w.N
    h = normal(gen, (B, d), 1.0, w.dtype, dev)
    W = normal(gen, (K, d, d), w.w_sigma, w.dtype, dev)
    bias = normal(gen, (K, d), bias_sigma, w.dtype, dev) if with_bias else None
    U = normal(gen, (V, d) if w.shared_vocab else (K, V, d), w.w_sigma, w.dtype, dev)
    L = committed_lengths(seed, B, *w.L_range)
    L_cap = cache_capacity(L, N)
    Q = normal(gen, (B, N, w.Hq, w.D), 1.0, w.dtype, dev)
    Kc = normal(gen, (B, w.Hkv, L_cap, w.D), 1.0, w.dtype, dev)
    Vc = normal(gen, (B, w.Hkv, L_cap, w.D), 1.0, w.dtype, dev)
    u_acc, u_res = uniforms_for_step(seed, B, K, w.s_max)
    return StepInputs(w=w, seed=seed, h=h, W=W, bias=bias, U=U,
                      root_token=root_tokens(seed, B, V), L=L, L_cap=L_cap,
                      Q=Q, Kc=Kc, Vc=Vc, u_acc=u_acc, u_res=u_res)


def target_logits(w: Workload, seed: int, device="cpu", zhat: Optional[torch.Tensor] = None,
                  depth: Optional[np.ndarray] = None) -> torch.Tensor:
    """Synthetic target logits [B][N][V] in the workload's element type.

    Independent workloads: N(0, sigma^2). Correlated workloads: for a node at
    depth e < K the row is ``sigma * (rho * std(zhat[b][e]) + sqrt(1-rho^2) * eps)``
    where ``std`` standardises the given head-logit row (zero mean, unit
    variance) and ``eps`` is N(0,1); nodes at depth K (leaves) use rho = 0.
    ``zhat`` is [B][K][V] and ``depth`` is [N], both supplied by the caller.
    """
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed + 7919)
    B, N, V, K = w.B, w.N, w.V, w.K
    rho = w.target_corr
    if rho == 0.0:
        return normal(gen, (B, N, V), w.target_sigma, w.dtype, dev)
    assert zhat is not None and depth is not None
    out = torch.empty((B, N, V), dtype=torch_dtype(w.dtype), device=dev)
    z = zhat.to(device=dev, dtype=torch.float32)
    zs = (z - z.mean(dim=-1, keepdim=True)) / z.std(dim=-1, keepdim=True)
    mix = float(np.sqrt(1.0 - rho * rho))
    for n in range(N):
        eps = torch.randn((B, V), generator=gen, device=dev, dtype=torch.float32)
        e = int(depth[n])
        if e < K:
            row = rho * zs[:, e, :] + mix * eps
        else:
            row = eps
        out[:, n, :] = (w.target_sigma * row).to(out.dtype)
    return out


def plant_tokens(logits: torch.Tensor, b: int, nodes, tokens, boost: float = 30.0) -> None:
    """Add ``boost`` to ``logits[b][node][token]`` for each given (node, token) pair, in place."""
    for n, t in zip(nodes, tokens):
        logits[b, int(n), int(t)] += boost
