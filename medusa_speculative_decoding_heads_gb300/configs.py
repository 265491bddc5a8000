"""The five synthetic Medusa verify-step workloads, by name and size.

Each workload fixes the shapes of one decoding step: batch ``B``, hidden size
``d``, vocabulary ``V``, the number of Medusa heads ``K`` with their branching
factors ``s_1..s_K`` (the candidate tree is the Cartesian product of the
per-head top-s lists), the attention shape (``Hq`` query heads, ``Hkv`` KV
heads, head dim ``D``), the committed KV length (fixed or drawn per sequence
from a range), the element type, the acceptance mode and the temperature.

This module holds sizes only: no arithmetic of the method.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Tuple

GREEDY = 0
REJECTION = 1

F32 = 0
BF16 = 1


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    d: int
    V: int
    branching: Tuple[int, ...]
    Hq: int
    Hkv: int
    D: int
    L_range: Tuple[int, int]          # committed KV length: inclusive [lo, hi]
    dtype: int                        # F32 or BF16 (weights, KV, Q, O, target logits)
    modes: Tuple[int, ...]            # acceptance modes the workload runs
    temperature: float
    target_sigma: float               # std of the synthetic target logits
    target_corr: float                # correlation of target logits with head logits
    compact: bool                     # KV compaction listed for the workload
    w_sigma: float = 0.02             # std of W_k and of the vocab projections
    shared_vocab: bool = False        # one vocab projection U for every head (U is [V][d])
    tree_paths: Optional[Tuple[Tuple[int, ...], ...]] = None   # a pruned tree's non-root rank paths
    note: str = ""

    @property
    def K(self) -> int:
        return len(self.branching)

    @property
    def N(self) -> int:
        """Node count: the pruned tree's, or the Cartesian tree's (root plus every level)."""
        if self.tree_paths is not None:
            return 1 + len(self.tree_paths)
        n, cnt = 1, 1
        for s in self.branching:
            cnt *= s
            n += cnt
        return n

    @property
    def tree_nodes(self):
        """(parent, rank) of every node of a pruned tree in breadth-first, rank-path
        lexicographic order (node 0 = root), or None for the Cartesian tree."""
        if self.tree_paths is None:
            return None
        order = [()] + sorted(self.tree_paths, key=lambda p: (len(p), p))
        at = {p: n for n, p in enumerate(order)}
        return [-1] + [at[p[:-1]] for p in order[1:]], [0] + [p[-1] for p in order[1:]]

    @property
    def s_max(self) -> int:
        return max(self.branching)

    @property
    def elt(self) -> int:
        return 4 if self.dtype == F32 else 2


WORKLOADS = {
    "tiny_fp32": Workload(
        name="tiny_fp32", B=1, d=256, V=1024, branching=(3, 2, 2), Hq=4, Hkv=4, D=64,
        L_range=(128, 128), dtype=F32, modes=(GREEDY, REJECTION), temperature=1.0,
        target_sigma=2.0, target_corr=0.0, compact=False,
        note="tiny fp32 step, batch 1, 22-node tree, greedy plus rejection sampling at T=1"),
    "vicuna7b_b1": Workload(
        name="vicuna7b_b1", B=1, d=4096, V=32000, branching=(4, 3, 2, 1), Hq=32, Hkv=32, D=128,
        L_range=(2048, 2048), dtype=BF16, modes=(GREEDY,), temperature=0.0,
        target_sigma=3.0, target_corr=0.0, compact=False,
        note="Vicuna-7B-shaped step, batch 1, bf16, 65-node tree, greedy"),
    "vicuna13b_b8": Workload(
        name="vicuna13b_b8", B=8, d=5120, V=32000, branching=(5, 3, 2, 1, 1), Hq=40, Hkv=40, D=128,
        L_range=(1024, 4096), dtype=BF16, modes=(REJECTION,), temperature=1.0,
        target_sigma=3.0, target_corr=0.8, compact=False,
        note="Vicuna-13B-shaped step, batch 8, bf16, 111-node tree, rejection sampling at T=1"),
    "vicuna33b_b16": Workload(
        name="vicuna33b_b16", B=16, d=6656, V=32000, branching=(4, 3, 2, 1), Hq=52, Hkv=52, D=128,
        L_range=(8192, 8192), dtype=BF16, modes=(GREEDY,), temperature=0.0,
        target_sigma=3.0, target_corr=0.0, compact=True,
        note="Vicuna-33B-shaped step, batch 16, bf16, 65-node tree, greedy plus KV compaction"),
    "gqa7b_b32": Workload(
        name="gqa7b_b32", B=32, d=4096, V=32000, branching=(4, 3, 2, 1), Hq=32, Hkv=8, D=128,
        L_range=(4096, 16384), dtype=BF16, modes=(REJECTION,), temperature=0.7,
        target_sigma=3.0, target_corr=0.8, compact=True,
        note="7B GQA-shaped step, batch 32, bf16, 65-node tree, rejection sampling at T=0.7 plus KV compaction"),
}

ORDER = ["tiny_fp32", "vicuna7b_b1", "vicuna13b_b8", "vicuna33b_b16", "gqa7b_b32"]

# The same steps with one frozen vocab projection shared by every head.
for _base in ("vicuna7b_b1", "vicuna13b_b8"):
    _w = WORKLOADS[_base]
    WORKLOADS[_base + "_shared"] = Workload(**dict(
        {k: getattr(_w, k) for k in _w.__dataclass_fields__}, name=_base + "_shared", shared_vocab=True,
        note=_w.note + "; every head projects with one shared (frozen LM-head) vocab matrix"))
SHARED = ["vicuna7b_b1_shared", "vicuna13b_b8_shared"]


def pruned_paths(K: int, s_max: int, count: int, decay: float = 0.5):
    """The `count` rank paths of highest estimated reach in a depth-K tree whose
    heads keep top-s_max lists, taking a candidate of rank r to be accepted with
    probability proportional to decay**r (so a path's score is the product over
    its ranks; prefixes always score higher, so the set is closed under prefixes).
    Ties go to the shorter, then lexicographically smaller path."""
    import heapq
    heap, out = [(-1.0, 0, ())], []
    while heap and len(out) < count + 1:
        neg, _, p = heapq.heappop(heap)
        out.append(p)
        if len(p) < K:
            for r in range(s_max):
                q = p + (r,)
                heapq.heappush(heap, (neg * decay ** r, len(q), q))
    return tuple(sorted((p for p in out if p), key=lambda p: (len(p), p)))


# Pruned 64-node trees (5 heads, top-8 lists) on the 7B and 13B step shapes.
for _base in ("vicuna7b_b1", "vicuna13b_b8"):
    _w = WORKLOADS[_base]
    _paths = pruned_paths(5, 8, 63)
    _br = tuple(1 + max(p[d] for p in _paths if len(p) > d) for d in range(5))
    WORKLOADS[_base + "_pruned64"] = Workload(**dict(
        {k: getattr(_w, k) for k in _w.__dataclass_fields__}, name=_base + "_pruned64", branching=_br,
        tree_paths=_paths, note=_w.note.split(",")[0] + f", pruned 64-node tree over 5 heads (top-s {_br})"))
PRUNED = ["vicuna7b_b1_pruned64", "vicuna13b_b8_pruned64"]


def get(name: str) -> Workload:
    return WORKLOADS[name]


def scaled(w: Workload, **overrides) -> Workload:
    """A copy of ``w`` with some sizes replaced (small parity cases of a workload)."""
    fields = {k: getattr(w, k) for k in w.__dataclass_fields__}
    fields.update(overrides)
    return Workload(**fields)
