"""CPU oracle for one Medusa verify step: plain, slow, float64, obviously correct.

TEST INFRASTRUCTURE ONLY. Nothing in the product imports, links or calls this
module; only the tests, the package's smoke check and the benchmark's CPU
baseline leg do. It shares no code with the CUDA path: it takes plain numpy
arrays (bf16 inputs already decoded exactly to float64) and returns numpy
arrays.

Sources (untrusted web pages, read for what the method computes):
  [MEDUSA-ARCH]  "Medusa 심층 아키텍처: 별도 초안 모델을 제거한 다중 헤드 추측 디코딩과
                  Tree Attention 3배 가속 원리" (techknowgenie.com)
  [VLLM-MEDUSA]  "[vLLM] Medusa: 다중 예측 헤드 투기적 디코딩" (blog.secrett2633.cloud)
  [SPEC-DEC]     "Speculative Decoding(투기적 디코딩) 원리와 가속 아키텍처: Draft Model과
                  Rejection Sampling부터 Medusa·EAGLE-3 및 vLLM 서빙 최적화까지" (blog.huny.dev)
  [OPT-2]        "최적화 2편. 추측 디코딩과 긴 컨텍스트 - Speculative Decoding과 MEDUSA·EAGLE,
                  Ring Attention" (beengineer500.github.io)

Readings where the pages are silent (each one repeated where it is used):
  R1  the tree root is the already committed next token, given per sequence;
      depth k (k = 1..K) draws its candidates from Medusa head k.
  R2  node order is breadth first; inside one depth, lexicographic in the
      rank path (first rank most significant).
  R3  the tree is the Cartesian product of per-head top-s lists, so a node's
      token is head[depth]'s candidate of the node's own rank.
  R4  top-s orders by value descending, ties to the lower index.
  R5  the residual-block output r is kept unrounded (float64 here).
  R7  position id of a node = committed length + depth.
  R8  attention scale 1/sqrt(D), no positional transform, GQA map
      kv = h // (Hq / Hkv).
  R9  greedy acceptance walks from the root to the child whose token equals the
      target argmax (ties to the lowest token id), then emits the target argmax
      at the last accepted node as the bonus/correction token.
  R10 tree rejection sampling applies the single-candidate rule at each depth,
      trying siblings in rank order and carrying the residual forward;
      inverse-CDF sampling picks the smallest y with cdf(y) > u * total.
  R11 compaction moves the accepted path's rows to the front of the tree
      region and advances the committed length by acc + 1.
  R13 a pruned tree is the prefix-closed set of its nodes' rank paths; R2's
      order and R3's tokens apply unchanged, and a leaf above depth K ends the
      walk there (the bonus comes from that leaf's target row).
  R14 a shared vocab projection is one matrix U [V][d] used by every head.
  R15 a paged cache is a storage layout of the same logical cache: logical row
      i of sequence b sits at offset i % P of page block_table[b][i // P]; the
      tree's own rows are staged apart and follow the committed prefix.

Parity status: every function below is pinned by tests under tests/ (closed
forms, brute force, library routines, the pages' worked examples) except the
rejection-sampling walk on *deterministic* top-s drafts, whose output law is
not fixed by the pages ("parity unpinned" for that case; its s=1 chain case
and its behaviour with drafts sampled from q are pinned).
"""
from __future__ import annotations

import itertools
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

# Flag bits written per sequence by the verify walks (same meaning as the C header).
FLAG_RS_NEAR_TIE = 1       # |u - r| < RS_TIE for some acceptance test on the walk
FLAG_CDF_NEAR_TIE = 2      # inverse-CDF draw within CDF_TIE * total of a boundary
FLAG_CAPACITY = 4          # L_b + N > L_cap

RS_TIE = 1e-6
CDF_TIE = 1e-6
TOPK_TIE = 1e-4


# --------------------------------------------------------------------------- heads
def silu(x: np.ndarray) -> np.ndarray:
    """SiLU(x) = x * sigmoid(x) = x / (1 + e^-x)."""
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def medusa_heads(h: np.ndarray, W: np.ndarray, b: Optional[np.ndarray], U: np.ndarray):
    """Residual block then vocab projection for every head.

    [MEDUSA-ARCH] "잔차 블록(Residual Block)을 포함한 Medusa 헤드 구조" section,
    equations for h_t^(k) and p_k:
    h^(k) = SiLU(h W_res^(k)) + h and p_k = softmax(h^(k) W_head^(k)); the
    "소스코드 레벨 구조 분석" section's MedusaHead applies Linear(d, d), SiLU,
    adds the residual, then Linear(d, V) without bias. A per-head bias b_k on
    the d x d layer is allowed (None means zero).

    Layouts: h [B][d]; W [K][d][d] with W[k][o][i] the weight from input i to
    output o (the nn.Linear convention); b [K][d] or None; U [K][V][d] with
    U[k][v][i] the weight from feature i to token v, or U [V][d]: one vocab
    projection shared by every head (the same section notes that W_head^(k)
    may be the base model's frozen unembedding W_lm_head, kept as is).
    Returns r [B][K][d] (R5: unrounded) and logits z [B][K][V].
    """
    B, d = h.shape
    K = W.shape[0]
    V = U.shape[-2]
    r = np.empty((B, K, d), dtype=np.float64)
    z = np.empty((B, K, V), dtype=np.float64)
    for k in range(K):
        pre = h @ W[k].T
        if b is not None:
            pre = pre + b[k][None, :]
        r[:, k, :] = h + silu(pre)
        Uk = U if U.ndim == 2 else U[k]
        z[:, k, :] = r[:, k, :] @ Uk.T
    return r, z


def top_s(row: np.ndarray, s: int, tie: float = TOPK_TIE) -> Tuple[np.ndarray, bool]:
    """Indices of the s largest entries, descending, ties to the lower index (R4).

    [MEDUSA-ARCH] "트리 어텐션" section (each head keeps its top-s candidates) and
    generate_candidates (torch.topk(...).indices per head). Also returns a
    near-tie flag: True when two neighbours among the first s+1 sorted values
    are closer than ``tie * max(1, |value|)``, where a float32 computation of
    the same row may order them differently.
    """
    V = row.shape[0]
    order = np.lexsort((np.arange(V), -row))
    m = min(s + 1, V)
    vals = row[order[:m]]
    near = False
    for i in range(m - 1):
        if vals[i] - vals[i + 1] < tie * max(1.0, abs(vals[i])):
            near = True
    return order[:s].astype(np.int64), near


def heads_top_s(z: np.ndarray, branching: Sequence[int]):
    """topk [B][K][s_max] int (-1 beyond s_k) and near-tie flags [B][K] bool."""
    B, K, V = z.shape
    s_max = max(branching)
    topk = np.full((B, K, s_max), -1, dtype=np.int64)
    near = np.zeros((B, K), dtype=bool)
    for b in range(B):
        for k in range(K):
            idx, nt = top_s(z[b, k], branching[k])
            topk[b, k, :branching[k]] = idx
            near[b, k] = nt
    return topk, near


# --------------------------------------------------------------------------- tree
def tree_layout(branching: Sequence[int]):
    """Node order and parent links of the Cartesian candidate tree.

    [MEDUSA-ARCH] "고정 트리 토폴로지와 2차원 어텐션 마스크": head k keeps top-s_k
    candidates and every candidate of depth k branches into the top-s_{k+1} of
    the next head (the pages' example is top-2 x top-3 x top-2). R1 puts a given
    root at depth 0; R2 orders nodes breadth first, lexicographically by rank
    path. Each node is named by its rank path, enumerated depth by depth.
    Returns dict with N, paths, parent, depth, rank, first_child.
    """
    levels: List[List[Tuple[int, ...]]] = [[()]]
    for s in branching:
        levels.append([p + (i,) for p in levels[-1] for i in range(s)])
    paths = [p for lvl in levels for p in lvl]
    index = {p: n for n, p in enumerate(paths)}
    N = len(paths)
    parent = [-1] + [index[p[:-1]] for p in paths[1:]]
    depth = [len(p) for p in paths]
    rank = [p[-1] if p else 0 for p in paths]
    first_child = []
    for n in range(N):
        kids = [c for c in range(N) if parent[c] == n]
        first_child.append(min(kids) if kids else -1)
    return {"N": N, "paths": paths, "parent": np.array(parent, dtype=np.int64),
            "depth": np.array(depth, dtype=np.int64), "rank": np.array(rank, dtype=np.int64),
            "first_child": np.array(first_child, dtype=np.int64)}


def tree_layout_from_paths(paths: Sequence[Sequence[int]], branching: Sequence[int]):
    """Node order and parent links of a pruned candidate tree given by its nodes' rank paths.

    [MEDUSA-ARCH] runs its benchmarks with 4 heads and 64 tree branches
    ("벤치마크 실측 지표: 도메인별 속도 향상 및 수용률") and calls a topology of
    about 32-64 nodes the usual optimum ("트리 크기(Tree Size)와 검증 오버헤드의
    균형"): a subset of the Cartesian tree rather than all of it. Reading (R13):
    the tree is given as the set of its non-root nodes' rank paths (i_1, ..., i_d)
    with 0 <= i_e < s_e, closed under prefixes; node order is R2's (breadth
    first, lexicographic by rank path), so each node's children are contiguous
    and in rank order, and a node's token is head d's candidate i_d (R3). The
    full Cartesian product gives back tree_layout(branching).
    Returns the same dict as tree_layout.
    """
    K = len(branching)
    ps = sorted({tuple(int(i) for i in p) for p in paths}, key=lambda p: (len(p), p))
    for p in ps:
        if not 1 <= len(p) <= K:
            raise ValueError(f"path {p}: depth outside 1..{K}")
        if any(not 0 <= p[e] < branching[e] for e in range(len(p))):
            raise ValueError(f"path {p}: rank outside the head's top-s")
        if len(p) > 1 and p[:-1] not in ps:
            raise ValueError(f"path {p}: its prefix is not a node")
    ordered = [()] + ps
    index = {p: n for n, p in enumerate(ordered)}
    N = len(ordered)
    parent = [-1] + [index[p[:-1]] for p in ordered[1:]]
    depth = [len(p) for p in ordered]
    rank = [p[-1] if p else 0 for p in ordered]
    first_child = []
    for n in range(N):
        kids = [c for c in range(N) if parent[c] == n]
        first_child.append(min(kids) if kids else -1)
    return {"N": N, "paths": ordered, "parent": np.array(parent, dtype=np.int64),
            "depth": np.array(depth, dtype=np.int64), "rank": np.array(rank, dtype=np.int64),
            "first_child": np.array(first_child, dtype=np.int64)}


def ancestor_mask(parent: np.ndarray) -> np.ndarray:
    """mask[i][j] = 1 iff j is an ancestor of i or j == i.

    [MEDUSA-ARCH] "트리 어텐션" section, TreeMask equation (0 where visible,
    -inf elsewhere; this returns the 0/1 visibility form). Built by walking
    each node's parent chain.
    """
    N = parent.shape[0]
    mask = np.zeros((N, N), dtype=np.uint8)
    for i in range(N):
        j = i
        while j >= 0:
            mask[i, j] = 1
            j = int(parent[j])
    return mask


def mask_bits(mask: np.ndarray) -> np.ndarray:
    """Pack mask rows into two 64-bit words per node (bit j of word j // 64)."""
    N = mask.shape[0]
    bits = np.zeros((N, 2), dtype=np.uint64)
    for i in range(N):
        for j in range(N):
            if mask[i, j]:
                bits[i, j // 64] |= np.uint64(1) << np.uint64(j % 64)
    return bits


def tree_build(branching: Sequence[int], root_token: np.ndarray, topk: np.ndarray,
               L: np.ndarray, L_cap: Optional[int] = None, paths: Optional[Sequence[Sequence[int]]] = None):
    """Tree arrays, per-sequence tokens and position ids (R1-R3, R7).

    tokens[b][0] = root_token[b]; tokens[b][n] = topk[b][depth-1][rank] (R3);
    pos[b][n] = L[b] + depth[n] (R7). flags[b] gets FLAG_CAPACITY when
    L[b] + N exceeds L_cap. `paths` selects a pruned tree (R13) instead of the
    full Cartesian one.
    """
    lay = tree_layout(branching) if paths is None else tree_layout_from_paths(paths, branching)
    N = lay["N"]
    B = root_token.shape[0]
    mask = ancestor_mask(lay["parent"])
    tokens = np.zeros((B, N), dtype=np.int64)
    pos = np.zeros((B, N), dtype=np.int64)
    flags = np.zeros(B, dtype=np.int64)
    for b in range(B):
        for n in range(N):
            dep = int(lay["depth"][n])
            tokens[b, n] = root_token[b] if dep == 0 else topk[b, dep - 1, lay["rank"][n]]
            pos[b, n] = int(L[b]) + dep
        if L_cap is not None and (int(L[b]) < 0 or int(L[b]) + N > L_cap):
            flags[b] = FLAG_CAPACITY
    return {"N": N, "parent": lay["parent"], "depth": lay["depth"], "rank": lay["rank"],
            "first_child": lay["first_child"], "mask": mask, "anc_bits": mask_bits(mask),
            "tokens": tokens, "pos": pos, "flags": flags}


# --------------------------------------------------------------------------- attention
def tree_attention(Q: np.ndarray, Kc: np.ndarray, Vc: np.ndarray, L: np.ndarray,
                   mask: np.ndarray, Hq: int, Hkv: int,
                   pairs: Optional[Sequence[Tuple[int, int]]] = None) -> np.ndarray:
    """Every tree node attends to the committed cache plus its own ancestors.

    [MEDUSA-ARCH] "트리 어텐션" section: with the TreeMask, all tree tokens are
    evaluated in one pass and branches do not see each other; [SPEC-DEC]
    "3. 최신 투기적 디코딩 아키텍처 진화" (Tree Attention item) says the same.
    R8: scores q.k / sqrt(D), plain softmax, GQA head map kv = h // (Hq/Hkv).

    Q [B][N][Hq][D]; Kc, Vc [B][Hkv][L_cap][D] with the tree's keys/values at
    rows L_b .. L_b+N-1. Node i sees rows [0, L_b) and L_b + j for mask[i][j].
    ``pairs`` restricts the work to the listed (b, h); other outputs are NaN.
    Returns O [B][N][Hq][D] float64.
    """
    B, N, _, D = Q.shape
    G = Hq // Hkv
    O = np.full(Q.shape, np.nan, dtype=np.float64)
    todo = pairs if pairs is not None else [(b, h) for b in range(B) for h in range(Hq)]
    for b, h in todo:
        Lb = int(L[b])
        kv = h // G
        keys = Kc[b, kv, :Lb + N, :].astype(np.float64)
        vals = Vc[b, kv, :Lb + N, :].astype(np.float64)
        visible = np.concatenate([np.ones((N, Lb), dtype=bool), mask.astype(bool)], axis=1)
        S = (Q[b, :, h, :].astype(np.float64) @ keys.T) / math.sqrt(D)
        S = np.where(visible, S, -np.inf)
        S = S - S.max(axis=1, keepdims=True)
        P = np.exp(S)
        P = P / P.sum(axis=1, keepdims=True)
        O[b, :, h, :] = P @ vals
    return O


def attention_block_partial(q: np.ndarray, keys: np.ndarray, vals: np.ndarray, visible: np.ndarray):
    """One key block's partial result for one query row, in the block-wise form of
    [OPT-2] section 3.3 (attention over key blocks merged through the running
    maximum and exp-sum): with s_j = q.k_j / sqrt(D) over the block's visible keys,
    m = max_j s_j, l = sum_j exp(s_j - m), o = sum_j exp(s_j - m) v_j (not yet
    divided by l). A block with no visible key gives (-inf, 0, 0)."""
    D = q.shape[0]
    s = (keys.astype(np.float64) @ q.astype(np.float64)) / math.sqrt(D)
    s = s[visible.astype(bool)]
    v = vals.astype(np.float64)[visible.astype(bool)]
    if s.size == 0:
        return -np.inf, 0.0, np.zeros(vals.shape[1])
    m = float(s.max())
    p = np.exp(s - m)
    return m, float(p.sum()), p @ v


def merge_attention_partials(parts) -> np.ndarray:
    """Exact merge of block partials (m_i, l_i, o_i) ([OPT-2] section 3.3):
    M = max_i m_i, l = sum_i exp(m_i - M) l_i, output = sum_i exp(m_i - M) o_i / l."""
    M = max(m for m, _, _ in parts)
    l = sum(math.exp(m - M) * li for m, li, _ in parts if m != -np.inf)
    o = sum(math.exp(m - M) * oi for m, _, oi in parts if m != -np.inf)
    return o / l


# --------------------------------------------------------------------------- acceptance
def children_of(parent: np.ndarray, node: int) -> List[int]:
    """Children in node-id order, which is rank order (R2)."""
    return [c for c in range(parent.shape[0]) if parent[c] == node]


def verify_greedy(tokens: np.ndarray, parent: np.ndarray, target_logits: np.ndarray, K: int):
    """Greedy longest-matching-path acceptance with the bonus/correction token (R9).

    [OPT-2] "1.3 검증 - 일치는 유지, 불일치는 폐기": drafts that match the
    target's own prediction are kept, everything after the first mismatch is
    dropped, the mismatch position takes the target's prediction, and an
    all-match yields one extra token; [SPEC-DEC] §5 Case 2 gives the worked
    example [1,2,3,4] -> [1,2,0]. On a tree the matching child is unique since
    siblings carry distinct tokens.

    One sequence: tokens [N], target_logits [N][V]. Returns (acc, path [K+1],
    out_tokens [K+1], n_out), -1 padded.
    """
    path = [0]
    out: List[int] = []
    cur = 0
    for _ in range(K):
        want = int(np.argmax(target_logits[cur]))     # first maximum = lowest id on ties
        nxt = [c for c in children_of(parent, cur) if int(tokens[c]) == want]
        if not nxt:
            break
        cur = nxt[0]
        path.append(cur)
        out.append(int(tokens[cur]))
    out.append(int(np.argmax(target_logits[cur])))
    acc = len(path) - 1
    return acc, _pad(path, K + 1), _pad(out, K + 1), acc + 1


def softmax_t(x: np.ndarray, T: float) -> np.ndarray:
    """softmax(x / T) in float64."""
    y = np.asarray(x, dtype=np.float64) / T
    y = y - y.max()
    e = np.exp(y)
    return e / e.sum()


def acceptance_ratio(p: np.ndarray, q: np.ndarray, x: int) -> float:
    """r = min(1, p(x) / q(x)).

    [MEDUSA-ARCH] "수학적 무손실 보장" section, equation alpha(x); [SPEC-DEC] §2.1,
    equation r.
    """
    return min(1.0, float(p[x]) / float(q[x]))


def residual(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """max(0, p - q) / sum max(0, p - q); p itself when that sum is below 1e-30.

    [MEDUSA-ARCH] "수학적 무손실 보장" section, equation p'(x); [SPEC-DEC] §2.1,
    equation p_res.
    """
    w = np.maximum(0.0, p - q)
    tot = float(w.sum())
    if tot < 1e-30:
        return p
    return w / tot


def inverse_cdf(w: np.ndarray, u: float, tie: float = CDF_TIE) -> Tuple[int, bool]:
    """Smallest y with sum_{v<=y} w_v > u * sum_v w_v (R10), sequential float64 sums.

    Also returns a near-boundary flag: u*total within CDF_TIE*total of the
    cumulative sum at y or at y-1.
    """
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    tot = float(c[-1])
    thr = u * tot
    y = int(np.argmax(c > thr))
    near = abs(thr - c[y]) < tie * tot or (y > 0 and abs(thr - c[y - 1]) < tie * tot)
    return y, near


def verify_rejection(tokens: np.ndarray, parent: np.ndarray, target_logits: np.ndarray,
                     head_logits: np.ndarray, u_acc: np.ndarray, u_res: np.ndarray,
                     K: int, T: float, rs_tie: float = RS_TIE, cdf_tie: float = CDF_TIE):
    """Tree rejection sampling with the residual carried across siblings (R10).

    The single-candidate rule is [MEDUSA-ARCH] "수학적 무손실 보장" and [SPEC-DEC]
    §2.1: accept x when u < min(1, p(x)/q(x)), otherwise resample from the
    residual max(0, p - q)/sum. On the tree: at the current node, p =
    softmax(target_logits[node] / T) and q = softmax(head_logits[depth] / T) for
    the head that drafted the next depth; children are tried in rank order
    with u_acc[depth][rank]; each rejection replaces p by the residual. When
    every child is rejected the bonus is drawn from the current p with
    u_res[depth]; after an accepted leaf it is drawn from softmax(target/T) at
    the leaf with u_res[K].

    One sequence: tokens [N], target_logits [N][V], head_logits [K][V],
    u_acc [K][s_max], u_res [K+1]. Returns (acc, path, out_tokens, n_out, flags).
    """
    flags = 0
    path = [0]
    out: List[int] = []
    cur = 0
    p = softmax_t(target_logits[cur], T)
    for dep in range(1, K + 1):
        q = softmax_t(head_logits[dep - 1], T)
        accepted = None
        for j, c in enumerate(children_of(parent, cur)):
            x = int(tokens[c])
            r = acceptance_ratio(p, q, x)
            u = float(u_acc[dep - 1, j])
            if abs(u - r) < rs_tie:
                flags |= FLAG_RS_NEAR_TIE
            if u < r:
                accepted = c
                break
            p = residual(p, q)
        if accepted is None:
            y, near = inverse_cdf(p, float(u_res[dep - 1]), cdf_tie)
            if near:
                flags |= FLAG_CDF_NEAR_TIE
            out.append(y)
            acc = len(path) - 1
            return acc, _pad(path, K + 1), _pad(out, K + 1), acc + 1, flags
        cur = accepted
        path.append(cur)
        out.append(int(tokens[cur]))
        p = softmax_t(target_logits[cur], T)
    y, near = inverse_cdf(p, float(u_res[K]), cdf_tie)
    if near:
        flags |= FLAG_CDF_NEAR_TIE
    out.append(y)
    acc = len(path) - 1
    return acc, _pad(path, K + 1), _pad(out, K + 1), acc + 1, flags


def verify_batch(mode: int, tree: dict, target_logits: np.ndarray, K: int,
                 head_logits: Optional[np.ndarray] = None, u_acc=None, u_res=None, T: float = 1.0,
                 rs_tie: float = RS_TIE, cdf_tie: float = CDF_TIE):
    """Run the walk for every sequence. mode 0 = greedy, 1 = rejection sampling."""
    B = target_logits.shape[0]
    acc = np.zeros(B, dtype=np.int64)
    path = np.full((B, K + 1), -1, dtype=np.int64)
    outt = np.full((B, K + 1), -1, dtype=np.int64)
    n_out = np.zeros(B, dtype=np.int64)
    flags = np.zeros(B, dtype=np.int64)
    for b in range(B):
        if mode == 0:
            a, pth, o, n = verify_greedy(tree["tokens"][b], tree["parent"], target_logits[b], K)
            f = 0
        else:
            a, pth, o, n, f = verify_rejection(tree["tokens"][b], tree["parent"], target_logits[b],
                                               head_logits[b], u_acc[b], u_res[b], K, T, rs_tie, cdf_tie)
        acc[b], path[b], outt[b], n_out[b], flags[b] = a, pth, o, n, f
    return {"acc": acc, "path": path, "out_tokens": outt, "n_out": n_out, "flags": flags}


# --------------------------------------------------------------------------- compaction
def kv_compact(Kc: np.ndarray, Vc: np.ndarray, L: np.ndarray, acc: np.ndarray, path: np.ndarray):
    """Keep the accepted path's tree rows, in path order, right after the committed prefix.

    [SPEC-DEC] §5 Case 2 (rejected drafts are rolled back) and §6 (the tree
    needs an extra KV buffer); [OPT-2] §1.3 (everything after the first
    mismatch is dropped). R11: for r = 0..acc_b, row L_b + r receives row
    L_b + path[b][r] in every KV head, then L_b grows by acc_b + 1. Sources are
    all read before any row is written. Returns new Kc, Vc, L and kv_map
    [B][K+1] (-1 padded).
    """
    Kc = Kc.copy()
    Vc = Vc.copy()
    B = Kc.shape[0]
    K1 = path.shape[1]
    L_new = L.astype(np.int64).copy()
    kv_map = np.full((B, K1), -1, dtype=np.int64)
    for b in range(B):
        Lb = int(L[b])
        n = int(acc[b]) + 1
        src = [Lb + int(path[b, r]) for r in range(n)]
        k_saved = Kc[b][:, src, :].copy()
        v_saved = Vc[b][:, src, :].copy()
        Kc[b][:, Lb:Lb + n, :] = k_saved
        Vc[b][:, Lb:Lb + n, :] = v_saved
        kv_map[b, :n] = path[b, :n]
        L_new[b] = Lb + n
    return Kc, Vc, L_new, kv_map


# --------------------------------------------------------------------------- paged cache (R15)
def paged_rows(pool: np.ndarray, block_table: np.ndarray, b: int, rows: int, page_rows: int) -> np.ndarray:
    """Logical rows [0, rows) of sequence b from a paged pool, [Hkv][rows][D].

    R15: a paged cache is a storage layout of the same logical cache: logical
    row i of sequence b lives in page block_table[b][i // P] at offset i % P,
    pool [num_pages][Hkv][P][D] (P = page_rows).
    """
    idx = np.arange(rows)
    pages = block_table[b, idx // page_rows]
    return pool[pages, :, idx % page_rows, :].transpose(1, 0, 2)


def tree_attention_paged(Q, Kp, Vp, block_table, page_rows, Kt, Vt, L, mask, Hq, Hkv, pairs=None):
    """Tree attention with the committed prefix in a paged pool and the tree's
    own keys/values in a staging buffer Kt, Vt [B][Hkv][N][D] (R15): the
    logical cache of each sequence is its paged prefix followed by its tree
    rows, and the result is tree_attention over that cache."""
    B, N = Q.shape[0], Q.shape[1]
    Hkv_, D = Kt.shape[1], Kt.shape[3]
    cap = int(np.max(L)) + N
    Kc = np.zeros((B, Hkv_, cap, D))
    Vc = np.zeros((B, Hkv_, cap, D))
    for b in range(B):
        Lb = int(L[b])
        Kc[b, :, :Lb] = paged_rows(Kp, block_table, b, Lb, page_rows)
        Vc[b, :, :Lb] = paged_rows(Vp, block_table, b, Lb, page_rows)
        Kc[b, :, Lb:Lb + N] = Kt[b]
        Vc[b, :, Lb:Lb + N] = Vt[b]
    return tree_attention(Q, Kc, Vc, L, mask, Hq, Hkv, pairs)


def kv_commit_paged(Kp_layers, Vp_layers, block_table, page_rows, Kt_layers, Vt_layers, L, acc, path):
    """Keep the accepted path in a paged cache, in every layer (R15, R11).

    For each layer and sequence b: logical row L_b + r (r = 0..acc_b) receives
    the tree row path[b][r] of that layer's staging buffer; then L_b grows by
    acc_b + 1. This is R11's compaction of the logical cache whose rows
    L_b .. L_b + N - 1 hold the tree. Returns new pools (one per layer), L and
    kv_map.
    """
    Kp_layers = [k.copy() for k in Kp_layers]
    Vp_layers = [v.copy() for v in Vp_layers]
    B, K1 = path.shape
    L_new = L.astype(np.int64).copy()
    kv_map = np.full((B, K1), -1, dtype=np.int64)
    for b in range(B):
        Lb, n = int(L[b]), int(acc[b]) + 1
        for r in range(n):
            row = Lb + r
            page, off = int(block_table[b, row // page_rows]), row % page_rows
            for Kp, Vp, Kt, Vt in zip(Kp_layers, Vp_layers, Kt_layers, Vt_layers):
                Kp[page, :, off, :] = Kt[b, :, int(path[b, r]), :]
                Vp[page, :, off, :] = Vt[b, :, int(path[b, r]), :]
        kv_map[b, :n] = path[b, :n]
        L_new[b] = Lb + n
    return Kp_layers, Vp_layers, L_new, kv_map


# --------------------------------------------------------------------------- helpers
def _pad(xs: Sequence[int], n: int) -> np.ndarray:
    out = np.full(n, -1, dtype=np.int64)
    out[:len(xs)] = xs
    return out


def expected_tokens_per_step(alpha: float, K: int) -> float:
    """E[N] = 1 + sum_{i=1..K} alpha^i = (1 - alpha^(K+1)) / (1 - alpha).

    [SPEC-DEC] §2.3, expected-tokens equation (i.i.d. acceptance alpha).
    """
    return sum(alpha ** i for i in range(K + 1))


def node_count(branching: Sequence[int]) -> int:
    return tree_layout(branching)["N"]
