"""Thin Python binding of libmedusa (ctypes): argument marshalling only.

Every function takes the same arguments as the C entry point of the same name
in include/medusa.h. Tensors are passed as raw device pointers (``data_ptr``);
``None`` becomes a null pointer. A non-zero status raises ``MedusaError``. No
computation happens here and there is no fallback: if the library cannot be
loaded, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmedusa.so")
# the same kernels built with device-side range checks (MEDUSA_CHECKED=1 in the environment selects it)
LIB_CHECKED_PATH = os.path.join(PKG, "libmedusa_checked.so")

F32, BF16 = 0, 1
GREEDY, REJECTION = 0, 1
FLAG_RS_NEAR_TIE, FLAG_CDF_NEAR_TIE, FLAG_CAPACITY = 1, 2, 4

ENTRY_POINTS = ("medusa_node_count", "medusa_workspace_size", "medusa_heads", "medusa_tree_build",
                "medusa_tree_attention", "medusa_verify", "medusa_kv_compact", "medusa_tree_attention_noalloc",
                "medusa_tree_attention_paged", "medusa_kv_commit_paged", "medusa_step_graph_create",
                "medusa_step_graph_launch", "medusa_step_graph_destroy", "medusa_poll_errors",
                "medusa_selftest_wait_timeout", "medusa_checked_build", "medusa_poll_checks", "medusa_step_fused",
                "medusa_launch_count", "medusa_status_string")
CHECK_TOKEN, CHECK_TREE, CHECK_PATH, CHECK_PAGE = 1, 2, 4, 8


class MedusaError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: {status} ({text})")
        self.status = status


class Cfg(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("d", ctypes.c_int32), ("V", ctypes.c_int32), ("K", ctypes.c_int32),
                ("branching", ctypes.c_int32 * 8), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("D", ctypes.c_int32), ("L_cap", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("temperature", ctypes.c_float), ("shared_vocab", ctypes.c_int32),
                ("tree_nodes", ctypes.c_int32), ("tree_parent", ctypes.c_int16 * 128), ("tree_rank", ctypes.c_uint8 * 128)]


def make_cfg(B: int, d: int, V: int, branching: Sequence[int], Hq: int, Hkv: int, D: int, L_cap: int,
             dtype: int, mode: int, temperature: float = 1.0, shared_vocab: bool = False,
             tree_nodes: Optional[Tuple[Sequence[int], Sequence[int]]] = None) -> Cfg:
    """tree_nodes: (parent, rank) of a pruned tree's nodes in breadth-first rank-path order, or None
    for the full Cartesian tree of ``branching``."""
    c = Cfg()
    c.B, c.d, c.V, c.K = B, d, V, len(branching)
    for i, s in enumerate(branching):
        c.branching[i] = int(s)
    c.Hq, c.Hkv, c.D, c.L_cap = Hq, Hkv, D, L_cap
    c.dtype, c.mode, c.temperature = dtype, mode, float(temperature)
    c.shared_vocab = 1 if shared_vocab else 0
    if tree_nodes is not None:
        parent, rank = tree_nodes
        c.tree_nodes = len(parent)
        for n, (p, r) in enumerate(zip(parent, rank)):
            c.tree_parent[n], c.tree_rank[n] = int(p), int(r)
    return c


class StepArgs(ctypes.Structure):
    """medusa_step_args: every buffer of the five calls, in the header's order."""
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "h", "W", "bias", "U", "logits", "topk", "root_token", "L", "parent", "depth", "first_child", "mask",
        "anc_bits", "tokens", "pos", "flags", "Q", "Kc", "Vc", "O", "target_logits", "u_acc", "u_res", "acc", "path",
        "out_tokens", "n_out", "kv_map", "workspace")] + [("kv_compact", ctypes.c_int32)]


_lib: Optional[ctypes.CDLL] = None
P = ctypes.c_void_p


def default_path() -> str:
    return LIB_CHECKED_PATH if os.environ.get("MEDUSA_CHECKED") == "1" else LIB_PATH


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libmedusa.so, or libmedusa_checked.so when MEDUSA_CHECKED=1 is set (build them
    first with ``_build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or default_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libmedusa not built: {path} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    cp = ctypes.POINTER(Cfg)
    sig = {
        "medusa_node_count": [cp, ctypes.POINTER(ctypes.c_int32)],
        "medusa_workspace_size": [cp, ctypes.POINTER(ctypes.c_size_t)],
        "medusa_heads": [cp, P, P, P, P, P, P, P, P],
        "medusa_tree_build": [cp, P, P, P, P, P, P, P, P, P, P, P, P],
        "medusa_tree_attention": [cp, P, P, P, P, P, P, P, P],
        "medusa_tree_attention_noalloc": [cp, P, P, P, P, P, P, P],
        "medusa_tree_attention_paged": [cp, P, P, P, ctypes.c_int32, ctypes.c_int32, P, P, P, P, P, P, P, P],
        "medusa_kv_commit_paged": [cp, P, P, ctypes.c_int32, P, P, P, ctypes.c_int32, ctypes.c_size_t,
                                   ctypes.c_size_t, P, P, P, P, P],
        "medusa_verify": [cp, P, P, P, P, P, P, P, P, P, P, P, P, P, P],
        "medusa_kv_compact": [cp, P, P, P, P, P, P, P],
        "medusa_poll_errors": [P, ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32)],
        "medusa_step_graph_create": [cp, ctypes.POINTER(StepArgs), ctypes.POINTER(ctypes.c_void_p)],
        "medusa_step_graph_launch": [P, P],
        "medusa_step_graph_destroy": [P],
        "medusa_selftest_wait_timeout": [ctypes.c_uint32, P],
        "medusa_checked_build": [],
        "medusa_step_fused": [cp, ctypes.POINTER(StepArgs), P],
        "medusa_poll_checks": [P, ctypes.POINTER(ctypes.c_uint32)],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.medusa_launch_count.argtypes = []
    lib.medusa_launch_count.restype = ctypes.c_uint64
    lib.medusa_status_string.argtypes = [ctypes.c_int]
    lib.medusa_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name: str, status: int) -> None:
    if status != 0:
        raise MedusaError(name, status, load().medusa_status_string(status).decode())


def status_string(status: int) -> str:
    return load().medusa_status_string(status).decode()


class StepGraph:
    """The whole step captured once as a CUDA graph over fixed buffers, replayed with one launch."""

    def __init__(self, cfg: "Cfg", **buffers):
        args = StepArgs(**{k: _ptr(v) for k, v in buffers.items() if k != "kv_compact"},
                        kv_compact=int(bool(buffers.get("kv_compact", 1))))
        self._cfg, self._args = cfg, args   # kept alive with the graph
        h = ctypes.c_void_p()
        _check("medusa_step_graph_create", load().medusa_step_graph_create(ctypes.byref(cfg), ctypes.byref(args),
                                                                            ctypes.byref(h)))
        self._h = h

    def launch(self, stream=None) -> None:
        _check("medusa_step_graph_launch", load().medusa_step_graph_launch(self._h, _stream(stream)))

    def close(self) -> None:
        if self._h is not None and self._h.value:
            _check("medusa_step_graph_destroy", load().medusa_step_graph_destroy(self._h))
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def step_args(**buffers) -> "StepArgs":
    """A medusa_step_args from tensors (None: NULL); kv_compact defaults to 1."""
    return StepArgs(**{k: _ptr(v) for k, v in buffers.items() if k != "kv_compact"},
                    kv_compact=int(bool(buffers.get("kv_compact", 1))))


def step_fused(cfg: "Cfg", args: "StepArgs", stream=None) -> None:
    """medusa_step_fused: the whole step as one persistent kernel launch."""
    _check("medusa_step_fused", load().medusa_step_fused(ctypes.byref(cfg), ctypes.byref(args), _stream(stream)))


WAIT_SELFTEST_CODE = 0x80000000
FUSED_WAIT_CODE = 0x40000000
STATUS_TIMEOUT = -5


def poll_errors(stream=None):
    """Read and clear the device words that record expired bounded waits (synchronises the stream).

    Returns (status, heads_codes, attention_codes); status is 0 or -5 (a wait expired)."""
    h, a = ctypes.c_uint32(), ctypes.c_uint32()
    s = load().medusa_poll_errors(_stream(stream), ctypes.byref(h), ctypes.byref(a))
    if s not in (0, STATUS_TIMEOUT):
        _check("medusa_poll_errors", s)
    return s, int(h.value), int(a.value)


STATUS_BOUNDS = -6


def checked_build() -> bool:
    """True when the loaded library is the range-checked build."""
    return bool(load().medusa_checked_build())


def poll_checks(stream=None):
    """Read and clear the checked build's range-check words (synchronises the stream).

    Returns (status, codes); status is 0 or -6 (an out-of-range index was met), codes the
    OR of the CHECK_* bits (always (0, 0) in the normal build)."""
    c = ctypes.c_uint32()
    s = load().medusa_poll_checks(_stream(stream), ctypes.byref(c))
    if s not in (0, STATUS_BOUNDS):
        _check("medusa_poll_checks", s)
    return s, int(c.value)


def selftest_wait_timeout(budget_us: int, stream=None) -> None:
    """Enqueue one bounded wait that nothing completes; the next poll_errors reports it."""
    _check("medusa_selftest_wait_timeout", load().medusa_selftest_wait_timeout(int(budget_us), _stream(stream)))


def launch_count() -> int:
    """Kernels libmedusa has enqueued in this process so far."""
    return int(load().medusa_launch_count())


def node_count(cfg: Cfg) -> int:
    n = ctypes.c_int32()
    _check("medusa_node_count", load().medusa_node_count(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def workspace_size(cfg: Cfg) -> int:
    n = ctypes.c_size_t()
    _check("medusa_workspace_size", load().medusa_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def heads(cfg, h, W, bias, U, logits, topk, workspace, stream=None):
    _check("medusa_heads", load().medusa_heads(ctypes.byref(cfg), _ptr(h), _ptr(W), _ptr(bias), _ptr(U),
                                                 _ptr(logits), _ptr(topk), _ptr(workspace), _stream(stream)))


def tree_build(cfg, root_token, topk, L, parent, depth, first_child, mask, anc_bits, tokens, pos, flags,
               stream=None):
    _check("medusa_tree_build", load().medusa_tree_build(
        ctypes.byref(cfg), _ptr(root_token), _ptr(topk), _ptr(L), _ptr(parent), _ptr(depth), _ptr(first_child),
        _ptr(mask), _ptr(anc_bits), _ptr(tokens), _ptr(pos), _ptr(flags), _stream(stream)))


def tree_attention(cfg, Q, Kc, Vc, L, anc_bits, O, workspace, stream=None):
    _check("medusa_tree_attention", load().medusa_tree_attention(
        ctypes.byref(cfg), _ptr(Q), _ptr(Kc), _ptr(Vc), _ptr(L), _ptr(anc_bits), _ptr(O), _ptr(workspace),
        _stream(stream)))


def tree_attention_paged(cfg, Q, Kp, Vp, num_pages, page_rows, block_table, Kt, Vt, L, anc_bits, O, workspace,
                         stream=None):
    """medusa_tree_attention over a paged pool, the tree's rows staged in Kt/Vt."""
    _check("medusa_tree_attention_paged", load().medusa_tree_attention_paged(
        ctypes.byref(cfg), _ptr(Q), _ptr(Kp), _ptr(Vp), int(num_pages), int(page_rows), _ptr(block_table), _ptr(Kt),
        _ptr(Vt), _ptr(L), _ptr(anc_bits), _ptr(O), _ptr(workspace), _stream(stream)))


def kv_commit_paged(cfg, Kp, Vp, page_rows, block_table, Kt, Vt, n_layers, pool_layer_elems, tree_layer_elems, L, acc,
                    path, kv_map, stream=None):
    """Write the accepted path's staged rows into the paged pools of n_layers layers."""
    _check("medusa_kv_commit_paged", load().medusa_kv_commit_paged(
        ctypes.byref(cfg), _ptr(Kp), _ptr(Vp), int(page_rows), _ptr(block_table), _ptr(Kt), _ptr(Vt), int(n_layers),
        int(pool_layer_elems), int(tree_layer_elems), _ptr(L), _ptr(acc), _ptr(path), _ptr(kv_map), _stream(stream)))


def tree_attention_noalloc(cfg, Q, Kc, Vc, L, anc_bits, O, stream=None):
    """medusa_tree_attention with the library's static scratch instead of a workspace."""
    _check("medusa_tree_attention_noalloc", load().medusa_tree_attention_noalloc(
        ctypes.byref(cfg), _ptr(Q), _ptr(Kc), _ptr(Vc), _ptr(L), _ptr(anc_bits), _ptr(O), _stream(stream)))


def verify(cfg, tokens, parent, first_child, target_logits, head_logits, u_acc, u_res, acc, path, out_tokens,
           n_out, flags, workspace, stream=None):
    _check("medusa_verify", load().medusa_verify(
        ctypes.byref(cfg), _ptr(tokens), _ptr(parent), _ptr(first_child), _ptr(target_logits), _ptr(head_logits),
        _ptr(u_acc), _ptr(u_res), _ptr(acc), _ptr(path), _ptr(out_tokens), _ptr(n_out), _ptr(flags),
        _ptr(workspace), _stream(stream)))


def kv_compact(cfg, Kc, Vc, L, acc, path, kv_map, stream=None):
    _check("medusa_kv_compact", load().medusa_kv_compact(
        ctypes.byref(cfg), _ptr(Kc), _ptr(Vc), _ptr(L), _ptr(acc), _ptr(path), _ptr(kv_map), _stream(stream)))


def raw_call(name: str, *args) -> int:
    """Call an entry point with already-marshalled arguments; returns the status."""
    return getattr(load(), name)(*args)
