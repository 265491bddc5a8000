"""The C ABI library loads on the host and exports what include/medusa.h declares (no GPU needed)."""
import ctypes
import os
import re

import pytest

from medusa_speculative_decoding_heads_gb300 import _build, binding as mb, configs
from medusa_speculative_decoding_heads_gb300.step import cfg_for

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return mb.load()


def declared_entry_points():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^MEDUSA_API\s+(?:int|uint64_t|const char\*)\s+(medusa_\w+)\s*\(", text, flags=re.M))
    return names


def test_header_declares_the_five_steps():
    names = declared_entry_points()
    for n in ("medusa_heads", "medusa_tree_build", "medusa_tree_attention", "medusa_verify", "medusa_kv_compact"):
        assert n in names


@pytest.mark.parametrize("lang,std", [("c", "-std=c11"), ("c++", "-std=c++17")])
def test_header_is_plain_c_and_cpp(lang, std):
    """include/medusa.h compiles on its own as C11 (pedantic) and as C++17: a C caller needs nothing else."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = '#include "medusa.h"\nint main(void) { medusa_cfg c; medusa_step_args a; (void)c; (void)a; return 0; }\n'
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    r = subprocess.run([cc, "-x", lang, std, "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only", "-I", inc, "-"],
                       input=src, text=True, capture_output=True)
    assert r.returncode == 0, r.stderr


def test_every_declared_symbol_is_exported(lib):
    for name in declared_entry_points():
        assert hasattr(lib, name), name


def test_binding_lists_every_declared_entry_point():
    assert set(mb.ENTRY_POINTS) == declared_entry_points()


def test_status_strings(lib):
    assert mb.status_string(0) == "ok"
    assert mb.status_string(-1) == "invalid argument"
    assert mb.status_string(-2) == "unsupported configuration"


def test_node_count_and_workspace(lib):
    for name in configs.ORDER:
        w = configs.get(name)
        cfg = cfg_for(w, L_cap=w.L_range[1] + w.N, mode=w.modes[0])
        assert mb.node_count(cfg) == w.N
        assert mb.workspace_size(cfg) > 0


def _cfg(**kw):
    w = configs.get("tiny_fp32")
    cfg = cfg_for(w, L_cap=256, mode=configs.GREEDY)
    for k, v in kw.items():
        setattr(cfg, k, v)
    return cfg


@pytest.mark.parametrize("field,value,status", [
    ("K", 0, -1), ("K", 9, -2), ("D", 96, -2), ("Hkv", 3, -2), ("dtype", 5, -1), ("mode", 7, -1),
    ("L_cap", 10, -3), ("B", 0, -1),
])
def test_bad_configs_are_rejected_before_any_launch(lib, field, value, status):
    cfg = _cfg(**{field: value})
    n = ctypes.c_size_t()
    assert lib.medusa_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == status


def test_too_many_nodes_and_wide_branching(lib):
    cfg = _cfg(K=4)
    for i, s in enumerate((8, 8, 1, 1)):
        cfg.branching[i] = s
    assert mb.raw_call("medusa_workspace_size", ctypes.byref(cfg), ctypes.byref(ctypes.c_size_t())) == -2
    cfg = _cfg()
    cfg.branching[0] = 9
    assert mb.raw_call("medusa_workspace_size", ctypes.byref(cfg), ctypes.byref(ctypes.c_size_t())) == -2


def test_null_pointers_are_rejected(lib):
    cfg = _cfg()
    assert lib.medusa_heads(ctypes.byref(cfg), None, None, None, None, None, None, None, None) == -1
    assert lib.medusa_tree_build(ctypes.byref(cfg), *([None] * 12)) == -1
    assert lib.medusa_tree_attention(ctypes.byref(cfg), *([None] * 8)) == -1
    assert lib.medusa_verify(ctypes.byref(cfg), *([None] * 14)) == -1
    assert lib.medusa_kv_compact(ctypes.byref(cfg), *([None] * 7)) == -1
    rs = _cfg(mode=configs.REJECTION, temperature=0.0)
    assert lib.medusa_workspace_size(ctypes.byref(rs), ctypes.byref(ctypes.c_size_t())) == -1


def test_rejection_mode_needs_logits_and_uniforms(lib):
    cfg = _cfg(mode=configs.REJECTION)
    fake = ctypes.c_void_p(256)   # never dereferenced: validation fails first
    assert lib.medusa_heads(ctypes.byref(cfg), fake, fake, None, fake, None, fake, fake, None) == -1
    assert lib.medusa_verify(ctypes.byref(cfg), fake, fake, fake, fake, None, None, None, fake, fake, fake, fake,
                             fake, fake, None) == -1


def test_pruned_and_shared_configs(lib):
    """The extra workloads (one shared vocab projection, pruned 64-node trees) pass
    the checks and report their own node counts."""
    for name in configs.SHARED + configs.PRUNED:
        w = configs.get(name)
        cfg = cfg_for(w, L_cap=w.L_range[1] + w.N, mode=w.modes[0])
        assert mb.node_count(cfg) == w.N
        assert mb.workspace_size(cfg) > 0
    assert configs.get("vicuna7b_b1_pruned64").N == 64


@pytest.mark.parametrize("edit", ["root_parent", "forward_parent", "rank_too_big", "too_deep", "sibling_order",
                                  "depth_order"])
def test_malformed_pruned_trees_are_rejected(lib, edit):
    w = configs.get("vicuna7b_b1_pruned64")
    parent, rank = (list(x) for x in w.tree_nodes)
    if edit == "root_parent":
        parent[0] = 0
    elif edit == "forward_parent":
        parent[5] = 7
    elif edit == "rank_too_big":
        rank[1] = w.branching[0]
    elif edit == "too_deep":
        w = configs.scaled(w, branching=w.branching[:4])   # the tree has depth-5 nodes
    elif edit == "sibling_order":
        rank[1], rank[2] = rank[2], rank[1]
    elif edit == "depth_order":
        parent[6] = 5          # node 6 drops to depth 3 while node 7 stays at depth 2: not breadth first
    cfg = mb.make_cfg(B=w.B, d=w.d, V=w.V, branching=w.branching, Hq=w.Hq, Hkv=w.Hkv, D=w.D, L_cap=4096,
                      dtype=w.dtype, mode=configs.GREEDY, tree_nodes=(parent, rank))
    assert mb.raw_call("medusa_workspace_size", ctypes.byref(cfg), ctypes.byref(ctypes.c_size_t())) == -1


def test_missing_library_fails_loudly(tmp_path):
    """Without the built library the binding raises instead of falling back to anything."""
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, %r)\n"
            "from medusa_speculative_decoding_heads_gb300 import binding\n"
            "try:\n    binding.load(%r)\nexcept RuntimeError as e:\n    print('raised:', e)\n    sys.exit(3)\n"
            % (ROOT, str(tmp_path / "libmedusa.so")))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 3 and "not built" in r.stdout, (r.stdout, r.stderr)


def test_step_fused_argument_checks():
    """medusa_step_fused returns INVALID_ARG for missing arguments and UNSUPPORTED outside its
    scope (float32, rejection sampling, B > 4) before any CUDA call."""
    import ctypes
    lib = mb.load()
    c = mb.make_cfg(B=1, d=256, V=500, branching=(2, 2), Hq=2, Hkv=2, D=128, L_cap=256, dtype=mb.BF16,
                    mode=mb.GREEDY)
    assert lib.medusa_step_fused(ctypes.byref(c), None, None) == -1
    args = mb.StepArgs()
    for kw in (dict(dtype=mb.F32), dict(mode=mb.REJECTION), dict(B=5)):
        cc = mb.make_cfg(**dict(dict(B=1, d=256, V=500, branching=(2, 2), Hq=2, Hkv=2, D=128, L_cap=256,
                                     dtype=mb.BF16, mode=mb.GREEDY), **kw))
        assert lib.medusa_step_fused(ctypes.byref(cc), ctypes.byref(args), None) == -2
    assert lib.medusa_step_fused(ctypes.byref(c), ctypes.byref(args), None) == -1   # null buffers
