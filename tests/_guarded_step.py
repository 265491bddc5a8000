"""Run small steps through the library with guard bytes around every buffer it writes.

Run as a script by tests/test_checked_build.py, once with the normal library and
once with the range-checked one (MEDUSA_CHECKED=1 selects libmedusa_checked.so).

1. Clean steps (float32 and bf16 workloads, greedy and rejection sampling): every
   output, the workspace, the attention output and the KV cache sit inside a
   larger buffer whose guard bytes must be untouched afterwards; the outputs
   must match the float64 oracle; neither the range checks nor the bounded
   waits may report anything.
2. Corrupted inputs that every build clamps or skips (a token id outside the
   vocabulary in a rejection-sampling walk, a path with a node id past the tree
   and an acc past K, a block-table page id past the pool): guards stay intact,
   the rows the corrupt entries would have addressed are untouched, and the
   checked build reports the matching MEDUSA_CHECK_* bit (the normal build
   reports nothing). A clean step afterwards must still match the oracle.
Prints one JSON line and exits non-zero on the first failed check.
"""
from __future__ import annotations

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from medusa_speculative_decoding_heads_gb300 import binding as mb, configs, synth  # noqa: E402
from medusa_speculative_decoding_heads_gb300.configs import GREEDY, REJECTION  # noqa: E402
from medusa_speculative_decoding_heads_gb300.step import DeviceStep, to_device_inputs  # noqa: E402
from oracle import medusa_oracle as O  # noqa: E402

from _helpers import assert_close, compare_verify, f64, gpu_ready, i64, planted_greedy_logits  # noqa: E402

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """A tensor view inside a byte buffer with GUARD pattern bytes on both sides."""

    def __init__(self, shape, dtype, dev, fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.n = n
        self.buf = torch.full((GUARD + (n + 255) // 256 * 256 + GUARD,), PATTERN, dtype=torch.uint8, device=dev)
        self.t = self.buf[GUARD:GUARD + n].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def intact(self) -> bool:
        b = self.buf.cpu().numpy()
        return bool((b[:GUARD] == PATTERN).all() and (b[GUARD + self.n:] == PATTERN).all())


def guard_step(st: DeviceStep, inp, w):
    """Replace the step's outputs, workspace and the cache by guarded copies; returns the guards."""
    dev = st.dev
    g = {}
    for name in ("logits", "topk", "parent", "depth", "first_child", "mask", "anc_bits", "tokens", "pos", "flags",
                 "acc", "path", "out_tokens", "n_out", "kv_map", "workspace"):
        t = getattr(st, name)
        g[name] = Guarded(t.shape, t.dtype, dev, fill=t)
        setattr(st, name, g[name].t)
    g["O"] = Guarded(inp.Q.shape, inp.Q.dtype, dev)
    st.O = g["O"].t
    for name in ("Kc", "Vc"):
        t = getattr(inp, name)
        g[name] = Guarded(t.shape, t.dtype, dev, fill=t)
        setattr(inp, name, g[name].t)
    return g


def expect(cond, what):
    if not cond:
        print(json.dumps({"ok": False, "failed": what}), flush=True)
        sys.exit(1)


def polls_clean(what):
    s, codes = mb.poll_checks()
    expect(s == 0 and codes == 0, f"{what}: range checks reported {codes:#x}")
    s, h, a = mb.poll_errors()
    expect(s == 0, f"{what}: bounded waits reported heads {h:#x} attention {a:#x}")


def clean_step(w, mode, dev, seed):
    si = synth.make_step_inputs(w, seed=seed, device=dev, with_bias=True)
    _, z = O.medusa_heads(f64(si.h), f64(si.W), f64(si.bias), f64(si.U))
    topk_ref, near = O.heads_top_s(z, w.branching)
    tree = O.tree_build(w.branching, si.root_token, topk_ref, si.L, si.L_cap)
    if mode == REJECTION:
        tl = synth.target_logits(configs.scaled(w, target_corr=0.8), seed, device=dev,
                                 zhat=torch.from_numpy(z).float(), depth=tree["depth"])
    else:
        tl = synth.target_logits(configs.scaled(w, target_corr=0.0), seed, device=dev)
        planted_greedy_logits(tl, tree, seed, w.K)
    inp = to_device_inputs(si, tl, dev)
    Kc0, Vc0 = f64(si.Kc), f64(si.Vc)
    st = DeviceStep(w, mode, si.L_cap, dev)
    g = guard_step(st, inp, w)
    st.run(inp, write_logits=True, compact=True)
    torch.cuda.synchronize()
    for name, gb in g.items():
        expect(gb.intact(), f"{w.name} mode={mode}: guard bytes around {name} overwritten")
    assert_close(st.logits.cpu().numpy(), z, w.dtype, "logits")
    ok_b = ~near.any(axis=1)
    expect(np.array_equal(i64(st.topk)[ok_b], topk_ref[ok_b]), f"{w.name}: top-s")
    Oref = O.tree_attention(f64(si.Q), Kc0, Vc0, si.L, tree["mask"], w.Hq, w.Hkv)
    assert_close(f64(st.O), Oref, w.dtype, "attention")
    ver, _ = compare_verify(st, mode, tree, f64(tl), w.K, head_logits=f64(st.logits), u_acc=si.u_acc,
                            u_res=si.u_res, T=w.temperature, eligible=ok_b, min_compared=1, what=w.name)
    ok = ok_b & (ver["flags"] == 0) & ((i64(st.flags) & 3) == 0)
    kr, vr, Lr, kv_map = O.kv_compact(Kc0, Vc0, si.L, ver["acc"], ver["path"])
    expect(np.array_equal(f64(inp.Kc)[ok], kr[ok]) and np.array_equal(f64(inp.Vc)[ok], vr[ok]), "compaction")
    expect(np.array_equal(i64(st.kv_map)[ok], kv_map[ok]), "kv_map")
    polls_clean(f"{w.name} mode={mode}")


def corrupt_token(w, dev, checked):
    """Top-s lists holding token ids V + 5 and -7: the tree copies them, the rejection walk clamps
    the index it reads the candidates' probabilities at."""
    w = configs.scaled(w, modes=(REJECTION,), temperature=0.8)
    si = synth.make_step_inputs(w, seed=3, device=dev)
    rng = np.random.default_rng(3)
    topk = np.full((w.B, w.K, w.s_max), -1, dtype=np.int32)
    for b in range(w.B):
        for k in range(w.K):
            topk[b, k, :w.branching[k]] = rng.choice(w.V, size=w.branching[k], replace=False)
    topk[0, 0, 0] = w.V + 5
    topk[1, 0, 1] = -7
    st = DeviceStep(w, REJECTION, si.L_cap, dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(3)
    z = torch.randn((w.B, w.K, w.V), generator=gen, device=dev)
    tl = synth.target_logits(configs.scaled(w, target_corr=0.0), 3, device=dev)
    g = guard_step(st, to_device_inputs(si, tl, dev), w)
    st.tree_build(torch.from_numpy(si.root_token).to(dev), torch.from_numpy(si.L).to(dev),
                  topk=torch.from_numpy(topk).to(dev))
    st.verify(tl, torch.from_numpy(si.u_acc).to(dev), torch.from_numpy(si.u_res).to(dev), head_logits=z)
    torch.cuda.synchronize()
    for name, gb in g.items():
        expect(gb.intact(), f"corrupt token: guard bytes around {name} overwritten")
    n = i64(st.n_out)
    expect(((n >= 1) & (n <= w.K + 1)).all(), "corrupt token: n_out out of range")
    s, codes = mb.poll_checks()
    expect((codes & mb.CHECK_TOKEN) != 0 if checked else (s == 0 and codes == 0),
           f"corrupt token: checks reported {codes:#x}")
    return codes


def corrupt_path(w, dev, checked):
    """A path slot naming node N + 5 and an acc of K + 2: compaction clamps the first and skips the second."""
    si = synth.make_step_inputs(w, seed=4, device=dev)
    st = DeviceStep(w, w.modes[0], si.L_cap, dev)
    inp = to_device_inputs(si, synth.target_logits(configs.scaled(w, target_corr=0.0), 4, device=dev), dev)
    g = guard_step(st, inp, w)
    lay = O.tree_layout(w.branching)
    acc = np.zeros(w.B, dtype=np.int32)
    path = np.full((w.B, w.K + 1), -1, dtype=np.int32)
    path[:, 0] = 0
    acc[0], path[0, 1] = 1, w.N + 5          # a node past the tree
    acc[1] = w.K + 2                          # more accepted drafts than heads
    acc[2], path[2, 1] = 1, O.children_of(lay["parent"], 0)[0]   # a valid path
    st.acc.copy_(torch.from_numpy(acc))
    st.path.copy_(torch.from_numpy(path))
    k_before = inp.Kc.clone()
    L = inp.L.clone()
    st.kv_compact(inp.Kc, inp.Vc, inp.L)
    torch.cuda.synchronize()
    for name, gb in g.items():
        expect(gb.intact(), f"corrupt path: guard bytes around {name} overwritten")
    Lh = i64(L)
    changed = (inp.Kc != k_before).any(dim=-1).cpu().numpy()   # [B][Hkv][L_cap]
    for b in range(w.B):
        rows = np.nonzero(changed[b].any(axis=0))[0]
        expect(all(Lh[b] <= r < Lh[b] + w.N for r in rows), f"corrupt path: b={b} wrote outside its tree rows")
    expect(not changed[1].any(), "corrupt path: a sequence with acc > K was not skipped")
    expect(int(inp.L[1]) == Lh[1] and int(inp.L[2]) == Lh[2] + 2, "corrupt path: lengths")
    s, codes = mb.poll_checks()
    expect((codes & mb.CHECK_PATH) != 0 if checked else (s == 0 and codes == 0),
           f"corrupt path: checks reported {codes:#x}")
    return codes


def corrupt_page(dev, checked):
    """A block table naming a page past the pool: the paged commit leaves that row unwritten."""
    w = configs.scaled(configs.get("vicuna13b_b8"), B=3, d=256, V=1000, Hq=2, Hkv=2, L_range=(100, 300))
    P = 128
    si = synth.make_step_inputs(w, seed=5, device=dev)
    cap = -(-si.L_cap // P) * P
    max_pages = cap // P
    num_pages = w.B * max_pages
    bt = np.arange(num_pages, dtype=np.int32).reshape(w.B, max_pages)
    L = np.array([150, 200, 250], dtype=np.int32)
    bad_page = num_pages + 3
    bt[1, L[1] // P] = bad_page              # sequence 1's tree rows land on a page past the pool
    Kp = Guarded((num_pages, w.Hkv, P, w.D), torch.bfloat16, dev, fill=torch.zeros((num_pages, w.Hkv, P, w.D)))
    Vp = Guarded((num_pages, w.Hkv, P, w.D), torch.bfloat16, dev, fill=torch.zeros((num_pages, w.Hkv, P, w.D)))
    Kt = torch.randn((w.B, w.Hkv, w.N, w.D), device=dev).to(torch.bfloat16)
    Vt = torch.randn((w.B, w.Hkv, w.N, w.D), device=dev).to(torch.bfloat16)
    st = DeviceStep(w, w.modes[0], cap, dev)
    acc = torch.tensor([1, 1, 1], dtype=torch.int32, device=dev)
    kid = O.children_of(O.tree_layout(w.branching)["parent"], 0)[0]
    path = torch.tensor([[0, kid] + [-1] * (w.K - 1)] * 3, dtype=torch.int32, device=dev)
    Ld = torch.from_numpy(L).to(dev)
    mb.kv_commit_paged(st.cfg, Kp.t, Vp.t, P, torch.from_numpy(bt).to(dev), Kt, Vt, 1, Kp.t.numel(), Kt.numel(),
                       Ld, acc, path, st.kv_map)
    torch.cuda.synchronize()
    expect(Kp.intact() and Vp.intact(), "corrupt page: guard bytes around the pool overwritten")
    written = (Kp.t.float() != 0).any(dim=-1).cpu().numpy()    # [pages][Hkv][P]
    for b in (0, 2):
        page, off = bt[b, L[b] // P], L[b] % P
        expect(written[page, :, off].all() and written[page, :, off + 1].all(), f"corrupt page: b={b} not committed")
    expect(int(written.sum()) == 2 * 2 * w.Hkv, "corrupt page: rows written beyond the two valid sequences")
    s, codes = mb.poll_checks()
    expect((codes & mb.CHECK_PAGE) != 0 if checked else (s == 0 and codes == 0),
           f"corrupt page: checks reported {codes:#x}")
    return codes


def main():
    dev = gpu_ready()
    checked = mb.checked_build()
    expect(checked == (os.environ.get("MEDUSA_CHECKED") == "1"), "wrong library loaded")
    tiny = configs.scaled(configs.get("tiny_fp32"), B=4, modes=(GREEDY, REJECTION))
    bf16 = configs.scaled(configs.get("gqa7b_b32"), B=4, d=512, V=1000, Hq=8, Hkv=2, L_range=(40, 300),
                          modes=(GREEDY, REJECTION), temperature=0.8)
    for w in (tiny, bf16):
        for mode in w.modes:
            clean_step(w, mode, dev, seed=17)
    codes = {"token": corrupt_token(bf16, dev, checked), "path": corrupt_path(bf16, dev, checked),
             "page": corrupt_page(dev, checked)}
    clean_step(bf16, REJECTION, dev, seed=18)   # the context is still usable and still right
    print(json.dumps({"ok": True, "checked": checked, "codes": codes}), flush=True)


if __name__ == "__main__":
    main()
