#!/usr/bin/env python
"""Medusa verify-step throughput on GB300 (steps/s), with the HBM roofline.

One step = the whole hot path on one batch of synthetic input, as five
library calls on one stream: Medusa heads (residual block, vocab projection,
top-s) -> candidate tree -> tree attention -> acceptance -> KV compaction.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

N > 1 runs one independent replica per GPU under torch.distributed.run (this
script starts the launcher itself when it is run plainly, and refuses a
launcher whose WORLD_SIZE differs from N); the step has no exchange, so there
is no collective on the data path and the scaling is weak. The default
workload is the largest one that fits one GPU (vicuna33b_b16). `--impl
reference` times the CPU oracle (plain float64 numpy, single-threaded BLAS) on
the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# The CPU oracle is timed single-threaded: its numpy matmuls would otherwise use every host
# core through the BLAS thread pool. Set before numpy loads its BLAS; a value already in the
# environment wins, and the line reports the thread count the pool actually has.
for _var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_var, "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

from medusa_speculative_decoding_heads_gb300 import configs, synth  # noqa: E402
from medusa_speculative_decoding_heads_gb300.configs import F32, GREEDY, REJECTION  # noqa: E402

METRIC = "Medusa verify steps/s (heads+tree-attn+accept); HBM GB/s vs 8 TB/s"
UNIT = "steps/s"
# the largest workload that fits one GPU: 33B-shaped heads over a batch of 16, 5.6 GB per step
DEFAULT_WORKLOAD = "vicuna33b_b16"
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + write) of one call of the step's dominant call, from full-size ncu captures
# of its kernels (one pass each; summarised in profiles/). Absent = not captured: traffic null.
NCU_TRAFFIC_BYTES = {"vicuna7b_b1": 1189250048, "vicuna7b_b1_shared": 402850048, "vicuna13b_b8": 1918169600}   # medusa_heads
NCU_ATTN_TRAFFIC_BYTES = {"gqa7b_b32": 1512010496, "vicuna33b_b16": 3573742592}   # medusa_tree_attention


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=configs.ORDER + configs.SHARED + configs.PRUNED)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time eager launches instead of one CUDA graph")
    ap.add_argument("--fused", action="store_true",
                    help="run each step as the one persistent kernel of medusa_step_fused (greedy, B <= 4)")
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of untimed steps before the timed region")
    ap.add_argument("--paged", type=int, default=0,
                    help="with --part attention: rows per page of a shuffled paged pool (0: contiguous cache)")
    ap.add_argument("--part", default="step", choices=["step", "heads", "attention", "verify"],
                    help="diagnostic: time one library call in a loop (for profiler captures)")
    ap.add_argument("--set", action="append", default=[], metavar="FIELD=VALUE",
                    help="diagnostic: override a workload field (e.g. V=8000, B=4)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(power) if power else None}


def algorithmic_bytes(w, L, acc, mode, with_bias=False):
    """Minimum bytes one step must move (each term counted once)."""
    elt = w.elt
    B, d, V, K, N = w.B, w.d, w.V, w.K, w.N
    vocab = (1 if w.shared_vocab else K) * d * V   # one shared projection is streamed once for all heads
    heads = (K * (d * d + (d if with_bias else 0)) + vocab) * elt + B * d * elt
    logits = 2 * B * K * V * 4 if mode == REJECTION else 0
    kv = int(np.sum(L)) * w.Hkv * w.D * 2 * elt
    tree = B * N * (w.Hq + 2 * w.Hkv) * w.D * elt
    out = B * N * w.Hq * w.D * elt
    visited = int(np.sum(np.asarray(acc) + 1)) * V * elt
    return {"heads": heads, "logits": logits, "kv": kv, "tree_qkv": tree, "attn_out": out, "target_rows": visited,
            "total": heads + logits + kv + tree + out + visited}


def replica_seed(seed, rank):
    """Each replica draws its own inputs (weak scaling: fixed work per GPU)."""
    return seed + 1000 * rank


def replica_throughput(elapsed_ms, steps, world, device):
    """Whole-job steps/s: every rank ran `steps` steps; the job time is the slowest rank's."""
    if world > 1:
        t = torch.tensor([float(elapsed_ms)], device=device, dtype=torch.float64)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    return elapsed_ms, world * steps / (elapsed_ms / 1000.0)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ----------------------------------------------------------------------------- CPU oracle timing
# At most this many sequences of a batch go through the oracle's per-sequence parts (tree,
# attention, acceptance, compaction) in one timed oracle step; the float64 copy of a 33B-shaped
# sequence's KV cache alone is 0.9 GB, and its attention takes about a second on one core. The
# heads always run over the whole batch.
ORACLE_SEQS = 1


def oracle_inputs_from(si, tl, seqs):
    """Host float64 inputs of the oracle: the heads' inputs for the whole batch, the
    per-sequence inputs (Q, cache, target logits, uniforms, lengths) of the first `seqs`."""
    f = lambda t: t.detach().to("cpu", torch.float32).double().numpy()
    n = seqs
    return {"h": f(si.h), "W": f(si.W), "b": None if si.bias is None else f(si.bias), "U": f(si.U),
            "Q": f(si.Q[:n]), "Kc": f(si.Kc[:n]), "Vc": f(si.Vc[:n]), "tl": f(tl[:n]), "root": si.root_token[:n],
            "L": si.L[:n], "L_cap": si.L_cap, "u_acc": si.u_acc[:n], "u_res": si.u_res[:n], "seqs": n,
            "B": int(si.h.shape[0])}


def oracle_step(O, w, mode, x):
    """One oracle step: heads over the whole batch, then the per-sequence parts over the
    sampled sequences. Returns (seconds in the heads, seconds in the rest)."""
    t0 = time.perf_counter()
    r, z = O.medusa_heads(x["h"], x["W"], x["b"], x["U"])
    t1 = time.perf_counter()
    z = z[:x["seqs"]]
    topk, _ = O.heads_top_s(z, w.branching)
    tree = O.tree_build(w.branching, x["root"], topk, x["L"], x["L_cap"], paths=w.tree_paths)
    O.tree_attention(x["Q"], x["Kc"], x["Vc"], x["L"], tree["mask"], w.Hq, w.Hkv)
    ver = O.verify_batch(mode, tree, x["tl"], w.K, head_logits=z, u_acc=x["u_acc"], u_res=x["u_res"],
                         T=w.temperature)
    # compaction moves rows inside each sequence's tree region only; the oracle gets that region
    # (committed length 0 there) instead of copying the whole float64 cache
    N = tree["N"]
    kr = np.stack([x["Kc"][b, :, int(x["L"][b]):int(x["L"][b]) + N] for b in range(x["seqs"])])
    vr = np.stack([x["Vc"][b, :, int(x["L"][b]):int(x["L"][b]) + N] for b in range(x["seqs"])])
    O.kv_compact(kr, vr, np.zeros(x["seqs"], dtype=np.int64), ver["acc"], ver["path"])
    return t1 - t0, time.perf_counter() - t1


def time_oracle(w, mode, x, steps, warmup=0, budget_s=None):
    """Seconds per whole-batch oracle step: the heads' time plus the sampled sequences'
    time scaled to the batch (B / seqs)."""
    from oracle import medusa_oracle as O
    for _ in range(warmup):
        oracle_step(O, w, mode, x)
    scale = x["B"] / x["seqs"]
    times = []
    t_all = time.perf_counter()
    for _ in range(steps):
        th, tr = oracle_step(O, w, mode, x)
        times.append(th + scale * tr)
        if budget_s is not None and time.perf_counter() - t_all > budget_s:
            break
    return times


def oracle_sample_text(w, x, n):
    if x["seqs"] == x["B"]:
        return (f"{n} full oracle steps of {w.name} (B={w.B}; compaction of the tree region), float64 numpy, "
                f"single-threaded BLAS, inputs pre-decoded")
    seqs = "sequence 0" if x["seqs"] == 1 else f"sequences 0..{x['seqs'] - 1}"
    return (f"{n} oracle steps of {w.name}: heads over all {x['B']} sequences, then tree, attention, acceptance "
            f"and compaction (of the tree region) for {seqs}, that part's time scaled by {x['B']}/{x['seqs']}; "
            f"float64 numpy, single-threaded BLAS, inputs pre-decoded")


def blas_threads():
    """Threads of the BLAS pool numpy uses (threadpoolctl when present, else the environment)."""
    try:
        import threadpoolctl
        n = [i["num_threads"] for i in threadpoolctl.threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except ImportError:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


# ----------------------------------------------------------------------------- reference arm
def workload_config(w, L, mode, world):
    """The `config` object of both arms' JSON lines: the workload, its sizes and lengths."""
    elt = 4 if w.dtype == F32 else 2
    weights = (w.K * w.d * w.d + (1 if w.shared_vocab else w.K) * w.d * w.V) * elt
    kv = int(np.sum(L)) * w.Hkv * w.D * 2 * elt
    return {"workload": w.name, "B": w.B, "d": w.d, "V": w.V, "K": w.K, "branching": list(w.branching),
            "N": w.N, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D, "L": [int(x) for x in L][:4],
            "L_sum": int(np.sum(L)), "mode": "greedy" if mode == GREEDY else "rejection",
            "temperature": w.temperature if mode == REJECTION else None, "shared_vocab": w.shared_vocab,
            "tree": "pruned" if w.tree_paths is not None else "cartesian",
            "l2": f"inputs larger than L2 ({(weights + kv) / 1e9:.2f} GB of weights and KV per step)",
            "parallelism": f"replicas x{world}"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = configs.get(args.workload)
    mode = w.modes[0]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    si = synth.make_step_inputs(w, seed=args.seed, device=dev)
    tl = make_targets(w, si, dev, mode, args.seed, via_library=False)
    x = oracle_inputs_from(si, tl, min(w.B, ORACLE_SEQS))
    L = np.asarray(si.L)
    del si, tl
    if dev == "cuda":
        torch.cuda.empty_cache()
    times = time_oracle(w, mode, x, args.steps, warmup=args.warmup)
    total = sum(times)
    value = len(times) / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": len(times), "warmup": args.warmup, "ms_per_step": 1000 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, L, mode, args.gpus),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                             "sample": oracle_sample_text(w, x, len(times))},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- our arm
def make_targets(w, si, dev, mode, seed, via_library=True):
    """Target logits: independent, or correlated with this step's head logits."""
    if w.target_corr == 0.0:
        return synth.target_logits(w, seed, device=dev)
    if via_library:
        # head logits and node depths from the library itself (setup, outside any timed region)
        from medusa_speculative_decoding_heads_gb300.step import DeviceStep
        st = DeviceStep(w, REJECTION, si.L_cap, dev)
        st.heads(si.h, si.W, si.bias, si.U, write_logits=True)
        st.tree_build(torch.from_numpy(si.root_token).to(dev), torch.from_numpy(si.L).to(dev))
        zhat, depth = st.logits, st.depth.cpu().numpy()
    else:
        # the reference arm: everything from the CPU oracle
        from oracle import medusa_oracle as O
        f = lambda t: t.detach().to("cpu", torch.float32).double().numpy()
        _, z = O.medusa_heads(f(si.h), f(si.W), None if si.bias is None else f(si.bias), f(si.U))
        lay = (O.tree_layout(w.branching) if w.tree_paths is None
               else O.tree_layout_from_paths(w.tree_paths, w.branching))
        zhat, depth = torch.from_numpy(z).float(), lay["depth"]
    return synth.target_logits(w, seed, device=dev, zhat=zhat, depth=depth)


def workload_of(args):
    w = configs.get(args.workload)
    if args.set:
        kv = {}
        for item in args.set:
            k, v = item.split("=", 1)
            kv[k] = type(getattr(w, k))(v) if not isinstance(getattr(w, k), tuple) else tuple(int(x) for x in v.split(","))
        w = configs.scaled(w, **kv)
    return w


def run_part(args):
    """Diagnostic: one library call of the workload, timed in a loop (eager launches)."""
    from medusa_speculative_decoding_heads_gb300 import _build, binding as mb
    from medusa_speculative_decoding_heads_gb300.step import DeviceStep, to_device_inputs
    _build.build()
    mb.load()
    dev = torch.device("cuda")
    w = workload_of(args)
    mode = w.modes[0]
    si = synth.make_step_inputs(w, seed=args.seed, device=dev)
    st = DeviceStep(w, mode, si.L_cap, dev)
    L = torch.from_numpy(si.L).to(dev)
    st.heads(si.h, si.W, si.bias, si.U, write_logits=True)
    st.tree_build(torch.from_numpy(si.root_token).to(dev), L)
    tl = make_targets(w, si, dev, mode, args.seed) if args.part == "verify" else None
    ua, ur = (torch.from_numpy(x).to(dev) for x in (si.u_acc, si.u_res))
    call = {"heads": lambda: st.heads(si.h, si.W, si.bias, si.U, write_logits=mode == REJECTION),
            "attention": lambda: st.tree_attention(si.Q, si.Kc, si.Vc, L),
            "verify": lambda: st.verify(tl, ua, ur)}[args.part]
    if args.part == "attention" and args.paged:
        # the same committed rows in a shuffled page pool, the tree rows staged
        P = args.paged
        cap = -(-si.L_cap // P) * P
        Kc = torch.nn.functional.pad(si.Kc, (0, 0, 0, cap - si.L_cap))
        Vc = torch.nn.functional.pad(si.Vc, (0, 0, 0, cap - si.L_cap))
        mp = cap // P
        gen = torch.Generator(device="cpu")
        gen.manual_seed(args.seed)
        perm = torch.randperm(w.B * mp, generator=gen).to(dev)             # pool slot of page (b, i)
        pool_k = torch.empty((w.B * mp, w.Hkv, P, w.D), dtype=Kc.dtype, device=dev)
        pool_v = torch.empty_like(pool_k)
        pool_k[perm] = Kc.view(w.B, w.Hkv, mp, P, w.D).permute(0, 2, 1, 3, 4).reshape(w.B * mp, w.Hkv, P, w.D)
        pool_v[perm] = Vc.view(w.B, w.Hkv, mp, P, w.D).permute(0, 2, 1, 3, 4).reshape(w.B * mp, w.Hkv, P, w.D)
        bt = perm.view(w.B, mp).to(torch.int32)
        Kt = torch.stack([si.Kc[b, :, int(si.L[b]):int(si.L[b]) + w.N] for b in range(w.B)]).contiguous()
        Vt = torch.stack([si.Vc[b, :, int(si.L[b]):int(si.L[b]) + w.N] for b in range(w.B)]).contiguous()
        del Kc, Vc
        st = DeviceStep(w, mode, cap, dev)
        st.tree_build(torch.from_numpy(si.root_token).to(dev), L)
        O_out = torch.empty_like(si.Q)
        call = lambda: mb.tree_attention_paged(st.cfg, si.Q, pool_k, pool_v, w.B * mp, P, bt, Kt, Vt, L,
                                               st.anc_bits, O_out, st.workspace)
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        call()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    print(json.dumps({"part": args.part, "workload": w.name, "overrides": args.set, "paged": args.paged,
                      "us_per_call": 1000 * ms}))
    return 0


def run_ours(args):
    from medusa_speculative_decoding_heads_gb300 import _build, binding as mb
    from medusa_speculative_decoding_heads_gb300.step import DeviceStep, to_device_inputs

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.build()
    mb.load()

    w = configs.get(args.workload)
    mode = w.modes[0]
    seed = replica_seed(args.seed, rank)
    si = synth.make_step_inputs(w, seed=seed, device=dev)
    tl = make_targets(w, si, dev, mode, seed)
    inp = to_device_inputs(si, tl, dev)
    L0 = inp.L.clone()
    stream = torch.cuda.current_stream(dev)
    st = DeviceStep(w, mode, si.L_cap, dev)
    write_logits = mode == REJECTION

    ev = lambda: torch.cuda.Event(enable_timing=True)

    calls = [
        lambda: st.heads(inp.h, inp.W, inp.bias, inp.U, write_logits=write_logits),
        lambda: st.tree_build(inp.root_token, inp.L),
        lambda: st.tree_attention(inp.Q, inp.Kc, inp.Vc, inp.L),
        lambda: st.verify(inp.target_logits, inp.u_acc, inp.u_res),
        lambda: st.kv_compact(inp.Kc, inp.Vc, inp.L),
    ]
    names = ["heads", "tree_build", "tree_attention", "verify", "kv_compact"]
    if args.fused:   # the same step as one persistent kernel (a memset of its barrier word, then the launch)
        fused_args = st.fused_args(inp, write_logits=False, compact=True)
        calls = [lambda: mb.step_fused(st.cfg, fused_args, st.stream)]
        names = ["fused_step"]

    def one_step(marks=None):
        inp.L.copy_(L0, non_blocking=True)
        for i, call in enumerate(calls):
            if marks is not None:
                marks[i].record()          # on the current stream (the capture stream inside a graph)
            call()
        if marks is not None:
            marks[len(calls)].record()

    for _ in range(max(3, args.warmup)):
        one_step()
    torch.cuda.synchronize()
    acc = st.acc.cpu().numpy()

    sampler = ClockSampler(local) if rank == 0 else None
    timed = None
    if not args.eager:
        try:
            timed = time_graph(one_step, len(calls), args.steps, stream, mb)
        except Exception as exc:  # graph capture unavailable: fall back to eager launches
            print(f"# CUDA graph capture failed ({exc!r}); timing eager launches", file=sys.stderr)
            timed = None
    if sampler:
        sampler.start()
    # Soak: ~1 s of the same step right before the timed region, so the clock
    # samples (every 200 ms) see the GPU under this load.
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak:
        if timed is not None:
            timed[0].replay()
        else:
            for _ in range(args.steps):
                one_step()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if timed is not None:
        graph, marked, marks, launches_per_step = timed
        t0, t1 = ev(), ev()
        t0.record(stream)
        graph.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        marked.replay()                 # per-call breakdown, outside the timed region
        torch.cuda.synchronize()
        launches = launches_per_step * args.steps
        launch_mode = "cuda_graph"
    else:
        marks = [[ev() for _ in range(len(calls) + 1)] for _ in range(args.steps)]
        t0, t1 = ev(), ev()
        n0 = mb.launch_count()
        t0.record(stream)
        for k in range(args.steps):
            one_step(marks[k])
        t1.record(stream)
        torch.cuda.synchronize()
        launches = mb.launch_count() - n0
        launch_mode = "eager"
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    elapsed_ms = t0.elapsed_time(t1)
    per_call = {n: statistics.mean(m[i].elapsed_time(m[i + 1]) for m in marks) for i, n in enumerate(names)}
    # the spread of single steps, from the event-marked replay (events end the launch overlap, so these
    # run a little above ms_per_step)
    q = np.percentile([m[0].elapsed_time(m[-1]) for m in marks], [10, 50, 90])
    step_spread = {"p10": float(q[0]), "p50": float(q[1]), "p90": float(q[2]), "source": "event-marked replay"}
    heads_ms = per_call.get("heads", 0.0)
    elapsed_ms, value = replica_throughput(elapsed_ms, args.steps, world, dev)
    ms_per_step = elapsed_ms / args.steps

    e2e = None if args.no_e2e else run_e2e(w, st, inp, L0, tl, si, args, stream, world)
    # every bounded device wait of the run completed (a wait that expired would have cut its work short)
    wait_status, heads_codes, attention_codes = mb.poll_errors()

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    hbm, peak_kind = peaks()
    by = algorithmic_bytes(w, si.L, acc, mode, with_bias=si.bias is not None)
    heads_bytes = by["heads"] + (w.B * w.K * w.V * 4 if write_logits else 0)
    attn_ms = per_call.get("tree_attention", 0.0)
    if args.fused:   # one kernel: the whole step's bytes over its duration
        kernel = "medusa_step_fused (the whole step as one persistent kernel)"
        dom_bytes, dom_ms, traffic = by["total"], per_call["fused_step"], None
    elif attn_ms > heads_ms:   # the dominant call is tree attention (long committed prefixes)
        kernel = "medusa_tree_attention (tcgen05 tree attention over the committed KV)"
        dom_bytes, dom_ms, traffic = by["kv"] + by["tree_qkv"] + by["attn_out"], attn_ms, NCU_ATTN_TRAFFIC_BYTES.get(w.name)
    else:
        kernel = "medusa_heads (residual + vocab projection GEMV, top-s)"
        dom_bytes, dom_ms, traffic = heads_bytes, heads_ms, NCU_TRAFFIC_BYTES.get(w.name)
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if w.dtype == F32 else "bf16", "data": "synthetic",
        "config": workload_config(w, si.L, mode, world),
        "clocks": dict(clocks or {}, window=f"{args.soak:.1f} s soak of the same step + the timed region"),
        "gpu_launches": launches,
        "roofline": {"bound": "hbm", "kernel": kernel,
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": traffic, "peak_source": f"hbm_gbs of {peak_kind}",
                     "algorithmic_bytes": dom_bytes, "avg_launch_ms": dom_ms},
        "step_roofline": {"algorithmic_bytes": by["total"], "achieved_gbs": by["total"] / (ms_per_step * 1e-3) / 1e9,
                          "frac": by["total"] / (ms_per_step * 1e-3) / 1e9 / hbm, "peak_source": f"hbm_gbs of {peak_kind}",
                          "frac_of_8000_gbs": by["total"] / (ms_per_step * 1e-3) / 1e9 / 8000.0,
                          "bytes_by_term": by},
        "breakdown_ms": dict(per_call, step=ms_per_step),
        "marked_step_ms": step_spread,
        "launch_mode": launch_mode + (", medusa_step_fused" if args.fused else ""),
        "accepted_per_step": float(np.mean(acc + 1)),
        "e2e": e2e,
        "expired_waits": {"status": wait_status, "heads": heads_codes, "attention": attention_codes},
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, mode, si, tl)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    if wait_status != 0:
        print(f"# a bounded device wait expired during the run (heads {heads_codes:#x}, attention "
              f"{attention_codes:#x}): the numbers above are not valid", file=sys.stderr)
        return 3
    return 0


def time_graph(one_step, ncalls, steps, stream, mb):
    """Capture `steps` consecutive steps as one CUDA graph (the timed one), and the
    same steps again with timing events recorded around every library call.

    The events are graph nodes between the kernels, and a kernel that follows an
    event node cannot start early under programmatic dependent launch; so the
    step time comes from the graph without them, and the events' graph only
    gives the per-call breakdown."""
    mk = lambda: torch.cuda.Event(enable_timing=True, external=True)
    marks = [[mk() for _ in range(ncalls + 1)] for _ in range(steps)]
    graph = torch.cuda.CUDAGraph()
    n0 = mb.launch_count()
    with torch.cuda.graph(graph):
        for k in range(steps):
            one_step()
    launches_per_step = (mb.launch_count() - n0) // steps
    marked = torch.cuda.CUDAGraph()
    with torch.cuda.graph(marked):
        for k in range(steps):
            one_step(marks[k])
    graph.replay()                      # one untimed replay of each
    marked.replay()
    torch.cuda.synchronize()
    return graph, marked, marks, launches_per_step


def run_e2e(w, st, inp, L0, tl, si, args, stream, world):
    """The same step with per-step inputs copied from pinned host memory and results read back.

    Every step copies all of its inputs host -> device (one copy of one packed
    pinned buffer) and reads its accepted tokens back inside the timed region.
    The copy of step k+1 runs on a copy stream into the second of two device
    input sets while step k computes on the other. The tree's K/V rows land in
    the staging part of the set and move into the cache at the start of their
    step (after the previous step's compaction), one indexed copy for K and one
    for V.
    """
    import dataclasses

    N = w.N
    dev = inp.h.device
    Lh = torch.from_numpy(np.asarray(si.L, dtype=np.int64)).to(dev)
    b_idx = torch.arange(w.B, device=dev).view(-1, 1).expand(w.B, N)
    t_idx = Lh.view(-1, 1) + torch.arange(N, device=dev).view(1, -1)
    parts = {
        "h": inp.h, "Q": inp.Q, "target_logits": inp.target_logits, "u_acc": inp.u_acc, "u_res": inp.u_res,
        "root_token": inp.root_token, "L": L0,
        # the tree rows of K and V, [B][N][Hkv][D] (the order an indexed write into the cache takes)
        "tk": inp.Kc[b_idx, :, t_idx].contiguous(), "tv": inp.Vc[b_idx, :, t_idx].contiguous(),
    }
    offs, total = {}, 0
    for key, t in parts.items():
        offs[key] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()

    def views(buf):
        out = {}
        for key, t in parts.items():
            n = t.numel() * t.element_size()
            out[key] = buf[offs[key]:offs[key] + n].view(t.dtype).view(t.shape)
        return out

    for key, v in views(host).items():
        v.copy_(parts[key].cpu())
    out_tok = torch.empty_like(st.out_tokens, device="cpu").pin_memory()
    h2d = total
    d2h = out_tok.numel() * 4
    # two device input sets (the cache Kc/Vc and the weights are shared state)
    sets = []
    for _ in range(2):
        buf = torch.empty(total, dtype=torch.uint8, device=dev)
        dv = views(buf)
        step_inp = dataclasses.replace(inp, h=dv["h"], Q=dv["Q"], target_logits=dv["target_logits"],
                                       u_acc=dv["u_acc"], u_res=dv["u_res"], root_token=dv["root_token"], L=dv["L"])
        sets.append((buf, dv, step_inp))
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    freed = [torch.cuda.Event(), torch.cuda.Event()]

    def run(steps):
        cur = torch.cuda.current_stream()
        copy_stream.wait_stream(cur)
        with torch.cuda.stream(copy_stream):
            sets[0][0].copy_(host, non_blocking=True)
            copied[0].record(copy_stream)
        for k in range(steps):
            if k + 1 < steps:
                with torch.cuda.stream(copy_stream):
                    if k >= 1:
                        copy_stream.wait_event(freed[(k + 1) % 2])   # step k-1 is done with that set
                    sets[(k + 1) % 2][0].copy_(host, non_blocking=True)
                    copied[(k + 1) % 2].record(copy_stream)
            cur.wait_event(copied[k % 2])
            _, dv, step_inp = sets[k % 2]
            if w.B <= 4:   # a few plain strided copies beat one indexed write for small batches
                for b in range(w.B):
                    lb = int(si.L[b])
                    inp.Kc[b, :, lb:lb + N].copy_(dv["tk"][b].transpose(0, 1))
                    inp.Vc[b, :, lb:lb + N].copy_(dv["tv"][b].transpose(0, 1))
            else:
                inp.Kc[b_idx, :, t_idx] = dv["tk"]
                inp.Vc[b_idx, :, t_idx] = dv["tv"]
            if args.fused:
                st.run_fused(step_inp, write_logits=False, compact=True)
            else:
                st.run(step_inp, write_logits=st.mode == REJECTION, compact=True)
            out_tok.copy_(st.out_tokens, non_blocking=True)
            freed[k % 2].record(cur)
        cur.wait_stream(copy_stream)

    run(3)
    torch.cuda.synchronize()
    steps = args.steps
    graph = None
    if not args.eager:
        try:   # the same launches and copies on both streams, captured once and replayed
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                run(steps)
            graph.replay()
            torch.cuda.synchronize()
        except Exception as exc:
            print(f"# e2e graph capture failed ({exc!r}); timing eager launches", file=sys.stderr)
            graph = None
    if world > 1:
        torch.distributed.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    if graph is not None:
        graph.replay()
    else:
        run(steps)
    b.record(stream)
    torch.cuda.synchronize()
    ms, e2e_value = replica_throughput(a.elapsed_time(b), steps, world, inp.h.device)
    return {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps, "launch_mode": "cuda_graph" if graph else "eager",
            "overlap": "H2D of step k+1 (one packed copy) on a copy stream during step k, two device input sets"}


def cpu_baseline(w, mode, si, tl):
    x = oracle_inputs_from(si, tl, min(w.B, ORACLE_SEQS))
    times = time_oracle(w, mode, x, steps=50, warmup=1, budget_s=15.0)
    return {"value": len(times) / sum(times), "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": oracle_sample_text(w, x, len(times))}


def launch_replicas(args):
    """`--gpus N` without a launcher: start N ranks of this script under torch.distributed.run
    (one per GPU, rendezvous on 127.0.0.1). Returns the launcher's exit status."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    args = parse()
    _, world, _ = dist_env()
    if args.gpus < 1:
        sys.exit("--gpus must be at least 1")
    if "WORLD_SIZE" in os.environ and world != args.gpus:
        sys.exit(f"--gpus {args.gpus} but the launcher started {world} ranks")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        if args.impl == "ours" and args.part == "step":
            return launch_replicas(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.part != "step":
        return run_part(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
