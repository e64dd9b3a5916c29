"""Benchmark: verified tree tokens/s for one tree-verification step on GB300.

One step = the whole hot path over one batch: ancestor mask, tree attention
(one attention layer over the request's KV prefix + tree), and verification
(vocab softmax, acceptance walk, bonus token).  Verification depends on none
of the other two, so it runs on a second branch of the step's CUDA graph,
side by side with the mask and attention.  The workload is the
LLaMA-7B-shaped tree-verify case: 1 request, 32 heads (MHA), head dim 128,
bf16 KV prefix 2048, a width-5 depth-3 draft tree pruned to 64 nodes, vocab
32000, stochastic verification at temperature 0.7.  Inputs are synthetic and
seeded; the step's inputs rotate over enough device copies (> 4x L2) that
every step reads them from HBM.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
Multi-GPU (torchrun, one rank per GPU) runs independent replicas: the path has
no exchange step, so there is no data-path collective (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified tree tokens/s; tree-attn + verify HBM GB/s as % of GB300 peak"
UNIT = "tree tokens/s"
WORKLOAD = "llama7b"   # the headline workload; --workload times the others the same way
WORKLOADS = {
    "llama7b": ("LLaMA-7B-shaped tree verify: B1, Hq=Hkv=32, D128, bf16 KV prefix 2048, "
                "w5 d3 draft tree pruned to 64 nodes, V32000 fp32 logits, T=0.7 stochastic"),
    "tiny": ("tiny: B1, Hq=Hkv=4, D64, fp32 Q/K/V, KV prefix 128, 8-node tree of depth 3, V1000, "
             "T=1 stochastic"),
    "dynamic": ("dynamic batch: B16, Hq=Hkv=32, D128, bf16 KV prefixes U[512,4096], trees of "
                "U[16,96] nodes and depth U[2,5] in one ragged launch, V32000, greedy"),
    "llama70b_gqa": ("LLaMA-2-70B-shaped GQA: B4, Hq=64, Hkv=8, D128, bf16 KV prefix 8192, "
                     "128-node trees of depth 5 and width <= 8, V32000, T=0.7 stochastic"),
    "long_chain": ("long context, chain: B8, Hq=Hkv=32, D128, bf16 KV prefix 32768, a chain of "
                   "K=5 speculated tokens (6 nodes), V32000, T=0.7 stochastic"),
    "long_tree": ("long context, tree: B8, Hq=Hkv=32, D128, bf16 KV prefix 32768, 128-node trees "
                  "of depth 6 and width <= 8, V32000, T=0.7 stochastic"),
}
MODEL_LAYERS = {"llama70b_gqa": 80}   # 32 for the LLaMA-7B-shaped rest


# --------------------------------------------------------------------------
# algorithmic bytes
# --------------------------------------------------------------------------
def attn_bytes(w) -> int:
    """KV of every prefix + tree slot read once per KV head, Q read once, O
    written once, in the inputs' dtype (O takes Q's)."""
    el = w.q.element_size()
    kv = sum(int(w.prefix_lens[b] + w.offsets[b + 1] - w.offsets[b]) for b in range(w.B)) * w.Hkv * w.D * el * 2
    return kv + 2 * w.T * w.Hq * w.D * el


def verify_bytes(w) -> int:
    """Every node's target row; internal nodes' draft rows when stochastic."""
    rows = w.T
    if w.temperature > 0:
        internal = 0
        for b in range(w.B):
            lo, hi = w.offsets[b], w.offsets[b + 1]
            internal += len(set(w.parents[lo + 1:hi].tolist()))
        rows += internal
    return rows * w.V * 4


def mask_bytes(w) -> int:
    return w.T * (4 + 16 + 4)


def attn_flops(w) -> int:
    """2 D flops for each score and 2 D for each weighted value, over the
    keys each (node, head) row sees: its request's prefix, its ancestors and
    itself."""
    total = 0
    for b in range(w.B):
        lo, hi = w.offsets[b], w.offsets[b + 1]
        par = w.parents[lo:hi]
        depth = np.zeros(hi - lo, np.int64)
        for i in range(1, hi - lo):
            depth[i] = depth[par[i]] + 1
        total += int((w.prefix_lens[b] + depth + 1).sum())
    return 4 * w.D * w.Hq * total


def describe(name: str, temperature, prefix=None) -> str:
    desc = WORKLOADS[name]
    if prefix is not None:
        desc = re.sub(r"KV prefix \d+", f"KV prefix {prefix}", desc)
    if temperature is None:
        return desc
    head, _, _ = desc.rpartition(", ")
    return f"{head}, " + ("greedy" if temperature == 0 else f"T={temperature:g} stochastic")


def prefix_override(args) -> dict:
    """--prefix sets the KV prefix length of the workloads whose requests
    share one (all but the dynamic batch, whose prefixes are drawn)."""
    if args.prefix is None:
        return {}
    if args.workload == "dynamic":
        raise SystemExit("--prefix does not apply to the dynamic batch (its prefixes are drawn)")
    return {"L": args.prefix}


# --------------------------------------------------------------------------
# environment helpers
# --------------------------------------------------------------------------
def measured_peaks(kind: str = "hbm"):
    """The roofline denominator: HBM copy GB/s, or dense bf16 TFLOP/s (burst:
    each kernel is timed alone)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    key, fallback = ("hbm_gbs", 6800.0) if kind == "hbm" else ("bf16_tflops", 1900.0)
    if os.path.exists(p):
        d = json.load(open(p))
        if key in d:
            return float(d[key]), "measured"
    return fallback, "fallback"


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key: str):
    """DRAM bytes per launch from a committed ncu summary, only while the
    kernel's source is unchanged since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d:
        return None
    srcs = [os.path.join(ROOT, s) for s in d["sources"]]
    if not all(os.path.exists(s) for s in srcs) or source_hash(srcs) != d["source_hash"]:
        return None
    return d["dram_bytes_per_launch"]


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = [l.split(",") for l in open(self.path).read().strip().splitlines() if l.strip()]
        os.unlink(self.path)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# the CUDA path
# --------------------------------------------------------------------------
class Step:
    """Device buffers for one workload and R rotating input copies."""

    def __init__(self, w, copies: int, seed: int):
        import torch
        import token_tree_verification_gb300 as ttv
        self.ttv, self.torch, self.w = ttv, torch, w
        dev = "cuda"
        self.par = torch.as_tensor(w.parents).to(dev)
        self.off = torch.as_tensor(w.offsets).to(dev)
        self.tok = torch.as_tensor(w.tokens).to(dev)
        self.pl = torch.as_tensor(w.prefix_lens).to(dev)
        self.status = torch.zeros(w.B, dtype=torch.int32, device=dev)
        self.mask = torch.empty((w.T, 4), dtype=torch.int32, device=dev)
        self.depth = torch.empty(w.T, dtype=torch.int32, device=dev)
        self.o = torch.empty((w.T, w.Hq, w.D), dtype=w.q.dtype, device=dev)
        self.W = w.max_depth + 1
        self.ws = ttv.make_verify_workspace(w.B, w.T, w.V)
        self.max_prefix = int(w.prefix_lens.max())
        na = ttv.tree_attn_workspace_size(w.B, w.T, w.Hq, w.Hkv, w.D, self.max_prefix)
        self.ws_attn = torch.zeros(max(na, 16), dtype=torch.uint8, device=dev)
        self.outs = dict(
            accept_len=torch.empty(w.B, dtype=torch.int32, device=dev),
            path_nodes=torch.empty((w.B, self.W), dtype=torch.int32, device=dev),
            out_tokens=torch.empty((w.B, self.W), dtype=torch.int32, device=dev),
            near_ties=torch.empty(w.B, dtype=torch.int32, device=dev))
        tl = torch.as_tensor(w.target_logits).to(dev)
        dl = torch.as_tensor(w.draft_logits).to(dev) if w.draft_logits is not None else None
        self.copies = []
        for _ in range(copies):
            self.copies.append(dict(q=w.q.to(dev).clone(), k=w.k_cache.to(dev).clone(),
                                    v=w.v_cache.to(dev).clone(), tl=tl.clone(),
                                    dl=None if dl is None else dl.clone()))
        self.max_prefix = int(w.prefix_lens.max())
        self.seed = seed
        self.side = torch.cuda.Stream()
        self.attn_ctas = attn_cta_budget(w, torch.cuda.get_device_properties(
            torch.cuda.current_device()).multi_processor_count)

    def run(self, i: int, stream=None):
        """Enqueue step i on ``stream`` (default: the current stream) over
        input copy i."""
        c = self.copies[i % len(self.copies)]
        self.launch(c["q"], c["k"], c["v"], c["tl"], c["dl"], self.par, self.off, self.tok, self.pl,
                    self.seed + i, self.outs, stream)

    def launch(self, q, k, v, tl, dl, par, off, tok, pl, seed, outs, stream=None):
        """One step: tree attention on ``stream``, building its rows' ancestor
        sets from the parent array itself, and on a second stream forked from
        it and joined back the mask kernel (its mask and depths, for the
        consumers after attention) then verification.  Verification reads only
        the logits and the tree, attention only Q, the caches and the
        parents, so the branches run side by side (under graph capture the
        fork and join become two branches of the graph)."""
        torch, ttv, w = self.torch, self.ttv, self.w
        cur = torch.cuda.current_stream() if stream is None else stream
        self.side.wait_stream(cur)
        ttv.tree_attn(q, k, v, pl, off, None, self.max_prefix, self.status, o=self.o,
                      workspace=self.ws_attn, stream=cur, max_ctas=self.attn_ctas, parents=par)
        with torch.cuda.stream(self.side):
            ttv.build_tree_mask(par, off, self.status, mask=self.mask, depth=self.depth,
                                stream=self.side)
            ttv.tree_verify(tl, dl, tok, par, off, w.temperature, seed, self.W, self.status, self.ws,
                            outputs=outs, stream=self.side)
        cur.wait_stream(self.side)


def verify_resident_ctas(w) -> int:
    """CTAs stochastic verification keeps resident while it works: two (one
    per 16384 vocabulary entries) for every internal node; leaves leave at
    once (their draw is taken by the walker when the walk reaches them).
    Greedy verification's CTAs are short and many; it gets no reservation."""
    if w.temperature <= 0 or w.V > 131072:
        return 0
    internal = 0
    for b in range(w.B):
        lo, hi = w.offsets[b], w.offsets[b + 1]
        internal += len(set(w.parents[lo + 1:hi].tolist()))
    return internal * ((w.V + 16383) // 16384)


def attn_cta_budget(w, sms: int) -> int:
    """The CTAs the step's attention may keep resident while verification
    runs beside it: the SMs verification's internal nodes do not hold, when
    they hold less than half of them (0: the whole GPU)."""
    need = verify_resident_ctas(w)
    return sms - need if 0 < need < sms // 2 else 0


def run_native(args, rank, world, local_rank):
    import torch
    from token_tree_verification_gb300 import synthetic
    torch.cuda.set_device(local_rank)
    import token_tree_verification_gb300 as ttv
    ttv.load()
    w = synthetic.make_workload(args.workload, seed=0, device="cuda", pad=0.0,
                                temperature=args.temperature, **prefix_override(args))
    l2 = torch.cuda.get_device_properties(local_rank).L2_cache_size
    per_copy = (w.q.numel() + w.k_cache.numel() + w.v_cache.numel()) * w.q.element_size() \
        + w.target_logits.nbytes + (w.draft_logits.nbytes if w.draft_logits is not None else 0)
    copies = max(2, math.ceil(4 * l2 / per_copy) + 1)
    st = Step(w, copies, seed=1000 * rank)
    stream = torch.cuda.Stream()
    K, Wm = args.steps, args.warmup

    # eager warm-up configures the kernels before any capture
    with torch.cuda.stream(stream):
        for i in range(max(1, Wm)):
            st.run(i)
    torch.cuda.synchronize()

    if args.eager:
        # profiler mode: plain stream launches, no graphs, no timing claims
        with torch.cuda.stream(stream):
            for i in range(K):
                st.run(i)
        torch.cuda.synchronize()
        status = st.status.cpu().numpy()
        return {"eager": True, "steps": K, "status": status.tolist(),
                "accept_len": st.outs["accept_len"].cpu().tolist()}

    # capture: a warm-up graph of W steps and the timed graph(s) of K steps
    # (nothing but the steps' own kernels: no event nodes between them)
    chunk = min(K, args.graph_steps)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                st.run(i)
        return g

    g_warm = capture(max(1, Wm))
    g_main = capture(chunk)
    reps, rem = divmod(K, chunk)
    g_rem = capture(rem) if rem else None
    with torch.cuda.stream(stream):
        g_warm.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.25)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    # graphs replay on the current stream: make it the timed stream
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(reps):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = t0.elapsed_time(t1)
    # If the timed region was shorter than a few clock samples, keep the same
    # work running briefly so the clock record covers this load.
    soak = False
    if elapsed_ms < 1500:
        soak = True
        tend = time.time() + 1.0
        with torch.cuda.stream(stream):
            while time.time() < tend:
                g_main.replay()
        torch.cuda.synchronize()
    clocks = sampler.stop()
    status = st.status.cpu().numpy()
    if (status != 0).any():
        raise RuntimeError(f"device status {status.tolist()}")

    # per-kernel durations: each kernel alone, back to back in a graph, on the
    # same stream and over the same rotating inputs
    d_mask, d_attn, d_ver, d_attn_step = per_kernel_graph_times(st, stream, chunk)
    _, w_attn, w_ver, _ = per_kernel_graph_times(st, stream, chunk, rotate=False)
    kernel_timing = ("each kernel kind timed alone: a CUDA graph of %d launches over the rotating "
                     "inputs, CUDA events on the launching stream" % chunk)

    elapsed_ms, value = combine_over_ranks(elapsed_ms, w.T, K, world, "cuda")
    ms_per_step = elapsed_ms / K
    peak, peak_kind = measured_peaks()
    ab, vb, mb = attn_bytes(w), verify_bytes(w), mask_bytes(w)
    attn_ms = float(d_attn.mean())
    ver_ms = float(d_ver.mean())
    mask_ms = float(d_mask.mean())
    achieved = ab / (attn_ms * 1e-3) / 1e9
    # the roofline block describes the kernel that takes the larger share of the step
    if ver_ms > attn_ms:
        kname = (("tree_verify_reg_kernel" if w.V <= 131072 else "tree_verify_cluster_kernel")
                 if w.temperature > 0 else "tree_verify_greedy_node_kernel")
        roof = {"bound": "hbm", "kernel": kname, "achieved": vb / (ver_ms * 1e-3) / 1e9, "peak": peak,
                "unit": "GB/s", "traffic": profiled_traffic(f"tree_verify_{args.workload}"),
                "algorithmic_bytes": vb, "launch_ms": ver_ms,
                "peak_kind": f"{peak_kind} (STREAM-style copy, burst)"}
    else:
        if w.q.dtype == torch.float32:
            kname = "tree_attn_f32_kernel"
        elif os.environ.get("SPEC_TREE_ATTN_KERNEL") == "mma":
            kname = "tree_attn_mma_kernel"
        else:
            kname = "tree_attn_tc_kernel"
        roof = {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peak, "unit": "GB/s",
                "traffic": profiled_traffic(f"tree_attn_{args.workload}"), "algorithmic_bytes": ab,
                "launch_ms": attn_ms, "peak_kind": f"{peak_kind} (STREAM-style copy, burst)"}
        fl = attn_flops(w)
        if fl / ab > 300:
            # a contraction with this many flops per byte is bound by the tensor pipe
            tpeak, tkind = measured_peaks("bf16")
            roof.update({"bound": "tensor", "achieved": fl / (attn_ms * 1e-3) / 1e12, "peak": tpeak,
                         "unit": "TFLOP/s", "algorithmic_flops": fl,
                         "peak_kind": f"{tkind} (cuBLAS bf16 GEMM, burst)"})
    roof["frac"] = roof["achieved"] / roof["peak"]

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if w.q.dtype == torch.float32 else "bf16",
        "data": "synthetic (seeded; no datasets or weights)",
        "config": {"workload": describe(args.workload, args.temperature, args.prefix), "T": w.T, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "prefix": int(w.prefix_lens[0]), "V": w.V, "temperature": w.temperature,
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs rotate over {copies} device copies ({copies * per_copy / 1e6:.0f} MB > 4x L2)",
                   "launch": f"CUDA graph of {chunk} steps, replayed"},
        "roofline": roof,
        "kernels": {
            "mask": {"ms": mask_ms, "bytes": mb},
            "attn": {"ms": attn_ms, "bytes": ab, "gbs": achieved, "plan": "whole GPU"},
            "attn_in_step": {"ms": float(d_attn_step.mean()), "max_ctas": st.attn_ctas,
                             "note": "the step's launch: ancestor sets from the parents, "
                                     "planned for the SMs verification leaves"},
            "verify": {"ms": ver_ms, "bytes": vb, "gbs": vb / (ver_ms * 1e-3) / 1e9},
            "step_gbs": (ab + vb + mb) / (ms_per_step * 1e-3) / 1e9,
            "step_frac": (ab + vb + mb) / (ms_per_step * 1e-3) / 1e9 / peak,
            "warm_l2": {"attn_ms": float(w_attn.mean()), "verify_ms": float(w_ver.mean()),
                        "note": "every launch reads one input copy, resident in L2; not the headline"},
        },
        "kernel_timing": kernel_timing,
        "gpu_launches": 3 * K,
        "clocks": clocks, "clock_window": "timed region + 1 s soak of the same graph" if soak else "timed region",
    }
    result.update(derived_rates(st, stream, ms_per_step, mask_ms, attn_ms, ver_ms,
                                layers=MODEL_LAYERS.get(args.workload, 32)))
    if args.workload == WORKLOAD:
        # the rows after the hot path, on the headline workload's shapes
        result["next_rows"] = {"kv_compact": time_kv_compact(st, stream, chunk),
                               "tree_build": time_tree_build(w, stream, chunk),
                               "top_p": time_verify_top_p(st, stream, chunk),
                               "tree_merge": time_tree_merge(st, stream, chunk)}
    if not args.no_e2e:
        result["e2e"] = run_e2e(st, w, stream, args.e2e_steps)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w)
    return result


def combine_over_ranks(elapsed_ms: float, units_per_step: int, steps: int, world: int, device):
    """Whole-job throughput of independent replicas: every rank processed
    ``units_per_step`` units per step, and the job took as long as the slowest
    rank.  Returns (max elapsed ms over ranks, units of all ranks / that time)."""
    if world > 1:
        import torch
        t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    return elapsed_ms, world * units_per_step * steps / (elapsed_ms / 1e3)


def deepest_paths(w):
    """Per request, the root-to-leaf path of a deepest node (request-local
    indices, -1 padded) and its length: the most a step can accept."""
    W = w.max_depth + 1
    pn = np.full((w.B, W), -1, np.int32)
    acc = np.zeros(w.B, np.int32)
    for b in range(w.B):
        lo, hi = w.offsets[b], w.offsets[b + 1]
        par = w.parents[lo:hi]
        depth = np.zeros(hi - lo, np.int32)
        for i in range(1, hi - lo):
            depth[i] = depth[par[i]] + 1
        x = int(np.argmax(depth))
        path = [x]
        while path[-1] != 0:
            path.append(int(par[path[-1]]))
        path = path[::-1]
        pn[b, :len(path)] = path
        acc[b] = len(path) - 1
    return pn, acc


def time_kv_compact(st, stream, n, reps=3):
    """The depth-first KV-cache update after verification, timed alone: a graph
    of n launches over the rotating caches, each moving the deepest accepted
    path a step can produce (2 x acc x Hkv rows of D elements per request, each
    read once and written once)."""
    import torch
    ttv, w = st.ttv, st.w
    pn_h, acc_h = deepest_paths(w)
    pn, acc = torch.as_tensor(pn_h).cuda(), torch.as_tensor(acc_h).cuda()
    newp = torch.empty(w.B, dtype=torch.int32, device="cuda")
    kst = torch.zeros(w.B, dtype=torch.int32, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            c = st.copies[i % len(st.copies)]
            ttv.kv_compact(c["k"], c["v"], st.pl, st.off, pn, acc, kst, new_prefix_lens=newp)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        best = ms if best is None else min(best, ms)
    if (kst.cpu().numpy() != 0).any():
        raise RuntimeError(f"kv_compact status {kst.cpu().tolist()}")
    moved = int(acc_h.sum()) * w.Hkv * w.D * w.k_cache.element_size() * 2 * 2
    return {"us": best * 1e3, "accept_len": acc_h.tolist(), "bytes": moved,
            "gbs": moved / (best * 1e-3) / 1e9,
            "timing": f"CUDA graph of {n} launches, events on the launching stream"}


def time_tree_merge(st, stream, n, reps=3):
    """Merging an n-gram speculator's chain into the step's draft tree (the
    mixed speculation of the developer article's deployment notes), timed
    alone: a graph of n launches.  The chain follows the tree's first path
    for two tokens, then leaves it for three new ones."""
    import torch
    ttv, w = st.ttv, st.w
    par_a, tok_a = st.par, st.tok
    path = [0]
    for i in range(1, w.T):
        if w.parents[i] == path[-1]:
            path.append(i)
    chain_tok = [0] + [int(w.tokens[i]) for i in path[1:3]] + [int(w.V) - 1 - j for j in range(3)]
    par_b = torch.tensor([-1] + list(range(len(chain_tok) - 1)), dtype=torch.int32, device="cuda")
    tok_b = torch.tensor(chain_tok, dtype=torch.int32, device="cuda")
    off_b = torch.tensor([0, len(chain_tok)], dtype=torch.int32, device="cuda")
    mst = torch.zeros(w.B, dtype=torch.int32, device="cuda")
    if w.B != 1:
        return None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(n):
            out = ttv.tree_merge(par_a, tok_a, st.off, par_b, tok_b, off_b, mst)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        best = ms if best is None else min(best, ms)
    if (mst.cpu().numpy() != 0).any():
        raise RuntimeError(f"tree_merge status {mst.cpu().tolist()}")
    return {"us": best * 1e3, "nodes": int(out["n_out"][0].item()),
            "shape": f"{w.T}-node draft tree + a {len(chain_tok)}-node n-gram chain",
            "timing": f"CUDA graph of {n} launches, events on the launching stream"}


def time_verify_top_p(st, stream, n, reps=3, top_p=0.9):
    """Stochastic verification with both distributions filtered to their
    top_p nucleus, timed alone like the step's verify kernel: a graph of n
    launches over the rotating logits copies."""
    import torch
    ttv, w = st.ttv, st.w
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            c = st.copies[i % len(st.copies)]
            ttv.tree_verify(c["tl"], c["dl"], st.tok, st.par, st.off, w.temperature, st.seed + i,
                            st.W, st.status, st.ws, outputs=st.outs, top_p=top_p)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        best = ms if best is None else min(best, ms)
    if (st.status.cpu().numpy() != 0).any():
        raise RuntimeError(f"verify status {st.status.cpu().tolist()}")
    rows = verify_bytes(w)
    return {"us": best * 1e3, "top_p": top_p, "bytes": rows, "gbs": rows / (best * 1e-3) / 1e9,
            "timing": f"CUDA graph of {n} launches, events on the launching stream"}


def time_tree_build(w, stream, n, reps=3):
    """Draft-tree construction for the workload's tree shape (width 5, depth 3,
    pruned to 64 nodes), timed alone: the last expansion level (25 frontier
    rows of the vocabulary, 5 i.i.d. draws each, reading 25 draft rows) and
    the pruning of the 156 candidates."""
    import torch
    import token_tree_verification_gb300 as ttv
    gen = torch.Generator(device="cuda")
    gen.manual_seed(7)
    Fr, width, cand = 25, 5, 156
    rows = [torch.randn((Fr, w.V), generator=gen, device="cuda") * 3 for _ in range(8)]
    ps = torch.zeros(Fr, device="cuda")
    nodes = torch.arange(6, 6 + Fr, dtype=torch.int32, device="cuda")
    reqs = torch.zeros(Fr, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(3)
    par = np.array([-1] + [(i - 1) // width for i in range(1, cand)], np.int32)
    sc = np.zeros(cand, np.float32)
    for i in range(1, cand):
        sc[i] = sc[par[i]] + np.float32(np.log(rng.uniform(1e-3, 1.0)))
    par_d = torch.as_tensor(par).cuda()
    tok_d = torch.as_tensor(rng.integers(0, w.V, cand).astype(np.int32)).cuda()
    sc_d = torch.as_tensor(sc).cuda()
    off_d = torch.tensor([0, cand], dtype=torch.int32, device="cuda")
    pst = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = {}
    for kind in ("expand", "prune"):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                if kind == "expand":
                    ttv.tree_expand(rows[i % len(rows)], ps, nodes, reqs, width, 0.7, i)
                else:
                    ttv.tree_prune(par_d, tok_d, sc_d, off_d, 64, pst)
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / n
            best = ms if best is None else min(best, ms)
        out[kind + "_us"] = best * 1e3
    if (pst.cpu().numpy() != 0).any():
        raise RuntimeError("tree_prune status")
    out["expand_bytes"] = Fr * w.V * 4
    out["expand_gbs"] = out["expand_bytes"] / (out["expand_us"] * 1e-6) / 1e9
    out["shape"] = "expand: 25 frontier rows x V, width 5, T=0.7; prune: 156 candidates -> 64"
    return out


def per_kernel_graph_times(st, stream, n, reps=3, rotate=True):
    """Mean duration per launch of each kernel kind, from a graph of n
    back-to-back launches of that kernel alone (best of `reps` replays).
    With ``rotate`` the launches cycle through the device input copies (cold
    L2); without it every launch reads the first copy, which then stays in
    L2 (warm)."""
    import torch
    ttv, w = st.ttv, st.w
    out = []
    for kind in range(4):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                c = st.copies[i % len(st.copies) if rotate else 0]
                if kind == 0:
                    ttv.build_tree_mask(st.par, st.off, st.status, mask=st.mask, depth=st.depth)
                elif kind == 1:
                    # planned for the whole GPU, from the mask array
                    ttv.tree_attn(c["q"], c["k"], c["v"], st.pl, st.off, st.mask, st.max_prefix,
                                  st.status, o=st.o, workspace=st.ws_attn)
                elif kind == 3:
                    # as the step launches it: from the parents, for the SMs verification leaves
                    ttv.tree_attn(c["q"], c["k"], c["v"], st.pl, st.off, None, st.max_prefix,
                                  st.status, o=st.o, workspace=st.ws_attn, max_ctas=st.attn_ctas,
                                  parents=st.par)
                else:
                    ttv.tree_verify(c["tl"], c["dl"], st.tok, st.par, st.off, w.temperature,
                                    st.seed + i, st.W, st.status, st.ws, outputs=st.outs)
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / n
            best = ms if best is None else min(best, ms)
        out.append(np.full(n, best))
    return out


def derived_rates(st, stream, ms_per_step, mask_ms, attn_ms, ver_ms, samples=64, layers=32):
    """Two rates derived from the measured times.  Accepted tokens/s: the mean
    over ``samples`` seeds of the tokens a step emits (accepted tokens plus
    the bonus token of every request) divided by the timed step.  Model-shaped
    tree tokens/s: a ``layers``-layer model runs the tree attention once per
    layer and the mask and verification once per step, so its step costs
    layers x attention + mask + verification (each kernel's own graph-timed
    mean)."""
    import torch
    w = st.w
    hist = torch.empty((samples, w.B), dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        for i in range(samples):
            st.run(i)
            hist[i].copy_(st.outs["accept_len"])
    torch.cuda.synchronize()
    if (st.status.cpu().numpy() != 0).any():
        raise RuntimeError(f"device status {st.status.cpu().tolist()}")
    acc = hist.cpu().numpy().astype(np.float64)
    emitted = float((acc + 1).sum(axis=1).mean())
    model_ms = layers * attn_ms + mask_ms + ver_ms
    return {
        "accepted": {"value": emitted / (ms_per_step * 1e-3), "unit": "emitted tokens/s",
                     "mean_accept_len": float(acc.mean()), "mean_emitted_per_step": emitted,
                     "samples": samples,
                     "note": "accepted + bonus tokens per step (mean over seeds) / timed step"},
        "model_shaped": {"value": w.T / (model_ms * 1e-3), "unit": UNIT, "layers": layers,
                         "ms_per_step": model_ms,
                         "note": f"{layers} x attention + mask + verification, per-kernel graph times"},
    }


def run_e2e(st, w, stream, steps):
    """Same metric through the public API with host buffers: every step copies
    all of its inputs (Q, K/V caches, target and draft logits, tree arrays)
    from pinned host memory and reads the verified tokens back.  The inputs sit
    in one pinned buffer (each at a 256-byte aligned offset), copied in two
    halves on two copy streams into the other of two device input buffers while
    step i's kernels run, as a serving loop would overlap them; the timed region
    spans every copy and every step.  The four outputs come back as one copy,
    since every copy pays a fixed start-up cost on the host-device link."""
    import torch
    ttv = st.ttv
    names = [k for k, v in st.copies[0].items() if v is not None]
    tree_parts = [("par", st.par), ("off", st.off), ("tok", st.tok), ("pl", st.pl)]
    parts = [(k, st.copies[0][k]) for k in names] + tree_parts
    # every input of a step at a 256-byte aligned offset of one byte buffer:
    # one pinned host buffer, two device buffers (double-buffered inputs)
    layout, at = [], 0
    for k, t in parts:
        nb = t.numel() * t.element_size()
        layout.append((k, at, nb, t.dtype, tuple(t.shape)))
        at = (at + nb + 255) // 256 * 256
    total = at

    def views(buf):
        return {k: buf[off:off + nb].view(dt).view(sh) for k, off, nb, dt, sh in layout}

    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    hv = views(host_buf)
    for k, t in parts:
        hv[k].copy_(t.cpu())
    dev_bufs = [torch.empty(total, dtype=torch.uint8, device="cuda") for _ in range(2)]
    sets = [views(b) for b in dev_bufs]
    # the outputs as views of one device buffer, read back with one copy
    shapes = [(k, tuple(v.shape)) for k, v in st.outs.items()]
    n_out = sum(int(np.prod(sh)) for _, sh in shapes)
    out_dev = torch.empty(n_out, dtype=torch.int32, device="cuda")
    outs, at = {}, 0
    for k, sh in shapes:
        n = int(np.prod(sh))
        outs[k] = out_dev[at:at + n].view(sh)
        at += n
    out_host = [torch.empty(n_out, dtype=torch.int32).pin_memory() for _ in range(2)]
    h2d = total
    d2h = out_dev.numel() * out_dev.element_size()
    cs = [torch.cuda.Stream(), torch.cuda.Stream()]
    # the buffer in two halves, one per copy stream (split on a 256-byte boundary)
    half = (total // 2 + 255) // 256 * 256
    ranges = [(0, half), (half, total)]
    free = [torch.cuda.Event() for _ in range(2)]

    def copy_in(i):
        dst = dev_bufs[i % 2]
        done = [torch.cuda.Event(), torch.cuda.Event()]
        for lane in range(2):
            cs[lane].wait_event(free[i % 2])
            a, b = ranges[lane]
            with torch.cuda.stream(cs[lane]):
                dst[a:b].copy_(host_buf[a:b], non_blocking=True)
            done[lane].record(cs[lane])
        stream.wait_event(done[0])
        stream.wait_event(done[1])

    def compute(i):
        d = sets[i % 2]
        with torch.cuda.stream(stream):
            st.launch(d["q"], d["k"], d["v"], d["tl"], d.get("dl"), d["par"], d["off"], d["tok"],
                      d["pl"], st.seed + i, outs, stream)
            free[i % 2].record(stream)
            out_host[i % 2].copy_(out_dev, non_blocking=True)

    def run_steps(n):
        for j in range(2):
            free[j].record(stream)
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)    # overlaps step i on the compute stream
            compute(i)

    run_steps(3)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for lane in range(2):
        cs[lane].wait_event(e0)
    run_steps(steps)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # the last step's tokens, as read back, equal the device path's for its seed
    if (st.status.cpu().numpy() != 0).any():
        raise RuntimeError(f"device status {st.status.cpu().tolist()}")
    last = out_host[(steps - 1) % 2].clone()
    with torch.cuda.stream(stream):
        st.run(steps - 1)
    torch.cuda.synchronize()
    ref = torch.cat([v.reshape(-1).cpu() for v in st.outs.values()])
    if not torch.equal(last, ref):
        raise RuntimeError("end-to-end outputs differ from the device path")
    return {"value": w.T / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms, "steps": steps,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipeline": ("every input of a step in one pinned buffer, copied in two halves on two "
                         "copy streams into double-buffered device inputs, overlapping the previous "
                         "step; outputs read back in one copy")}


# --------------------------------------------------------------------------
# the oracle as CPU baseline / reference arm
# --------------------------------------------------------------------------
class OracleInputs:
    def __init__(self, w):
        self.w = w
        self.q = w.q.float().cpu().numpy()
        self.k = w.k_cache.float().cpu().numpy()
        self.v = w.v_cache.float().cpu().numpy()


def oracle_step_time(oi, nsel: int, seed: int):
    """Wall time of one oracle step on a bounded sample: the full mask, the
    full verification walk, and attention for ``nsel`` seeded (node, head)
    rows, scaled to all rows."""
    import oracle
    w, q, k, v = oi.w, oi.q, oi.k, oi.v
    n_rows = w.T * w.Hq
    rng = np.random.default_rng(seed)
    nsel = max(1, min(n_rows, nsel))
    rows = np.sort(rng.choice(n_rows, size=nsel, replace=False)).astype(np.int64)
    t0 = time.perf_counter()
    oracle.build_mask(w.parents, w.offsets)
    t1 = time.perf_counter()
    oracle.tree_attn(q, k, v, w.prefix_lens, w.offsets, w.parents, rows=rows)
    t2 = time.perf_counter()
    oracle.tree_verify(w.target_logits, w.draft_logits, w.tokens, w.parents, w.offsets,
                       w.temperature, seed, w.max_depth + 1)
    t3 = time.perf_counter()
    return (t1 - t0) + (t2 - t1) * (n_rows / nsel) + (t3 - t2), nsel, n_rows


def cpu_baseline(w, nsel=512):
    import oracle
    oracle.build()
    t, nsel, n_rows = oracle_step_time(OracleInputs(w), nsel, 0)
    return {"value": w.T / t, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"one step: full mask and verification walk, attention on {nsel} of {n_rows} "
                      f"(node, head) rows scaled to all rows; plain C fp64, 1 thread",
            "host_cores": os.cpu_count()}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step a bounded sample of the
    same workload, timed on the host cores (rank 0 only)."""
    if rank != 0:
        return None
    import oracle
    from token_tree_verification_gb300 import synthetic
    oracle.build()
    w = synthetic.make_workload(args.workload, seed=0, device="cpu", pad=0.0,
                                temperature=args.temperature, **prefix_override(args))
    oi = OracleInputs(w)
    n_rows = w.T * w.Hq
    # size each step's attention sample so that K + W steps take ~2 minutes
    t_row = oracle_step_time(oi, 64, 999)[0] / n_rows      # scaled time per row
    budget = 120.0 / max(1, args.steps + args.warmup)
    nsel = int(max(1, min(n_rows, budget / max(t_row, 1e-9) * 0.5)))
    for i in range(args.warmup):
        oracle_step_time(oi, nsel, 100 + i)
    times = [oracle_step_time(oi, nsel, i)[0] for i in range(args.steps)]
    ms = 1e3 * float(np.mean(times))
    value = w.T / (ms * 1e-3)
    sample = (f"each step: full mask and verification walk, attention on {nsel} "
              f"of {n_rows} (node, head) rows scaled to all rows; plain C fp64, 1 thread")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(args.workload, args.temperature, args.prefix),
                       "parallelism": "1 host thread"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def relaunch_ranks(n: int, argv: list) -> int:
    """Run this script as ``n`` local ranks (one per GPU) under
    torch.distributed.run on 127.0.0.1 and return its exit code; rank 0
    prints the job's line."""
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs of this node, one independent replica each; without torchrun's "
                         "environment the script starts the ranks itself")
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--graph-steps", type=int, default=200)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(WORKLOADS),
                    help="the workload to time (default: the headline LLaMA-7B-shaped step)")
    ap.add_argument("--prefix", type=int, default=None,
                    help="KV prefix length (every workload but the dynamic batch); default: the workload's own")
    ap.add_argument("--temperature", type=float, default=None,
                    help="verification temperature (0 = greedy); default: the workload's own")
    ap.add_argument("--eager", action="store_true",
                    help="plain stream launches without graphs or timing (for profilers)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "native":
        args.warmup = 3

    if args.gpus < 1:
        raise SystemExit("--gpus must be at least 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # one process per GPU: start the ranks under torch.distributed.run
        raise SystemExit(relaunch_ranks(args.gpus, sys.argv[1:]))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit(f"WORLD_SIZE={world} disagrees with --gpus {args.gpus}")
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_native(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
