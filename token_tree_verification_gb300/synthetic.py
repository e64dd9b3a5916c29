"""Seeded synthetic workloads for tree attention + verification.

This module is the one piece shared by the CUDA path's tests/benchmark and the
CPU oracle: it only draws inputs.  It contains none of the verification
method's arithmetic (no masks, no attention, no acceptance rule).  The only
arithmetic here plays the *draft model*: it samples each node's children from
the draft distribution softmax(draft/T) and, for the LLaMA-7B-shaped tree,
keeps the 63 speculated nodes of highest cumulative draft log-probability.

Shapes follow the model shapes named in the SpecInfer pages (LLaMA-7B target;
LLaMA-2-70B with 8 KV heads) and the tree knobs of the SpecInfer developer
article §4.1 config (tree_width 5, max_depth 3, temperature 0.7).  The value
distributions are this library's own choices (the pages give none):

    Q, K, V ~ N(0, 1) * 0.5 (bf16), or N(0, 1) fp32 for the tiny case
    target logits ~ N(0, sigma_t^2), draft = target + N(0, sigma_d^2)

Tree topology, token choice and logits use numpy PCG64; dense Q/K/V use a
seeded ``torch.Generator`` on the requested device so multi-GB caches can be
drawn directly in device memory.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

CONFIGS = ("tiny", "llama7b", "dynamic", "llama70b_gqa", "long_chain", "long_tree")


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    S_cap: int
    V: int
    temperature: float
    seed: int
    prefix_lens: np.ndarray      # [B] int32
    offsets: np.ndarray          # [B+1] int32
    parents: np.ndarray          # [T] int32, request-local, parent[0] = -1
    tokens: np.ndarray           # [T] int32, root token unused
    q: torch.Tensor              # [T, Hq, D]
    k_cache: torch.Tensor        # [B, Hkv, S_cap, D]
    v_cache: torch.Tensor        # [B, Hkv, S_cap, D]
    target_logits: np.ndarray    # [T, V] float32
    draft_logits: np.ndarray | None  # [T, V] float32 (None for greedy-only workloads)
    max_depth: int

    @property
    def T(self) -> int:
        return int(self.offsets[-1])

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def node_counts(self) -> np.ndarray:
        return np.diff(self.offsets)


# --------------------------------------------------------------------------
# tree topologies
# --------------------------------------------------------------------------

def random_tree(rng: np.random.Generator, n: int, depth: int, width: int | None) -> np.ndarray:
    """Random rooted tree of ``n`` nodes (root included) of exactly ``depth``
    levels below the root.  A spine guarantees every depth; every other node
    picks a uniform depth among those with room and a parent uniformly among
    the nodes one level up that have fewer than ``width`` children.  Nodes are
    returned in breadth-first order, so parent[i] < i."""
    assert n >= depth + 1
    node_depth = [0]
    parent = [-1]
    nchild = [0]
    by_depth: list[list[int]] = [[0]] + [[] for _ in range(depth)]

    def add(d: int, p: int):
        idx = len(node_depth)
        node_depth.append(d)
        parent.append(p)
        nchild.append(0)
        nchild[p] += 1
        by_depth[d].append(idx)

    for d in range(1, depth + 1):          # the spine
        add(d, by_depth[d - 1][-1])
    while len(node_depth) < n:
        open_depths = [d for d in range(1, depth + 1)
                       if any(width is None or nchild[p] < width for p in by_depth[d - 1])]
        if not open_depths:
            raise ValueError("tree too large for the given width and depth")
        d = int(rng.choice(open_depths))
        cands = [p for p in by_depth[d - 1] if width is None or nchild[p] < width]
        add(d, int(rng.choice(cands)))
    # breadth-first renumbering (stable within a depth)
    order = sorted(range(n), key=lambda i: (node_depth[i], i))
    new_id = {old: new for new, old in enumerate(order)}
    out = np.empty(n, dtype=np.int32)
    for new, old in enumerate(order):
        out[new] = -1 if parent[old] < 0 else new_id[parent[old]]
    return out


def chain_tree(n: int) -> np.ndarray:
    return np.arange(-1, n - 1, dtype=np.int32)


def tree_depth(parents: np.ndarray) -> int:
    d = np.zeros(parents.size, dtype=np.int64)
    for i in range(1, parents.size):
        d[i] = d[parents[i]] + 1
    return int(d.max())


# --------------------------------------------------------------------------
# the draft model's part: choose children tokens
# --------------------------------------------------------------------------

def _draft_probs(draft_row: np.ndarray, temperature: float) -> np.ndarray:
    z = draft_row.astype(np.float64) / max(temperature, 1e-6)
    z -= z.max()
    e = np.exp(z)
    return e / e.sum()


def draw_children_tokens(rng, parents, draft_logits, temperature, mode: str) -> np.ndarray:
    """Tokens proposed by the draft for every non-root node.  ``iid``: each
    child of u is an independent sample of softmax(draft_u / T); ``topk``: the
    children of u take u's most likely draft tokens in order (greedy draft)."""
    n = parents.size
    tokens = np.zeros(n, dtype=np.int32)
    children: dict[int, list[int]] = {}
    for i in range(1, n):
        children.setdefault(int(parents[i]), []).append(i)
    for u, cs in children.items():
        if mode == "iid":
            pr = _draft_probs(draft_logits[u], temperature)
            tokens[cs] = rng.choice(pr.size, size=len(cs), p=pr)
        else:
            order = np.argsort(-draft_logits[u], kind="stable")
            tokens[cs] = order[: len(cs)]
    return tokens


def _logits(rng, n, V, sigma_t, sigma_d, with_draft=True):
    tgt = (rng.standard_normal((n, V), dtype=np.float32) * np.float32(sigma_t)).astype(np.float32)
    if not with_draft:
        return tgt, None
    drf = (tgt + rng.standard_normal((n, V), dtype=np.float32) * np.float32(sigma_d)).astype(np.float32)
    return tgt, drf


def pruned_beam_tree(rng, width, depth, keep, V, sigma_t, sigma_d, temperature):
    """Full ``width``-ary tree of ``depth`` levels whose children are i.i.d.
    draft samples, pruned to the root plus the ``keep - 1`` nodes with the
    highest cumulative draft log-probability (ties to the lower breadth-first
    index).  Scores never increase along a path, so the kept set is closed
    under ancestors.  Returns parents, tokens, target rows, draft rows."""
    parents = [-1]
    lvl = [0]
    for d in range(depth):
        nxt = []
        for p in lvl:
            for _ in range(width):
                parents.append(p)
                nxt.append(len(parents) - 1)
        lvl = nxt
    parents = np.asarray(parents, dtype=np.int32)
    n = parents.size
    tgt, drf = _logits(rng, n, V, sigma_t, sigma_d)
    tokens = draw_children_tokens(rng, parents, drf, temperature, "iid")
    score = np.zeros(n, dtype=np.float64)
    for i in range(1, n):
        pr = _draft_probs(drf[parents[i]], temperature)
        score[i] = score[parents[i]] + math.log(max(pr[tokens[i]], 1e-300))
    order = sorted(range(1, n), key=lambda i: (-score[i], i))
    kept = sorted([0] + order[: keep - 1])
    remap = {old: new for new, old in enumerate(kept)}
    par = np.array([-1] + [remap[int(parents[o])] for o in kept[1:]], dtype=np.int32)
    return par, tokens[kept].astype(np.int32), tgt[kept], drf[kept]


# --------------------------------------------------------------------------
# dense tensors
# --------------------------------------------------------------------------

def _randn(shape, gen, device, dtype, scale):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(dtype)


def _fill_caches(B, Hkv, S_cap, D, lens, gen, device, dtype, scale, pad):
    """K/V caches with slots [0, L_b + N_b) drawn and the rest set to ``pad``
    (NaN by default: a kernel that lets a slot outside the request's keys into
    its sums returns NaN)."""
    k = torch.empty((B, Hkv, S_cap, D), device=device, dtype=dtype)
    v = torch.empty((B, Hkv, S_cap, D), device=device, dtype=dtype)
    for b in range(B):
        n = int(lens[b])
        k[b, :, :n] = _randn((Hkv, n, D), gen, device, dtype, scale)
        v[b, :, :n] = _randn((Hkv, n, D), gen, device, dtype, scale)
        if n < S_cap:
            k[b, :, n:] = pad
            v[b, :, n:] = pad
    return k, v


def make_workload(name: str, seed: int = 0, device: str | torch.device = "cpu",
                  pad: float = float("nan"), temperature: float | None = None,
                  **overrides) -> Workload:
    """Build one of the named workloads (see ``CONFIGS``).  ``overrides`` may
    shrink sizes for fast tests (B, L, V, D, Hq, Hkv, N, depth, width)."""
    rng = np.random.default_rng(seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    o = overrides

    if name == "tiny":
        B, Hq, Hkv, D, V = o.get("B", 1), o.get("Hq", 4), o.get("Hkv", 4), o.get("D", 64), o.get("V", 1000)
        L = o.get("L", 128)
        temp = 1.0 if temperature is None else temperature
        trees = [random_tree(rng, o.get("N", 8), o.get("depth", 3), o.get("width", 3)) for _ in range(B)]
        lens = np.full(B, L, dtype=np.int32)
        dtype, scale, sig = torch.float32, 1.0, (2.0, 1.0)
        child_mode = "iid"
        logit_rows = None
    elif name == "llama7b":
        B, Hq, Hkv, D, V = o.get("B", 1), o.get("Hq", 32), o.get("Hkv", 32), o.get("D", 128), o.get("V", 32000)
        L = o.get("L", 2048)
        temp = 0.7 if temperature is None else temperature
        trees, logit_rows, toks = [], [], []
        for _ in range(B):
            par, tk, tg, dr = pruned_beam_tree(rng, o.get("width", 5), o.get("depth", 3), o.get("N", 64),
                                               V, 3.0, 1.5, 0.7)
            trees.append(par); toks.append(tk); logit_rows.append((tg, dr))
        lens = np.full(B, L, dtype=np.int32)
        dtype, scale, sig = torch.bfloat16, 0.5, (3.0, 1.5)
        child_mode = "given"
    elif name == "dynamic":
        B, Hq, Hkv, D, V = o.get("B", 16), o.get("Hq", 32), o.get("Hkv", 32), o.get("D", 128), o.get("V", 32000)
        lo, hi = o.get("L_range", (512, 4096))
        nlo, nhi = o.get("N_range", (16, 96))
        dlo, dhi = o.get("depth_range", (2, 5))
        temp = 0.0 if temperature is None else temperature
        lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
        trees = []
        for _ in range(B):
            n = int(rng.integers(nlo, nhi + 1))
            dep = int(rng.integers(dlo, dhi + 1))
            trees.append(random_tree(rng, n, dep, None))
        dtype, scale, sig = torch.bfloat16, 0.5, (3.0, 1.5)
        child_mode = "topk"
        logit_rows = None
    elif name == "llama70b_gqa":
        B, Hq, Hkv, D, V = o.get("B", 4), o.get("Hq", 64), o.get("Hkv", 8), o.get("D", 128), o.get("V", 32000)
        L = o.get("L", 8192)
        temp = 0.7 if temperature is None else temperature
        trees = [random_tree(rng, o.get("N", 128), o.get("depth", 5), o.get("width", 8)) for _ in range(B)]
        lens = np.full(B, L, dtype=np.int32)
        dtype, scale, sig = torch.bfloat16, 0.5, (3.0, 1.5)
        child_mode = "iid"
        logit_rows = None
    elif name in ("long_chain", "long_tree"):
        B, Hq, Hkv, D, V = o.get("B", 8), o.get("Hq", 32), o.get("Hkv", 32), o.get("D", 128), o.get("V", 32000)
        L = o.get("L", 32768)
        temp = 0.7 if temperature is None else temperature
        if name == "long_chain":
            trees = [chain_tree(o.get("N", 6)) for _ in range(B)]
        else:
            trees = [random_tree(rng, o.get("N", 128), o.get("depth", 6), o.get("width", 8)) for _ in range(B)]
        lens = np.full(B, L, dtype=np.int32)
        dtype, scale, sig = torch.bfloat16, 0.5, (3.0, 2.0)
        child_mode = "iid"
        logit_rows = None
    else:
        raise ValueError(f"unknown workload {name!r}; choose from {CONFIGS}")

    counts = np.array([t.size for t in trees], dtype=np.int32)
    offsets = np.zeros(B + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    T = int(offsets[-1])
    parents = np.concatenate(trees).astype(np.int32)

    if logit_rows is not None:
        target = np.concatenate([r[0] for r in logit_rows]).astype(np.float32)
        draft = np.concatenate([r[1] for r in logit_rows]).astype(np.float32)
        tokens = np.concatenate(toks).astype(np.int32)
    else:
        target, draft = _logits(rng, T, V, sig[0], sig[1])
        tokens = np.zeros(T, dtype=np.int32)
        sample_temp = temp if temp > 0 else 1.0
        for b in range(B):
            s, e = offsets[b], offsets[b + 1]
            tokens[s:e] = draw_children_tokens(rng, parents[s:e], draft[s:e], sample_temp, child_mode)
    if temp == 0.0 and name == "dynamic":
        draft = None          # greedy verification never reads draft rows

    lens_total = lens + counts
    align = 64
    S_cap = int(o.get("S_cap", int(math.ceil(lens_total.max() / align) * align)))
    q = _randn((T, Hq, D), gen, device, dtype, scale)
    k, v = _fill_caches(B, Hkv, S_cap, D, lens_total, gen, device, dtype, scale, pad)
    return Workload(name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, S_cap=S_cap, V=V, temperature=float(temp),
                    seed=seed, prefix_lens=lens.astype(np.int32), offsets=offsets, parents=parents,
                    tokens=tokens, q=q, k_cache=k, v_cache=v, target_logits=target,
                    draft_logits=draft, max_depth=max(tree_depth(t) for t in trees))
