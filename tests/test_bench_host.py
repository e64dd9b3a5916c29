"""Host-side logic of bench.py: the algorithmic bytes and flops behind the
roofline, counted here independently from the tree itself, and the workload
description and prefix override."""
import argparse
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from token_tree_verification_gb300 import synthetic  # noqa: E402


def _ancestors(par, i):
    out = [i]
    while par[out[-1]] >= 0:
        out.append(int(par[out[-1]]))
    return out


@pytest.fixture(scope="module", params=["tiny", "ragged"])
def w(request):
    if request.param == "tiny":
        return synthetic.make_workload("tiny", seed=0)
    return synthetic.make_workload("tiny", seed=5, B=3, L=77, N=20, depth=4, width=4, Hq=8, Hkv=2, D=128)


def test_attention_bytes_are_the_visible_slots_once_per_kv_head(w):
    el = w.q.element_size()
    touched = set()
    for b in range(w.B):
        lo, hi = w.offsets[b], w.offsets[b + 1]
        par = w.parents[lo:hi]
        L = int(w.prefix_lens[b])
        for i in range(hi - lo):
            for g in range(w.Hkv):
                touched.update((b, g, j) for j in range(L))
                touched.update((b, g, L + a) for a in _ancestors(par, i))
    expect = len(touched) * w.D * el * 2 + 2 * w.T * w.Hq * w.D * el   # K and V; Q in, O out
    assert bench.attn_bytes(w) == expect


def test_verify_bytes_count_target_rows_and_internal_draft_rows(w):
    internal = 0
    for b in range(w.B):
        lo, hi = w.offsets[b], w.offsets[b + 1]
        par = w.parents[lo:hi]
        internal += sum(1 for u in range(hi - lo) if any(par[c] == u for c in range(hi - lo)))
    assert bench.verify_bytes(w) == (w.T + internal) * w.V * 4
    w.temperature, t = 0.0, w.temperature
    try:
        assert bench.verify_bytes(w) == w.T * w.V * 4   # greedy reads no draft row
    finally:
        w.temperature = t


def test_attention_flops_count_each_rows_visible_keys(w):
    keys = 0
    for b in range(w.B):
        lo, hi = w.offsets[b], w.offsets[b + 1]
        par = w.parents[lo:hi]
        for i in range(hi - lo):
            keys += int(w.prefix_lens[b]) + len(_ancestors(par, i))
    assert bench.attn_flops(w) == 4 * w.D * w.Hq * keys


def test_description_follows_the_overrides():
    base = bench.WORKLOADS["llama7b"]
    assert bench.describe("llama7b", None) == base
    assert bench.describe("llama7b", 0.0).endswith(", greedy")
    assert bench.describe("llama7b", 1.0).endswith(", T=1 stochastic")
    d = bench.describe("long_tree", None, 4096)
    assert "KV prefix 4096" in d and "32768" not in d


def test_prefix_override():
    ns = argparse.Namespace(prefix=None, workload="llama7b")
    assert bench.prefix_override(ns) == {}
    ns.prefix = 448
    assert bench.prefix_override(ns) == {"L": 448}
    ns.workload = "dynamic"
    with pytest.raises(SystemExit):
        bench.prefix_override(ns)
