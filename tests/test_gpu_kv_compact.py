"""GPU parity of spec_kv_compact (the depth-first KV-cache update after
verification) against the oracle: bit-exact bytes, new prefix lengths and
status codes."""
import numpy as np
import pytest
import torch

import oracle
import token_tree_verification_gb300 as ttv
from parity import dev, gpu_verify
from token_tree_verification_gb300 import synthetic

pytestmark = pytest.mark.gpu


def _run(k, v, L, off, pn, acc, status=None):
    B = len(L)
    st = torch.as_tensor(np.zeros(B, np.int32) if status is None else status, dtype=torch.int32).cuda()
    kk, vv = k.clone().cuda(), v.clone().cuda()
    newp = ttv.kv_compact(kk, vv, dev(L, torch.int32), dev(off, torch.int32), dev(pn, torch.int32),
                          dev(acc, torch.int32), st)
    torch.cuda.synchronize()
    return kk.cpu(), vv.cpu(), newp.cpu().numpy(), st.cpu().numpy()


def _oracle(k, v, L, off, pn, acc, status=None):
    as_np = (lambda t: t.view(torch.int16).numpy()) if k.dtype == torch.bfloat16 else (lambda t: t.numpy())
    ko, newp, st = oracle.kv_compact(as_np(k), L, off, pn, acc, status)
    vo, _, _ = oracle.kv_compact(as_np(v), L, off, pn, acc, status)
    return ko, vo, newp, st


def _check(k, v, L, off, pn, acc, status=None):
    kg, vg, npg, stg = _run(k, v, L, off, pn, acc, status)
    ko, vo, npo, sto = _oracle(k, v, L, off, pn, acc, status)
    view = (lambda t: t.view(torch.int16).numpy()) if k.dtype == torch.bfloat16 else (lambda t: t.numpy())
    np.testing.assert_array_equal(stg, sto)
    np.testing.assert_array_equal(npg, npo)
    np.testing.assert_array_equal(view(kg), ko)
    np.testing.assert_array_equal(view(vg), vo)
    return npg


def test_after_verification_llama7b():
    w = synthetic.make_workload("llama7b", seed=2, L=300, Hq=8, Hkv=8)
    g = gpu_verify(w, 5)
    assert (g["status"] == 0).all()
    _check(w.k_cache, w.v_cache, w.prefix_lens, w.offsets, g["path_nodes"], g["accept_len"])


def test_accepting_trees_many_requests():
    # one-hot logits: every child accepted greedily -> long paths
    rng = np.random.default_rng(0)
    B, H, D, V = 5, 4, 128, 50
    w = synthetic.make_workload("dynamic", seed=7, B=B, Hq=H, Hkv=H, D=D, V=V, L_range=(20, 60),
                                N_range=(8, 40), depth_range=(2, 5))
    tgt = np.full((w.T, V), -30.0, np.float32)
    for b in range(B):
        lo, hi = w.offsets[b], w.offsets[b + 1]
        for i in range(lo, hi):
            kids = [c for c in range(i + 1, hi) if w.parents[c] == i - lo]
            tgt[i, w.tokens[kids[-1]] if kids else 0] = 10.0
    g = gpu_verify(w, 1, target=tgt, temperature=0.0)
    assert (g["status"] == 0).all() and g["accept_len"].max() >= 2
    _check(w.k_cache, w.v_cache, w.prefix_lens, w.offsets, g["path_nodes"], g["accept_len"])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_synthetic_paths_overlap_and_edges(dtype):
    rng = np.random.default_rng(4)
    B, H, S, D = 4, 3, 80, 64
    k = torch.randn(B, H, S, D).to(dtype)
    v = torch.randn(B, H, S, D).to(dtype)
    off = np.array([0, 9, 30, 31, 60], np.int32)
    L = np.array([3, 40, 0, 17], np.int32)
    W = 8
    pn = np.full((B, W), -1, np.int32)
    pn[0, :3] = [0, 2, 3]                 # overlapping source / destination
    pn[1, :8] = [0, 1, 5, 6, 9, 12, 18, 20]
    pn[2, :1] = [0]                       # a one-node tree
    pn[3, :4] = [0, 4, 10, 28]
    acc = np.array([2, 7, 0, 3], np.int32)
    _check(k, v, L, off, pn, acc)


def test_errors_and_skipped_requests():
    B, H, S, D = 4, 2, 40, 64
    k = torch.randn(B, H, S, D).to(torch.bfloat16)
    v = torch.randn(B, H, S, D).to(torch.bfloat16)
    off = np.array([0, 6, 12, 18, 24], np.int32)
    L = np.array([2, 2, 36, 2], np.int32)
    pn = np.array([[0, 3, 3, -1], [1, 2, -1, -1], [0, 1, -1, -1], [0, 1, 2, -1]], np.int32)
    acc = np.array([2, 1, 1, 2], np.int32)
    status = np.array([0, 0, 0, -9], np.int32)
    npg = _check(k, v, L, off, pn, acc, status)
    assert npg.tolist() == L.tolist()
