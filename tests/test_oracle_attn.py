"""Pins for the oracle's step A2 (tree attention).

The SpecInfer developer article §2.1 gives tree attention as masked scores,
softmax, times V over the request's keys; the SpecInfer news write-up ("Token
樹驗證器", "研究現狀") says tree decoding generalises incremental decoding with
a KV cache.  Pins:
  * a chain-shaped tree equals ordinary causal incremental attention, computed
    by torch's scaled_dot_product_attention in float64 (library routine);
  * any tree equals SDPA with a mask built from networkx ancestor sets;
  * every root-to-leaf path run alone as a chain gives bit-identical rows;
  * a root-only tree equals single-token decode attention;
  * with an empty prefix the root's output is exactly its own value row."""
import networkx as nx
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from token_tree_verification_gb300 import synthetic


def make_case(rng, trees, prefix, Hq, Hkv, D, pad=np.nan):
    B = len(trees)
    off = np.zeros(B + 1, dtype=np.int32)
    off[1:] = np.cumsum([t.size for t in trees])
    T = int(off[-1])
    par = np.concatenate(trees).astype(np.int32)
    L = np.asarray(prefix, dtype=np.int32)
    S_cap = int((L + np.diff(off)).max()) + 3
    q = rng.standard_normal((T, Hq, D)).astype(np.float32)
    k = np.full((B, Hkv, S_cap, D), pad, dtype=np.float32)
    v = np.full((B, Hkv, S_cap, D), pad, dtype=np.float32)
    for b in range(B):
        n = L[b] + trees[b].size
        k[b, :, :n] = rng.standard_normal((Hkv, n, D))
        v[b, :, :n] = rng.standard_normal((Hkv, n, D))
    return q, k, v, L, off, par


def sdpa_reference(q, k, v, L, off, par, visible_fn, scale=None):
    """float64 SDPA per request with a boolean visibility mask."""
    B, Hkv = k.shape[0], k.shape[1]
    T, Hq, D = q.shape
    G = Hq // Hkv
    out = np.zeros((T, Hq, D))
    for b in range(B):
        s, e = off[b], off[b + 1]
        n = e - s
        nk = L[b] + n
        vis = np.zeros((n, nk), dtype=bool)
        for i in range(n):
            vis[i] = visible_fn(b, i, L[b], nk)
        qb = torch.from_numpy(q[s:e].astype(np.float64)).permute(1, 0, 2)          # [Hq, n, D]
        kb = torch.from_numpy(k[b, :, :nk].astype(np.float64)).repeat_interleave(G, 0)
        vb = torch.from_numpy(v[b, :, :nk].astype(np.float64)).repeat_interleave(G, 0)
        o = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=torch.from_numpy(vis), scale=scale)
        out[s:e] = o.permute(1, 0, 2).numpy()
    return out


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2)])
def test_chain_equals_causal_incremental(Hq, Hkv):
    rng = np.random.default_rng(0)
    trees = [synthetic.chain_tree(4), synthetic.chain_tree(6), synthetic.chain_tree(1)]
    q, k, v, L, off, par = make_case(rng, trees, [5, 9, 3], Hq, Hkv, 16)
    got = oracle.tree_attn(q, k, v, L, off, par)
    ref = sdpa_reference(q, k, v, L, off, par, lambda b, i, Lb, nk: np.arange(nk) <= Lb + i)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_random_tree_equals_sdpa_with_networkx_mask():
    rng = np.random.default_rng(1)
    trees = [synthetic.random_tree(rng, 12, 3, 3), synthetic.random_tree(rng, 20, 4, None),
             synthetic.random_tree(rng, 1, 0, None)]
    q, k, v, L, off, par = make_case(rng, trees, [7, 0, 4], 4, 2, 8)
    anc = []
    for t in trees:
        g = nx.DiGraph([(int(t[i]), i) for i in range(1, t.size)])
        g.add_nodes_from(range(t.size))
        anc.append([nx.ancestors(g, i) | {i} for i in range(t.size)])

    def vis(b, i, Lb, nk):
        m = np.arange(nk) < Lb
        for a in anc[b][i]:
            m[Lb + a] = True
        return m
    got = oracle.tree_attn(q, k, v, L, off, par)
    np.testing.assert_allclose(got, sdpa_reference(q, k, v, L, off, par, vis), rtol=1e-11, atol=1e-12)
    # an explicit softmax scale is honoured, 1.0 included (the unscaled
    # scores of the developer article's tree_attention snippet)
    for sc in (0.3, 1.0):
        got2 = oracle.tree_attn(q, k, v, L, off, par, scale=sc)
        np.testing.assert_allclose(got2, sdpa_reference(q, k, v, L, off, par, vis, scale=sc),
                                   rtol=1e-11, atol=1e-12)


def test_each_path_alone_is_bit_identical():
    rng = np.random.default_rng(2)
    tree = synthetic.random_tree(rng, 24, 4, 4)
    q, k, v, L, off, par = make_case(rng, [tree], [11], 4, 4, 16)
    full = oracle.tree_attn(q, k, v, L, off, par)
    leaves = set(range(tree.size)) - set(tree[1:].tolist())
    for leaf in sorted(leaves):
        path = []
        a = leaf
        while a != -1:
            path.append(a)
            a = tree[a]
        path = path[::-1]
        n = len(path)
        slots = list(range(L[0])) + [L[0] + a for a in path]
        k1 = np.full((1, 4, len(slots) + 2, 16), np.nan, dtype=np.float32)
        v1 = np.full_like(k1, np.nan)
        k1[0, :, :len(slots)] = k[0][:, slots]
        v1[0, :, :len(slots)] = v[0][:, slots]
        o1 = oracle.tree_attn(q[path], k1, v1, L, np.array([0, n], np.int32), synthetic.chain_tree(n))
        assert np.array_equal(o1, full[path]), f"path to leaf {leaf}"


def test_root_only_is_decode_attention():
    rng = np.random.default_rng(3)
    q, k, v, L, off, par = make_case(rng, [synthetic.chain_tree(1)] * 2, [17, 1], 8, 4, 32)
    got = oracle.tree_attn(q, k, v, L, off, par)
    ref = sdpa_reference(q, k, v, L, off, par, lambda b, i, Lb, nk: np.ones(nk, dtype=bool))
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_empty_prefix_root_returns_its_value():
    rng = np.random.default_rng(4)
    tree = synthetic.random_tree(rng, 6, 2, 3)
    q, k, v, L, off, par = make_case(rng, [tree], [0], 4, 2, 8)
    got = oracle.tree_attn(q, k, v, L, off, par)
    for h in range(4):
        assert np.array_equal(got[0, h], v[0, h // 2, 0].astype(np.float64))


def test_selected_rows_match_full():
    rng = np.random.default_rng(5)
    tree = synthetic.random_tree(rng, 10, 3, 3)
    q, k, v, L, off, par = make_case(rng, [tree, tree], [6, 3], 4, 4, 8)
    full = oracle.tree_attn(q, k, v, L, off, par).reshape(-1, 8)
    rows = np.array([0, 5, 17, 39, 79], dtype=np.int64)
    assert np.array_equal(oracle.tree_attn(q, k, v, L, off, par, rows=rows), full[rows])
