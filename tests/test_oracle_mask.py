"""Pins for the oracle's step A1 (ancestor-or-self mask and depth).

The SpecInfer news write-up ("Token 樹驗證器") and the SpecInfer developer
article §2.1 (tree_attention snippet, parent pointers) define the mask as the
ancestor relation of the token tree.  Pinned against networkx's ancestor sets
and shortest-path depths (an independent library routine), exhaustively for
every parent array with up to 7 nodes, and by invariants on random trees."""
import itertools

import networkx as nx
import numpy as np

import oracle
from token_tree_verification_gb300 import synthetic


def all_parent_arrays(n):
    ranges = [range(i) for i in range(1, n)]
    for choice in itertools.product(*ranges):
        yield np.array((-1,) + choice, dtype=np.int32)


def nx_mask_depth(par):
    g = nx.DiGraph()
    g.add_nodes_from(range(par.size))
    g.add_edges_from((int(par[i]), i) for i in range(1, par.size))
    n = par.size
    mask = np.zeros((n, 4), dtype=np.uint32)
    depth = np.zeros(n, dtype=np.int32)
    for i in range(n):
        for a in nx.ancestors(g, i) | {i}:
            mask[i, a // 32] |= np.uint32(1 << (a % 32))
        depth[i] = nx.shortest_path_length(g, 0, i)
    return mask, depth


def pack(trees):
    off = np.zeros(len(trees) + 1, dtype=np.int32)
    off[1:] = np.cumsum([t.size for t in trees])
    return np.concatenate(trees), off


def test_exhaustive_small_trees():
    for n in range(1, 8):
        trees = list(all_parent_arrays(n))
        par, off = pack(trees)
        mask, depth, status = oracle.build_mask(par, off)
        assert (status == 0).all()
        for b, t in enumerate(trees):
            m_ref, d_ref = nx_mask_depth(t)
            s, e = off[b], off[b + 1]
            np.testing.assert_array_equal(mask[s:e], m_ref)
            np.testing.assert_array_equal(depth[s:e], d_ref)
    assert len(list(all_parent_arrays(7))) == 720


def test_random_trees_invariants_and_networkx():
    rng = np.random.default_rng(1)
    trees = []
    for n, d, w in zip(rng.integers(1, 129, 40), rng.integers(1, 9, 40), [None, 3, 8, 16] * 10):
        d = int(min(d, n - 1))
        while w is not None and sum(w ** j for j in range(d + 1)) < n:
            d += 1
        trees.append(synthetic.random_tree(rng, int(n), d, w))
    par, off = pack(trees)
    mask, depth, status = oracle.build_mask(par, off)
    assert (status == 0).all()
    for b, t in enumerate(trees):
        s, e = off[b], off[b + 1]
        m, d = mask[s:e], depth[s:e]
        m_ref, d_ref = nx_mask_depth(t)
        np.testing.assert_array_equal(m, m_ref)
        np.testing.assert_array_equal(d, d_ref)
        bits = np.unpackbits(m.view(np.uint8), bitorder="little").reshape(t.size, 128)
        for i in range(t.size):
            assert bits[i, i] == 1                       # a node sees itself
            assert bits[i].sum() == d[i] + 1             # itself plus its ancestors
            assert not bits[i, i + 1:].any()             # only lower indices
            if i:
                assert (bits[i] >= bits[t[i]]).all()     # contains the parent's set


def test_bad_trees_flagged():
    good = np.array([-1, 0, 0, 1], dtype=np.int32)
    cases = {
        "root not -1": np.array([0, 0, 0, 1], dtype=np.int32),
        "forward parent": np.array([-1, 2, 0, 1], dtype=np.int32),
        "self parent": np.array([-1, 1, 0, 1], dtype=np.int32),
        "negative": np.array([-1, 0, -3, 1], dtype=np.int32),
    }
    for name, bad in cases.items():
        par, off = pack([good, bad, good])
        mask, depth, status = oracle.build_mask(par, off)
        assert status.tolist() == [0, -5, 0], name
    # more than 128 nodes in one request
    par, off = pack([synthetic.chain_tree(129)])
    _, _, status = oracle.build_mask(par, off)
    assert status.tolist() == [-4]
