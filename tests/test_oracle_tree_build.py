"""Pins for the oracle's draft-tree construction (SpecInfer developer article
§2.1: the speculator proposes candidate tokens from each node's draft
distribution; each node keeps its parent; the deployment configuration sets
the tree width): level expansion (greedy top-w and i.i.d. inverse-CDF draws)
and pruning to the best-scoring ancestor-closed subtree."""
import numpy as np
import pytest
from scipy.special import log_softmax

import oracle


def test_greedy_expansion_is_stable_argsort_with_log_softmax_scores():
    rng = np.random.default_rng(0)
    F, V, w = 6, 50, 5
    d = rng.standard_normal((F, V)).astype(np.float32) * 3
    d[2, [4, 9, 11]] = d[2].max() + 1.0      # a three-way tie at the top: lower index first
    ps = rng.standard_normal(F)
    tok, sc, ties = oracle.tree_expand(d, ps, np.arange(F), np.zeros(F), w, 0.0, 7)
    for f in range(F):
        order = np.argsort(-d[f].astype(np.float64), kind="stable")[:w]
        np.testing.assert_array_equal(tok[f], order)
        np.testing.assert_allclose(sc[f], ps[f] + log_softmax(d[f].astype(np.float64))[order], rtol=0, atol=1e-12)
    assert (ties == 0).all()
    assert tok[2, :3].tolist() == [4, 9, 11]


def test_sampled_expansion_matches_searchsorted_at_the_same_uniforms():
    rng = np.random.default_rng(1)
    F, V, w, T, seed = 5, 40, 4, 0.7, 123
    d = rng.standard_normal((F, V)).astype(np.float32) * 2
    nodes, reqs = np.array([0, 3, 7, 2, 9]), np.array([0, 0, 1, 2, 2])
    tok, sc, ties = oracle.tree_expand(d, np.zeros(F), nodes, reqs, w, T, seed)
    for f in range(F):
        z = d[f].astype(np.float64) / T
        q = np.exp(z - z.max())
        cdf = np.cumsum(q) / q.sum()
        lq = np.log(q / q.sum())
        for j in range(w):
            # counter (node, request, 2, child slot), key (seed, 0), top 24 bits of word 0
            word = oracle.philox4x64_10([nodes[f], reqs[f], 2, j], [seed, 0])[0]
            u = float(int(word) >> 40) / 2**24
            assert tok[f, j] == int(np.searchsorted(cdf, u, side="right"))
            assert abs(sc[f, j] - lq[tok[f, j]]) < 1e-12


def test_sampled_expansion_draws_from_q():
    V, T, n = 8, 1.3, 40000
    logits = np.array([1.0, 0.2, -0.5, 2.0, 0.0, -1.0, 1.5, 0.7], np.float32)
    d = np.tile(logits, (n, 1))
    tok, _, _ = oracle.tree_expand(d, np.zeros(n), np.arange(n), np.zeros(n), 1, T, 99)
    q = np.exp(logits / T); q /= q.sum()
    counts = np.bincount(tok[:, 0], minlength=V)
    chi2 = ((counts - n * q) ** 2 / (n * q)).sum()
    dof = V - 1
    assert chi2 < dof + 3 * np.sqrt(2 * dof), chi2


def _random_candidates(rng, n):
    par = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)], np.int32)
    sc = np.zeros(n)
    for i in range(1, n):
        sc[i] = sc[par[i]] + np.log(rng.uniform(1e-3, 1.0))
    return par, sc


@pytest.mark.parametrize("n,keep", [(30, 10), (156, 64), (7, 7), (5, 12), (40, 1)])
def test_pruning_keeps_the_best_ancestor_closed_subtree(n, keep):
    rng = np.random.default_rng(n + keep)
    par, sc = _random_candidates(rng, n)
    sc[5 % n] = sc[par[5 % n]] if n > 5 else sc[0]      # a child as good as its parent
    tok = rng.integers(0, 1000, n).astype(np.int32)
    out = oracle.tree_prune(par, tok, sc, [0, n], keep)
    k = min(keep, n)
    assert out["status"].tolist() == [0] and out["n_out"].tolist() == [k]
    expect = sorted([0] + sorted(range(1, n), key=lambda i: (-sc[i], i))[: keep - 1])
    kept = out["kept"][0, :k]
    assert kept.tolist() == expect
    # renumbered parents are the kept parents' new indices; tokens follow
    new = {int(o): i for i, o in enumerate(kept)}
    for i, o in enumerate(kept):
        assert out["tokens"][0, i] == tok[o]
        assert out["parents"][0, i] == (-1 if o == 0 else new[int(par[o])])
    assert (out["parents"][0, k:] == -2).all()


def test_expand_then_prune_builds_a_valid_tree():
    rng = np.random.default_rng(5)
    V, w, depth, keep, T = 64, 3, 3, 12, 0.8
    parents, tokens, scores = [-1], [0], [0.0]
    frontier = [0]
    for _ in range(depth):
        d = rng.standard_normal((len(frontier), V)).astype(np.float32) * 2
        tok, sc, _ = oracle.tree_expand(d, [scores[u] for u in frontier], frontier,
                                        np.zeros(len(frontier)), w, T, 11)
        nxt = []
        for f, u in enumerate(frontier):
            for j in range(w):
                parents.append(u); tokens.append(int(tok[f, j])); scores.append(float(sc[f, j]))
                nxt.append(len(parents) - 1)
        frontier = nxt
    out = oracle.tree_prune(parents, tokens, scores, [0, len(parents)], keep)
    par = out["parents"][0]
    assert par[0] == -1 and all(0 <= par[i] < i for i in range(1, keep))


def test_pruning_non_monotone_scores_orphans_and_the_mask_rejects_it():
    # a chain 0 -> 1 -> 2 whose grandchild outscores its parent: with keep 2 the
    # root and node 2 survive, node 2's parent (1) is dropped
    par = np.array([-1, 0, 1], np.int32)
    sc = np.array([0.0, -3.0, -1.0])
    out = oracle.tree_prune(par, np.array([5, 6, 7], np.int32), sc, [0, 3], 2)
    assert out["status"].tolist() == [0]
    assert out["kept"][0].tolist() == [0, 2]
    assert out["parents"][0].tolist() == [-1, -1]
    _, _, st = oracle.build_mask(out["parents"][0], np.array([0, 2], np.int32))
    assert st.tolist() == [-5]   # bad parent
