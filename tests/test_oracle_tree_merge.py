"""Pins for the oracle's merge of two speculators' token trees (developer
article, §7.2 混合推测策略: an LLM speculator's tree merged with an n-gram
speculator's, tree.merge(other)).

  * brute force over token paths: the merged tree's paths are the union of
    both trees' paths, A's nodes stay where they are, each B node maps to
    the lowest merged node with the same path, and the merged size is n_a
    plus the distinct paths of B absent from A;
  * a tree merged with itself, and with a root-only tree, is unchanged;
  * a hand-worked example (an LLM speculator's tree and an n-gram chain);
  * the merged tree is a tree (parent < index), and greedy verification on
    it accepts at least as much as on either input (the target's argmax
    depends only on the token path);
  * errors: a merged tree over the cap, malformed parents."""
import numpy as np
import pytest

import oracle
from test_oracle_verify import pack
from token_tree_verification_gb300 import synthetic


def paths(par, tok):
    out = []
    for i in range(len(par)):
        p, a = [], i
        while a > 0:
            p.append(int(tok[a]))
            a = par[a]
        out.append(tuple(reversed(p)))
    return out


def check_merge(pa, ta, pb, tb, res, b=0):
    n = int(res["n_out"][b])
    mp, mt = res["parents"][b][:n], res["tokens"][b][:n]
    assert mp[0] == -1 and all(0 <= mp[i] < i for i in range(1, n))
    PA, PB, PM = paths(pa, ta), paths(pb, tb), paths(mp, mt)
    assert PM[:len(pa)] == PA and (mp[:len(pa)] == pa).all()
    assert set(PM) == set(PA) | set(PB)
    assert n == len(pa) + len(set(PB) - set(PA))
    first = {}
    for j, pth in enumerate(PM):
        first.setdefault(pth, j)
    for i in range(len(pb)):
        assert PM[res["map_b"][b][i]] == PB[i]
        assert res["map_b"][b][i] == first[PB[i]]
    assert (res["parents"][b][n:] == -2).all() and (res["tokens"][b][n:] == -1).all()
    assert (res["map_b"][b][len(pb):] == -1).all()


def random_pair(rng, vocab=6):
    na, nb = int(rng.integers(4, 40)), int(rng.integers(4, 40))
    pa = synthetic.random_tree(rng, na, int(rng.integers(1, min(6, na - 1) + 1)), None)
    pb = synthetic.random_tree(rng, nb, int(rng.integers(1, min(6, nb - 1) + 1)), None)
    ta = rng.integers(0, vocab, na).astype(np.int32)
    tb = rng.integers(0, vocab, nb).astype(np.int32)
    return pa, ta, pb, tb


def test_merge_matches_path_brute_force():
    rng = np.random.default_rng(1)
    for _ in range(60):
        pa, ta, pb, tb = random_pair(rng)
        res = oracle.tree_merge(pa, ta, [0, len(pa)], pb, tb, [0, len(pb)])
        assert res["status"][0] == 0
        check_merge(pa, ta, pb, tb, res)


def test_ragged_batch_matches_one_by_one():
    rng = np.random.default_rng(2)
    pairs = [random_pair(rng) for _ in range(7)]
    PA, OA = pack([p[0] for p in pairs])
    PB, OB = pack([p[2] for p in pairs])
    TA = np.concatenate([p[1] for p in pairs])
    TB = np.concatenate([p[3] for p in pairs])
    res = oracle.tree_merge(PA, TA, OA, PB, TB, OB)
    for b, (pa, ta, pb, tb) in enumerate(pairs):
        one = oracle.tree_merge(pa, ta, [0, len(pa)], pb, tb, [0, len(pb)])
        for k in ("parents", "tokens", "map_b"):
            np.testing.assert_array_equal(res[k][b], one[k][0])
        check_merge(pa, ta, pb, tb, res, b)


def test_self_merge_and_root_only():
    rng = np.random.default_rng(3)
    pa, ta, _, _ = random_pair(rng, vocab=50)
    res = oracle.tree_merge(pa, ta, [0, len(pa)], pa, ta, [0, len(pa)])
    assert res["n_out"][0] == len(pa)
    first = {}
    for j, pth in enumerate(paths(pa, ta)):
        first.setdefault(pth, j)
    assert [first[p] for p in paths(pa, ta)] == res["map_b"][0][:len(pa)].tolist()
    res = oracle.tree_merge(pa, ta, [0, len(pa)], [-1], [9], [0, 1])
    assert res["n_out"][0] == len(pa) and res["map_b"][0][0] == 0


def test_hand_worked_merge():
    # LLM speculator: root -> 7 -> 11, root -> 3; n-gram chain: root -> 7 -> 12 -> 15
    pa, ta = np.array([-1, 0, 0, 1], np.int32), np.array([0, 7, 3, 11], np.int32)
    pb, tb = np.array([-1, 0, 1, 2], np.int32), np.array([0, 7, 12, 15], np.int32)
    res = oracle.tree_merge(pa, ta, [0, 4], pb, tb, [0, 4])
    n = res["n_out"][0]
    assert n == 6
    assert res["parents"][0][:n].tolist() == [-1, 0, 0, 1, 1, 4]
    assert res["tokens"][0][1:n].tolist() == [7, 3, 11, 12, 15]
    assert res["map_b"][0][:4].tolist() == [0, 1, 4, 5]


def test_merging_never_shortens_greedy_acceptance():
    """With the target's argmax a function of the token path, greedy
    verification on the merged tree accepts at least the longer of the two
    inputs' accepted paths."""
    rng = np.random.default_rng(4)
    V = 5
    def logits_for(par, tok):
        rows = []
        for pth in paths(par, tok):
            h = np.random.default_rng(abs(hash(pth)) % (2**32))
            rows.append(h.normal(0, 1, V))
        return np.array(rows, np.float32)
    for _ in range(40):
        pa, ta, pb, tb = random_pair(rng, vocab=V)
        res = oracle.tree_merge(pa, ta, [0, len(pa)], pb, tb, [0, len(pb)])
        n = int(res["n_out"][0])
        mp, mt = res["parents"][0][:n], res["tokens"][0][:n]
        acc = []
        for par, tok in ((pa, ta), (pb, tb), (mp, mt)):
            r = oracle.tree_verify(logits_for(par, tok), None, tok, par, [0, len(par)], 0.0, 0, 64)
            acc.append(int(r["accept_len"][0]))
        assert acc[2] >= max(acc[0], acc[1]), acc


def test_merge_errors():
    pa, ta = np.array([-1, 0, 0], np.int32), np.array([0, 1, 2], np.int32)
    pb = np.array([-1] + list(range(0, 7)), np.int32)          # a chain of 8 new tokens
    tb = np.arange(10, 18).astype(np.int32)
    res = oracle.tree_merge(pa, ta, [0, 3], pb, tb, [0, 8], cap=8)   # 3 + 7 > 8
    assert res["status"][0] == -4
    bad = np.array([-1, 0, 3], np.int32)
    res = oracle.tree_merge(bad, ta, [0, 3], pa, ta, [0, 3])
    assert res["status"][0] == -5
