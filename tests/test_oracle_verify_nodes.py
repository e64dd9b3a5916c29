"""Pins for the oracle's per-node decisions and margins, which the GPU parity
tests use to decide whether a GPU decision that differs from the oracle's is
a legitimate near-tie.

Sources: speculative-decoding explainer §2.2 (stage 2 alpha = min(1, p/q),
stage 3 rejection and a new target prediction); developer article,
deployment configuration (top_p).  Pins:
  * the per-node decisions reproduce the oracle's walk on random trees
    (greedy, stochastic, top-p): a decision at a node depends only on that
    node's rows, children and uniforms;
  * margins on the hand-worked example, from its hand-derived alpha values
    (1/2 and 0) and residuals;
  * the plausible top-p nuclei against a brute-force numpy enumeration of
    the same rule;
  * a value-band swap at the nucleus boundary makes the node fragile;
  * the draw gaps of expansion against numpy's cumulative sums."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from test_oracle_verify import GOLDEN, np_uniform, pack
from token_tree_verification_gb300 import synthetic

MASS_BAND = 5e-6
VALUE_BAND = 2.0 ** -16


def walk_from_nodes(nodes, tokens, offsets, W):
    B = len(offsets) - 1
    acc = np.zeros(B, np.int32)
    pn = np.full((B, W), -1, np.int32)
    ot = np.full((B, W), -1, np.int32)
    for b in range(B):
        lo = int(offsets[b])
        u, a = 0, 0
        pn[b, 0] = 0
        while True:
            nxt = int(nodes["next"][lo + u])
            if nxt < 0:
                ot[b, a] = nodes["token"][lo + u]
                break
            ot[b, a] = tokens[lo + nxt]
            a += 1
            pn[b, a] = nxt
            u = nxt
        acc[b] = a
    return acc, pn, ot


@pytest.mark.parametrize("temp,top_p", [(0.0, 1.0), (0.8, 1.0), (1.3, 1.0), (0.8, 0.9), (1.0, 0.5)])
def test_node_decisions_reproduce_the_walk(temp, top_p):
    rng = np.random.default_rng(int(temp * 10 + top_p * 100))
    trees = [synthetic.random_tree(rng, int(rng.integers(4, 14)), 3, 4) for _ in range(60)]
    par, off = pack(trees)
    V = 50
    tl = rng.normal(0, 2, (par.size, V)).astype(np.float32)
    dl = (tl + rng.normal(0, 1, tl.shape)).astype(np.float32)
    tok = rng.integers(0, V, par.size).astype(np.int32)
    tok[off[:-1]] = 0
    r = oracle.tree_verify(tl, dl if temp > 0 else None, tok, par, off, temp, 21, 4, top_p=top_p)
    nodes = oracle.verify_nodes(tl, dl if temp > 0 else None, tok, par, off, temp, 21, 4, top_p=top_p)
    assert (r["status"] == 0).all() and (nodes["status"] == 0).all()
    acc, pn, ot = walk_from_nodes(nodes, tok, off, 4)
    np.testing.assert_array_equal(acc, r["accept_len"])
    np.testing.assert_array_equal(pn, r["path_nodes"])
    np.testing.assert_array_equal(ot, r["out_tokens"])
    if temp == 0.0:
        assert np.isinf(nodes["margin"]).all() and (nodes["n_close"] == 0).all()
    else:
        assert (nodes["margin"] >= 0).all() and np.isfinite(nodes["margin"]).all()


def test_want_restricts_the_evaluated_nodes():
    rng = np.random.default_rng(3)
    par, off = pack([synthetic.random_tree(rng, 9, 3, 3) for _ in range(4)])
    tl = rng.normal(0, 2, (par.size, 20)).astype(np.float32)
    tok = rng.integers(0, 20, par.size).astype(np.int32)
    want = np.zeros(par.size, np.uint8)
    want[[0, 5, 11]] = 1
    nodes = oracle.verify_nodes(tl, tl, tok, par, off, 1.0, 2, 4, want=want)
    assert (nodes["next"][want == 0] == -2).all() and (nodes["next"][want == 1] != -2).all()


def test_margins_of_the_hand_worked_example():
    """Root of the hand example: alpha of child 1 is 1/2, alpha of child 2 is
    0, and after both rejections the residual is one-hot at token 0, so the
    draw's interval is [0, 1).  The margin is the smallest of |u1 - 1/2|
    and, when child 1 is rejected, |u2 - 0| and min(u_fb, 1 - u_fb)."""
    g = json.load(open(os.path.join(GOLDEN, "verify_hand_example.json")))
    tl = np.array([[math.log(0.5), math.log(0.25), math.log(0.125), math.log(0.125)]]
                  + g["target_logits"][1:], dtype=np.float32)
    dl = np.array(g["draft_logits"], dtype=np.float32)
    par = np.array(g["parents"], np.int32)
    tok = np.array(g["tokens"], np.int32)
    off = np.array([0, 3], np.int32)
    for seed in range(30):
        nodes = oracle.verify_nodes(tl, dl, tok, par, off, 1.0, seed, 3, band=0.05)
        u1, u2, ufb = np_uniform(seed, 1, 0, 0), np_uniform(seed, 2, 0, 0), np_uniform(seed, 0, 0, 1)
        if u1 < 0.5:
            want = [abs(u1 - 0.5)]
            assert nodes["next"][0] == 1
        else:
            want = [abs(u1 - 0.5), u2, min(ufb, 1 - ufb)]
            assert nodes["next"][0] == -1 and nodes["token"][0] == 0
        # fp32 logits of ln 1/8 etc. are exact to ~1e-8 relative
        assert abs(nodes["margin"][0] - min(want)) < 1e-7, (seed, nodes["margin"][0], want)
        assert nodes["n_close"][0] == sum(x < 0.05 for x in want)


def brute_force_nuclei(d, top_p):
    """The plausible nuclei of the stated rule, enumerated directly: exact
    tau by trying every distinct value, the mass-band cuts by testing every
    distinct value, and every subset of the distinct values within the value
    band of tau (when there are at least two)."""
    d = np.asarray(d, np.float64)
    vals = np.unique(d)[::-1]
    tails = np.array([d[d >= t].sum() for t in vals])
    above = np.array([d[d > t].sum() for t in vals])
    ok = np.nonzero(tails >= top_p)[0]
    tau = vals[ok[0]] if ok.size else vals[-1]
    sets = {frozenset(np.nonzero(d >= tau)[0])}
    cuts = [t for t, ge, ab in zip(vals, tails, above)
            if t != tau and ge >= top_p - MASS_BAND and ab < top_p + MASS_BAND]
    lo, hi = tau * (1 - VALUE_BAND), tau * (1 + VALUE_BAND)
    near = [t for t in vals if lo <= t <= hi]
    if len(cuts) > 16 or len(near) > 4:
        return tau, None          # more than the enumeration takes
    for t in cuts:
        sets.add(frozenset(np.nonzero(d >= t)[0]))
    if len(near) > 1:
        base = set(np.nonzero(d > hi)[0])
        for s in range(1 << len(near)):
            keep = set(base)
            for j, t in enumerate(near):
                if (s >> j) & 1:
                    keep |= set(np.nonzero(d == t)[0])
            sets.add(frozenset(keep))
    return tau, sets


def _cases():
    rng = np.random.default_rng(8)
    out = []
    for V in (3, 7, 40, 300):
        for _ in range(6):
            d = rng.exponential(1.0, V) ** 3
            d /= d.sum()
            out.append((d, float(rng.uniform(0.2, 0.99))))
    # the boundary mass exactly at top_p (the hand example of the top-p pins)
    out.append((np.array([0.5, 0.3, 0.2]), 0.8))
    # ties at tau
    out.append((np.array([0.4, 0.3, 0.3]), 0.5))
    # two entries within the value band of tau, in either order
    d = np.array([0.3, 0.2, 0.2 * (1 + 3e-6), 0.15, 0.1499999, 0.05])
    out.append((d / d.sum(), 0.55))
    out.append((d / d.sum(), 0.7))
    # dense values near the boundary (many mass-band cuts)
    d = np.full(2000, 1.0) + rng.uniform(0, 1e-3, 2000)
    out.append((d / d.sum(), 0.9))
    return out


@pytest.mark.parametrize("case", range(len(_cases())))
def test_nucleus_alternatives_match_brute_force(case):
    d, top_p = _cases()[case]
    tau, keeps = oracle.nucleus_alternatives(d, top_p)
    tau_bf, sets = brute_force_nuclei(d, top_p)
    assert tau == tau_bf
    # more cuts or near values than the enumeration takes (the node then
    # counts as fragile) on both sides, or the same plausible sets
    assert (keeps is None) == (sets is None)
    if keeps is None:
        return
    assert frozenset(np.nonzero(keeps[0])[0]) == frozenset(np.nonzero(d >= tau)[0])
    got = {frozenset(np.nonzero(k)[0]) for k in keeps}
    assert got == sets


def test_value_band_swap_makes_a_node_fragile():
    """Two target entries 4e-6 apart (relative) straddle tau: in float32 they
    may come out in either order, so a nucleus that keeps the lower one and
    drops the upper one is plausible.  A leaf whose draw lands on one of them
    differs between the two nuclei: the node is fragile (margin 0, counted)
    exactly when the draw's token changes."""
    p = np.array([0.35, 0.25, 0.2, 0.2 * (1 - 4e-6), 0.1])
    p /= p.sum()
    logits = np.log(p).astype(np.float64)
    # tau is the upper of the close pair at top_p 0.75 (0.35 + 0.25 + 0.2 = 0.8)
    tau, keeps = oracle.nucleus_alternatives(np.exp(logits.astype(np.float32).astype(np.float64)) /
                                             np.exp(logits.astype(np.float32).astype(np.float64)).sum(), 0.75)
    assert keeps is not None and len(keeps) > 1
    n = 400
    tl = np.tile(logits.astype(np.float32), (n, 1))
    par = np.full(n, -1, np.int32)
    off = np.arange(n + 1, dtype=np.int32)
    nodes = oracle.verify_nodes(tl, tl, np.zeros(n, np.int32), par, off, 1.0, 4, 1, top_p=0.75)
    r = oracle.tree_verify(tl, tl, np.zeros(n, np.int32), par, off, 1.0, 4, 1, top_p=0.75)
    fragile = nodes["margin"] == 0.0
    assert 0 < fragile.sum() < n
    np.testing.assert_array_equal(fragile, r["near_ties"] > 0)


def test_expansion_gaps_against_cumulative_sums():
    rng = np.random.default_rng(5)
    F, V, width, T = 6, 300, 8, 0.9
    d = (rng.standard_normal((F, V)) * 2).astype(np.float32)
    nodes, reqs = np.arange(F), np.zeros(F)
    tok, _, ties, gaps = oracle.tree_expand(d, np.zeros(F), nodes, reqs, width, T, 3, with_gaps=True)
    for f in range(F):
        w = np.exp((d[f].astype(np.float64) - d[f].max()) / T)
        c = np.cumsum(w)
        for j in range(width):
            x = tok[f, j]
            lo = c[x - 1] if x > 0 else 0.0
            # the draw's target lies in [lo, c[x]); its gap is the distance to
            # the nearer end, relative to the total
            assert gaps[f, j] <= (c[x] - lo) / c[-1] + 1e-12
            assert (gaps[f, j] < 1e-6) == bool(ties[f, j])
    # greedy children have no draw
    _, _, _, g0 = oracle.tree_expand(d, np.zeros(F), nodes, reqs, width, 0.0, 3, with_gaps=True)
    assert np.isinf(g0).all()
