"""Pins for the oracle's verification (steps V1-V4 and R).

Sources: SpecInfer developer article §2.1 (accept the longest verified
prefix); speculative-decoding explainer §2.2 (stage 1 greedy draft, stage 2
alpha = min(1, p/q), stage 3 left-to-right rejection with a new target
prediction, output distribution identical to the target's); SpecInfer news
write-up (lossless tree verification).  Pins:
  * a hand-worked example (tests/golden/verify_hand_example.json);
  * greedy: brute-force enumeration of root-to-node paths, and the
    first-mismatch length of a chain;
  * stochastic single-child chain: empirical accept rate equals the closed
    form sum_x min(p, q) within 3 sigma; the second sibling's accept rate
    equals the closed form of the residual;
  * q = p accepts every first child; a one-hot p rejects every other token
    and emits argmax p;
  * losslessness: over 10^6 seeded trials the first emitted token follows
    p_root and the first two tokens follow p(x1) p(x2 | x1) (chi-square at
    dof + 3 sqrt(2 dof))."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from token_tree_verification_gb300 import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def np_uniform(seed, node, req, kind):
    bg = np.random.Philox(key=seed, counter=(node + (req << 64) + (kind << 128) - 1) % 2**256)
    return (int(bg.random_raw(1)[0]) >> 40) / 2.0**24


def softmax64(row, temp):
    z = np.asarray(row, dtype=np.float64) / temp
    e = np.exp(z - z.max())
    return e / e.sum()


def pack(trees):
    off = np.zeros(len(trees) + 1, dtype=np.int32)
    off[1:] = np.cumsum([t.size for t in trees])
    return np.concatenate(trees).astype(np.int32), off


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "verify_hand_example.json")))
    V = g["V"]
    tl = np.array([[math.log(0.5), math.log(0.25), math.log(0.125), math.log(0.125)]]
                  + g["target_logits"][1:], dtype=np.float32)
    dl = np.array(g["draft_logits"], dtype=np.float32)
    par = np.array(g["parents"], np.int32)
    tok = np.array(g["tokens"], np.int32)
    seen = set()
    for seed in range(40):
        u = np_uniform(seed, 1, 0, 0)
        if abs(u - 0.5) < 1e-3 or np_uniform(seed, 1, 0, 1) == 0.0:
            continue
        res = oracle.tree_verify(tl, dl, tok, par, np.array([0, 3], np.int32), g["temperature"], seed, 3)
        exp = g["expect_if_u_below_half"] if u < 0.5 else g["expect_otherwise"]
        n = exp["accept_len"] + 1
        assert res["status"][0] == 0
        assert res["accept_len"][0] == exp["accept_len"]
        assert res["path_nodes"][0, :n].tolist() == exp["path_nodes"]
        assert res["out_tokens"][0, :n].tolist() == exp["out_tokens"]
        assert (res["out_tokens"][0, n:] == -1).all()
        assert res["near_ties"][0] == 0
        seen.add(u < 0.5)
    assert seen == {True, False}


def greedy_brute_force(par, tok, logits):
    """Longest root-to-node path whose every token equals the target argmax
    at its parent; emitted = path tokens + argmax at the path's end."""
    n = par.size
    best = None
    for v in range(n):
        path = []
        a = v
        while a != -1:
            path.append(a)
            a = par[a]
        path = path[::-1]
        if all(tok[c] == int(np.argmax(logits[p])) for p, c in zip(path, path[1:])):
            if best is None or len(path) > len(best) or (len(path) == len(best) and path < best):
                best = path
    return best, [int(tok[c]) for c in best[1:]] + [int(np.argmax(logits[best[-1]]))]


def test_greedy_matches_brute_force():
    rng = np.random.default_rng(0)
    V = 6
    trees, toks = [], []
    for _ in range(300):
        n = int(rng.integers(1, 30))
        d = int(rng.integers(1, 6)) if n > 1 else 0
        while sum(V ** j for j in range(d + 1)) < n:
            d += 1
        t = synthetic.random_tree(rng, n, min(d, n - 1), V)
        tk = np.zeros(n, np.int32)
        for u in range(n):                   # distinct sibling tokens
            cs = np.nonzero(t == u)[0]
            tk[cs] = rng.permutation(V)[: cs.size]
        trees.append(t); toks.append(tk)
    par, off = pack(trees)
    tok = np.concatenate(toks)
    # integer logits: frequent ties exercise the lowest-index rule
    logits = rng.integers(-3, 3, size=(par.size, V)).astype(np.float32)
    res = oracle.tree_verify(logits, None, tok, par, off, 0.0, 0, 32)
    assert (res["status"] == 0).all()
    for b, t in enumerate(trees):
        s = off[b]
        path, emitted = greedy_brute_force(t, tok[s:s + t.size], logits[s:s + t.size])
        a = res["accept_len"][b]
        assert a == len(path) - 1
        assert res["path_nodes"][b, :a + 1].tolist() == path
        assert res["out_tokens"][b, :a + 1].tolist() == emitted
        assert res["near_ties"][b] == 0


def test_greedy_duplicate_siblings_first_child_wins():
    par = np.array([-1, 0, 0, 2], np.int32)
    tok = np.array([0, 3, 3, 1], np.int32)
    logits = np.zeros((4, 4), np.float32)
    logits[0, 3] = 1.0          # root predicts 3: both children match
    logits[2, 1] = 1.0          # only the second child would continue
    res = oracle.tree_verify(logits, None, tok, par, np.array([0, 4], np.int32), 0.0, 0, 4)
    assert res["accept_len"][0] == 1
    assert res["path_nodes"][0, :2].tolist() == [0, 1]


def test_greedy_chain_first_mismatch():
    rng = np.random.default_rng(3)
    B, K, V = 500, 5, 4
    logits = rng.standard_normal((B * (K + 1), V)).astype(np.float32)
    am = logits.reshape(B, K + 1, V).argmax(-1)
    tok = np.where(rng.random((B, K + 1)) < 0.7, np.roll(am, 1, axis=1), rng.integers(0, V, (B, K + 1)))
    tok[:, 0] = 0
    par, off = pack([synthetic.chain_tree(K + 1)] * B)
    res = oracle.tree_verify(logits, None, tok.reshape(-1).astype(np.int32), par, off, 0.0, 0, K + 1)
    match = tok[:, 1:] == am[:, :-1]
    first_miss = np.where(match.all(1), K, np.argmin(match, axis=1))
    np.testing.assert_array_equal(res["accept_len"], first_miss)
    bonus = am[np.arange(B), first_miss]
    np.testing.assert_array_equal(res["out_tokens"][np.arange(B), first_miss], bonus)


def _rate_test(accepted, expected):
    n = accepted.size
    sigma = math.sqrt(expected * (1 - expected) / n)
    assert abs(accepted.mean() - expected) <= 3 * sigma + 1e-12, (accepted.mean(), expected, sigma)


@pytest.mark.parametrize("temp", [1.0, 0.7])
def test_single_child_accept_rate_closed_form(temp):
    rng = np.random.default_rng(4)
    B, V = 40000, 16
    tl = rng.normal(0, 1.5, V).astype(np.float32)
    dl = (tl + rng.normal(0, 1.0, V)).astype(np.float32)
    p, q = softmax64(tl, temp), softmax64(dl, temp)
    toks = np.zeros((B, 2), np.int32)
    toks[:, 1] = rng.choice(V, size=B, p=q)
    par, off = pack([synthetic.chain_tree(2)] * B)
    res = oracle.tree_verify(np.tile(tl, (2 * B, 1)), np.tile(dl, (2 * B, 1)), toks.reshape(-1),
                             par, off, temp, 99, 2)
    _rate_test(res["accept_len"] >= 1, float(np.minimum(p, q).sum()))


def test_second_sibling_accept_rate_uses_residual():
    rng = np.random.default_rng(5)
    B, V = 40000, 8
    tl = rng.normal(0, 1.5, V).astype(np.float32)
    tl[0] = -1000.0                              # p(0) = 0: the first child (token 0) is always rejected
    dl = rng.normal(0, 1.0, V).astype(np.float32)
    p, q = softmax64(tl, 1.0), softmax64(dl, 1.0)
    r1 = np.maximum(p - q, 0.0)
    r1 /= r1.sum()
    toks = np.zeros((B, 3), np.int32)
    toks[:, 2] = rng.choice(V, size=B, p=q)
    par, off = pack([np.array([-1, 0, 0], np.int32)] * B)
    res = oracle.tree_verify(np.tile(tl, (3 * B, 1)), np.tile(dl, (3 * B, 1)), toks.reshape(-1),
                             par, off, 1.0, 7, 2)
    assert not (res["path_nodes"][:, 1] == 1).any()
    expected = float(np.sum(q * np.minimum(1.0, r1 / q)))
    _rate_test(res["path_nodes"][:, 1] == 2, expected)


def test_q_equals_p_accepts_first_children():
    rng = np.random.default_rng(6)
    trees = [synthetic.random_tree(rng, int(n), 3, 4) for n in rng.integers(4, 30, 50)]
    par, off = pack(trees)
    V = 10
    tl = rng.normal(0, 2, (par.size, V)).astype(np.float32)
    tok = rng.integers(0, V, par.size).astype(np.int32)
    res = oracle.tree_verify(tl, tl.copy(), tok, par, off, 0.8, 1, 8)
    for b, t in enumerate(trees):
        u, path = 0, [0]
        while True:
            cs = np.nonzero(t == u)[0]
            if cs.size == 0:
                break
            u = int(cs[0]); path.append(u)
        assert res["accept_len"][b] == len(path) - 1
        assert res["path_nodes"][b, :len(path)].tolist() == path


def test_one_hot_target_rejects_and_emits_argmax():
    rng = np.random.default_rng(7)
    trees = [synthetic.random_tree(rng, 8, 2, 4) for _ in range(100)]
    par, off = pack(trees)
    V = 12
    a = rng.integers(0, V, par.size)
    tl = np.full((par.size, V), -1000.0, np.float32)
    tl[np.arange(par.size), a] = 0.0
    dl = rng.normal(0, 1, (par.size, V)).astype(np.float32)
    tok = np.zeros(par.size, np.int32)
    for b, t in enumerate(trees):
        s = off[b]
        for c in range(1, t.size):
            tok[s + c] = (a[s + t[c]] + 1 + rng.integers(0, V - 1)) % V   # never the parent's argmax
    res = oracle.tree_verify(tl, dl, tok, par, off, 1.0, 3, 4)
    assert (res["accept_len"] == 0).all()
    np.testing.assert_array_equal(res["out_tokens"][:, 0], a[off[:-1]])


# ---------------------------------------------------------------------------
# losslessness (chi-square), V = 8, 10^6 trials
# ---------------------------------------------------------------------------
LOSSLESS_PARENTS = np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3, 4, 5, 6, 7, 8, 9], np.int32)
LOSSLESS_DEPTH = np.array([0, 1, 1, 1, 2, 2, 2, 2, 2, 2, 3, 3, 3, 3, 3, 3])
PATH_OFF = [0, 1, 9, 73, 585, 4681]           # path ids by length for V = 8


def lossless_tables(seed, V=8):
    rng = np.random.default_rng(seed)
    tab_t = rng.normal(0, 1.5, (PATH_OFF[-1], V)).astype(np.float32)
    tab_d = (tab_t + rng.normal(0, 1.0, tab_t.shape)).astype(np.float32)
    return tab_t, tab_d


def nucleus_np(prob, top_p):
    """Top-p nucleus of each row of ``prob`` by sorting: the largest value tau
    whose upper tail {prob >= tau} holds at least top_p of the mass; the tail
    (ties at tau included) renormalised, the rest zero."""
    prob = np.atleast_2d(np.asarray(prob, np.float64))
    out = np.zeros_like(prob)
    for i, row in enumerate(prob):
        srt = np.sort(row)[::-1]
        k = int(np.searchsorted(np.cumsum(srt), top_p))   # first index with cumsum >= top_p
        tau = srt[min(k, srt.size - 1)]
        keep = row >= tau
        out[i] = np.where(keep, row, 0.0) / row[keep].sum()
    return out


def lossless_trial_batch(rng, tab_t, tab_d, ctx_pid, ctx_len, temp, V=8, top_p=1.0):
    """One speculated tree per trial: node logits are a function of the node's
    token path; each child is an i.i.d. draft sample from its parent's q (its
    top-p nucleus when top_p < 1)."""
    n_tr = ctx_pid.size
    nn = LOSSLESS_PARENTS.size
    pid = np.zeros((n_tr, nn), np.int64)
    tok = np.zeros((n_tr, nn), np.int32)
    pid[:, 0] = ctx_pid
    q = np.exp(tab_d.astype(np.float64) / temp - (tab_d.astype(np.float64) / temp).max(1, keepdims=True))
    q /= q.sum(1, keepdims=True)
    if top_p < 1.0:
        q = nucleus_np(q, top_p)
    qcum = np.cumsum(q, axis=1)
    qcum /= qcum[:, -1:]
    for c in range(1, nn):
        u = LOSSLESS_PARENTS[c]
        pp = pid[:, u]
        x = (rng.random(n_tr)[:, None] >= qcum[pp]).sum(1).clip(max=V - 1)
        tok[:, c] = x
        l = ctx_len + LOSSLESS_DEPTH[u]
        pid[:, c] = PATH_OFF[l + 1] + (pp - PATH_OFF[l]) * V + x
    return tok, tab_t[pid].reshape(-1, V), tab_d[pid].reshape(-1, V)


def run_lossless(verify, trials, temp, seed, chunk=100000, V=8, top_p=1.0):
    """Returns counts of the first emitted token [V] and of the first two
    emitted tokens [V, V] (a second verification step, rooted after the first
    token, supplies the second token when the first step emits only one)."""
    tab_t, tab_d = lossless_tables(seed)
    rng = np.random.default_rng(seed + 1)
    c1 = np.zeros(V, np.int64)
    c2 = np.zeros((V, V), np.int64)
    nn = LOSSLESS_PARENTS.size
    done = 0
    step = 0
    while done < trials:
        n_tr = min(chunk, trials - done)
        par = np.tile(LOSSLESS_PARENTS, n_tr)
        off = (np.arange(n_tr + 1) * nn).astype(np.int32)
        tok, tl, dl = lossless_trial_batch(rng, tab_t, tab_d, np.zeros(n_tr, np.int64), 0, temp, top_p=top_p)
        r = verify(tl, dl, tok.reshape(-1), par, off, temp, 1000 * seed + 2 * step, 4, top_p=top_p)
        x1 = r["out_tokens"][:, 0]
        x2 = r["out_tokens"][:, 1].copy()
        need = r["accept_len"] == 0
        if need.any():
            m = int(need.sum())
            tok2, tl2, dl2 = lossless_trial_batch(rng, tab_t, tab_d, 1 + x1[need].astype(np.int64), 1, temp,
                                                  top_p=top_p)
            off2 = (np.arange(m + 1) * nn).astype(np.int32)
            r2 = verify(tl2, dl2, tok2.reshape(-1), np.tile(LOSSLESS_PARENTS, m), off2, temp,
                        1000 * seed + 2 * step + 1, 4, top_p=top_p)
            x2[need] = r2["out_tokens"][:, 0]
        np.add.at(c1, x1, 1)
        np.add.at(c2, (x1, x2), 1)
        done += n_tr
        step += 1
    p1 = softmax64(tab_t[0], temp)
    p2 = np.stack([softmax64(tab_t[1 + x], temp) for x in range(V)])
    if top_p < 1.0:
        p1 = nucleus_np(p1, top_p)[0]
        p2 = nucleus_np(p2, top_p)
    return c1, c2, p1, p1[:, None] * p2


def chi2_ok(counts, probs):
    """Pearson chi-square over the cells of positive probability (cells of
    probability zero must be empty) and its 3-sigma bound."""
    counts = counts.reshape(-1)
    probs = probs.reshape(-1)
    assert (counts[probs == 0] == 0).all(), "a draw landed outside the support"
    m = probs > 0
    n = counts.sum()
    e = n * probs[m]
    chi2 = float((((counts[m] - e) ** 2) / e).sum())
    dof = int(m.sum()) - 1
    return chi2, dof + 3 * math.sqrt(2 * dof)


def test_lossless_chi_square_oracle():
    c1, c2, p1, p12 = run_lossless(oracle.tree_verify, 1_000_000, 1.0, seed=0)
    chi, bound = chi2_ok(c1, p1)
    assert chi <= bound, (chi, bound)
    chi, bound = chi2_ok(c2, p12)
    assert chi <= bound, (chi, bound)


def test_lossless_chi_square_oracle_temperature():
    c1, c2, p1, p12 = run_lossless(oracle.tree_verify, 200_000, 0.7, seed=1)
    for c, p in ((c1, p1), (c2, p12)):
        chi, bound = chi2_ok(c, p)
        assert chi <= bound, (chi, bound)


# ---------------------------------------------------------------------------
# top-p (nucleus) filtering of p and q (developer article, deployment
# configuration: top_p)
# ---------------------------------------------------------------------------
def _leaf_draws(probs, top_p, trials, seed=0):
    """Bonus tokens of root-only trees whose target is ``probs`` (T = 1):
    draws from the target's nucleus."""
    logits = np.log(np.asarray(probs, np.float64)).astype(np.float32)
    V = logits.size
    tl = np.tile(logits, (trials, 1))
    par = np.full(trials, -1, np.int32)
    off = np.arange(trials + 1, dtype=np.int32)
    r = oracle.tree_verify(tl, tl, np.zeros(trials, np.int32), par, off, 1.0, seed, 1, top_p=top_p)
    assert (r["accept_len"] == 0).all()
    return np.bincount(r["out_tokens"][:, 0], minlength=V), r["near_ties"]


def test_top_p_hand_example_draws_from_the_nucleus():
    # [0.5, 0.3, 0.2], top_p = 0.7: the tail {0.5, 0.3} holds 0.8 >= 0.7, {0.5}
    # only 0.5 -> nucleus {0, 1}, renormalised to 5/8, 3/8
    counts, ties = _leaf_draws([0.5, 0.3, 0.2], 0.7, 40000)
    assert counts[2] == 0 and (ties == 0).all()
    chi, bound = chi2_ok(counts, np.array([5 / 8, 3 / 8, 0.0]))
    assert chi <= bound, (chi, bound)


def test_top_p_keeps_ties_at_the_threshold():
    # [0.4, 0.3, 0.3], top_p = 0.5: tau = 0.3 and both entries tied at 0.3 stay
    counts, _ = _leaf_draws([0.4, 0.3, 0.3], 0.5, 40000)
    chi, bound = chi2_ok(counts, np.array([0.4, 0.3, 0.3]))
    assert chi <= bound, (chi, bound)


def test_top_p_one_is_no_filter():
    rng = np.random.default_rng(4)
    trees = [synthetic.random_tree(rng, 10, 3, 3) for _ in range(50)]
    par, off = pack(trees)
    V = 30
    tl = rng.normal(0, 2, (par.size, V)).astype(np.float32)
    dl = (tl + rng.normal(0, 1, tl.shape)).astype(np.float32)
    tok = rng.integers(0, V, par.size).astype(np.int32)
    a = oracle.tree_verify(tl, dl, tok, par, off, 0.8, 9, 4)
    b = oracle.tree_verify(tl, dl, tok, par, off, 0.8, 9, 4, top_p=1.0)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


def test_top_p_boundary_near_tie_is_flagged():
    # [0.5, 0.3, 0.2] with top_p = 0.8: the tail {0.5, 0.3} holds 0.8 up to
    # rounding, so both {0, 1} (renormalised to 5/8, 3/8) and {0, 1, 2} are
    # nuclei a finite-precision run may find.  A draw is a near-tie exactly
    # when its uniform gives different tokens under the two; otherwise it is
    # the token both give.
    n, seed = 4000, 0
    r = None
    logits = np.log(np.array([0.5, 0.3, 0.2])).astype(np.float32)
    tl = np.tile(logits, (n, 1))
    par = np.full(n, -1, np.int32)
    off = np.arange(n + 1, dtype=np.int32)
    r = oracle.tree_verify(tl, tl, np.zeros(n, np.int32), par, off, 1.0, seed, 1, top_p=0.8)
    u = np.array([oracle.uniform(seed, 0, b, 1) for b in range(n)])
    two = np.where(u < 0.625, 0, 1)
    three = np.where(u < 0.5, 0, np.where(u < 0.8, 1, 2))
    differ = two != three
    away = np.minimum.reduce([abs(u - 0.5), abs(u - 0.625), abs(u - 0.8)]) > 1e-5
    np.testing.assert_array_equal((r["near_ties"] > 0)[away], differ[away])
    same = away & ~differ
    np.testing.assert_array_equal(r["out_tokens"][same, 0], two[same])
    assert 0.25 < differ.mean() < 0.4            # u in [0.5, 0.625) or [0.8, 1)


def test_top_p_spread_nucleus_rarely_ties():
    # thousands of entries near the boundary: the nuclei a rounding may pick
    # differ by entries of mass ~1e-6, which rarely changes a decision
    rng = np.random.default_rng(12)
    trees = [synthetic.random_tree(rng, 12, 3, 4) for _ in range(40)]
    par, off = pack(trees)
    V = 4000
    tl = rng.normal(0, 1.0, (par.size, V)).astype(np.float32)
    dl = (tl + rng.normal(0, 0.5, tl.shape)).astype(np.float32)
    tok = rng.integers(0, V, par.size).astype(np.int32)
    r = oracle.tree_verify(tl, dl, tok, par, off, 1.0, 3, 4, top_p=0.9)
    assert (r["status"] == 0).all()
    assert (r["near_ties"] > 0).sum() <= 2


def test_lossless_chi_square_oracle_top_p():
    c1, c2, p1, p12 = run_lossless(oracle.tree_verify, 200_000, 1.0, seed=5, top_p=0.8)
    assert (p1 == 0).any()            # the nucleus really removes tokens
    for c, p in ((c1, p1), (c2, p12)):
        chi, bound = chi2_ok(c, p)
        assert chi <= bound, (chi, bound)
