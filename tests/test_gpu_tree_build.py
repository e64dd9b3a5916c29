"""GPU parity of draft-tree construction (spec_tree_expand, spec_tree_prune)
against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import token_tree_verification_gb300 as ttv
from parity import BAND, dev

pytestmark = pytest.mark.gpu


def _expand_gpu(d, ps, nodes, reqs, width, T, seed):
    tok, sc, ties = ttv.tree_expand(dev(d, torch.float32), dev(ps, torch.float32), dev(nodes, torch.int32),
                                    dev(reqs, torch.int32), width, T, seed)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), sc.cpu().numpy(), ties.cpu().numpy()


@pytest.mark.parametrize("V,width", [(32000, 5), (1000, 16), (16, 16), (1, 1), (4097, 3),
                                     (8193, 4), (100000, 7)])
def test_greedy_expansion(V, width):
    # V > 8192 splits each row over a cluster of CTAs (one slice each)
    rng = np.random.default_rng(V)
    F = 7
    d = (rng.standard_normal((F, V)) * 3).astype(np.float32)
    if V > 20:
        d[1, [5, 17, 3]] = d[1].max() + 2.0          # tie at the top: lower index first
    if V > 30000:
        d[2, [30000, 9000, 20]] = d[2].max() + 3.0   # the same across slices
    ps = rng.standard_normal(F).astype(np.float32)
    nodes, reqs = np.arange(F), np.zeros(F)
    tg, sg, _ = _expand_gpu(d, ps, nodes, reqs, width, 0.0, 1)
    to, so, _ = oracle.tree_expand(d, ps.astype(np.float64), nodes, reqs, width, 0.0, 1)
    np.testing.assert_array_equal(tg, to)
    np.testing.assert_allclose(sg, so, rtol=0, atol=2e-4)


@pytest.mark.parametrize("V,width,T", [(32000, 5, 0.7), (1000, 16, 1.0), (50, 8, 2.5), (65536, 4, 0.3),
                                       (8193, 6, 1.0), (131077, 3, 0.8)])
def test_sampled_expansion(V, width, T):
    rng = np.random.default_rng(V + width)
    F = 12
    d = (rng.standard_normal((F, V)) * 3).astype(np.float32)
    ps = np.zeros(F, np.float32)
    nodes, reqs = rng.integers(0, 128, F), rng.integers(0, 4, F)
    tg, sg, tiesg = _expand_gpu(d, ps, nodes, reqs, width, T, 77)
    to, so, tieso, gap = oracle.tree_expand(d, ps.astype(np.float64), nodes, reqs, width, T, 77,
                                            with_gaps=True)
    assert (tiesg >= 0).all(), "an exchange between the CTAs of a row timed out"
    assert ((tg >= 0) & (tg < V)).all()
    # A draw may differ from the oracle's only where the oracle's exact gap to
    # the nearer inverse-CDF boundary is below BAND (at most one per case),
    # and the GPU may flag a near-tie only where that gap is below BAND.  (A
    # draw that lands on an entry of mass below 1e-6 of the total is a
    # near-tie by definition; with V = 131077 at T = 0.8 such entries carry
    # enough mass in total to be drawn now and then.)
    differ = tg != to
    assert (gap[differ] < BAND).all(), gap[differ]
    assert (gap[tiesg != 0] < BAND).all(), gap[tiesg != 0]
    assert differ.sum() <= 1
    same = ~differ
    np.testing.assert_allclose(sg[same], so[same], rtol=0, atol=2e-4)


def _prune_both(par, tok, sc32, off, keep):
    st = torch.zeros(len(off) - 1, dtype=torch.int32, device="cuda")
    g = ttv.tree_prune(dev(par, torch.int32), dev(tok, torch.int32), dev(sc32, torch.float32),
                       dev(off, torch.int32), keep, st)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    g["status"] = st.cpu().numpy()
    o = oracle.tree_prune(par, tok, sc32.astype(np.float64), off, keep)
    return g, o


def test_pruning_ragged_batch_matches_oracle():
    rng = np.random.default_rng(2)
    pars, toks, scs, off = [], [], [], [0]
    for n in (156, 1, 40, 1024, 64):
        p = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)], np.int32)
        s = np.zeros(n, np.float32)
        for i in range(1, n):
            s[i] = s[p[i]] + np.float32(np.log(rng.uniform(1e-3, 1.0)))
        if n > 10:
            s[7] = s[p[7]]        # a child as good as its parent (ties to the lower index)
        pars.append(p); toks.append(rng.integers(0, 32000, n).astype(np.int32)); scs.append(s)
        off.append(off[-1] + n)
    g, o = _prune_both(np.concatenate(pars), np.concatenate(toks), np.concatenate(scs), np.array(off, np.int32), 64)
    for k in ("parents", "tokens", "kept", "n_out", "status"):
        np.testing.assert_array_equal(g[k], o[k], err_msg=k)


def test_pruning_errors():
    par = np.array([-1, 0, 0, 5, -1, 0], np.int32)      # request 0: forward parent
    tok = np.zeros(6, np.int32)
    sc = np.zeros(6, np.float32)
    g, o = _prune_both(par, tok, sc, np.array([0, 4, 6], np.int32), 3)
    assert g["status"].tolist() == [-5, 0]
    np.testing.assert_array_equal(g["parents"][1], o["parents"][1])


def test_build_a_pruned_tree_level_by_level():
    """Width 5, depth 3, i.i.d. draft samples, pruned to 64 nodes: the GPU and
    the oracle build the same tree (parents, tokens) unless a draw differs,
    which it may only within BAND of an inverse-CDF boundary."""
    rng = np.random.default_rng(11)
    V, w, depth, keep, T, seed = 4000, 5, 3, 64, 0.7, 5
    par_g, tok_g, sc_g = [-1], [0], [0.0]
    par_o, tok_o, sc_o = [-1], [0], [0.0]
    frontier = [0]
    any_tie = False
    for _ in range(depth):
        d = (rng.standard_normal((len(frontier), V)) * 3).astype(np.float32)
        tg, sg, tiesg = _expand_gpu(d, np.array([sc_g[u] for u in frontier], np.float32), frontier,
                                    np.zeros(len(frontier)), w, T, seed)
        to, so, tieso, gap = oracle.tree_expand(d, [sc_o[u] for u in frontier], frontier,
                                                np.zeros(len(frontier)), w, T, seed, with_gaps=True)
        assert (tiesg >= 0).all()
        assert (gap[tg != to] < BAND).all()
        any_tie |= bool((tg != to).any())
        nxt = []
        for f, u in enumerate(frontier):
            for j in range(w):
                par_g.append(u); tok_g.append(int(tg[f, j])); sc_g.append(float(sg[f, j]))
                par_o.append(u); tok_o.append(int(to[f, j])); sc_o.append(float(so[f, j]))
                nxt.append(len(par_g) - 1)
        frontier = nxt
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = ttv.tree_prune(dev(par_g, torch.int32), dev(tok_g, torch.int32), dev(np.float32(sc_g), torch.float32),
                       dev([0, len(par_g)], torch.int32), keep, st)
    o = oracle.tree_prune(par_o, tok_o, sc_o, [0, len(par_o)], keep)
    gp = g["parents"].cpu().numpy()[0]
    assert gp[0] == -1 and all(0 <= gp[i] < i for i in range(1, keep))
    if not any_tie:
        np.testing.assert_array_equal(g["tokens"].cpu().numpy(), o["tokens"])
        np.testing.assert_array_equal(gp, o["parents"][0])
