"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding and the oracle on the same seeded inputs, and compare them with the
bars the method's correctness statement fixes:
  * mask, depth, greedy accept length and tokens: bit-exact;
  * stochastic decisions: every decision on the GPU's walk equals the
    oracle's decision at that node, except where the oracle's exact (fp64)
    margin there is below BAND; such exemptions are counted and bounded, and
    the GPU may only report a near-tie where the oracle finds a decision
    within BAND (the GPU's own flag exempts nothing);
  * attention: max|d| <= 1e-2 max|ref| and relative error <= 2e-2 wherever
    |ref| >= 1e-2 max|ref|."""
import numpy as np
import torch

import oracle
import token_tree_verification_gb300 as ttv

ATOL_FRAC = 1e-2
RTOL = 2e-2


def dev(x, dtype=None):
    t = torch.as_tensor(x) if not isinstance(x, torch.Tensor) else x
    if dtype is not None:
        t = t.to(dtype)
    return t.contiguous().cuda()


def gpu_mask(parents, offsets):
    B = len(offsets) - 1
    status = torch.zeros(B, dtype=torch.int32, device="cuda")
    m, d = ttv.build_tree_mask(dev(parents, torch.int32), dev(offsets, torch.int32), status)
    torch.cuda.synchronize()
    return m.cpu().numpy().view(np.uint32), d.cpu().numpy(), status.cpu().numpy()


def gpu_attn(w, mask_dev=None, status=None, max_prefix=None):
    parents = dev(w.parents, torch.int32)
    offsets = dev(w.offsets, torch.int32)
    if status is None:
        status = torch.zeros(w.B, dtype=torch.int32, device="cuda")
    if mask_dev is None:
        mask_dev, _ = ttv.build_tree_mask(parents, offsets, status)
    o = ttv.tree_attn(w.q.cuda(), w.k_cache.cuda(), w.v_cache.cuda(), dev(w.prefix_lens, torch.int32),
                      offsets, mask_dev, int(w.prefix_lens.max()) if max_prefix is None else max_prefix,
                      status)
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64), status.cpu().numpy()


def oracle_attn_rows(w, rows):
    """Oracle rows (flat node*Hq + head) computed per (request, KV head) slice,
    so caches of any size never need a full float copy."""
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.size, w.D))
    G = w.G
    node = rows // w.Hq
    head = rows % w.Hq
    req = np.searchsorted(w.offsets, node, side="right") - 1
    for b in np.unique(req):
        lo, hi = int(w.offsets[b]), int(w.offsets[b + 1])
        L = int(w.prefix_lens[b])
        for g in np.unique(head[req == b] // G):
            sel = np.nonzero((req == b) & (head // G == g))[0]
            n = hi - lo
            k = w.k_cache[b, g, :L + n].float().cpu().numpy()[None, None]
            v = w.v_cache[b, g, :L + n].float().cpu().numpy()[None, None]
            q = w.q[lo:hi, g * G:(g + 1) * G].float().cpu().numpy()
            sub_rows = (node[sel] - lo) * G + (head[sel] - g * G)
            out[sel] = oracle.tree_attn(q, k, v, np.array([L], np.int32), np.array([0, n], np.int32),
                                        w.parents[lo:hi], rows=sub_rows)
    return out


def assert_attn_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    scale = np.abs(ref).max()
    diff = np.abs(got - ref)
    assert diff.max() <= ATOL_FRAC * scale, f"{what}: max|d| {diff.max():.3e} > {ATOL_FRAC}*{scale:.3e}"
    big = np.abs(ref) >= 1e-2 * scale
    rel = diff[big] / np.abs(ref[big])
    assert rel.max() <= RTOL, f"{what}: max rel {rel.max():.3e} on {big.sum()} elements"
    return dict(max_abs=float(diff.max()), max_rel=float(rel.max()), excluded=int((~big).sum()))


def gpu_verify(w, seed, W=None, temperature=None, target=None, draft="auto", tokens=None,
               parents=None, offsets=None, top_p=1.0):
    target = w.target_logits if target is None else target
    if isinstance(draft, str):
        draft = w.draft_logits
    temp = w.temperature if temperature is None else temperature
    tokens = w.tokens if tokens is None else tokens
    parents = w.parents if parents is None else parents
    offsets = w.offsets if offsets is None else offsets
    B = len(offsets) - 1
    T, V = np.asarray(target).shape
    W = (w.max_depth + 1) if W is None else W
    status = torch.zeros(B, dtype=torch.int32, device="cuda")
    ws = ttv.make_verify_workspace(B, T, V)
    r = ttv.tree_verify(dev(target, torch.float32), None if (draft is None or temp == 0) else dev(draft, torch.float32),
                        dev(tokens, torch.int32), dev(parents, torch.int32), dev(offsets, torch.int32),
                        temp, seed, W, status, ws, top_p=top_p)
    torch.cuda.synchronize()
    out = {k: v.cpu().numpy() for k, v in r.items()}
    out["status"] = status.cpu().numpy()
    return out


def oracle_verify(w, seed, W=None, temperature=None, top_p=1.0):
    temp = w.temperature if temperature is None else temperature
    return oracle.tree_verify(w.target_logits, w.draft_logits if temp > 0 else None, w.tokens,
                              w.parents, w.offsets, temp, seed, (w.max_depth + 1) if W is None else W,
                              top_p=top_p)


# A float32 implementation of the accept test and the inverse-CDF draw is
# accurate to a few 1e-6 of the exact threshold (fp32 sums over up to 1.5e5
# entries, ~4-ulp exponentials, the closed-form residual); a decision whose
# exact fp64 distance from its threshold is below BAND may legitimately be
# taken the other way.  BAND is 10x the near-tie band of the method.
BAND = 1e-5


def walk_nodes(res, offsets):
    """Global node ids on each request's walk: the root, the accepted nodes
    (the last one is where the walk stopped)."""
    out = []
    for b in range(len(offsets) - 1):
        if res["status"][b] != 0:
            out.append([])
            continue
        a = int(res["accept_len"][b])
        out.append([int(offsets[b]) + int(u) for u in res["path_nodes"][b][:a + 1]])
    return out


def assert_verify_match(g, o, parents, tokens, offsets, what="", nodes=None, max_exempt=1):
    """Compare a GPU verification result ``g`` with the oracle's walk ``o``.

    ``nodes`` is the oracle's per-node evaluation (``oracle.verify_nodes``)
    covering every node on both walks.  Each decision on the GPU's walk must
    equal the oracle's decision at that node unless the oracle's margin there
    is below BAND (an exemption; at most ``max_exempt`` over the call); the
    GPU's walk must be a valid path; the GPU's near-tie count on a request
    must not exceed the number of decisions the oracle finds within BAND on
    that walk.  Returns the number of exemptions."""
    np.testing.assert_array_equal(g["status"], o["status"], err_msg=what)
    off = np.asarray(offsets)
    exempt = 0
    ow = walk_nodes(o, off)
    gw = walk_nodes(g, off)
    for b in np.nonzero(o["status"] == 0)[0]:
        lo = int(off[b])
        # the oracle's walk follows its own per-node decisions
        for j, t in enumerate(ow[b]):
            nxt = ow[b][j + 1] - lo if j + 1 < len(ow[b]) else -1
            assert nodes["next"][t] == nxt, f"{what}: oracle walk / node decisions, request {b}"
            if nxt < 0:
                assert nodes["token"][t] == o["out_tokens"][b, j], what
        a = int(g["accept_len"][b])
        pn = g["path_nodes"][b]
        assert pn[0] == 0, what
        assert (pn[a + 1:] == -1).all() and (g["out_tokens"][b, a + 1:] == -1).all(), what
        support = 0
        for j, t in enumerate(gw[b]):
            assert nodes["next"][t] != -2, f"{what}: node {t} not evaluated"
            if j < a:
                nxt = int(pn[j + 1])
                assert parents[lo + nxt] == pn[j], f"{what}: request {b} path is not a tree path"
                assert g["out_tokens"][b, j] == tokens[lo + nxt], what
                same = nodes["next"][t] == nxt
            else:
                same = nodes["next"][t] == -1 and nodes["token"][t] == g["out_tokens"][b, j]
            if not same:
                assert nodes["margin"][t] < BAND, (
                    f"{what}: request {b} node {t - lo}: GPU decision differs from the oracle's, "
                    f"oracle margin {nodes['margin'][t]:.3e} >= {BAND}")
                exempt += 1
                support += 1 << 20     # the GPU took other decisions at this node
            support += int(nodes["n_close"][t])
        assert g["near_ties"][b] <= support, (
            f"{what}: request {b}: GPU reports {g['near_ties'][b]} near-ties, the oracle finds "
            f"{support} decisions within {BAND} on that walk")
    assert exempt <= max_exempt, f"{what}: {exempt} exempted decisions > {max_exempt}"
    return exempt


def oracle_nodes_for(g, o, target, draft, tokens, parents, offsets, temperature, seed, W, top_p=1.0):
    """The oracle's per-node decisions on every node of both walks."""
    want = np.zeros(np.asarray(target).shape[0], np.uint8)
    for walk in walk_nodes(o, offsets) + walk_nodes(g, offsets):
        want[walk] = 1
    return oracle.verify_nodes(target, draft if temperature > 0 else None, tokens, parents, offsets,
                               temperature, seed, W, top_p=top_p, band=BAND, want=want)


def check_verify(w, seed, W=None, temperature=None, top_p=1.0, max_exempt=1, what=None, **kw):
    """GPU verification of workload ``w`` against the oracle (walk and
    per-node decisions).  Returns (gpu result, oracle result, exemptions)."""
    temp = w.temperature if temperature is None else temperature
    W = (w.max_depth + 1) if W is None else W
    g = gpu_verify(w, seed, W=W, temperature=temp, top_p=top_p, **kw)
    target = kw.get("target", w.target_logits)
    tokens = kw.get("tokens", w.tokens)
    parents = kw.get("parents", w.parents)
    offsets = kw.get("offsets", w.offsets)
    draft = w.draft_logits if kw.get("draft", "auto") == "auto" else kw["draft"]
    o = oracle.tree_verify(target, draft if temp > 0 else None, tokens, parents, offsets, temp, seed,
                           W, top_p=top_p)
    nodes = oracle_nodes_for(g, o, target, draft, tokens, parents, offsets, temp, seed, W, top_p)
    what = what or f"{w.name} seed {seed} T={temp} top_p={top_p}"
    ex = assert_verify_match(g, o, parents, tokens, offsets, what, nodes=nodes, max_exempt=max_exempt)
    return g, o, ex
