"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding and the oracle on the same seeded inputs, and compare them with the
bars the method's correctness statement fixes:
  * mask, depth, greedy accept length and tokens: bit-exact;
  * stochastic decisions: bit-exact except requests where either side saw a
    near-tie (|u - alpha| < 1e-6, or an inverse-CDF draw within 1e-6 of a
    bucket edge), whose results must still be valid paths;
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


def assert_verify_match(g, o, parents, tokens, offsets, what=""):
    """Bit-exact on every request without a near-tie on either side; the
    near-tie requests must still return a valid accepted path."""
    np.testing.assert_array_equal(g["status"], o["status"], err_msg=what)
    ok = o["status"] == 0
    tie = (g["near_ties"] > 0) | (o["near_ties"] > 0)
    exact = ok & ~tie
    np.testing.assert_array_equal(g["accept_len"][exact], o["accept_len"][exact], err_msg=what)
    np.testing.assert_array_equal(g["path_nodes"][exact], o["path_nodes"][exact], err_msg=what)
    np.testing.assert_array_equal(g["out_tokens"][exact], o["out_tokens"][exact], err_msg=what)
    for b in np.nonzero(ok & tie)[0]:
        a = int(g["accept_len"][b])
        lo = int(offsets[b])
        pn = g["path_nodes"][b]
        assert pn[0] == 0
        for j in range(1, a + 1):
            assert parents[lo + pn[j]] == pn[j - 1], what
            assert g["out_tokens"][b, j - 1] == tokens[lo + pn[j]], what
        assert (pn[a + 1:] == -1).all() and (g["out_tokens"][b, a + 1:] == -1).all()
    return int(tie.sum())
