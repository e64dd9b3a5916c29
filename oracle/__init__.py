"""CPU oracle for token-tree verification (ctypes wrapper over ``oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline leg.  The product library never imports,
links or calls anything here, and this package never imports the product.

All arithmetic lives in ``oracle.c`` (plain single-threaded C, IEEE double);
this module only marshals numpy arrays.  Inputs are taken as float32 (bf16
values widen to float32 exactly), so the oracle reads the same numbers as the
GPU path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` with plain gcc (-O2, no
    OpenMP, no BLAS, no -march flags: the same source builds on x86 and Arm)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
             "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    P = ctypes.c_void_p
    i32, i64, u64 = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
    lib.oracle_philox4x64_10.argtypes = [P, P, P]
    lib.oracle_philox4x64_10.restype = None
    lib.oracle_uniform.argtypes = [u64, i64, i64, i64]
    lib.oracle_uniform.restype = ctypes.c_double
    lib.oracle_uniforms.argtypes = [u64, P, i64, P]
    lib.oracle_uniforms.restype = None
    lib.oracle_build_mask.argtypes = [P, P, i32, i32, P, P, P]
    lib.oracle_build_mask.restype = i32
    lib.oracle_tree_attn.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32,
                                     P, P, P, ctypes.c_double, P, i64]
    lib.oracle_tree_attn.restype = i32
    lib.oracle_tree_verify.argtypes = [P, P, P, P, P, i32, i32, i32, ctypes.c_float,
                                       u64, P, P, P, P, i32, P]
    lib.oracle_tree_verify.restype = i32
    lib.oracle_tree_verify_top_p.argtypes = [P, P, P, P, P, i32, i32, i32, ctypes.c_float,
                                             ctypes.c_double, u64, P, P, P, P, i32, P]
    lib.oracle_tree_verify_top_p.restype = i32
    lib.oracle_kv_compact.argtypes = [P, i32, i32, i32, i32, i32, P, P, P, P, i32, P, P]
    lib.oracle_kv_compact.restype = i32
    lib.oracle_tree_expand.argtypes = [P, P, P, P, i32, i32, i32, ctypes.c_double, u64, P, P, P, P]
    lib.oracle_tree_expand.restype = i32
    lib.oracle_tree_prune.argtypes = [P, P, P, P, i32, i32, P, P, P, P, P]
    lib.oracle_tree_prune.restype = i32
    lib.oracle_tree_merge.argtypes = [P, P, P, P, P, P, i32, i32, P, P, P, P, P]
    lib.oracle_tree_merge.restype = i32
    lib.oracle_verify_nodes.argtypes = [P, P, P, P, P, i32, i32, i32, ctypes.c_float,
                                        ctypes.c_double, u64, i32, ctypes.c_double, P, P, P, P, P, P]
    lib.oracle_verify_nodes.restype = i32
    lib.oracle_nucleus_alternatives.argtypes = [P, i32, ctypes.c_double, P, P]
    lib.oracle_nucleus_alternatives.restype = i32
    lib.oracle_nucleus_max_alternatives.argtypes = []
    lib.oracle_nucleus_max_alternatives.restype = i32
    _lib = lib
    return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def philox4x64_10(counter, key) -> np.ndarray:
    """One Philox4x64-10 block: counter = 4 uint64 words, key = 2 uint64 words."""
    ctr = _c(counter, np.uint64)
    k = _c(key, np.uint64)
    out = np.zeros(4, dtype=np.uint64)
    _load().oracle_philox4x64_10(_ptr(ctr), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, node: int, request: int, kind: int) -> float:
    """The method's uniform for (request, node, kind), in [0, 1)."""
    return float(_load().oracle_uniform(seed & (2**64 - 1), node, request, kind))


def uniforms(seed: int, counters) -> np.ndarray:
    """The uniform of every counter row (c0, c1, c2, c3) of ``counters`` [n, 4]
    (any integer dtype; words taken as uint64), key (seed, 0)."""
    ctr = np.ascontiguousarray(np.asarray(counters).astype(np.int64).view(np.uint64))
    n = ctr.shape[0]
    out = np.zeros(n, np.float64)
    _load().oracle_uniforms(seed & (2**64 - 1), _ptr(ctr), n, _ptr(out))
    return out


def build_mask(parents, offsets):
    """Ancestor-or-self bitmask [T, 4] uint32, depth [T] int32, status [B]."""
    par = _c(parents, np.int32)
    off = _c(offsets, np.int32)
    B, T = off.size - 1, par.size
    mask = np.zeros((T, 4), dtype=np.uint32)
    depth = np.full(T, -1, dtype=np.int32)
    status = np.zeros(B, dtype=np.int32)
    rc = _load().oracle_build_mask(_ptr(par), _ptr(off), B, T, _ptr(mask), _ptr(depth), _ptr(status))
    if rc != 0:
        raise ValueError(f"oracle_build_mask: status {rc}")
    return mask, depth, status


def tree_attn(q, k, v, prefix_lens, offsets, parents, scale: float = 0.0, rows=None):
    """Dense masked attention per (node, head) in float64.

    q [T, Hq, D]; k, v [B, Hkv, S_cap, D] (float32 or anything that widens to
    it exactly).  Returns [T, Hq, D] float64, or [len(rows), D] when ``rows``
    (flat node*Hq + head indices) is given."""
    qa = _c(q, np.float32)
    ka = _c(k, np.float32)
    va = _c(v, np.float32)
    T, Hq, D = qa.shape
    B, Hkv, S_cap, D2 = ka.shape
    assert D2 == D and va.shape == ka.shape
    pl = _c(prefix_lens, np.int32)
    off = _c(offsets, np.int32)
    par = _c(parents, np.int32)
    if rows is None:
        out = np.zeros((T, Hq, D), dtype=np.float64)
        rows_a, nrows = None, T * Hq
    else:
        rows_a = _c(rows, np.int64)
        nrows = rows_a.size
        out = np.zeros((nrows, D), dtype=np.float64)
    rc = _load().oracle_tree_attn(_ptr(qa), _ptr(ka), _ptr(va), _ptr(out), B, T, Hq, Hkv, D,
                                  S_cap, _ptr(pl), _ptr(off), _ptr(par), float(scale),
                                  _ptr(rows_a), nrows)
    if rc != 0:
        raise ValueError(f"oracle_tree_attn: status {rc}")
    return out


def tree_verify(target_logits, draft_logits, tokens, parents, offsets, temperature: float,
                seed: int, max_depth_plus1: int, top_p: float = 1.0):
    """Sequential root-to-leaf verification walk per request (with the target
    and draft distributions filtered to their top_p nucleus when top_p < 1).

    Returns a dict of numpy arrays: accept_len [B], path_nodes [B, W],
    out_tokens [B, W], near_ties [B], status [B]."""
    tl = _c(target_logits, np.float32)
    T, V = tl.shape
    dl = None if draft_logits is None else _c(draft_logits, np.float32)
    tok = _c(tokens, np.int32)
    par = _c(parents, np.int32)
    off = _c(offsets, np.int32)
    B = off.size - 1
    W = int(max_depth_plus1)
    res = dict(
        accept_len=np.full(B, -1, dtype=np.int32),
        path_nodes=np.full((B, W), -1, dtype=np.int32),
        out_tokens=np.full((B, W), -1, dtype=np.int32),
        near_ties=np.zeros(B, dtype=np.int32),
        status=np.zeros(B, dtype=np.int32),
    )
    if top_p >= 1.0:
        rc = _load().oracle_tree_verify(
            _ptr(tl), _ptr(dl), _ptr(tok), _ptr(par), _ptr(off), B, T, V,
            ctypes.c_float(temperature), seed & (2**64 - 1),
            _ptr(res["accept_len"]), _ptr(res["path_nodes"]), _ptr(res["out_tokens"]),
            _ptr(res["near_ties"]), W, _ptr(res["status"]))
    else:
        rc = _load().oracle_tree_verify_top_p(
            _ptr(tl), _ptr(dl), _ptr(tok), _ptr(par), _ptr(off), B, T, V,
            ctypes.c_float(temperature), float(top_p), seed & (2**64 - 1),
            _ptr(res["accept_len"]), _ptr(res["path_nodes"]), _ptr(res["out_tokens"]),
            _ptr(res["near_ties"]), W, _ptr(res["status"]))
    if rc != 0:
        raise ValueError(f"oracle_tree_verify: status {rc}")
    return res


def verify_nodes(target_logits, draft_logits, tokens, parents, offsets, temperature: float,
                 seed: int, max_depth_plus1: int, top_p: float = 1.0, band: float = 1e-5,
                 want=None):
    """The decisions at every node (or every node with ``want[t]``) as if the
    walk reached it: dict of next [T] (accepted child, request-local, or -1 to
    stop; -2 when not evaluated), token [T] (the emitted token when stopping),
    margin [T] (smallest distance of a decision from its threshold; inf for
    greedy, 0 for a fragile top-p node), n_close [T] (decisions within
    ``band``, top-p: plus those involving an entry near tau), status [B]."""
    tl = _c(target_logits, np.float32)
    T, V = tl.shape
    dl = None if draft_logits is None else _c(draft_logits, np.float32)
    tok = _c(tokens, np.int32)
    par = _c(parents, np.int32)
    off = _c(offsets, np.int32)
    B = off.size - 1
    wa = None if want is None else _c(want, np.uint8)
    res = dict(next=np.zeros(T, np.int32), token=np.zeros(T, np.int32),
               margin=np.zeros(T, np.float64), n_close=np.zeros(T, np.int32),
               status=np.zeros(B, np.int32))
    rc = _load().oracle_verify_nodes(
        _ptr(tl), _ptr(dl), _ptr(tok), _ptr(par), _ptr(off), B, T, V, ctypes.c_float(temperature),
        float(top_p), seed & (2**64 - 1), int(max_depth_plus1), float(band), _ptr(wa),
        _ptr(res["next"]), _ptr(res["token"]), _ptr(res["margin"]), _ptr(res["n_close"]),
        _ptr(res["status"]))
    if rc != 0:
        raise ValueError(f"oracle_verify_nodes: status {rc}")
    return res


def nucleus_alternatives(d, top_p: float):
    """The plausible top-p nuclei of distribution ``d`` (float64 [V]):
    (tau, keep-flags [n][V] bool, row 0 the exact nucleus), or (tau, None)
    when there are more than the enumeration takes."""
    lib = _load()
    da = _c(d, np.float64)
    V = da.size
    keeps = np.zeros((lib.oracle_nucleus_max_alternatives(), V), np.uint8)
    tau = ctypes.c_double(0.0)
    n = lib.oracle_nucleus_alternatives(_ptr(da), V, float(top_p), _ptr(keeps), ctypes.byref(tau))
    if n < -1:
        raise ValueError("oracle_nucleus_alternatives: allocation failed")
    return tau.value, (None if n < 0 else keeps[:n].astype(bool))


def kv_compact(cache, prefix_lens, offsets, path_nodes, accept_len, status=None):
    """Depth-first KV-cache update (oracle_kv_compact) on a copy of ``cache``
    ([B][H][S_cap][D], any fixed-size dtype).  Returns (new_cache,
    new_prefix_lens, status)."""
    lib = _load()
    c = np.array(cache, copy=True, order="C")
    B, H, S_cap, D = c.shape
    pn = _c(path_nodes, np.int32)
    W = pn.shape[1]
    st = np.zeros(B, np.int32) if status is None else _c(status, np.int32).copy()
    newp = np.zeros(B, np.int32)
    rc = lib.oracle_kv_compact(_ptr(c), c.dtype.itemsize, B, H, S_cap, D,
                               _ptr(_c(prefix_lens, np.int32)), _ptr(_c(offsets, np.int32)),
                               _ptr(pn), _ptr(_c(accept_len, np.int32)), W, _ptr(newp), _ptr(st))
    if rc != 0:
        raise ValueError(f"oracle_kv_compact: {rc}")
    return c, newp, st


def tree_expand(draft, parent_scores, node_ids, reqs, width: int, temperature: float, seed: int,
                with_gaps: bool = False):
    """One level of draft-tree expansion (oracle_tree_expand).  Returns
    (tokens [F][width], scores [F][width], ties [F][width]), plus gaps
    [F][width] (each draw's relative distance from the nearer inverse-CDF
    boundary) with ``with_gaps``."""
    lib = _load()
    d = _c(draft, np.float32)
    F, V = d.shape
    tok = np.zeros((F, width), np.int32)
    sc = np.zeros((F, width), np.float64)
    ties = np.zeros((F, width), np.int32)
    gaps = np.zeros((F, width), np.float64)
    rc = lib.oracle_tree_expand(_ptr(d), _ptr(_c(parent_scores, np.float64)), _ptr(_c(node_ids, np.int32)),
                                _ptr(_c(reqs, np.int32)), F, V, width, float(temperature),
                                int(seed) & (2**64 - 1), _ptr(tok), _ptr(sc), _ptr(ties), _ptr(gaps))
    if rc != 0:
        raise ValueError(f"oracle_tree_expand: {rc}")
    return (tok, sc, ties, gaps) if with_gaps else (tok, sc, ties)


def tree_prune(parents, tokens, scores, cand_offsets, keep: int):
    """Pruning of candidate trees to `keep` nodes (oracle_tree_prune).  Returns
    dict(parents, tokens, kept, n_out, status) with [B][keep] rows."""
    lib = _load()
    off = _c(cand_offsets, np.int32)
    B = off.size - 1
    out = {k: np.zeros((B, keep), np.int32) for k in ("parents", "tokens", "kept")}
    out["n_out"] = np.zeros(B, np.int32)
    out["status"] = np.zeros(B, np.int32)
    rc = lib.oracle_tree_prune(_ptr(_c(parents, np.int32)), _ptr(_c(tokens, np.int32)),
                               _ptr(_c(scores, np.float64)), _ptr(off), B, keep, _ptr(out["parents"]),
                               _ptr(out["tokens"]), _ptr(out["kept"]), _ptr(out["n_out"]), _ptr(out["status"]))
    if rc != 0:
        raise ValueError(f"oracle_tree_prune: {rc}")
    return out


def tree_merge(parents_a, tokens_a, off_a, parents_b, tokens_b, off_b, cap: int = 128):
    """Merge two speculators' token trees per request (oracle_tree_merge).
    Returns dict(parents, tokens, map_b [B][cap], n_out [B], status [B])."""
    lib = _load()
    oa, ob = _c(off_a, np.int32), _c(off_b, np.int32)
    B = oa.size - 1
    out = {k: np.zeros((B, cap), np.int32) for k in ("parents", "tokens", "map_b")}
    out["n_out"] = np.zeros(B, np.int32)
    out["status"] = np.zeros(B, np.int32)
    rc = lib.oracle_tree_merge(_ptr(_c(parents_a, np.int32)), _ptr(_c(tokens_a, np.int32)), _ptr(oa),
                               _ptr(_c(parents_b, np.int32)), _ptr(_c(tokens_b, np.int32)), _ptr(ob),
                               B, cap, _ptr(out["parents"]), _ptr(out["tokens"]), _ptr(out["map_b"]),
                               _ptr(out["n_out"]), _ptr(out["status"]))
    if rc != 0:
        raise ValueError(f"oracle_tree_merge: {rc}")
    return out
