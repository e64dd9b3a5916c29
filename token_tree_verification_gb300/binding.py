"""ctypes binding of ``libspec_tree.so`` (declared in include/spec_tree.h).

Argument marshalling only: torch tensors are checked for device, dtype and
contiguity, and their device pointers plus the current CUDA stream are passed
to the C ABI.  Every step of the computation runs in the library's CUDA
kernels; if the library cannot be loaded the calls raise, there is no CPU
fallback.

The library launches on the current CUDA device, so a call's tensors must
live there (``torch.cuda.set_device`` or ``with torch.cuda.device(...)``
around calls on another GPU).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None

STATUS = {
    0: "SPEC_OK", -1: "SPEC_ERR_NULL", -2: "SPEC_ERR_SHAPE", -3: "SPEC_ERR_DTYPE",
    -4: "SPEC_ERR_TREE_TOO_LARGE", -5: "SPEC_ERR_BAD_PARENT", -6: "SPEC_ERR_TOKEN_RANGE",
    -7: "SPEC_ERR_WORKSPACE", -8: "SPEC_ERR_CUDA", -9: "SPEC_ERR_TIMEOUT",
    -10: "SPEC_ERR_PREFIX_RANGE", -11: "SPEC_ERR_ALIGNMENT", -12: "SPEC_ERR_INDEX",
}
SPEC_F32, SPEC_BF16 = 0, 1
MAX_TREE_NODES = 128


class SpecError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)}")


def lib_path() -> str:
    """The library ``load()`` opens: the bounds-checked build when the
    environment sets ``SPEC_TREE_CHECKED=1`` (built by ``build(checked=True)``),
    the normal one otherwise."""
    if os.environ.get("SPEC_TREE_CHECKED", "0") == "1":
        return os.path.join(_HERE, "libspec_tree_checked.so")
    return os.path.join(_HERE, "libspec_tree.so")


def load():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with token_tree_verification_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I, U64, SZ, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t, ctypes.c_float
    lib.spec_build_tree_mask.argtypes = [P, P, I, I, P, P, P, P]
    lib.spec_build_tree_mask.restype = I
    lib.spec_tree_attn_workspace_size.argtypes = [I, I, I, I, I, I]
    lib.spec_tree_attn_workspace_size.restype = SZ
    lib.spec_tree_attn.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, P, P, P, F, P, SZ, P, P]
    lib.spec_tree_attn.restype = I
    lib.spec_tree_attn_ex.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, P, P, P, P, F, P, SZ, I, P, P]
    lib.spec_tree_attn_ex.restype = I
    lib.spec_tree_verify_workspace_size.argtypes = [I, I, I]
    lib.spec_tree_verify_workspace_size.restype = SZ
    lib.spec_tree_verify.argtypes = [P, P, P, P, P, I, I, I, F, U64, P, P, P, P, I, P, SZ, P, P]
    lib.spec_tree_verify.restype = I
    lib.spec_tree_verify_top_p.argtypes = [P, P, P, P, P, I, I, I, F, F, U64, P, P, P, P, I, P, SZ, P, P]
    lib.spec_tree_verify_top_p.restype = I
    lib.spec_kv_compact.argtypes = [P, P, I, I, I, I, I, P, P, P, P, I, P, P, P]
    lib.spec_kv_compact.restype = I
    lib.spec_tree_expand.argtypes = [P, P, P, P, I, I, I, F, U64, P, P, P, P]
    lib.spec_tree_expand.restype = I
    lib.spec_tree_prune.argtypes = [P, P, P, P, I, I, P, P, P, P, P, P]
    lib.spec_tree_prune.restype = I
    lib.spec_tree_merge.argtypes = [P, P, P, P, P, P, I, I, I, P, P, P, P, P, P]
    lib.spec_tree_merge.restype = I
    lib.spec_philox_uniforms.argtypes = [U64, P, I, P, P]
    lib.spec_philox_uniforms.restype = I
    lib.spec_status_string.argtypes = [I]
    lib.spec_status_string.restype = ctypes.c_char_p
    lib.spec_build_checked.argtypes = []
    lib.spec_build_checked.restype = I
    _lib = lib
    return lib


def status_string(code: int) -> str:
    try:
        return load().spec_status_string(int(code)).decode()
    except Exception:  # library absent: fall back to the name table
        return STATUS.get(int(code), f"status {code}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, dtype, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _check(code: int, where: str):
    if code != 0:
        raise SpecError(code, where)


def build_tree_mask(parents, offsets, status, mask=None, depth=None, stream=None):
    """Step A1.  parents [T] int32, offsets [B+1] int32, status [B] int32 (zeroed
    by the caller).  Returns (mask [T, 4] int32 view of the uint32 bits, depth [T])."""
    lib = load()
    _dev(parents, torch.int32, "parents")
    _dev(offsets, torch.int32, "offsets")
    _dev(status, torch.int32, "status")
    T, B = parents.numel(), offsets.numel() - 1
    if mask is None:
        mask = torch.empty((T, 4), dtype=torch.int32, device=parents.device)
    if depth is None:
        depth = torch.empty(T, dtype=torch.int32, device=parents.device)
    _check(lib.spec_build_tree_mask(_ptr(parents), _ptr(offsets), B, T, _ptr(mask), _ptr(depth),
                                    _ptr(status), _stream(stream)), "spec_build_tree_mask")
    return mask, depth


def tree_attn_workspace_size(B, T, Hq, Hkv, D, max_prefix) -> int:
    return int(load().spec_tree_attn_workspace_size(B, T, Hq, Hkv, D, max_prefix))


def tree_attn(q, k_cache, v_cache, prefix_lens, offsets, mask, max_prefix, status, o=None,
              softmax_scale: float = 0.0, workspace=None, stream=None, max_ctas: int = 0,
              parents=None):
    """Steps A2-A3.  q [T, Hq, D]; k_cache, v_cache [B, Hkv, S_cap, D]; bf16 or fp32.
    ``max_ctas`` > 0 plans the launch for that many resident CTAs, leaving
    the other SMs to concurrent work; with ``mask=None`` the kernel builds
    every row's ancestor set from ``parents`` (both spec_tree_attn_ex)."""
    lib = load()
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise TypeError("q must be bfloat16 or float32")
    _dev(q, dt, "q")
    _dev(k_cache, dt, "k_cache")
    _dev(v_cache, dt, "v_cache")
    _dev(prefix_lens, torch.int32, "prefix_lens")
    _dev(offsets, torch.int32, "offsets")
    if mask is None:
        if parents is None:
            raise ValueError("tree_attn needs a mask or the parent array")
        _dev(parents, torch.int32, "parents")
    else:
        _dev(mask, torch.int32, "mask")
    _dev(status, torch.int32, "status")
    T, Hq, D = q.shape
    B, Hkv, S_cap, D2 = k_cache.shape
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("q / k_cache / v_cache shapes disagree")
    if o is None:
        o = torch.empty_like(q)
    ws_need = tree_attn_workspace_size(B, T, Hq, Hkv, D, max_prefix)
    if ws_need and workspace is None:
        workspace = torch.zeros(ws_need, dtype=torch.uint8, device=q.device)
    _check(lib.spec_tree_attn_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o),
                                 SPEC_BF16 if dt == torch.bfloat16 else SPEC_F32, B, T, Hq, Hkv, D,
                                 S_cap, int(max_prefix), _ptr(prefix_lens), _ptr(offsets),
                                 _ptr(mask), _ptr(parents) if mask is None else None,
                                 float(softmax_scale), _ptr(workspace),
                                 0 if workspace is None else workspace.numel(), int(max_ctas),
                                 _ptr(status), _stream(stream)), "spec_tree_attn_ex")
    return o


def tree_verify_workspace_size(B, T, V) -> int:
    return int(load().spec_tree_verify_workspace_size(B, T, V))


def make_verify_workspace(B, T, V, device="cuda"):
    """A zero-filled verification workspace (reusable across calls on one stream)."""
    return torch.zeros(tree_verify_workspace_size(B, T, V), dtype=torch.uint8, device=device)


def tree_verify(target_logits, draft_logits, tokens, parents, offsets, temperature: float,
                seed: int, max_depth_plus1: int, status, workspace, outputs=None, stream=None,
                top_p: float = 1.0):
    """Steps V1-V4 (top_p < 1: on the top_p nucleus of p and of q).  Returns
    dict(accept_len, path_nodes, out_tokens, near_ties) of device tensors."""
    lib = load()
    _dev(target_logits, torch.float32, "target_logits")
    if draft_logits is not None:
        _dev(draft_logits, torch.float32, "draft_logits")
    _dev(tokens, torch.int32, "tokens")
    _dev(parents, torch.int32, "parents")
    _dev(offsets, torch.int32, "offsets")
    _dev(status, torch.int32, "status")
    _dev(workspace, torch.uint8, "workspace")
    T, V = target_logits.shape
    B = offsets.numel() - 1
    W = int(max_depth_plus1)
    dev = target_logits.device
    if outputs is None:
        outputs = dict(
            accept_len=torch.empty(B, dtype=torch.int32, device=dev),
            path_nodes=torch.empty((B, W), dtype=torch.int32, device=dev),
            out_tokens=torch.empty((B, W), dtype=torch.int32, device=dev),
            near_ties=torch.empty(B, dtype=torch.int32, device=dev),
        )
    if top_p >= 1.0:
        _check(lib.spec_tree_verify(_ptr(target_logits), _ptr(draft_logits), _ptr(tokens),
                                    _ptr(parents), _ptr(offsets), B, T, V, float(temperature),
                                    int(seed) & (2**64 - 1), _ptr(outputs["accept_len"]),
                                    _ptr(outputs["path_nodes"]), _ptr(outputs["out_tokens"]),
                                    _ptr(outputs["near_ties"]), W, _ptr(workspace),
                                    workspace.numel(), _ptr(status), _stream(stream)),
               "spec_tree_verify")
        return outputs
    _check(lib.spec_tree_verify_top_p(_ptr(target_logits), _ptr(draft_logits), _ptr(tokens),
                                      _ptr(parents), _ptr(offsets), B, T, V, float(temperature),
                                      float(top_p), int(seed) & (2**64 - 1),
                                      _ptr(outputs["accept_len"]), _ptr(outputs["path_nodes"]),
                                      _ptr(outputs["out_tokens"]), _ptr(outputs["near_ties"]), W,
                                      _ptr(workspace), workspace.numel(), _ptr(status),
                                      _stream(stream)), "spec_tree_verify_top_p")
    return outputs


def kv_compact(k_cache, v_cache, prefix_lens, offsets, path_nodes, accept_len, status,
               new_prefix_lens=None, stream=None):
    """Depth-first KV-cache update after verification (in place).  Returns the
    new prefix lengths (device int32 [B])."""
    lib = load()
    if k_cache.dtype != v_cache.dtype or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must match")
    dt = {torch.bfloat16: SPEC_BF16, torch.float32: SPEC_F32}.get(k_cache.dtype)
    if dt is None:
        raise ValueError(f"unsupported cache dtype {k_cache.dtype}")
    for t, name in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _dev(t, k_cache.dtype, name)
    for t, name in ((prefix_lens, "prefix_lens"), (offsets, "offsets"), (path_nodes, "path_nodes"),
                    (accept_len, "accept_len"), (status, "status")):
        _dev(t, torch.int32, name)
    B, H, S_cap, D = k_cache.shape
    W = path_nodes.shape[-1]
    if new_prefix_lens is None:
        new_prefix_lens = torch.empty(B, dtype=torch.int32, device=k_cache.device)
    _check(lib.spec_kv_compact(_ptr(k_cache), _ptr(v_cache), dt, B, H, D, S_cap, _ptr(prefix_lens),
                               _ptr(offsets), _ptr(path_nodes), _ptr(accept_len), W,
                               _ptr(new_prefix_lens), _ptr(status), _stream(stream)),
           "spec_kv_compact")
    return new_prefix_lens


def tree_expand(draft_logits, parent_scores, node_ids, requests, width: int, temperature: float,
                seed: int, stream=None):
    """One level of draft-tree expansion.  Returns (child_tokens [F][width],
    child_scores [F][width], near_ties [F][width]) as device tensors."""
    lib = load()
    _dev(draft_logits, torch.float32, "draft_logits")
    _dev(parent_scores, torch.float32, "parent_scores")
    _dev(node_ids, torch.int32, "node_ids")
    _dev(requests, torch.int32, "requests")
    F, V = draft_logits.shape
    dev_ = draft_logits.device
    tok = torch.empty((F, width), dtype=torch.int32, device=dev_)
    sc = torch.empty((F, width), dtype=torch.float32, device=dev_)
    ties = torch.empty((F, width), dtype=torch.int32, device=dev_)
    _check(lib.spec_tree_expand(_ptr(draft_logits), _ptr(parent_scores), _ptr(node_ids), _ptr(requests),
                                F, V, width, float(temperature), int(seed) & (2**64 - 1), _ptr(tok),
                                _ptr(sc), _ptr(ties), _stream(stream)), "spec_tree_expand")
    return tok, sc, ties


def tree_prune(parents, tokens, scores, cand_offsets, keep: int, status, stream=None):
    """Prune candidate trees to `keep` nodes.  Returns dict(parents, tokens,
    kept, n_out) of device tensors ([B][keep] rows)."""
    lib = load()
    for t, name in ((parents, "parents"), (tokens, "tokens"), (cand_offsets, "cand_offsets"),
                    (status, "status")):
        _dev(t, torch.int32, name)
    _dev(scores, torch.float32, "scores")
    B = cand_offsets.numel() - 1
    dev_ = parents.device
    out = {k: torch.empty((B, keep), dtype=torch.int32, device=dev_) for k in ("parents", "tokens", "kept")}
    out["n_out"] = torch.empty(B, dtype=torch.int32, device=dev_)
    _check(lib.spec_tree_prune(_ptr(parents), _ptr(tokens), _ptr(scores), _ptr(cand_offsets), B, keep,
                               _ptr(out["parents"]), _ptr(out["tokens"]), _ptr(out["kept"]),
                               _ptr(out["n_out"]), _ptr(status), _stream(stream)), "spec_tree_prune")
    return out


def philox_uniforms(seed: int, counters, out=None, stream=None):
    """Step R: the uniform for each counter row (c0, c1, c2, c3) of the int64
    device tensor ``counters`` [n, 4].  Returns a float32 device tensor [n]."""
    lib = load()
    _dev(counters, torch.int64, "counters")
    if counters.dim() != 2 or counters.shape[1] != 4:
        raise ValueError("counters must be [n, 4]")
    n = counters.shape[0]
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=counters.device)
    _check(lib.spec_philox_uniforms(int(seed) & (2**64 - 1), _ptr(counters), n, _ptr(out),
                                    _stream(stream)), "spec_philox_uniforms")
    return out


def tree_merge(parents_a, tokens_a, offsets_a, parents_b, tokens_b, offsets_b, status,
               stream=None):
    """Merge two speculators' token trees per request.  Returns dict(parents,
    tokens, map_b [B][128], n_out [B]) of device tensors."""
    lib = load()
    for t, name in ((parents_a, "parents_a"), (tokens_a, "tokens_a"), (offsets_a, "offsets_a"),
                    (parents_b, "parents_b"), (tokens_b, "tokens_b"), (offsets_b, "offsets_b"),
                    (status, "status")):
        _dev(t, torch.int32, name)
    B = offsets_a.numel() - 1
    if offsets_b.numel() - 1 != B:
        raise ValueError("both trees need the same number of requests")
    dev_ = parents_a.device
    out = {k: torch.empty((B, MAX_TREE_NODES), dtype=torch.int32, device=dev_)
           for k in ("parents", "tokens", "map_b")}
    out["n_out"] = torch.empty(B, dtype=torch.int32, device=dev_)
    _check(lib.spec_tree_merge(_ptr(parents_a), _ptr(tokens_a), _ptr(offsets_a), _ptr(parents_b),
                               _ptr(tokens_b), _ptr(offsets_b), B, parents_a.numel(),
                               parents_b.numel(), _ptr(out["parents"]), _ptr(out["tokens"]),
                               _ptr(out["map_b"]), _ptr(out["n_out"]), _ptr(status),
                               _stream(stream)), "spec_tree_merge")
    return out
