"""spec_tree_verify_static, the verification entry point that allocates
nothing: its scratch is a fixed array inside the library, for callers (engine
plugins, runtimes without a CUDA allocator) that can pass only inputs and
outputs.

It must agree exactly with spec_tree_verify (same kernels, integer outputs)
on consecutive calls, since every call reuses the array and finds the
previous call's contents in it, and with the oracle decision by decision,
as spec_tree_verify does.  This file is collected last so that a run
stopping at the first failure has run every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from parity import assert_verify_match, dev, gpu_verify, oracle_nodes_for
from token_tree_verification_gb300 import binding, synthetic

SCRATCH_BYTES = 256 * 1024
SPEC_ERR_WORKSPACE = -7


def _fn(lib):
    P, I, U64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float
    fn = lib.spec_tree_verify_static
    fn.argtypes = [P, P, P, P, P, I, I, I, F, U64, P, P, P, P, I, P, P]
    fn.restype = I
    return fn


def _call_static(fn, w, seed, temperature):
    B = len(w.offsets) - 1
    T, V = w.target_logits.shape
    W = w.max_depth + 1
    target = dev(w.target_logits, torch.float32)
    draft = dev(w.draft_logits, torch.float32) if temperature > 0 else None
    tokens, parents = dev(w.tokens, torch.int32), dev(w.parents, torch.int32)
    offsets = dev(w.offsets, torch.int32)
    out = dict(accept_len=torch.full((B,), -7, dtype=torch.int32, device="cuda"),
               path_nodes=torch.full((B, W), -7, dtype=torch.int32, device="cuda"),
               out_tokens=torch.full((B, W), -7, dtype=torch.int32, device="cuda"),
               near_ties=torch.full((B,), -7, dtype=torch.int32, device="cuda"))
    status = torch.zeros(B, dtype=torch.int32, device="cuda")
    rc = fn(target.data_ptr(), None if draft is None else draft.data_ptr(), tokens.data_ptr(),
            parents.data_ptr(), offsets.data_ptr(), B, T, V, float(temperature), seed,
            out["accept_len"].data_ptr(), out["path_nodes"].data_ptr(),
            out["out_tokens"].data_ptr(), out["near_ties"].data_ptr(), W, status.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, binding.status_string(rc)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["status"] = status.cpu().numpy()
    return res


def test_static_scratch_limit_rejected_on_host():
    """Sizes beyond the fixed scratch are refused before any device work
    (this runs without a GPU: the refusal precedes every CUDA call)."""
    lib = binding.load()
    fn = _fn(lib)
    B, T, V = 512, 65536, 32000
    assert lib.spec_tree_verify_workspace_size(B, T, V) > SCRATCH_BYTES
    fake = ctypes.c_void_p(256)  # never dereferenced: the call returns first
    rc = fn(fake, fake, fake, fake, fake, B, T, V, 0.0, 0, fake, fake, fake, fake, 8, fake, None)
    assert rc == SPEC_ERR_WORKSPACE


@pytest.mark.gpu
def test_static_matches_workspace_entry_point_on_consecutive_calls():
    fn = _fn(binding.load())
    # only the logits and trees matter here: keep the (unused) KV caches small
    cases = [("llama7b", 0.7, 11, dict(L=64, Hq=1, Hkv=1)),
             ("dynamic", 0.7, 12, dict(L_range=(16, 32), Hq=1, Hkv=1)),
             ("llama7b", 0.0, 13, dict(L=64, Hq=1, Hkv=1))]
    for name, temp, seed, small in cases:
        w = synthetic.make_workload(name, seed=seed, temperature=temp, **small)
        got = _call_static(fn, w, seed, temp)
        ref = gpu_verify(w, seed, temperature=temp)
        for k in ("status", "accept_len", "path_nodes", "out_tokens", "near_ties"):
            np.testing.assert_array_equal(got[k], ref[k], err_msg=f"{name} T={temp}: {k}")
        assert (got["status"] == 0).all()
        W = w.max_depth + 1
        draft = w.draft_logits if temp > 0 else None
        o = oracle.tree_verify(w.target_logits, draft, w.tokens, w.parents, w.offsets, temp, seed, W)
        nodes = oracle_nodes_for(got, o, w.target_logits, draft, w.tokens, w.parents, w.offsets,
                                 temp, seed, W)
        assert_verify_match(got, o, w.parents, w.tokens, w.offsets, f"static {name} T={temp}",
                            nodes=nodes)
