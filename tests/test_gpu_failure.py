"""Verification's failure path on the GPU without a fault: one request's
first statistics exchange is withheld (spec_test_verify_timeout), so the
bounded waits on it, limited to 1 ms, run out.  The kernel returns, that
request reports SPEC_ERR_TIMEOUT and keeps its outputs as they were, the
other requests are verified exactly as by spec_tree_verify, and the same
workspace serves a normal call afterwards."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from parity import assert_verify_match, dev, oracle_nodes_for
from token_tree_verification_gb300 import binding, synthetic

pytestmark = pytest.mark.gpu
SPEC_ERR_TIMEOUT = -9


def _fn(lib):
    P, I, U64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t
    fn = lib.spec_test_verify_timeout
    fn.argtypes = [P, P, P, P, P, I, I, I, F, U64, P, P, P, P, I, P, SZ, P, P, U64, I]
    fn.restype = I
    return fn


def test_withheld_exchange_times_out_one_request(gpu_lib):
    fn = _fn(binding.load())
    w = synthetic.make_workload("llama7b", seed=4, B=3, L=32, Hq=1, Hkv=1)
    B, (T, V), W = w.B, w.target_logits.shape, w.max_depth + 1
    tl, dl = dev(w.target_logits, torch.float32), dev(w.draft_logits, torch.float32)
    tok, par, off = dev(w.tokens, torch.int32), dev(w.parents, torch.int32), dev(w.offsets, torch.int32)
    ws = gpu_lib.make_verify_workspace(B, T, V)
    seed = 21
    o = oracle.tree_verify(w.target_logits, w.draft_logits, w.tokens, w.parents, w.offsets,
                           w.temperature, seed, W)
    for rep in range(2):
        out = dict(accept_len=torch.full((B,), -7, dtype=torch.int32, device="cuda"),
                   path_nodes=torch.full((B, W), -7, dtype=torch.int32, device="cuda"),
                   out_tokens=torch.full((B, W), -7, dtype=torch.int32, device="cuda"),
                   near_ties=torch.full((B,), -7, dtype=torch.int32, device="cuda"))
        status = torch.zeros(B, dtype=torch.int32, device="cuda")
        rc = fn(tl.data_ptr(), dl.data_ptr(), tok.data_ptr(), par.data_ptr(), off.data_ptr(), B, T,
                V, w.temperature, seed, out["accept_len"].data_ptr(), out["path_nodes"].data_ptr(),
                out["out_tokens"].data_ptr(), out["near_ties"].data_ptr(), W, ws.data_ptr(),
                ws.numel(), status.data_ptr(), torch.cuda.current_stream().cuda_stream,
                1_000_000, 1)
        assert rc == 0, binding.status_string(rc)
        torch.cuda.synchronize()
        g = {k: v.cpu().numpy() for k, v in out.items()}
        g["status"] = status.cpu().numpy()
        assert g["status"].tolist() == [0, SPEC_ERR_TIMEOUT, 0], (rep, g["status"])
        # the timed-out request's outputs are untouched
        assert (g["accept_len"][1] == -7) and (g["path_nodes"][1] == -7).all()
        assert (g["out_tokens"][1] == -7).all() and g["near_ties"][1] == -7
        # the other requests match the oracle (request ids enter the uniforms,
        # so the whole batch is evaluated and the timed-out request's rows are
        # replaced by the oracle's before the comparison)
        g2 = {k: v.copy() for k, v in g.items()}
        for k in ("accept_len", "path_nodes", "out_tokens", "near_ties", "status"):
            g2[k][1] = o[k][1]
        nodes = oracle_nodes_for(g2, o, w.target_logits, w.draft_logits, w.tokens, w.parents,
                                 w.offsets, w.temperature, seed, W)
        assert_verify_match(g2, o, w.parents, w.tokens, w.offsets, f"timeout test rep {rep}",
                            nodes=nodes)
    # the workspace's counters were left at zero: a normal call still verifies
    status = torch.zeros(B, dtype=torch.int32, device="cuda")
    r = gpu_lib.tree_verify(tl, dl, tok, par, off, w.temperature, seed, W, status, ws)
    torch.cuda.synchronize()
    assert (status.cpu().numpy() == 0).all()
    np.testing.assert_array_equal(r["accept_len"].cpu().numpy(), o["accept_len"])


def test_timeout_hook_rejects_what_it_does_not_cover(gpu_lib):
    fn = _fn(binding.load())
    fake = ctypes.c_void_p(256)
    # greedy, and an out-of-range request or limit, are refused on the host
    for temp, wait_ns, drop in ((0.0, 1000, 0), (0.7, 0, 0), (0.7, 1000, 5), (0.7, 3_000_000_000, 0)):
        rc = fn(fake, fake, fake, fake, fake, 2, 4, 100, temp, 0, fake, fake, fake, fake, 4, fake,
                4096, fake, None, wait_ns, drop)
        assert rc == -2
