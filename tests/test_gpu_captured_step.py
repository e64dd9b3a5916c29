"""The step bench.py times, as it times it: tree attention (its masks built
from the parents) on one branch and the mask kernel then verification on the
other, captured in one CUDA graph and replayed, compared with the oracle.

Source: speculative-decoding explainer (intelliparadigm.com) §3.2
并行验证的CUDA优化 (capture the whole verification flow in a CUDA graph).
Several steps with different seeds go into one graph; each step's outputs
are copied out inside the graph, so every replayed step is checked: the
mask bit-exact, attention within the tolerance, verification decision by
decision against the oracle."""
import numpy as np
import pytest
import torch

import bench
import oracle
from parity import assert_attn_close, assert_verify_match, oracle_attn_rows, oracle_nodes_for
from token_tree_verification_gb300 import synthetic

pytestmark = pytest.mark.gpu

CASES = [("llama7b", 0.7, dict(L=512)),
         ("dynamic", 0.0, dict(B=4, L_range=(64, 300))),
         ("dynamic", 0.9, dict(B=4, L_range=(64, 300))),
         ("llama70b_gqa", 0.7, dict(B=2, L=200, N=48, depth=4))]


@pytest.mark.parametrize("name,temp,kw", CASES)
def test_captured_step_matches_oracle(gpu_lib, name, temp, kw):
    w = synthetic.make_workload(name, seed=3, device="cuda", pad=float("nan"), temperature=temp, **kw)
    st = bench.Step(w, copies=2, seed=100)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        st.run(0)                      # eager: configures the kernels before capture
    torch.cuda.synchronize()
    steps = 3
    outs = dict(mask=st.mask, depth=st.depth, o=st.o, **st.outs)
    saved = [{k: torch.empty_like(v) for k, v in outs.items()} for _ in range(steps)]
    st.status.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(steps):
            st.run(i)
            for k, v in outs.items():
                saved[i][k].copy_(v)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    assert (st.status.cpu().numpy() == 0).all()

    m_ref, d_ref, _ = oracle.build_mask(w.parents, w.offsets)
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(w.T * w.Hq, size=min(w.T * w.Hq, 768), replace=False))
    a_ref = oracle_attn_rows(w, rows)
    W = w.max_depth + 1
    draft = w.draft_logits if temp > 0 else None
    for i in range(steps):
        s = {k: v.cpu() for k, v in saved[i].items()}
        np.testing.assert_array_equal(s["mask"].numpy().view(np.uint32), m_ref)
        np.testing.assert_array_equal(s["depth"].numpy(), d_ref)
        got = s["o"].float().numpy().reshape(w.T * w.Hq, w.D)[rows]
        assert_attn_close(got, a_ref, f"{name} step {i}")
        gv = {k: s[k].numpy() for k in ("accept_len", "path_nodes", "out_tokens", "near_ties")}
        gv["status"] = np.zeros(w.B, np.int32)
        seed = st.seed + i
        o = oracle.tree_verify(w.target_logits, draft, w.tokens, w.parents, w.offsets, temp, seed, W)
        nodes = oracle_nodes_for(gv, o, w.target_logits, draft, w.tokens, w.parents, w.offsets,
                                 temp, seed, W)
        assert_verify_match(gv, o, w.parents, w.tokens, w.offsets, f"{name} captured step {i}",
                            nodes=nodes)
