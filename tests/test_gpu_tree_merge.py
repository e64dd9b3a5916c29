"""GPU parity of spec_tree_merge (merging two speculators' token trees)
against the oracle: bit-exact on ragged batches with shared and duplicate
paths, deep chains, self-merges, root-only trees, and the error cases."""
import numpy as np
import pytest
import torch

import oracle
import token_tree_verification_gb300 as ttv
from parity import dev
from test_oracle_tree_merge import random_pair
from test_oracle_verify import pack

pytestmark = pytest.mark.gpu


def _both(pairs):
    PA, OA = pack([p[0] for p in pairs])
    PB, OB = pack([p[2] for p in pairs])
    TA = np.concatenate([p[1] for p in pairs]).astype(np.int32)
    TB = np.concatenate([p[3] for p in pairs]).astype(np.int32)
    st = torch.zeros(len(pairs), dtype=torch.int32, device="cuda")
    g = ttv.tree_merge(dev(PA, torch.int32), dev(TA, torch.int32), dev(OA, torch.int32),
                       dev(PB, torch.int32), dev(TB, torch.int32), dev(OB, torch.int32), st)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    g["status"] = st.cpu().numpy()
    o = oracle.tree_merge(PA, TA, OA, PB, TB, OB)
    return g, o


def test_merge_matches_oracle(gpu_lib):
    rng = np.random.default_rng(11)
    for vocab in (2, 6, 50):
        pairs = [random_pair(rng, vocab=vocab) for _ in range(33)]
        pairs.append((pairs[0][0], pairs[0][1], pairs[0][0], pairs[0][1]))        # self-merge
        pairs.append((pairs[1][0], pairs[1][1], np.array([-1], np.int32), np.array([5], np.int32)))
        chain = np.array([-1] + list(range(0, 60)), np.int32)                       # deep chains
        pairs.append((chain, rng.integers(0, 3, 61).astype(np.int32), chain,
                      rng.integers(0, 3, 61).astype(np.int32)))
        g, o = _both(pairs)
        np.testing.assert_array_equal(g["status"], o["status"])
        ok = o["status"] == 0
        for k in ("parents", "tokens", "map_b", "n_out"):
            np.testing.assert_array_equal(g[k][ok], o[k][ok], err_msg=k)


def test_merge_errors(gpu_lib):
    full = np.array([-1] + list(range(0, 99)), np.int32)          # 100-node chain
    other = np.array([-1] + [0] * 49, np.int32)                   # 50 distinct children of the root
    bad = np.array([-1, 0, 3, 1], np.int32)
    pairs = [(full, np.arange(100).astype(np.int32), other, (1000 + np.arange(50)).astype(np.int32)),
             (bad, np.zeros(4, np.int32), bad, np.zeros(4, np.int32)),
             (full[:5], np.arange(5).astype(np.int32), full[:5], np.arange(5).astype(np.int32))]
    g, o = _both(pairs)
    assert g["status"].tolist() == [-4, -5, 0] == o["status"].tolist()
    np.testing.assert_array_equal(g["parents"][2], o["parents"][2])
