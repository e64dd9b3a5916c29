"""Step R on the device (spec_philox_uniforms) against the oracle's
generator, itself pinned to numpy's Philox: bit-exact on 10^6 counters that
cover the kinds the method draws (accept tests, fallback draws, expansion
slots), large request ids and the full node range, plus a chi-square test of
uniformity of the device's draws."""
import numpy as np
import pytest
import torch

import oracle
import token_tree_verification_gb300 as ttv

pytestmark = pytest.mark.gpu


def test_device_uniforms_match_the_oracle(gpu_lib):
    rng = np.random.default_rng(17)
    n = 1_000_000
    ctr = np.empty((n, 4), np.int64)
    ctr[:, 0] = rng.integers(0, 128, n)                    # request-local node
    ctr[:, 1] = rng.integers(0, 2**31 - 1, n)              # request id, up to the int32 range
    ctr[:, 2] = rng.integers(0, 3, n)                      # kind: 0 accept, 1 draw, 2 expansion
    ctr[:, 3] = np.where(ctr[:, 2] == 2, rng.integers(0, 16, n), 0)   # expansion child slot
    ctr[:8] = [[127, 2**31 - 2, 1, 0], [0, 0, 0, 0], [5, 2**20, 2, 15], [64, 7, 0, 0],
               [1, 1, 2, 0], [126, 2**30, 1, 0], [3, 12345, 2, 7], [127, 2**31 - 2, 0, 0]]
    for seed in (0, 1234, 2**64 - 1):
        got = ttv.philox_uniforms(seed, torch.as_tensor(ctr).cuda()).cpu().numpy()
        ref = oracle.uniforms(seed, ctr)
        np.testing.assert_array_equal(got.astype(np.float64), ref)
    bins = 64
    h = np.bincount((got.astype(np.float64) * bins).astype(int), minlength=bins)
    chi2 = ((h - n / bins) ** 2 / (n / bins)).sum()
    dof = bins - 1
    assert chi2 <= dof + 3 * np.sqrt(2 * dof), chi2
    assert (got >= 0).all() and (got < 1).all()
