"""GPU step A1 (spec_build_tree_mask) against the oracle, bit-exact."""
import numpy as np
import pytest

import oracle
from parity import gpu_mask
from test_oracle_mask import all_parent_arrays, pack
from token_tree_verification_gb300 import synthetic

pytestmark = pytest.mark.gpu


def test_exhaustive_small_trees(gpu_lib):
    trees = [t for n in range(1, 8) for t in all_parent_arrays(n)]
    par, off = pack(trees)
    m, d, s = gpu_mask(par, off)
    mo, do, so = oracle.build_mask(par, off)
    assert (s == 0).all() and (so == 0).all()
    np.testing.assert_array_equal(m, mo)
    np.testing.assert_array_equal(d, do)


def test_random_trees_up_to_128_nodes(gpu_lib):
    rng = np.random.default_rng(11)
    trees = [synthetic.chain_tree(128), synthetic.chain_tree(1),
             np.array([-1] + [0] * 127, np.int32)]
    for n in rng.integers(2, 129, 200):
        trees.append(synthetic.random_tree(rng, int(n), int(rng.integers(1, min(n - 1, 12) + 1)), None))
    par, off = pack(trees)
    m, d, s = gpu_mask(par, off)
    mo, do, so = oracle.build_mask(par, off)
    assert (s == 0).all()
    np.testing.assert_array_equal(m, mo)
    np.testing.assert_array_equal(d, do)


def test_errors_reported_per_request(gpu_lib):
    good = np.array([-1, 0, 0, 1], np.int32)
    bad = np.array([-1, 2, 0, 1], np.int32)
    big = synthetic.chain_tree(129)
    par, off = pack([good, bad, good, big, good])
    m, d, s = gpu_mask(par, off)
    assert s.tolist() == [0, -5, 0, -4, 0]
    mo, do, _ = oracle.build_mask(*pack([good]))
    for b in (0, 2, 4):
        np.testing.assert_array_equal(m[off[b]:off[b + 1]], mo)
