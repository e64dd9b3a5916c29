"""Pins for the oracle's counter-based generator (step R).

The method draws its uniforms from Philox4x64-10 (Salmon et al., SC'11).  The
oracle's C implementation is pinned to numpy's independent implementation of
the same generator (numpy.random.Philox advances its counter by one before
producing a block, hence the ``- 1``), and the uniform conversion is checked
for range and a chi-square uniformity bound."""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("ctr,key", [
    ((1, 0, 0, 0), (0, 0)),
    ((5, 3, 1, 0), (0x0123456789ABCDEF, 0)),
    ((2**64 - 1, 7, 2**63, 12345), (2**64 - 1, 2**64 - 1)),
    ((99, 2**40, 0, 1), (42, 7)),
])
def test_philox_matches_numpy(ctr, key):
    c_int = sum(int(w) << (64 * i) for i, w in enumerate(ctr))
    k_int = int(key[0]) | (int(key[1]) << 64)
    bg = np.random.Philox(key=k_int, counter=(c_int - 1) % 2**256)
    ref = bg.random_raw(4)
    got = oracle.philox4x64_10(np.array(ctr, dtype=np.uint64), np.array(key, dtype=np.uint64))
    np.testing.assert_array_equal(got, ref)


def test_uniform_is_top24_bits_of_word0():
    for seed, node, req, kind in [(0, 0, 0, 0), (7, 5, 3, 1), (2**63 + 5, 127, 1000, 0)]:
        bg = np.random.Philox(key=seed, counter=(node + (req << 64) + (kind << 128) - 1) % 2**256)
        w0 = int(bg.random_raw(1)[0])
        assert oracle.uniform(seed, node, req, kind) == (w0 >> 40) / 2.0**24


def test_uniform_chi_square():
    n, bins = 20000, 64
    u = np.array([oracle.uniform(11, i % 128, i // 128, i & 1) for i in range(n)])
    assert (u >= 0).all() and (u < 1).all()
    h = np.bincount((u * bins).astype(int), minlength=bins)
    chi2 = ((h - n / bins) ** 2 / (n / bins)).sum()
    dof = bins - 1
    assert chi2 <= dof + 3 * np.sqrt(2 * dof)


def test_batch_uniforms_match_numpy_and_the_single_counter_form():
    rng = np.random.default_rng(3)
    ctr = np.stack([rng.integers(0, 128, 50), rng.integers(0, 2**31 - 1, 50),
                    rng.integers(0, 3, 50), rng.integers(0, 16, 50)], axis=1).astype(np.int64)
    ctr[0] = (2**62, 2**40, 2, 15)
    seed = 0x5EED
    u = oracle.uniforms(seed, ctr)
    for i, (c0, c1, c2, c3) in enumerate(ctr.tolist()):
        c_int = c0 + (c1 << 64) + (c2 << 128) + (c3 << 192)
        bg = np.random.Philox(key=seed, counter=(c_int - 1) % 2**256)
        assert u[i] == (int(bg.random_raw(1)[0]) >> 40) / 2.0**24
        if c3 == 0:
            assert u[i] == oracle.uniform(seed, c0, c1, c2)
