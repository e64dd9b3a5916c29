"""Pins for the oracle's depth-first KV-cache update (SpecInfer news
write-up, "Token 樹驗證器": the verifier's KV cache is updated depth-first, so
the accepted path becomes the next step's prefix without extra storage).

Slot L + j receives the old slot L + path[j] (j = 1 .. acc); every other slot
keeps its value; the committed prefix becomes L + 1 + acc."""
import numpy as np

import oracle


def _cache(B=1, H=2, S=12, D=4, seed=0):
    # every element distinct, so any wrong source row is visible
    return np.arange(B * H * S * D, dtype=np.float32).reshape(B, H, S, D) + 1000 * seed


def test_chain_accepted_in_place_is_identity():
    c = _cache()
    off = np.array([0, 6], np.int32)
    pn = np.array([[0, 1, 2, 3, -1, -1, -1]], np.int32)
    new, newp, st = oracle.kv_compact(c, [3], off, pn, [3])
    assert st.tolist() == [0]
    assert newp.tolist() == [3 + 1 + 3]
    np.testing.assert_array_equal(new, c)


def test_hand_example_with_overlapping_source_and_destination():
    # L = 2, tree of 5 nodes at slots 2..6, accepted path root -> 2 -> 3:
    # slot 3 <- old slot 4, slot 4 <- old slot 5 (slot 4 is both a destination
    # and the previous entry's source: the copy must read the old cache)
    c = _cache(S=9)
    off = np.array([0, 5], np.int32)
    pn = np.array([[0, 2, 3, -1]], np.int32)
    new, newp, st = oracle.kv_compact(c, [2], off, pn, [2])
    assert st.tolist() == [0] and newp.tolist() == [5]
    expect = c.copy()
    expect[:, :, 3] = c[:, :, 4]
    expect[:, :, 4] = c[:, :, 5]
    np.testing.assert_array_equal(new, expect)


def test_nothing_accepted_keeps_everything():
    c = _cache()
    new, newp, st = oracle.kv_compact(c, [4], np.array([0, 5], np.int32),
                                      np.array([[0, -1, -1]], np.int32), [0])
    np.testing.assert_array_equal(new, c)
    assert newp.tolist() == [5] and st.tolist() == [0]


def test_untouched_regions_and_ragged_batch():
    rng = np.random.default_rng(3)
    B, H, S, D = 3, 2, 40, 8
    c = rng.standard_normal((B, H, S, D)).astype(np.float32)
    off = np.array([0, 7, 19, 24], np.int32)
    L = np.array([5, 10, 0], np.int32)
    pn = np.full((B, 6), -1, np.int32)
    pn[0, :3] = [0, 3, 6]
    pn[1, :5] = [0, 1, 4, 9, 11]
    pn[2, :1] = [0]
    acc = np.array([2, 4, 0], np.int32)
    new, newp, st = oracle.kv_compact(c, L, off, pn, acc)
    assert st.tolist() == [0, 0, 0]
    assert newp.tolist() == (L + 1 + acc).tolist()
    for b in range(B):
        lo, hi = L[b] + 1, L[b] + 1 + acc[b]
        np.testing.assert_array_equal(new[b, :, :lo], c[b, :, :lo])     # prefix and root
        np.testing.assert_array_equal(new[b, :, hi:], c[b, :, hi:])     # the rest
        for j in range(1, acc[b] + 1):
            np.testing.assert_array_equal(new[b, :, L[b] + j], c[b, :, L[b] + pn[b, j]])


def test_invalid_paths_and_preset_status():
    c = _cache(B=4, S=16)
    off = np.array([0, 5, 10, 15, 20], np.int32)
    L = np.array([1, 1, 1, 1], np.int32)
    pn = np.array([[0, 2, 2, -1],     # not increasing
                   [0, 7, -1, -1],    # node outside the tree
                   [0, 1, 2, 3],      # acc = 4 needs 5 entries (W = 4)
                   [0, 1, -1, -1]], np.int32)
    acc = np.array([2, 1, 4, 1], np.int32)
    status = np.array([0, 0, 0, -6], np.int32)   # request 3 already failed
    new, newp, st = oracle.kv_compact(c, L, off, pn, acc, status)
    assert st.tolist() == [-5, -5, -4, -6]
    assert newp.tolist() == [1, 1, 1, 1]
    np.testing.assert_array_equal(new, c)


def test_bf16_bits_copied_exactly():
    import torch
    c = torch.randn(1, 2, 10, 8).to(torch.bfloat16).view(torch.int16).numpy()
    new, newp, st = oracle.kv_compact(c, [1], np.array([0, 6], np.int32),
                                      np.array([[0, 4, 5]], np.int32), [2])
    np.testing.assert_array_equal(new[:, :, 2], c[:, :, 5])
    np.testing.assert_array_equal(new[:, :, 3], c[:, :, 6])
