"""Pins for the oracle's paged-cache definition (``oracle.paged``; page tables of
"Enabling dynamic computation in Looped LMs", §"Ragged KV" and Appendix A.1).

The gather is pinned to a hand-written layout, to its inverse (scatter then gather
is the identity on stored tokens), to aliasing (two table entries naming one page
read the same rows), to the one-token page of the page's own vLLM implementation
(plain per-token indexing) and to the slot formula.
"""
import numpy as np

from oracle import paged


def test_hand_written_layout():
    # P = 2, pages hold 10 * page + row
    pool = np.zeros((4, 1, 2, 1))
    for pg in range(4):
        for row in range(2):
            pool[pg, 0, row, 0] = 10 * pg + row
    bt = np.array([[2, 0, -1], [1, 3, -1]])
    dense = paged.gather(pool, bt, 2, [3, 4])
    assert dense.shape == (2, 1, 6, 1)
    np.testing.assert_array_equal(dense[0, 0, :4, 0], [20, 21, 0, 1])
    np.testing.assert_array_equal(dense[1, 0, :4, 0], [10, 11, 30, 31])
    assert np.all(np.isnan(dense[:, :, 4:, :]))          # logical page 2 holds no token


def test_scatter_then_gather_is_identity_on_stored_tokens():
    g = np.random.default_rng(5)
    B, H, P, r, max_pages = 3, 2, 4, 3, 5
    lens = [17, 4, 0]
    used = [(L + P - 1) // P for L in lens]
    num_pages = sum(used) + 2
    perm = g.permutation(num_pages)
    bt = np.full((B, max_pages), -1)
    k = 0
    for b in range(B):
        for lp in range(used[b]):
            bt[b, lp] = perm[k]
            k += 1
    dense = g.standard_normal((B, H, max_pages * P, r))
    pool = paged.scatter(dense, bt, P, lens, num_pages)
    back = paged.gather(pool, bt, P, lens)
    for b in range(B):
        np.testing.assert_array_equal(back[b, :, :lens[b]], dense[b, :, :lens[b]])
    # the two pages nobody names are untouched
    named = set(bt[bt >= 0].tolist())
    for pg in range(num_pages):
        if pg not in named:
            assert np.all(np.isnan(pool[pg]))


def test_aliased_entries_read_the_same_rows():
    g = np.random.default_rng(6)
    pool = g.standard_normal((3, 2, 8, 4))
    bt = np.array([[1, 2], [1, 0]])                      # both sequences start on page 1
    dense = paged.gather(pool, bt, 8, [16, 16])
    np.testing.assert_array_equal(dense[0, :, :8], dense[1, :, :8])
    np.testing.assert_array_equal(dense[0, :, 8:], pool[2])
    np.testing.assert_array_equal(dense[1, :, 8:], pool[0])


def test_one_token_pages_are_per_token_indexing():
    g = np.random.default_rng(7)
    pool = g.standard_normal((9, 2, 1, 3))
    bt = np.array([[4, 0, 8, 1], [2, 2, 7, 5]])
    dense = paged.gather(pool, bt, 1, [4, 3])
    for b, L in ((0, 4), (1, 3)):
        for j in range(L):
            np.testing.assert_array_equal(dense[b, :, j], pool[bt[b, j], :, 0])


def test_slot_formula_matches_gather():
    g = np.random.default_rng(8)
    P = 3
    pool = g.standard_normal((6, 2, P, 2))
    bt = np.array([[5, 1, 3], [0, 2, 4]])
    dense = paged.gather(pool, bt, P, [8, 9])
    for b, L in ((0, 8), (1, 9)):
        for j in range(L):
            pg, row = paged.slot(bt, P, b, j)
            assert (pg, row) == (bt[b, j // P], j % P)
            np.testing.assert_array_equal(dense[b, :, j], pool[pg, :, row])
