"""Pins for the oracle's token eviction (``oracle.evict``; LLA paper, Appendix D
"Token-eviction composition table" and Appendix J "Eviction and long-context
prefill": a StreamingLLM/H2O-style sink + window budget composed with LLA).

Pinned to a hand-written budget, the no-op at or below the budget, idempotence, the
kept rows being the original rows in order, and the composition with decode: the C
oracle's decode over the evicted latent cache equals a numpy brute force attention
over exactly the kept tokens' reconstructions at positions 0.. within the kept cache.
"""
import math

import numpy as np

import oracle
from oracle import brute, evict


def test_hand_written_budget():
    assert evict.kept_tokens(10, 2, 3) == [0, 1, 7, 8, 9]
    assert evict.kept_tokens(5, 2, 3) == [0, 1, 2, 3, 4]
    assert evict.kept_tokens(6, 0, 4) == [2, 3, 4, 5]
    assert evict.kept_tokens(6, 4, 0) == [0, 1, 2, 3]
    cache = np.arange(2 * 1 * 12 * 1, dtype=np.float64).reshape(2, 1, 12, 1)
    out, lens = evict.evict(cache, [10, 4], 2, 3)
    np.testing.assert_array_equal(out[0, 0, :5, 0], [0, 1, 7, 8, 9])
    np.testing.assert_array_equal(out[0, 0, 5:, 0], cache[0, 0, 5:, 0])   # rows past the budget as they were
    np.testing.assert_array_equal(out[1], cache[1])                       # under budget: untouched
    assert list(lens) == [5, 4]


def test_idempotent_and_rows_in_order():
    g = np.random.default_rng(21)
    cache = g.standard_normal((3, 2, 40, 5))
    lens = [40, 9, 23]
    once, l1 = evict.evict(cache, lens, 4, 8)
    twice, l2 = evict.evict(once, l1, 4, 8)
    np.testing.assert_array_equal(once, twice)
    assert list(l1) == list(l2) == [12, 9, 12]
    for b, L in enumerate(lens):
        keep = evict.kept_tokens(L, 4, 8)
        np.testing.assert_array_equal(once[b, :, :len(keep)], cache[b][:, keep])


def test_eviction_composes_with_decode():
    g = np.random.default_rng(22)
    B, H, T, d, rk, rv, L_max = 2, 2, 2, 128, 16, 32, 30
    sink, window = 3, 9
    ck = g.standard_normal((B, H, L_max, rk))
    cv = g.standard_normal((B, H, L_max, rv))
    wk = g.standard_normal((T, H, d, rk)) / math.sqrt(rk)
    wv = g.standard_normal((T, H, d, rv)) / math.sqrt(rv)
    mk = g.standard_normal((H, T * d)) * math.sqrt(0.1)
    mv = g.standard_normal((H, T * d)) * math.sqrt(0.1)
    q = g.standard_normal((B, H, d))
    lens = [30, 11]
    ek, lens2 = evict.evict(ck, lens, sink, window)
    ev, _ = evict.evict(cv, lens, sink, window)
    q_pos = np.array(lens2) - 1                          # the newest kept slot
    dm = oracle.dims(T, H, d, rk, rv)
    for t in range(T):
        o, l, _ = oracle.decode(dm, t, q, ek, ev, lens2, q_pos, wk, wv, mk, mv)
        for b in range(B):
            keep = evict.kept_tokens(lens[b], sink, window)
            for h in range(H):
                K = brute.reconstruct(ck[b, h, keep], wk[t, h], mk[h, t * d:(t + 1) * d])
                V = brute.reconstruct(cv[b, h, keep], wv[t, h], mv[h, t * d:(t + 1) * d])
                qr = brute.rotation_matrix(d, len(keep) - 1, 10000.0) @ q[b, h]
                s = np.array([(brute.rotation_matrix(d, j, 10000.0) @ K[j]) @ qr for j in range(len(keep))])
                s /= math.sqrt(d)
                p = np.exp(s - s.max())
                np.testing.assert_allclose(o[b, h], (p / p.sum()) @ V, rtol=0, atol=1e-12)
                np.testing.assert_allclose(l[b, h], s.max() + np.log(p.sum()), rtol=0, atol=1e-12)
