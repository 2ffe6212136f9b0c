"""Pins for the oracle's hybrid attention with an exact window ("Hybrid Latent
Attention for Looped Language Models", §3.4 "Exact sliding window", Eq. (4)).

The oracle's ``hybrid`` is pinned to: an independent numpy brute force; the page's
own reduction (with no window tokens it is pure latent attention); a window holding
the latent tokens' own reconstructions (then the split point cannot matter); the
teacher's attention under the full-rank orthonormal codec; and the log-sum-exp
merge of two separate softmaxes that the page's serving path (Appendix I) uses.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import brute


def _case(seed, B=2, H=2, T=2, d=128, rk=16, rv=32, L_max=9, W=6):
    g = np.random.default_rng(seed)
    return dict(
        q=g.standard_normal((B, H, d)),
        cache_k=g.standard_normal((B, H, L_max, rk)),
        cache_v=g.standard_normal((B, H, L_max, rv)),
        w_up_k=g.standard_normal((T, H, d, rk)) / math.sqrt(rk),
        w_up_v=g.standard_normal((T, H, d, rv)) / math.sqrt(rv),
        mu_k=g.standard_normal((H, T * d)) * math.sqrt(0.1),
        mu_v=g.standard_normal((H, T * d)) * math.sqrt(0.1),
        k_win=g.standard_normal((B, H, W, d)),
        v_win=g.standard_normal((B, H, W, d)),
    )


def _hyb(dm, t, c, n_lat, q_pos, n_win, win_pos):
    return oracle.hybrid(dm, t, c["q"], c["cache_k"], c["cache_v"], np.array(n_lat, np.int32),
                         np.array(q_pos, np.int32), c["w_up_k"], c["w_up_v"], c["mu_k"], c["mu_v"],
                         c["k_win"], c["v_win"], np.array(n_win, np.int32), np.array(win_pos, np.int32))


@pytest.mark.parametrize("style", [0, 1])
def test_hybrid_matches_brute_force(style):
    dm = oracle.dims(2, 2, 128, 16, 32, 0, 10000.0, style)
    c = _case(1)
    n_lat, n_win = [9, 3], [6, 2]
    win_pos = [9, 40]                      # right after the latent tokens / further on
    q_pos = [14, 41]
    for t in range(2):
        o, l = _hyb(dm, t, c, n_lat, q_pos, n_win, win_pos)
        ob, lb = brute.hybrid_per_head(t, c["q"], c["cache_k"], c["cache_v"], n_lat, q_pos, c["w_up_k"],
                                       c["w_up_v"], c["mu_k"], c["mu_v"], c["k_win"], c["v_win"], n_win,
                                       win_pos, style=style)
        np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, lb, rtol=0, atol=1e-12)


def test_no_window_is_latent_attention():
    """The page: with W = 0, Eq. (4) reduces to pure latent attention."""
    dm = oracle.dims(2, 2, 128, 16, 32)
    c = _case(2)
    n_lat, q_pos = [9, 4], [8, 3]
    o, l = _hyb(dm, 1, c, n_lat, q_pos, [0, 0], [0, 0])
    ob, lb = brute.decode_per_head(1, c["q"], c["cache_k"], c["cache_v"], n_lat, q_pos, c["w_up_k"],
                                   c["w_up_v"], c["mu_k"], c["mu_v"])
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, lb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("split", [0, 3, 7, 9])
def test_window_of_reconstructions_matches_all_latent(split):
    """Window tokens that carry the latent tokens' own reconstructions, at the same
    positions: the result cannot depend on where the window starts."""
    dm = oracle.dims(2, 2, 128, 16, 32)
    c = _case(3, W=9)
    L, t, B, H = 9, 1, 2, 2
    for b in range(B):
        for h in range(H):
            for w in range(L - split):
                j = split + w
                c["k_win"][b, h, w] = brute.reconstruct(c["cache_k"][b, h, j:j + 1], c["w_up_k"][t, h],
                                                        c["mu_k"][h, t * 128:(t + 1) * 128])[0]
                c["v_win"][b, h, w] = brute.reconstruct(c["cache_v"][b, h, j:j + 1], c["w_up_v"][t, h],
                                                        c["mu_v"][h, t * 128:(t + 1) * 128])[0]
    o, l = _hyb(dm, t, c, [split] * B, [L - 1] * B, [L - split] * B, [split] * B)
    of, lf, _ = oracle.decode(dm, t, c["q"], c["cache_k"], c["cache_v"], np.array([L] * B, np.int32),
                              np.array([L - 1] * B, np.int32), c["w_up_k"], c["w_up_v"], c["mu_k"], c["mu_v"])
    np.testing.assert_allclose(o, of, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, lf, rtol=0, atol=1e-12)


def test_window_only_is_the_teacher_attention():
    """No latent tokens: the window alone is ordinary attention over exact K/V."""
    dm = oracle.dims(2, 2, 128, 16, 32)
    c = _case(4)
    o, l = _hyb(dm, 0, c, [0, 0], [12, 12], [6, 4], [7, 7])
    os_, ls_ = oracle.sdpa(dm, c["q"], c["k_win"], c["v_win"], np.array([6, 4], np.int32),
                           np.array([5, 5], np.int32), pos_offset=7)
    np.testing.assert_allclose(o, os_, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, ls_, rtol=0, atol=1e-12)


def test_full_rank_codec_with_window_is_the_teacher():
    """Orthonormal codec of rank T d (exact latents) plus an exact window over the
    newest tokens: together the teacher's attention over every token."""
    T, H, d, B, L = 2, 2, 128, 2, 8
    r = T * d
    g = np.random.default_rng(5)
    dm = oracle.dims(T, H, d, r, r)
    Kt = g.standard_normal((B, H, L, T, d))
    Vt = g.standard_normal((B, H, L, T, d))
    mu_k = g.standard_normal((H, T * d)) * 0.3
    mu_v = g.standard_normal((H, T * d)) * 0.3
    wd = [np.stack([np.linalg.qr(g.standard_normal((r, r)))[0] for _ in range(H)]) for _ in range(2)]
    wu = [np.stack([w[:, t * d:(t + 1) * d, :] for t in range(T)]) for w in wd]
    ck, cv = np.zeros((B, H, L, r)), np.zeros((B, H, L, r))
    seq_idx = np.repeat(np.arange(B, dtype=np.int32), L)
    pos = np.tile(np.arange(L, dtype=np.int32), B)
    oracle.encode(dm, Kt.transpose(0, 2, 1, 3, 4).reshape(B * L, H, T * d), seq_idx, pos, wd[0], mu_k, r, ck)
    oracle.encode(dm, Vt.transpose(0, 2, 1, 3, 4).reshape(B * L, H, T * d), seq_idx, pos, wd[1], mu_v, r, cv)
    q = g.standard_normal((B, H, d))
    t, split = 1, 5
    o, l = oracle.hybrid(dm, t, q, ck, cv, np.array([split] * B, np.int32), np.array([L - 1] * B, np.int32),
                         wu[0], wu[1], mu_k, mu_v, np.ascontiguousarray(Kt[:, :, split:, t]),
                         np.ascontiguousarray(Vt[:, :, split:, t]), np.array([L - split] * B, np.int32),
                         np.array([split] * B, np.int32))
    os_, ls_ = oracle.sdpa(dm, q, np.ascontiguousarray(Kt[:, :, :, t]), np.ascontiguousarray(Vt[:, :, :, t]),
                           np.array([L] * B, np.int32), np.array([L - 1] * B, np.int32))
    np.testing.assert_allclose(o, os_, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, ls_, rtol=0, atol=1e-12)


def test_log_sum_exp_merge_of_two_softmaxes_is_the_single_softmax():
    """Appendix I "Serving Implementation": the latent part and the window part,
    each normalised by its own softmax, merged with their log-sum-exps, equal the
    single softmax of Eq. (4).  (The merge the GPU path applies.)"""
    dm = oracle.dims(2, 2, 128, 16, 32)
    c = _case(6)
    n_lat, n_win, win_pos, q_pos = [9, 0], [6, 3], [9, 2], [14, 4]
    ol, ll, _ = oracle.decode(dm, 1, c["q"], c["cache_k"], c["cache_v"], np.array(n_lat, np.int32),
                              np.array(q_pos, np.int32), c["w_up_k"], c["w_up_v"], c["mu_k"], c["mu_v"])
    ow = np.zeros_like(ol)
    lw = np.zeros_like(ll)
    for b in range(2):
        # sdpa rotates keys at j + offset and the query at q_pos + offset
        o1, l1 = oracle.sdpa(dm, c["q"][b:b + 1], c["k_win"][b:b + 1], c["v_win"][b:b + 1],
                             np.array([n_win[b]], np.int32), np.array([q_pos[b] - win_pos[b]], np.int32),
                             pos_offset=win_pos[b])
        ow[b], lw[b] = o1[0], l1[0]
    M = np.maximum(ll, lw)
    a = np.where(np.isneginf(ll), 0.0, np.exp(ll - M))
    w = np.where(np.isneginf(lw), 0.0, np.exp(lw - M))
    om = (a[..., None] * ol + w[..., None] * ow) / (a + w)[..., None]
    lm = M + np.log(a + w)
    o, l = _hyb(dm, 1, c, n_lat, q_pos, n_win, win_pos)
    np.testing.assert_allclose(om, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lm, l, rtol=0, atol=1e-12)
