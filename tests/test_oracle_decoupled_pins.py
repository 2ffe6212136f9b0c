"""Pins for the oracle's absorbed decoupled-RoPE decode (LLA page, Appendix J
"Absorbed attention": NoPE content path on the latents plus a small explicit rotary
branch shared across the loops, d_rope = 64 as in Table 14).

``oracle.decoupled`` is pinned to an independent numpy brute force (explicit rotation
matrices over the rotary branch, concatenated keys), to the closed form of the score
difference between two tokens (read back through a two-token softmax with one-hot
values), to position-shift invariance of the rotary branch, and to the single-token
case.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import brute

D_ROPE = 64


def _case(seed, B=2, H=2, T=2, d=128, rk=16, rv=32, L_max=7):
    g = np.random.default_rng(seed)
    return dict(
        q=g.standard_normal((B, H, d + D_ROPE)),
        cache_k=g.standard_normal((B, H, L_max, rk)),
        cache_v=g.standard_normal((B, H, L_max, rv)),
        k_rope=g.standard_normal((B, H, L_max, D_ROPE)),
        w_up_k=g.standard_normal((T, H, d, rk)) / math.sqrt(rk),
        w_up_v=g.standard_normal((T, H, d, rv)) / math.sqrt(rv),
        mu_k=g.standard_normal((H, T * d)) * math.sqrt(0.1),
        mu_v=g.standard_normal((H, T * d)) * math.sqrt(0.1),
    )


def _dec(dm, t, c, lens, q_pos, pos_offset=0):
    return oracle.decoupled(dm, t, c["q"], c["cache_k"], c["cache_v"], c["k_rope"], np.array(lens, np.int32),
                            np.array(q_pos, np.int32), c["w_up_k"], c["w_up_v"], c["mu_k"], c["mu_v"],
                            pos_offset=pos_offset)


@pytest.mark.parametrize("style", [0, 1])
def test_decoupled_matches_brute_force(style):
    dm = oracle.dims(2, 2, 128, 16, 32, 0, 10000.0, style)
    c = _case(11)
    lens, q_pos = [7, 3], [6, 40]
    for t in range(2):
        o, l = _dec(dm, t, c, lens, q_pos)
        ob, lb = brute.decoupled_per_head(t, c["q"], c["cache_k"], c["cache_v"], c["k_rope"], lens, q_pos,
                                          c["w_up_k"], c["w_up_v"], c["mu_k"], c["mu_v"], style=style)
        np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, lb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("style", [0, 1])
def test_score_difference_closed_form(style):
    """Two tokens, one-hot values (token j's value is e_j), so out[j] = p_j and
    ln(p_1 / p_0) = s_1 - s_0 with s_j = (q_c . k_j + sum_f [cos((j - q_pos) th_f)
    (q_a r_a + q_b r_b) + sin((j - q_pos) th_f) (q_b r_a - q_a r_b)]) / sqrt(d + d_rope)
    over the rotary pairs (a, b) of frequency f, th_f = base^(-2f / d_rope)."""
    T, H, d, rk, rv = 1, 1, 128, 16, 16
    dm = oracle.dims(T, H, d, rk, rv, 0, 10000.0, style)
    g = np.random.default_rng(12)
    q = g.standard_normal((1, 1, d + D_ROPE))
    ck = g.standard_normal((1, 1, 2, rk))
    kr = g.standard_normal((1, 1, 2, D_ROPE))
    wk = g.standard_normal((T, H, d, rk)) / 4.0
    mk = g.standard_normal((H, T * d)) * 0.3
    cv = np.zeros((1, 1, 2, rv))
    cv[0, 0, 0, 0] = cv[0, 0, 1, 1] = 1.0
    wv = np.zeros((T, H, d, rv))
    wv[0, 0, 0, 0] = wv[0, 0, 1, 1] = 1.0
    qp = 9
    o, _ = oracle.decoupled(dm, 0, q, ck, cv, kr, np.array([2], np.int32), np.array([qp], np.int32), wk, wv, mk,
                            np.zeros((H, T * d)))
    s = []
    for j in range(2):
        content = q[0, 0, :d] @ (wk[0, 0] @ ck[0, 0, j] + mk[0, :d])
        rot = 0.0
        for f in range(D_ROPE // 2):
            a, b = (f, f + D_ROPE // 2) if style == 0 else (2 * f, 2 * f + 1)
            th = 10000.0 ** (-2.0 * f / D_ROPE)
            qa, qb, ra, rb = q[0, 0, d + a], q[0, 0, d + b], kr[0, 0, j, a], kr[0, 0, j, b]
            ang = (j - qp) * th
            rot += math.cos(ang) * (qa * ra + qb * rb) + math.sin(ang) * (qb * ra - qa * rb)
        s.append((content + rot) / math.sqrt(d + D_ROPE))
    assert abs(math.log(o[0, 0, 1] / o[0, 0, 0]) - (s[1] - s[0])) < 1e-12
    assert abs(o[0, 0, 0] + o[0, 0, 1] - 1.0) < 1e-14


def test_shift_invariance_of_the_rotary_branch():
    dm = oracle.dims(2, 2, 128, 16, 32)
    c = _case(13)
    o0, l0 = _dec(dm, 1, c, [7, 5], [6, 4])
    o1, l1 = _dec(dm, 1, c, [7, 5], [6, 4], pos_offset=1234)
    np.testing.assert_allclose(o0, o1, rtol=0, atol=1e-9)
    np.testing.assert_allclose(l0, l1, rtol=0, atol=1e-9)


def test_single_token_returns_its_value():
    dm = oracle.dims(2, 2, 128, 16, 32)
    c = _case(14)
    o, _ = _dec(dm, 0, c, [1, 1], [0, 0])
    for b in range(2):
        for h in range(2):
            v = brute.reconstruct(c["cache_v"][b, h, :1], c["w_up_v"][0, h], c["mu_v"][h, :128])[0]
            np.testing.assert_allclose(o[b, h], v, rtol=0, atol=1e-12)
